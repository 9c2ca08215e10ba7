/*
 * ssd_oracle.c -- plain, slow, double-precision CPU reference for the Mamba-2
 * selective-state-space (SSD) forward pass and single-token decode.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and the CPU
 * baseline leg of bench.py may load this library.  The GPU product path never
 * calls it and shares no code with it.
 *
 * Source of every formula: NVIDIA developer blog "Accelerating Mamba-2 with
 * High-Performance Forward Pass Kernels in NVIDIA CUDA Tile" (Korean edition,
 * mirrored in Chinese), section "Mamba-2 architecture":
 *
 *   h_t = exp(A * dt_t) h_{t-1} + dt_t B_t x_t^T          (recurrence)
 *   y_t = c_t^T h_t + D x_t                                 (output line)
 *
 * with x_t in R^H (value-like), B_t, c_t in R^S (key/query-like), a matrix
 * state h of S x H entries, and A, D per-head scalars.  The state is stored
 * head-dim major, h[p][s] (p < H, s < S), the layout of the blog's
 * init_state / final_state tensors (section "Kernel 2: fwd_pass_state").
 *
 * Readings taken where the pages are ambiguous (each is listed in the design
 * notes of the repository):
 *   - the output uses h_t (token t's own update included), not h_{t-1};
 *   - heads map to B/C groups as group = head / (nheads / ngroups);
 *   - dt is given already positive (no softplus inside the operation);
 *   - the in-chunk cumulative sum is inclusive and restarts at every chunk.
 *
 * Layouts (all contiguous, row-major):
 *   x, y   [batch][seqlen][nheads][H]
 *   dt     [batch][seqlen][nheads]
 *   Bm, Cm [batch][seqlen][ngroups][S]
 *   A, D   [nheads]
 *   h0, hf [batch][nheads][H][S]     (h0 may be NULL: zeros)
 *
 * Each (batch, head) pair is an independent recurrence; the only parallelism
 * is a plain pthread split over those pairs.  No blocking, no fusion, no
 * reordering of the arithmetic inside a pair.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    int64_t batch, seqlen, nheads, H, S, ngroups, chunk;
    const double *x, *dt, *A, *Bm, *Cm, *D, *h0;
    double *y, *hf;
    /* chunked form only (nullable) */
    double *gcum;        /* [batch][nheads][seqlen]: in-chunk cumsum of A*dt */
    double *s_local;     /* [batch][nheads][nchunks][H][S] */
    double *h_start;     /* [batch][nheads][nchunks][H][S] */
    int mode;            /* 0 = sequential recurrence, 1 = chunked form */
    int64_t next_unit;   /* work counter, guarded by lock */
    pthread_mutex_t lock;
} job_t;

#define IX_X(j, b, t, h, p) ((((b) * (j)->seqlen + (t)) * (j)->nheads + (h)) * (j)->H + (p))
#define IX_DT(j, b, t, h) (((b) * (j)->seqlen + (t)) * (j)->nheads + (h))
#define IX_BC(j, b, t, g, s) ((((b) * (j)->seqlen + (t)) * (j)->ngroups + (g)) * (j)->S + (s))
#define IX_H(j, b, h, p, s) ((((b) * (j)->nheads + (h)) * (j)->H + (p)) * (j)->S + (s))

/* ---------------------------------------------------------------------------
 * Sequential recurrence for one (batch, head) pair: the plain definition.
 * Blog section "Mamba-2 architecture", recurrence and output line.
 * ------------------------------------------------------------------------- */
static void seq_unit(const job_t *j, int64_t b, int64_t h, double *st)
{
    const int64_t H = j->H, S = j->S;
    const int64_t g = h / (j->nheads / j->ngroups);
    if (j->h0) {
        for (int64_t p = 0; p < H; ++p)
            for (int64_t s = 0; s < S; ++s) st[p * S + s] = j->h0[IX_H(j, b, h, p, s)];
    } else {
        memset(st, 0, (size_t)(H * S) * sizeof(double));
    }
    for (int64_t t = 0; t < j->seqlen; ++t) {
        const double dtv = j->dt[IX_DT(j, b, t, h)];
        const double alpha = exp(j->A[h] * dtv);          /* exp(A dt_t) */
        for (int64_t p = 0; p < H; ++p) {
            const double xp = j->x[IX_X(j, b, t, h, p)];
            double acc = 0.0;
            for (int64_t s = 0; s < S; ++s) {
                /* h_t = exp(A dt_t) h_{t-1} + dt_t * (B_t x_t^T), entry [p][s] */
                double v = alpha * st[p * S + s] + dtv * j->Bm[IX_BC(j, b, t, g, s)] * xp;
                st[p * S + s] = v;
                /* y_t[p] = sum_s c_t[s] h_t[p][s] */
                acc += j->Cm[IX_BC(j, b, t, g, s)] * v;
            }
            j->y[IX_X(j, b, t, h, p)] = acc + j->D[h] * xp;   /* + D x_t */
        }
    }
    if (j->hf) {
        for (int64_t p = 0; p < H; ++p)
            for (int64_t s = 0; s < S; ++s) j->hf[IX_H(j, b, h, p, s)] = st[p * S + s];
    }
}

/* ---------------------------------------------------------------------------
 * Chunked form for one (batch, head) pair, written in the blog's notation
 * (section "Mamba-2 architecture", the log-space jump and the chunk output):
 *
 *   a_t = A dt_t,  b_t = dt_t B_t,  G = inclusive in-chunk cumsum of a
 *   h_{k+1} = exp(G_last) h_k + (exp(G_last - G) o b)^T X
 *   Y_k     = exp(G) o (C h_k) + (exp(G - G^T) o (C b^T) o M) X + D X
 *
 * M is the causal mask with the diagonal kept (i >= j).  Natural exp, no
 * log2 scaling.  The last chunk may be shorter than `chunk`.
 * ------------------------------------------------------------------------- */
static void chunked_unit(const job_t *j, int64_t b, int64_t h, double *st, double *G)
{
    double *P = G + j->chunk;      /* scratch: one masked, decayed row of C b^T */
    const int64_t H = j->H, S = j->S, L = j->seqlen, T = j->chunk;
    const int64_t g = h / (j->nheads / j->ngroups);
    const int64_t nc = (L + T - 1) / T;
    double *snew = st + H * S;     /* scratch: next state */
    if (j->h0) {
        for (int64_t p = 0; p < H; ++p)
            for (int64_t s = 0; s < S; ++s) st[p * S + s] = j->h0[IX_H(j, b, h, p, s)];
    } else {
        memset(st, 0, (size_t)(H * S) * sizeof(double));
    }
    for (int64_t k = 0; k < nc; ++k) {
        const int64_t t0 = k * T;
        const int64_t n = (L - t0 < T) ? (L - t0) : T;
        /* G: inclusive cumsum of a_t = A dt_t inside the chunk (kernel 1) */
        double run = 0.0;
        for (int64_t i = 0; i < n; ++i) {
            run += j->A[h] * j->dt[IX_DT(j, b, t0 + i, h)];
            G[i] = run;
            if (j->gcum) j->gcum[((b * j->nheads + h) * L) + t0 + i] = run;
        }
        const double Glast = G[n - 1];
        if (j->h_start) {
            double *dst = j->h_start + (((b * j->nheads + h) * nc + k) * H) * S;
            memcpy(dst, st, (size_t)(H * S) * sizeof(double));
        }
        /* chunk output Y_k */
        for (int64_t i = 0; i < n; ++i) {
            const int64_t ti = t0 + i;
            const double *ci = &j->Cm[IX_BC(j, b, ti, g, 0)];
            /* row i of (C b^T) masked to j <= i, with its decay exp(G_i - G_j) */
            for (int64_t jj = 0; jj <= i; ++jj) {
                const int64_t tj = t0 + jj;
                const double *bj = &j->Bm[IX_BC(j, b, tj, g, 0)];
                double cb = 0.0;
                for (int64_t s = 0; s < S; ++s) cb += ci[s] * bj[s];
                const double bdt = j->dt[IX_DT(j, b, tj, h)];       /* b_j = dt_j B_j */
                P[jj] = exp(G[i] - G[jj]) * cb * bdt;
            }
            for (int64_t p = 0; p < H; ++p) {
                /* exp(G_i) (C h_k)_i */
                double carried = 0.0;
                for (int64_t s = 0; s < S; ++s) carried += ci[s] * st[p * S + s];
                carried *= exp(G[i]);
                /* sum_{j <= i} exp(G_i - G_j) (c_i . b_j) x_j */
                double intra = 0.0;
                for (int64_t jj = 0; jj <= i; ++jj) intra += P[jj] * j->x[IX_X(j, b, t0 + jj, h, p)];
                j->y[IX_X(j, b, ti, h, p)] = carried + intra + j->D[h] * j->x[IX_X(j, b, ti, h, p)];
            }
        }
        /* local chunk state (exp(G_last - G) o b)^T X, entry [p][s] */
        for (int64_t p = 0; p < H; ++p) {
            for (int64_t s = 0; s < S; ++s) {
                double acc = 0.0;
                for (int64_t i = 0; i < n; ++i) {
                    const int64_t ti = t0 + i;
                    acc += exp(Glast - G[i]) * j->dt[IX_DT(j, b, ti, h)] *
                           j->Bm[IX_BC(j, b, ti, g, s)] * j->x[IX_X(j, b, ti, h, p)];
                }
                snew[p * S + s] = acc;
            }
        }
        if (j->s_local) {
            double *dst = j->s_local + (((b * j->nheads + h) * nc + k) * H) * S;
            memcpy(dst, snew, (size_t)(H * S) * sizeof(double));
        }
        /* jump: h_{k+1} = exp(G_last) h_k + local state */
        const double decay = exp(Glast);
        for (int64_t e = 0; e < H * S; ++e) st[e] = decay * st[e] + snew[e];
    }
    if (j->hf) {
        for (int64_t p = 0; p < H; ++p)
            for (int64_t s = 0; s < S; ++s) j->hf[IX_H(j, b, h, p, s)] = st[p * S + s];
    }
}

static void *worker(void *arg)
{
    job_t *j = (job_t *)arg;
    const int64_t units = j->batch * j->nheads;
    double *st = (double *)malloc((size_t)(2 * j->H * j->S) * sizeof(double));
    double *G = (double *)malloc((size_t)(2 * (j->chunk > 0 ? j->chunk : 1)) * sizeof(double));
    if (!st || !G) { free(st); free(G); return (void *)1; }
    for (;;) {
        pthread_mutex_lock(&j->lock);
        const int64_t u = j->next_unit++;
        pthread_mutex_unlock(&j->lock);
        if (u >= units) break;
        const int64_t b = u / j->nheads, h = u % j->nheads;
        if (j->mode == 0) seq_unit(j, b, h, st);
        else chunked_unit(j, b, h, st, G);
    }
    free(st);
    free(G);
    return NULL;
}

static int run_job(job_t *j, int nthreads)
{
    if (j->batch < 0 || j->seqlen < 0 || j->nheads < 0 || j->H <= 0 || j->S <= 0) return -1;
    if (j->ngroups <= 0 || (j->nheads % j->ngroups) != 0) return -1;
    if (j->mode == 1 && j->chunk <= 0) return -1;
    const int64_t units = j->batch * j->nheads;
    /* empty sequence: h_final = h0 (or zeros), no output rows */
    if (j->seqlen == 0) {
        if (j->hf) {
            const size_t n = (size_t)(units * j->H * j->S);
            if (j->h0) memcpy(j->hf, j->h0, n * sizeof(double));
            else memset(j->hf, 0, n * sizeof(double));
        }
        return 0;
    }
    if (units == 0) return 0;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > units) nthreads = (int)units;
    j->next_unit = 0;
    pthread_mutex_init(&j->lock, NULL);
    pthread_t *tid = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
    int rc = 0;
    for (int i = 0; i < nthreads; ++i) pthread_create(&tid[i], NULL, worker, j);
    for (int i = 0; i < nthreads; ++i) {
        void *ret = NULL;
        pthread_join(tid[i], &ret);
        if (ret) rc = -2;
    }
    free(tid);
    pthread_mutex_destroy(&j->lock);
    return rc;
}

/* Sequential recurrence over the whole sequence.  Returns 0 on success. */
int oracle_ssd_fwd_seq(int64_t batch, int64_t seqlen, int64_t nheads, int64_t H, int64_t S,
                       int64_t ngroups, const double *x, const double *dt, const double *A,
                       const double *Bm, const double *Cm, const double *D, const double *h0,
                       double *y, double *h_final, int nthreads)
{
    job_t j;
    memset(&j, 0, sizeof j);
    j.batch = batch; j.seqlen = seqlen; j.nheads = nheads; j.H = H; j.S = S;
    j.ngroups = ngroups; j.chunk = 1;
    j.x = x; j.dt = dt; j.A = A; j.Bm = Bm; j.Cm = Cm; j.D = D; j.h0 = h0;
    j.y = y; j.hf = h_final; j.mode = 0;
    return run_job(&j, nthreads);
}

/* Chunked form.  gcum, s_local, h_start are optional outputs (NULL: skipped):
 *   gcum    [batch][nheads][seqlen]            natural-log in-chunk cumsum of A dt
 *   s_local [batch][nheads][nchunks][H][S]     local chunk states (zero start)
 *   h_start [batch][nheads][nchunks][H][S]     state entering each chunk       */
int oracle_ssd_fwd_chunked(int64_t batch, int64_t seqlen, int64_t nheads, int64_t H, int64_t S,
                           int64_t ngroups, int64_t chunk, const double *x, const double *dt,
                           const double *A, const double *Bm, const double *Cm, const double *D,
                           const double *h0, double *y, double *h_final, double *gcum,
                           double *s_local, double *h_start, int nthreads)
{
    job_t j;
    memset(&j, 0, sizeof j);
    j.batch = batch; j.seqlen = seqlen; j.nheads = nheads; j.H = H; j.S = S;
    j.ngroups = ngroups; j.chunk = chunk;
    j.x = x; j.dt = dt; j.A = A; j.Bm = Bm; j.Cm = Cm; j.D = D; j.h0 = h0;
    j.y = y; j.hf = h_final; j.gcum = gcum; j.s_local = s_local; j.h_start = h_start;
    j.mode = 1;
    return run_job(&j, nthreads);
}

/* One recurrent decode step (blog section "Mamba-2 architecture": the
 * recurrent form suits sequential inference; the final state of a call feeds
 * the next one, section "Kernel 2: fwd_pass_state").
 *   x [batch][nheads][H], dt [batch][nheads], Bm, Cm [batch][ngroups][S],
 *   h [batch][nheads][H][S] updated in place, y [batch][nheads][H].        */
int oracle_ssd_step(int64_t batch, int64_t nheads, int64_t H, int64_t S, int64_t ngroups,
                    const double *x, const double *dt, const double *A, const double *Bm,
                    const double *Cm, const double *D, double *h, double *y)
{
    if (batch < 0 || nheads < 0 || H <= 0 || S <= 0 || ngroups <= 0 || nheads % ngroups) return -1;
    const int64_t hpg = nheads / ngroups;
    for (int64_t b = 0; b < batch; ++b) {
        for (int64_t hh = 0; hh < nheads; ++hh) {
            const int64_t g = hh / hpg;
            const double dtv = dt[b * nheads + hh];
            const double alpha = exp(A[hh] * dtv);
            const double *Bv = Bm + (b * ngroups + g) * S;
            const double *Cv = Cm + (b * ngroups + g) * S;
            for (int64_t p = 0; p < H; ++p) {
                const double xp = x[(b * nheads + hh) * H + p];
                double *row = h + ((b * nheads + hh) * H + p) * S;
                double acc = 0.0;
                for (int64_t s = 0; s < S; ++s) {
                    row[s] = alpha * row[s] + dtv * Bv[s] * xp;
                    acc += Cv[s] * row[s];
                }
                y[(b * nheads + hh) * H + p] = acc + D[hh] * xp;
            }
        }
    }
    return 0;
}

/* ---------------------------------------------------------------------------
 * Gradients of the forward pass (reverse mode of the plain recurrence).
 *
 * Source: "Sasha Rush: Mamba: The Hard Way" (Korean translation), Part 3,
 * deriving the derivatives: for the scalar scan h_k = a_k h_{k-1} + b_k x_k, y_k = c_k h_k
 * the adjoint runs the same scan backwards, dh_k = c_k dy_k + a_{k+1} dh_{k+1},
 * and then dx_k = b_k dh_k, db_k = x_k dh_k, dc_k = h_k dy_k,
 * da_k = dh_k h_{k-1}.  Here the same steps are taken for the matrix state of
 * the blog's recurrence (a_t = exp(A dt_t), b_t = dt_t B_t, with c_t^T h_t
 * contracting over the state index), and the chain rule carries da_t and db_t
 * to dt_t, A and B:
 *
 *   lam_t  = dy_t c_t^T + exp(A dt_{t+1}) lam_{t+1},   lam_{L-1} = dy c^T + dh_final
 *   dx_t[p]  = dt_t sum_s lam_t[p][s] B_t[s] + D dy_t[p]
 *   dB_t[s] += dt_t sum_p lam_t[p][s] x_t[p]               (summed over the group's heads)
 *   dC_t[s] += sum_p h_t[p][s] dy_t[p]                     (summed over the group's heads)
 *   ddt_t   = <lam_t, x_t B_t^T> + A exp(A dt_t) <lam_t, h_{t-1}>
 *   dA     += dt_t exp(A dt_t) <lam_t, h_{t-1}>
 *   dD     += dy_t . x_t
 *   dh0     = exp(A dt_0) lam_0
 *
 * The loss is sum(dy * y) + sum(dh_final * h_final); dh_final may be NULL
 * (zeros).  The forward states h_t of the pair are kept in full (plain
 * definition, no recomputation), so memory is (L + 1) H S doubles per thread.
 * ------------------------------------------------------------------------- */
typedef struct {
    int64_t batch, seqlen, nheads, H, S, ngroups;
    const double *x, *dt, *A, *Bm, *Cm, *D, *h0, *dy, *dhf;
    double *dx, *ddt, *dh0;
    double *dB_head, *dC_head;   /* [batch][seqlen][nheads][S]: per-head parts of dB, dC */
    double *dA_pair, *dD_pair;   /* [batch][nheads] */
    int64_t next_unit;
    pthread_mutex_t lock;
} bwd_job_t;

#define BIX_X(j, b, t, h, p) ((((b) * (j)->seqlen + (t)) * (j)->nheads + (h)) * (j)->H + (p))
#define BIX_DT(j, b, t, h) (((b) * (j)->seqlen + (t)) * (j)->nheads + (h))
#define BIX_BC(j, b, t, g, s) ((((b) * (j)->seqlen + (t)) * (j)->ngroups + (g)) * (j)->S + (s))
#define BIX_HS(j, b, t, h, s) ((((b) * (j)->seqlen + (t)) * (j)->nheads + (h)) * (j)->S + (s))
#define BIX_H(j, b, h, p, s) ((((b) * (j)->nheads + (h)) * (j)->H + (p)) * (j)->S + (s))

/* hs: (seqlen + 1) * H * S doubles, hs[0] = h_{-1} = h0; lam: H * S doubles */
static void bwd_unit(const bwd_job_t *j, int64_t b, int64_t h, double *hs, double *lam)
{
    const int64_t H = j->H, S = j->S, L = j->seqlen, HS = H * S;
    const int64_t g = h / (j->nheads / j->ngroups);
    const double Ah = j->A[h];
    /* forward: every state h_t, t = -1 .. L-1 */
    for (int64_t p = 0; p < H; ++p)
        for (int64_t s = 0; s < S; ++s) hs[p * S + s] = j->h0 ? j->h0[BIX_H(j, b, h, p, s)] : 0.0;
    for (int64_t t = 0; t < L; ++t) {
        const double dtv = j->dt[BIX_DT(j, b, t, h)];
        const double alpha = exp(Ah * dtv);
        const double *prev = hs + t * HS;
        double *cur = hs + (t + 1) * HS;
        for (int64_t p = 0; p < H; ++p) {
            const double xp = j->x[BIX_X(j, b, t, h, p)];
            for (int64_t s = 0; s < S; ++s)
                cur[p * S + s] = alpha * prev[p * S + s] + dtv * j->Bm[BIX_BC(j, b, t, g, s)] * xp;
        }
    }
    /* backward: lam = dh_final, then t = L-1 .. 0 */
    for (int64_t p = 0; p < H; ++p)
        for (int64_t s = 0; s < S; ++s) lam[p * S + s] = j->dhf ? j->dhf[BIX_H(j, b, h, p, s)] : 0.0;
    double dA = 0.0, dD = 0.0;
    for (int64_t t = L - 1; t >= 0; --t) {
        const double dtv = j->dt[BIX_DT(j, b, t, h)];
        const double alpha = exp(Ah * dtv);
        const double *hprev = hs + t * HS;        /* h_{t-1} */
        const double *hcur = hs + (t + 1) * HS;   /* h_t */
        /* lam_t: add the output's contribution dy_t c_t^T */
        for (int64_t p = 0; p < H; ++p) {
            const double dyp = j->dy[BIX_X(j, b, t, h, p)];
            for (int64_t s = 0; s < S; ++s) lam[p * S + s] += dyp * j->Cm[BIX_BC(j, b, t, g, s)];
        }
        /* dC_t (this head's part): h_t^T dy_t */
        for (int64_t s = 0; s < S; ++s) {
            double acc = 0.0;
            for (int64_t p = 0; p < H; ++p) acc += hcur[p * S + s] * j->dy[BIX_X(j, b, t, h, p)];
            j->dC_head[BIX_HS(j, b, t, h, s)] = acc;
        }
        /* dx_t = dt_t lam_t B_t + D dy_t */
        for (int64_t p = 0; p < H; ++p) {
            double acc = 0.0;
            for (int64_t s = 0; s < S; ++s) acc += lam[p * S + s] * j->Bm[BIX_BC(j, b, t, g, s)];
            const double dyp = j->dy[BIX_X(j, b, t, h, p)];
            j->dx[BIX_X(j, b, t, h, p)] = dtv * acc + j->D[h] * dyp;
            dD += dyp * j->x[BIX_X(j, b, t, h, p)];
        }
        /* dB_t (this head's part): dt_t lam_t^T x_t */
        for (int64_t s = 0; s < S; ++s) {
            double acc = 0.0;
            for (int64_t p = 0; p < H; ++p) acc += lam[p * S + s] * j->x[BIX_X(j, b, t, h, p)];
            j->dB_head[BIX_HS(j, b, t, h, s)] = dtv * acc;
        }
        /* d(dt_t): through b_t = dt_t B_t, and through a_t = exp(A dt_t) */
        double via_b = 0.0, lam_hprev = 0.0;
        for (int64_t p = 0; p < H; ++p) {
            const double xp = j->x[BIX_X(j, b, t, h, p)];
            for (int64_t s = 0; s < S; ++s) {
                via_b += lam[p * S + s] * xp * j->Bm[BIX_BC(j, b, t, g, s)];
                lam_hprev += lam[p * S + s] * hprev[p * S + s];
            }
        }
        const double da = alpha * lam_hprev;      /* dL/da_t times a_t: d/d(A dt_t) */
        j->ddt[BIX_DT(j, b, t, h)] = via_b + Ah * da;
        dA += dtv * da;
        /* lam_{t-1} gets exp(A dt_t) lam_t */
        for (int64_t e = 0; e < HS; ++e) lam[e] *= alpha;
    }
    if (j->dh0)
        for (int64_t p = 0; p < H; ++p)
            for (int64_t s = 0; s < S; ++s) j->dh0[BIX_H(j, b, h, p, s)] = lam[p * S + s];
    j->dA_pair[b * j->nheads + h] = dA;
    j->dD_pair[b * j->nheads + h] = dD;
}

static void *bwd_worker(void *arg)
{
    bwd_job_t *j = (bwd_job_t *)arg;
    const int64_t units = j->batch * j->nheads;
    const int64_t HS = j->H * j->S;
    double *hs = (double *)malloc((size_t)((j->seqlen + 1) * HS) * sizeof(double));
    double *lam = (double *)malloc((size_t)HS * sizeof(double));
    if (!hs || !lam) { free(hs); free(lam); return (void *)1; }
    for (;;) {
        pthread_mutex_lock(&j->lock);
        const int64_t u = j->next_unit++;
        pthread_mutex_unlock(&j->lock);
        if (u >= units) break;
        bwd_unit(j, u / j->nheads, u % j->nheads, hs, lam);
    }
    free(hs);
    free(lam);
    return NULL;
}

/* Gradients of sum(dy * y) + sum(dh_final * h_final) with respect to every
 * input of oracle_ssd_fwd_seq.  dh_final and h0 may be NULL (zeros); dh0 may be
 * NULL (not written).  Output layouts match the inputs':
 *   dx [batch][seqlen][nheads][H], ddt [batch][seqlen][nheads], dA, dD [nheads],
 *   dB, dC [batch][seqlen][ngroups][S], dh0 [batch][nheads][H][S].
 * The sums over heads (dB, dC) and over batch and time (dA, dD) are taken
 * serially in index order after the parallel part.  Returns 0 on success. */
int oracle_ssd_bwd_seq(int64_t batch, int64_t seqlen, int64_t nheads, int64_t H, int64_t S,
                       int64_t ngroups, const double *x, const double *dt, const double *A,
                       const double *Bm, const double *Cm, const double *D, const double *h0,
                       const double *dy, const double *dh_final, double *dx, double *ddt,
                       double *dA, double *dB, double *dC, double *dD, double *dh0, int nthreads)
{
    if (batch < 0 || seqlen < 0 || nheads < 0 || H <= 0 || S <= 0) return -1;
    if (ngroups <= 0 || (nheads % ngroups) != 0) return -1;
    const int64_t units = batch * nheads, hpg = ngroups ? nheads / ngroups : 1;
    const int64_t HS = H * S;
    for (int64_t h = 0; h < nheads; ++h) { dA[h] = 0.0; dD[h] = 0.0; }
    memset(dB, 0, (size_t)(batch * seqlen * ngroups * S) * sizeof(double));
    memset(dC, 0, (size_t)(batch * seqlen * ngroups * S) * sizeof(double));
    if (units == 0) return 0;
    if (seqlen == 0) {   /* no tokens: h_final = h0, so dh0 = dh_final */
        if (dh0) {
            if (dh_final) memcpy(dh0, dh_final, (size_t)(units * HS) * sizeof(double));
            else memset(dh0, 0, (size_t)(units * HS) * sizeof(double));
        }
        return 0;
    }
    bwd_job_t j;
    memset(&j, 0, sizeof j);
    j.batch = batch; j.seqlen = seqlen; j.nheads = nheads; j.H = H; j.S = S; j.ngroups = ngroups;
    j.x = x; j.dt = dt; j.A = A; j.Bm = Bm; j.Cm = Cm; j.D = D; j.h0 = h0; j.dy = dy; j.dhf = dh_final;
    j.dx = dx; j.ddt = ddt; j.dh0 = dh0;
    const size_t nhs = (size_t)(batch * seqlen * nheads * S);
    j.dB_head = (double *)malloc(nhs * sizeof(double));
    j.dC_head = (double *)malloc(nhs * sizeof(double));
    j.dA_pair = (double *)malloc((size_t)units * sizeof(double));
    j.dD_pair = (double *)malloc((size_t)units * sizeof(double));
    int rc = 0;
    if (!j.dB_head || !j.dC_head || !j.dA_pair || !j.dD_pair) rc = -2;
    if (rc == 0) {
        if (nthreads < 1) nthreads = 1;
        if (nthreads > units) nthreads = (int)units;
        pthread_mutex_init(&j.lock, NULL);
        pthread_t *tid = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
        for (int i = 0; i < nthreads; ++i) pthread_create(&tid[i], NULL, bwd_worker, &j);
        for (int i = 0; i < nthreads; ++i) {
            void *ret = NULL;
            pthread_join(tid[i], &ret);
            if (ret) rc = -2;
        }
        free(tid);
        pthread_mutex_destroy(&j.lock);
    }
    if (rc == 0) {
        for (int64_t b = 0; b < batch; ++b)
            for (int64_t t = 0; t < seqlen; ++t)
                for (int64_t h = 0; h < nheads; ++h) {
                    const int64_t g = h / hpg;
                    for (int64_t s = 0; s < S; ++s) {
                        dB[BIX_BC(&j, b, t, g, s)] += j.dB_head[BIX_HS(&j, b, t, h, s)];
                        dC[BIX_BC(&j, b, t, g, s)] += j.dC_head[BIX_HS(&j, b, t, h, s)];
                    }
                }
        for (int64_t b = 0; b < batch; ++b)
            for (int64_t h = 0; h < nheads; ++h) {
                dA[h] += j.dA_pair[b * nheads + h];
                dD[h] += j.dD_pair[b * nheads + h];
            }
    }
    free(j.dB_head);
    free(j.dC_head);
    free(j.dA_pair);
    free(j.dD_pair);
    return rc;
}

/* ---------------------------------------------------------------------------
 * Mamba-1 selective scan (S6), forward: "Sasha Rush: Mamba: The Hard Way"
 * (Korean translation), Part 5.  Each channel d carries a vector state of N
 * entries with its own continuous-time A[d][n]; the step size delta and the
 * input-dependent B, C vary per token.  Per token the parameters are first
 * discretised (the page's discretize):
 *     abar = exp(delta_t A[d][n]),   bbar = delta_t B_t[n]
 * and then the plain recurrence runs (the page's mamba_torch loop):
 *     h[n] = abar h[n] + bbar x_t,   y_t = sum_n C_t[n] h[n]  (+ D[d] x_t)
 * Channels map to B/C groups as group = d / (dim / ngroups).  The skip term
 * D is an addition of this library's interface (NULL: none), as are h0 and
 * h_final (NULL: zeros / not written).
 *
 * Layouts (time innermost, the page's (batch, ., channel, token) order):
 *   x, delta, y  [batch][dim][seqlen]
 *   A            [dim][dstate]
 *   Bm, Cm       [batch][ngroups][dstate][seqlen]
 *   D            [dim]
 *   h0, hf       [batch][dim][dstate]
 * ------------------------------------------------------------------------- */
int oracle_s6_fwd_seq(int64_t batch, int64_t seqlen, int64_t dim, int64_t N, int64_t ngroups,
                      const double *x, const double *delta, const double *A, const double *Bm,
                      const double *Cm, const double *D, const double *h0, double *y, double *h_final)
{
    if (batch < 0 || seqlen < 0 || dim < 0 || N <= 0 || ngroups <= 0 || (dim % ngroups) != 0) return -1;
    const int64_t cpg = ngroups ? dim / ngroups : 1;
    double *h = (double *)malloc((size_t)N * sizeof(double));
    if (!h) return -2;
    for (int64_t b = 0; b < batch; ++b) {
        for (int64_t d = 0; d < dim; ++d) {
            const int64_t g = d / cpg;
            for (int64_t n = 0; n < N; ++n) h[n] = h0 ? h0[(b * dim + d) * N + n] : 0.0;
            for (int64_t t = 0; t < seqlen; ++t) {
                const double xt = x[(b * dim + d) * seqlen + t];
                const double dl = delta[(b * dim + d) * seqlen + t];
                double acc = 0.0;
                for (int64_t n = 0; n < N; ++n) {
                    const double abar = exp(dl * A[d * N + n]);
                    const double bbar = dl * Bm[((b * ngroups + g) * N + n) * seqlen + t];
                    h[n] = abar * h[n] + bbar * xt;
                    acc += Cm[((b * ngroups + g) * N + n) * seqlen + t] * h[n];
                }
                y[(b * dim + d) * seqlen + t] = acc + (D ? D[d] * xt : 0.0);
            }
            if (h_final)
                for (int64_t n = 0; n < N; ++n) h_final[(b * dim + d) * N + n] = h[n];
        }
    }
    free(h);
    return 0;
}
