// ssd_api.cu -- the extern "C" entry points of libssd.so (declared in include/ssd.h):
// argument validation, workspace carving and the stage sequence of the forward pass.
#include <cuda.h>
#include <stdint.h>
#include <string.h>

#include <math.h>

#include <algorithm>
#include <mutex>

#include "ssd_common.cuh"
#include "ssd_tc.cuh"

namespace {

using ssd::Problem;

constexpr size_t kWsAlign = 256;

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

bool aligned(const void *p, size_t a) { return ((uintptr_t)p % a) == 0; }

// Validate a descriptor; fills `pr` on success.  `need_seq` is false for the
// decode step, which ignores seqlen and chunk.
ssd_status check_desc(const ssd_desc *d, Problem *pr, bool need_seq)
{
    if (!d) return SSD_ERR_INVALID_ARG;
    if (d->batch < 0 || d->nheads < 0 || d->headdim < 1 || d->dstate < 1 || d->ngroups < 1)
        return SSD_ERR_INVALID_ARG;
    if (d->nheads % d->ngroups != 0) return SSD_ERR_INVALID_ARG;
    if (d->in_dtype != SSD_F32 && d->in_dtype != SSD_BF16) return SSD_ERR_INVALID_ARG;
    if (d->out_dtype != SSD_F32 && d->out_dtype != SSD_BF16) return SSD_ERR_INVALID_ARG;
    if ((d->dt_dtype != SSD_DT_AS_INPUTS && d->dt_dtype != SSD_DT_FLOAT32) ||
        (d->flags & ~(SSD_FLAG_FORCE_SIMT | SSD_FLAG_EXPIRE_WAITS)) != 0)
        return SSD_ERR_INVALID_ARG;
    if (need_seq && (d->seqlen < 0 || d->chunk < 1)) return SSD_ERR_INVALID_ARG;
    if (d->dstate > 256 || d->headdim > 1024) return SSD_ERR_UNSUPPORTED;
    if (need_seq && d->chunk > 1024) return SSD_ERR_UNSUPPORTED;
    // grid-dimension limits of the launches (y and z are at most 65535)
    if (d->batch > 65535) return SSD_ERR_UNSUPPORTED;
    if (d->nheads * ((d->headdim + 31) / 32) * ((d->dstate + 63) / 64) > 65535) return SSD_ERR_UNSUPPORTED;
    // sequence ((batch, head) pair) indices are 32-bit inside the kernels
    if (d->batch * d->nheads > 0x7fffffffLL) return SSD_ERR_UNSUPPORTED;
    pr->B = d->batch;
    pr->L = need_seq ? d->seqlen : 1;
    pr->nh = d->nheads;
    pr->H = d->headdim;
    pr->S = d->dstate;
    pr->G = d->ngroups;
    pr->T = need_seq ? d->chunk : 1;
    pr->nc = need_seq ? (d->seqlen + d->chunk - 1) / d->chunk : 1;
    pr->hpg = d->ngroups ? d->nheads / d->ngroups : 1;
    pr->in_dt = d->in_dtype;
    pr->out_dt = d->out_dtype;
    pr->dt_f32 = d->dt_dtype == SSD_DT_FLOAT32 && d->in_dtype == SSD_BF16;
    pr->wait_ns = (d->flags & SSD_FLAG_EXPIRE_WAITS) ? 0ull : 250000000ull;
    if (need_seq && pr->nc > 0x7fffffffLL) return SSD_ERR_UNSUPPORTED;
    // every array size (workspace, buffers, the offsets the kernels compute) is formed in 64-bit
    // arithmetic: a problem whose largest arrays need 2^62 bytes or more is refused before any
    // size is formed, so that no size can wrap around
    const double lim = 4611686018427387904.0;   // 2^62
    const double rows = (double)pr->B * (double)pr->L;
    const double states = (double)pr->B * (double)pr->nh * (double)pr->nc * (double)pr->H * (double)pr->S;
    if (16.0 * states >= lim || 16.0 * rows * (double)pr->nh * (double)pr->H >= lim ||
        16.0 * rows * (double)pr->G * (double)pr->S >= lim)
        return SSD_ERR_UNSUPPORTED;
    return SSD_OK;
}

size_t esize(int dt) { return dt == SSD_BF16 ? 2 : 4; }

// Workspace: [error word, count of finished cumsum CTAs (a 256-byte header) | G [B][nh][L] |
// dtT [B][nh][L] | s_local [B][nh][nc][H][S] | h_start [B][nh][nc][H][S] | dt16 [B][L][nh]],
// float32 but dt16, states sized for one per chunk (the largest any path uses).
struct Workspace {
    int *err;
    float *G;
    float *dtT;       // dt as float32, [b][h][L] (written by the cumsum, read by chunk_state)
    float *s_local;
    float *h_start;
    __nv_bfloat16 *dt16;   // SSD_DT_FLOAT32 only: dt rounded to bfloat16 in dt's layout (written by the cumsum)
    size_t bytes;
};

Workspace carve(const Problem &pr, void *base)
{
    Workspace w;
    const size_t e_bytes = kWsAlign;
    const size_t g_bytes = align_up(sizeof(float) * (size_t)(pr.B * pr.nh * pr.L), kWsAlign);
    const size_t states = (size_t)(pr.B * pr.nh * pr.nc * pr.H * pr.S);
    const size_t s_bytes = align_up(sizeof(float) * states, kWsAlign);
    char *p = (char *)base;
    w.err = (int *)p;
    w.G = (float *)(p + e_bytes);
    w.dtT = (float *)(p + e_bytes + g_bytes);
    w.s_local = (float *)(p + e_bytes + 2 * g_bytes);
    w.h_start = (float *)(p + e_bytes + 2 * g_bytes + s_bytes);
    w.bytes = e_bytes + 2 * g_bytes + 2 * s_bytes;
    w.dt16 = nullptr;
    if (pr.dt_f32) {
        w.dt16 = (__nv_bfloat16 *)(p + w.bytes);
        w.bytes += align_up(sizeof(__nv_bfloat16) * (size_t)(pr.B * pr.L * pr.nh), kWsAlign);
    }
    return w;
}

bool overlaps(const void *a, size_t na, const void *b, size_t nb)
{
    if (!a || !b || na == 0 || nb == 0) return false;
    const uintptr_t a0 = (uintptr_t)a, b0 = (uintptr_t)b;
    return a0 < b0 + nb && b0 < a0 + na;
}

ssd_status cuda_status(cudaError_t e) { return e == cudaSuccess ? SSD_OK : SSD_ERR_CUDA; }

bool use_tensor_cores(const ssd_desc *desc, const Problem &pr)
{
    return !(desc->flags & SSD_FLAG_FORCE_SIMT) && ssd::tc_supported(pr);
}

// The float32 inputs that the kind::tf32 kernel takes (one launch for the whole pass).
bool use_tf32(const ssd_desc *desc, const Problem &pr)
{
    return !(desc->flags & SSD_FLAG_FORCE_SIMT) && ssd::tf32_supported(pr);
}

int device_sms()
{
    static std::mutex mu;
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    std::lock_guard<std::mutex> lock(mu);
    if (!cache[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
        cache[dev] = n;
    }
    return cache[dev];
}

// Chunks per super-chunk for the tensor-core path.  Each scan CTA walks one
// super-chunk of one (batch, head, 64-column block) with the state on chip, one CTA per
// SM; more super-chunks give more CTAs but cost an extra read of x and B (the
// chunk_state pass) and state traffic.  Pick the count that minimises estimated bytes /
// wave efficiency.
int choose_chunks_per_super(const Problem &pr, double sms)
{
    const double es = (double)esize(pr.in_dt);
    // scan CTAs of one super-chunk over all sequences
    const double units1 = (double)(pr.B * pr.nh * (pr.H / 64)) / ssd::scan_seqs_per_cta(pr);
    const double x_bytes = (double)(pr.B * pr.L * pr.nh * pr.H) * es;
    const double bc_bytes = (double)(pr.B * pr.L * pr.G * pr.S) * es;
    const double alg = 2.0 * x_bytes + 2.0 * bc_bytes;
    const double state_bytes = (double)(pr.B * pr.nh * pr.H * pr.S) * 4.0;
    int best_R = (int)pr.nc;
    double best = 1e300;
    const int max_sup = (int)(pr.nc < 256 ? pr.nc : 256);
    for (int want = 1; want <= max_sup; ++want) {
        const int R = (int)((pr.nc + want - 1) / want);
        if (R > 256) continue;
        const int nsup = (int)((pr.nc + R - 1) / R);
        const double units = units1 * nsup;
        const double waves = units / sms;
        const double eff = waves / ceil(waves);
        const double extra = (nsup - 1.0) / nsup * (x_bytes + bc_bytes) + 4.0 * (nsup - 1.0) * state_bytes;
        const double cost = (alg + extra) / eff;
        if (cost < best * 0.999) { best = cost; best_R = R; }
    }
    return best_R;
}

// How the tensor-core path cuts the sequences into super-chunks (ssd::ScanSplit).
// Every sequence is first cut into super-chunks of R chunks (choose_chunks_per_super).
// When that leaves the last wave of scan CTAs less than a third full, its few CTAs
// would run alone for a whole super-chunk while the other SMs idle; instead, the
// sequences of that last wave (rounded up to whole chunk_state head groups) are cut
// again into super-chunks short enough that their CTAs spread over all SMs.  The short
// super-chunks need their entering states (a chunk_state and a state_passing pass over
// those sequences only), which costs far less than the idle wave.
ssd::ScanSplit choose_tc_plan(const Problem &pr)
{
    const int64_t sms = device_sms();
    // a scan "row" is the spc sequences one CTA walks together (two heads of a group, or one)
    const int64_t spc = ssd::scan_seqs_per_cta(pr);
    const int64_t nseq = pr.B * pr.nh, npb = spc == 2 ? 1 : pr.H / 64;   // CTAs per row and super-chunk
    const int R = choose_chunks_per_super(pr, (double)sms);
    const int nsup = (int)((pr.nc + R - 1) / R);
    ssd::ScanSplit sp{nseq, R, nsup, R, nsup, 1, nseq * nsup};
    const int64_t per_row = (int64_t)nsup * npb;             // scan CTAs per row
    const int64_t ctas = nseq / spc * per_row;
    const int64_t last = ctas % sms;                          // CTAs in the last, partial wave
    if (ctas <= sms || last == 0 || 3 * last >= sms) return sp;
    // the tail is whole chunk_state head groups and whole scan rows (both powers of two)
    const int64_t sh = ssd::state_heads_per_cta(pr);
    const int64_t align = sh > spc ? sh : spc;
    int64_t tail = (last + per_row - 1) / per_row * spc;      // sequences of the last wave
    tail = (tail + align - 1) / align * align;
    if (tail >= nseq) return sp;
    // the tail's chunks over all SMs, at least two chunks per super-chunk where the first
    // part's are longer: a scan CTA's start-up costs about two 128-token periods, so one-chunk
    // super-chunks would nearly double the tail's time (B = 4, L = 4096, 80 heads of 64 x 128:
    // 124.9 us per pass with two, 126.6 us with one, 126.3 us with four)
    const int64_t tail_chunks = tail / spc * (int64_t)pr.nc * npb;
    int R1 = (int)((tail_chunks + sms - 1) / sms);
    if (R1 < 1) R1 = 1;
    if (R1 < 2 && R > 2) R1 = 2;
    if (R1 >= R) return sp;
    sp.split = nseq - tail;
    sp.R1 = R1;
    sp.nsup1 = (int)((pr.nc + R1 - 1) / R1);
    sp.base1 = sp.split * nsup;
    return sp;
}

// The two parts of a plan as sequence runs with their cuts and state-array offsets.
struct PlanPart {
    ssd::SeqRange seqs;
    int R, nsup;
    int64_t base;        // first state index of the part in s_local / h_start
};

void plan_parts(const Problem &pr, const ssd::ScanSplit &sp, PlanPart out[2])
{
    out[0] = PlanPart{ssd::SeqRange{0, sp.split}, sp.R0, sp.nsup0, 0};
    out[1] = PlanPart{ssd::SeqRange{sp.split, pr.B * pr.nh - sp.split}, sp.R1, sp.nsup1, sp.base1};
}

ssd_status fwd_impl(const ssd_desc *desc, const void *x, const void *dt, const float *A,
                    const void *Bm, const void *Cm, const float *D, const float *h0, void *y,
                    float *h_final, void *workspace, size_t ws_bytes, cudaStream_t st,
                    ssd_event_t const *events)
{
    Problem pr;
    ssd_status s = check_desc(desc, &pr, true);
    if (s != SSD_OK) return s;
    const size_t nstate = (size_t)(pr.B * pr.nh * pr.H * pr.S);
    const bool empty = pr.B == 0 || pr.nh == 0 || pr.L == 0;
    if (!empty) {
        if (!x || !dt || !A || !Bm || !Cm || !D || !y) return SSD_ERR_INVALID_ARG;
        if (!aligned(x, 16) || !aligned(dt, 16) || !aligned(Bm, 16) || !aligned(Cm, 16) || !aligned(y, 16))
            return SSD_ERR_INVALID_ARG;
        if (!aligned(A, 4) || !aligned(D, 4)) return SSD_ERR_INVALID_ARG;
        const size_t ny = (size_t)(pr.B * pr.L * pr.nh * pr.H) * esize(pr.out_dt);
        const size_t nx = (size_t)(pr.B * pr.L * pr.nh * pr.H) * esize(pr.in_dt);
        const size_t nbc = (size_t)(pr.B * pr.L * pr.G * pr.S) * esize(pr.in_dt);
        if (overlaps(y, ny, x, nx) || overlaps(y, ny, Bm, nbc) || overlaps(y, ny, Cm, nbc))
            return SSD_ERR_INVALID_ARG;
    }
    if ((h0 && !aligned(h0, 4)) || (h_final && !aligned(h_final, 4))) return SSD_ERR_INVALID_ARG;
    if (empty) {
        // Nothing to scan: the final state is the initial state (zeros if absent).
        if (h_final && nstate) {
            cudaError_t e = h0 ? cudaMemcpyAsync(h_final, h0, nstate * sizeof(float), cudaMemcpyDeviceToDevice, st)
                               : cudaMemsetAsync(h_final, 0, nstate * sizeof(float), st);
            return cuda_status(e);
        }
        return SSD_OK;
    }
    Workspace w = carve(pr, workspace);
    if (!workspace || !aligned(workspace, kWsAlign) || ws_bytes < w.bytes) return SSD_ERR_WORKSPACE;

    auto rec = [&](int i) -> bool { return !events || cudaEventRecord((cudaEvent_t)events[i], st) == cudaSuccess; };
    if (use_tf32(desc, pr)) {
        // one launch: the kernel takes its own cumsum; the events of the first three stages
        // bracket nothing
        if (cudaMemsetAsync(w.err, 0, 2 * sizeof(int), st) != cudaSuccess) return SSD_ERR_CUDA;
        for (int i = 0; i < 7; ++i)
            if (!rec(i)) return SSD_ERR_CUDA;
        if (ssd::launch_ssd_tf32(pr, x, dt, A, Bm, Cm, D, h0, y, h_final, w.err, st) != cudaSuccess || !rec(7))
            return SSD_ERR_CUDA;
        return SSD_OK;
    }
    const bool tc = use_tensor_cores(desc, pr);
    // the error word and, next to it, the count of finished cumsum CTAs
    if (cudaMemsetAsync(w.err, 0, 2 * sizeof(int), st) != cudaSuccess) return SSD_ERR_CUDA;
    unsigned *g_count = reinterpret_cast<unsigned *>(w.err + 1);
    ssd::ScanSplit sp{};
    PlanPart parts[2];
    // the float32 copy of dt is read by chunk_state only: the sequences of the parts it runs for.
    // chunk_state fetches G and that copy by bulk copies of 64-token row pieces, which need
    // 16-byte aligned starts: the rows of a sequence start at (b * nh + h) * L floats, so for L
    // not a multiple of 4 chunk_state loads them per thread instead (no copy).
    const bool staged = pr.L % 4 == 0;
    int64_t dtT_lo = 0, dtT_hi = 0;
    if (tc) {
        sp = choose_tc_plan(pr);
        sp.g_count = g_count;
        sp.g_target = ssd::cumsum_ctas(pr);
        plan_parts(pr, sp, parts);
        for (const PlanPart &p : parts) {
            if (!staged) break;
            if (p.seqs.n <= 0 || p.nsup <= 1) continue;
            if (dtT_hi == dtT_lo) { dtT_lo = p.seqs.lo; dtT_hi = p.seqs.lo + p.seqs.n; }
            else { dtT_lo = std::min(dtT_lo, p.seqs.lo); dtT_hi = std::max(dtT_hi, p.seqs.lo + p.seqs.n); }
        }
    }
    if (!rec(0) ||
        ssd::launch_chunk_cumsum(pr, dt, A, w.G, dtT_hi > dtT_lo ? w.dtT : nullptr, dtT_lo, dtT_hi, st,
                                 tc ? g_count : nullptr, w.dt16) != cudaSuccess ||
        !rec(1))
        return SSD_ERR_CUDA;
    // with a float32 dt beside bfloat16 inputs, the stages after the cumsum read its bfloat16 copy
    if (pr.dt_f32) dt = w.dt16;

    if (tc) {
        const int64_t HS = pr.H * pr.S;
        // per part: states of super-chunks 0 .. nsup-2 (the last one's state is produced by the scan)
        if (!rec(2)) return SSD_ERR_CUDA;
        for (const PlanPart &p : parts)
            if (p.seqs.n > 0 && p.nsup > 1 &&
                ssd::launch_chunk_state_tc(pr, p.seqs, x, dt, staged ? w.dtT : nullptr, Bm, w.G,
                                           w.s_local + p.base * HS, p.R, p.nsup, p.nsup - 1, w.err, st) != cudaSuccess)
                return SSD_ERR_CUDA;
        if (!rec(3) || !rec(4)) return SSD_ERR_CUDA;
        for (const PlanPart &p : parts)
            if (p.seqs.n > 0 && p.nsup > 1 &&
                ssd::launch_state_passing(pr, p.seqs, w.G, w.s_local + p.base * HS, h0, w.h_start + p.base * HS,
                                          nullptr, p.R, p.nsup, p.nsup - 1, st) != cudaSuccess)
                return SSD_ERR_CUDA;
        if (!rec(5) || !rec(6)) return SSD_ERR_CUDA;
        if (ssd::launch_chunk_scan_tc(pr, x, dt, Bm, Cm, D, w.G, h0, w.h_start, h_final, y, sp, w.err, st) !=
            cudaSuccess)
            return SSD_ERR_CUDA;
        if (!rec(7)) return SSD_ERR_CUDA;
        return SSD_OK;
    }
    const int nc = (int)pr.nc;
    if (!rec(2) || ssd::launch_chunk_state_simt(pr, x, dt, Bm, w.G, w.s_local, st) != cudaSuccess || !rec(3))
        return SSD_ERR_CUDA;
    if (!rec(4) ||
        ssd::launch_state_passing(pr, ssd::SeqRange{0, pr.B * pr.nh}, w.G, w.s_local, h0, w.h_start, h_final, 1, nc,
                                  nc, st) != cudaSuccess ||
        !rec(5))
        return SSD_ERR_CUDA;
    if (!rec(6) || ssd::launch_chunk_scan_simt(pr, x, dt, Bm, Cm, D, w.G, w.h_start, y, st) != cudaSuccess || !rec(7))
        return SSD_ERR_CUDA;
    return SSD_OK;
}

bool nonempty(const Problem &pr) { return pr.B > 0 && pr.nh > 0 && pr.L > 0; }

// ---- forward pass on host buffers (ssd_fwd_host) -------------------------------------------
// The problem is cut into up to kHostParts slices: runs of whole batch rows when there are
// enough rows, else token ranges of whole chunks within each row (a row's ranges run in order;
// each range enters from the state the one before it left, through the device buffer).  Slice
// k's inputs go to the device on the library's copy-in stream, its forward pass runs on the
// caller's stream once they have landed, and its outputs come back on the copy-out stream once
// it is done: the copies of one slice overlap the computation and the copies of the others.
// Every slice has its own 256-byte-aligned device regions (a slice of dt need not start on a
// 16-byte boundary in a packed layout); the slices share one workspace.  Device buffer:
// [error words of the slices | A | D | per slice: x, dt, B, C, h0, y, h_final | workspace].
constexpr int kHostParts = 16;    // the most slices (error words, events)
constexpr int kHostTarget = 8;    // slices aimed at: each one costs about 20 API calls to enqueue

struct HostLayout {
    int64_t parts = 0;                       // slices
    int64_t rows = 0, toks = 0;              // batch rows and tokens of a full slice
    int64_t ranges = 1;                      // token ranges per row (1: slices of whole rows)
    size_t a = 0, d = 0, slice0 = 0, slice = 0, ws = 0, ws_bytes = 0, bytes = 0;
    size_t x = 0, dt = 0, bm = 0, cm = 0, h0 = 0, y = 0, hf = 0;   // offsets inside a slice
    size_t x_t = 0, dt_t = 0, bc_t = 0, y_t = 0, st_b = 0;          // bytes per token (of one row), per state
    // small inputs copied in whole, in one copy each before the slices (every slice's part of
    // them then starts on a 16-byte boundary): dt, B and C, h0; their regions
    bool m_dt = false, m_bc = false, m_h0 = false;
    size_t dt_all = 0, b_all = 0, c_all = 0, h0_all = 0;
};

// Slice k: batch rows [b0, b0 + nb), tokens [t0, t0 + nt).
struct HostSlice {
    int64_t b0, nb, t0, nt;
};

HostSlice host_slice(const HostLayout &h, const Problem &pr, int64_t k)
{
    if (h.ranges == 1) {
        const int64_t b0 = k * h.rows;
        return HostSlice{b0, std::min<int64_t>(h.rows, pr.B - b0), 0, pr.L};
    }
    const int64_t b0 = k / h.ranges, t0 = (k % h.ranges) * h.toks;
    return HostSlice{b0, 1, t0, std::min<int64_t>(h.toks, pr.L - t0)};
}

HostLayout host_layout(const ssd_desc *desc, const Problem &pr)
{
    HostLayout h;
    // whole rows when there are enough of them, else token ranges (the 2.7B-shaped layer, 4 rows:
    // 8 ranges measured 1.38 ms per call against 1.48 ms for 4 row slices)
    if (pr.B >= kHostTarget || pr.L <= pr.T) {
        h.parts = std::min<int64_t>(pr.B, kHostTarget);
        h.rows = h.parts > 0 ? (pr.B + h.parts - 1) / h.parts : 0;
        if (h.rows > 0) h.parts = (pr.B + h.rows - 1) / h.rows;
        h.toks = pr.L;
    } else {
        // each row in ranges of whole chunks, about kHostTarget slices in all
        const int64_t want = std::max<int64_t>(1, kHostTarget / pr.B);
        h.toks = std::max<int64_t>(1, (pr.L + want - 1) / want);
        h.toks = (h.toks + pr.T - 1) / pr.T * pr.T;
        h.ranges = (pr.L + h.toks - 1) / h.toks;
        h.rows = 1;
        h.parts = pr.B * h.ranges;
    }
    const size_t es = esize(pr.in_dt), eo = esize(pr.out_dt), ed = pr.dt_f32 ? 4 : es;
    h.x_t = (size_t)(pr.nh * pr.H) * es;
    h.dt_t = (size_t)pr.nh * ed;
    h.bc_t = (size_t)(pr.G * pr.S) * es;
    h.y_t = (size_t)(pr.nh * pr.H) * eo;
    h.st_b = (size_t)(pr.nh * pr.H * pr.S) * sizeof(float);
    const size_t nt = (size_t)(h.rows * h.toks), nr = (size_t)h.rows;
    size_t o = 0;
    h.x = o;  o += align_up(nt * h.x_t, kWsAlign);
    h.dt = o; o += align_up(nt * h.dt_t, kWsAlign);
    h.bm = o; o += align_up(nt * h.bc_t, kWsAlign);
    h.cm = o; o += align_up(nt * h.bc_t, kWsAlign);
    h.h0 = o; o += align_up(nr * h.st_b, kWsAlign);
    h.y = o;  o += align_up(nt * h.y_t, kWsAlign);
    h.hf = o; o += align_up(nr * h.st_b, kWsAlign);
    h.slice = o;
    h.a = kWsAlign;                                        // after the slices' error words
    h.d = h.a + align_up((size_t)pr.nh * sizeof(float), kWsAlign);
    h.slice0 = h.d + align_up((size_t)pr.nh * sizeof(float), kWsAlign);
    h.ws = h.slice0 + (size_t)h.parts * h.slice;
    // An input small next to x (a 16th of it at most) goes in one copy when every slice's part of
    // it starts on a 16-byte boundary: each copy costs a few microseconds however small it is.
    const size_t rows_t = (size_t)(pr.B * pr.L), x_all = rows_t * h.x_t;
    auto slices_aligned = [&](size_t per_token) {
        for (int64_t k = 0; k < h.parts; ++k) {
            const HostSlice c = host_slice(h, pr, k);
            if ((((size_t)c.b0 * pr.L + c.t0) * per_token) % 16 != 0) return false;
        }
        return true;
    };
    h.m_dt = rows_t * h.dt_t * 16 <= x_all && slices_aligned(h.dt_t);
    h.m_bc = rows_t * h.bc_t * 16 <= x_all && slices_aligned(h.bc_t);
    h.m_h0 = (size_t)pr.B * h.st_b * 16 <= x_all;          // h0 parts start at whole rows
    size_t w = h.ws;
    if (h.m_dt) { h.dt_all = w; w += align_up(rows_t * h.dt_t, kWsAlign); }
    if (h.m_bc) {
        h.b_all = w; w += align_up(rows_t * h.bc_t, kWsAlign);
        h.c_all = w; w += align_up(rows_t * h.bc_t, kWsAlign);
    }
    if (h.m_h0) { h.h0_all = w; w += align_up((size_t)pr.B * h.st_b, kWsAlign); }
    h.ws = w;
    ssd_desc sub = *desc;
    sub.batch = h.rows;
    sub.seqlen = h.toks;
    Problem ps;
    if (h.rows > 0 && check_desc(&sub, &ps, true) == SSD_OK && nonempty(ps)) h.ws_bytes = carve(ps, nullptr).bytes;
    h.bytes = h.ws + h.ws_bytes;
    return h;
}

// The copy streams of ssd_fwd_host and their events, one set per device, created on first use.
// Callers hold host_mutex() while they enqueue.
struct HostStreams {
    cudaStream_t in = nullptr, out = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr, landed[kHostParts] = {}, done[kHostParts] = {};
};

std::mutex &host_mutex()
{
    static std::mutex mu;
    return mu;
}

HostStreams *host_streams()
{
    static HostStreams cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    HostStreams &r = cache[dev];
    if (r.join) return &r;
    HostStreams n;
    bool ok = cudaStreamCreateWithFlags(&n.in, cudaStreamNonBlocking) == cudaSuccess &&
              cudaStreamCreateWithFlags(&n.out, cudaStreamNonBlocking) == cudaSuccess &&
              cudaEventCreateWithFlags(&n.fork, cudaEventDisableTiming) == cudaSuccess;
    for (int k = 0; ok && k < kHostParts; ++k)
        ok = cudaEventCreateWithFlags(&n.landed[k], cudaEventDisableTiming) == cudaSuccess &&
             cudaEventCreateWithFlags(&n.done[k], cudaEventDisableTiming) == cudaSuccess;
    ok = ok && cudaEventCreateWithFlags(&n.join, cudaEventDisableTiming) == cudaSuccess;
    if (!ok) {
        for (cudaStream_t s : {n.in, n.out})
            if (s) cudaStreamDestroy(s);
        for (cudaEvent_t e : {n.fork, n.join})
            if (e) cudaEventDestroy(e);
        for (int k = 0; k < kHostParts; ++k)
            for (cudaEvent_t e : {n.landed[k], n.done[k]})
                if (e) cudaEventDestroy(e);
        return nullptr;
    }
    r = n;
    return &r;
}

}  // namespace

extern "C" {

const char *ssd_status_string(ssd_status s)
{
    switch (s) {
    case SSD_OK: return "SSD_OK";
    case SSD_ERR_INVALID_ARG: return "SSD_ERR_INVALID_ARG: invalid argument (null/misaligned pointer, bad size or dtype)";
    case SSD_ERR_UNSUPPORTED: return "SSD_ERR_UNSUPPORTED: problem size outside what this library handles";
    case SSD_ERR_WORKSPACE: return "SSD_ERR_WORKSPACE: workspace missing, too small or not 256-byte aligned";
    case SSD_ERR_CUDA: return "SSD_ERR_CUDA: a CUDA call or kernel launch failed";
    case SSD_ERR_TOO_LARGE: return "SSD_ERR_TOO_LARGE: problem needs more scratch than the built-in no-alloc array";
    case SSD_ERR_TIMEOUT: return "SSD_ERR_TIMEOUT: a bounded wait inside a kernel expired; results are invalid";
    }
    return "unknown ssd_status";
}

ssd_status ssd_fwd_workspace_size(const ssd_desc *desc, size_t *bytes)
{
    Problem pr;
    if (!bytes) return SSD_ERR_INVALID_ARG;
    ssd_status s = check_desc(desc, &pr, true);
    if (s != SSD_OK) return s;
    *bytes = nonempty(pr) ? carve(pr, nullptr).bytes : 0;
    return SSD_OK;
}

ssd_status ssd_fwd_path(const ssd_desc *desc, int32_t *uses_tensor_cores)
{
    Problem pr;
    if (!uses_tensor_cores) return SSD_ERR_INVALID_ARG;
    ssd_status s = check_desc(desc, &pr, true);
    if (s != SSD_OK) return s;
    *uses_tensor_cores = (use_tensor_cores(desc, pr) || use_tf32(desc, pr)) ? 1 : 0;
    return SSD_OK;
}

ssd_status ssd_fwd_plan(const ssd_desc *desc, ssd_plan *plan)
{
    Problem pr;
    if (!plan) return SSD_ERR_INVALID_ARG;
    ssd_status s = check_desc(desc, &pr, true);
    if (s != SSD_OK) return s;
    ssd_plan p = {};
    p.tensor_cores = (use_tensor_cores(desc, pr) || use_tf32(desc, pr)) ? 1 : 0;
    if (pr.B == 0 || pr.nh == 0 || pr.L == 0) {
        // nothing to scan: at most one copy or memset of h_final, issued only if h_final is given
        p.super_tokens = (int32_t)std::min<int64_t>(pr.T, 0x7fffffff);
        *plan = p;
        return SSD_OK;
    }
    const int32_t nseq = (int32_t)(pr.B * pr.nh);
    if (use_tf32(desc, pr)) {
        // one launch, one CTA per sequence walking it whole
        p.super_tokens = p.tail_super_tokens = (int32_t)pr.L;
        p.n_super = p.tail_n_super = 1;
        p.split_sequences = nseq;
        p.kernel_launches = 1;
        p.memsets = 1;
        *plan = p;
        return SSD_OK;
    }
    if (p.tensor_cores) {        const ssd::ScanSplit sp = choose_tc_plan(pr);
        PlanPart parts[2];
        plan_parts(pr, sp, parts);
        p.super_tokens = (int32_t)std::min<int64_t>(sp.R0 * pr.T, pr.L);
        p.n_super = sp.nsup0;
        p.split_sequences = (int32_t)sp.split;
        p.tail_super_tokens = (int32_t)std::min<int64_t>(sp.R1 * pr.T, pr.L);
        p.tail_n_super = sp.nsup1;
        p.kernel_launches = 2;                 // cumsum and scan
        p.memsets = 1;                         // the error word
        for (const PlanPart &q : parts) {
            if (q.seqs.n == 0 || q.nsup <= 1) continue;
            p.kernel_launches += 2;            // chunk_state and state_passing of the part
            if (ssd::chunk_state_tc_memsets(pr, q.seqs, q.R, q.nsup - 1)) p.memsets += 1;
        }
    } else {
        p.super_tokens = (int32_t)std::min<int64_t>(pr.T, pr.L);
        p.n_super = (int32_t)pr.nc;
        p.split_sequences = nseq;
        p.tail_super_tokens = p.super_tokens;
        p.tail_n_super = (int32_t)pr.nc;
        p.kernel_launches = 4;
        p.memsets = 1;
    }
    *plan = p;
    return SSD_OK;
}

ssd_status ssd_fwd(const ssd_desc *desc, const void *x, const void *dt, const float *A,
                   const void *Bm, const void *Cm, const float *D, const float *h0, void *y,
                   float *h_final, void *workspace, size_t ws_bytes, ssd_stream_t stream)
{
    return fwd_impl(desc, x, dt, A, Bm, Cm, D, h0, y, h_final, workspace, ws_bytes,
                    (cudaStream_t)stream, nullptr);
}

ssd_status ssd_fwd_timed(const ssd_desc *desc, const void *x, const void *dt, const float *A,
                         const void *Bm, const void *Cm, const float *D, const float *h0, void *y,
                         float *h_final, void *workspace, size_t ws_bytes, ssd_stream_t stream,
                         ssd_event_t const *events)
{
    if (!events) return SSD_ERR_INVALID_ARG;
    for (int i = 0; i < 8; ++i)
        if (!events[i]) return SSD_ERR_INVALID_ARG;
    return fwd_impl(desc, x, dt, A, Bm, Cm, D, h0, y, h_final, workspace, ws_bytes,
                    (cudaStream_t)stream, events);
}

ssd_status ssd_fwd_host_buffer_size(const ssd_desc *desc, size_t *bytes)
{
    Problem pr;
    if (!bytes) return SSD_ERR_INVALID_ARG;
    ssd_status s = check_desc(desc, &pr, true);
    if (s != SSD_OK) return s;
    *bytes = host_layout(desc, pr).bytes;
    return SSD_OK;
}

ssd_status ssd_fwd_host(const ssd_desc *desc, const void *x, const void *dt, const float *A, const void *Bm,
                        const void *Cm, const float *D, const float *h0, void *y, float *h_final, void *device_buffer,
                        size_t buffer_bytes, ssd_stream_t stream)
{
    Problem pr;
    ssd_status s = check_desc(desc, &pr, true);
    if (s != SSD_OK) return s;
    const HostLayout h = host_layout(desc, pr);
    if (!device_buffer || !aligned(device_buffer, kWsAlign) || buffer_bytes < h.bytes) return SSD_ERR_WORKSPACE;
    const bool empty = !nonempty(pr);
    if (!empty && (!x || !dt || !A || !Bm || !Cm || !D || !y)) return SSD_ERR_INVALID_ARG;
    cudaStream_t st = (cudaStream_t)stream;
    char *base = (char *)device_buffer;
    int *errs = (int *)base;
    if (cudaMemsetAsync(errs, 0, kHostParts * sizeof(int), st) != cudaSuccess) return SSD_ERR_CUDA;
    if (empty) {
        // nothing to scan: h_final is h0 (zeros if absent), through the slices' state regions
        if (!h_final || h.st_b == 0) return SSD_OK;
        for (int64_t k = 0; k < h.parts; ++k) {
            const HostSlice c = host_slice(h, pr, k);
            const size_t n = (size_t)c.nb * h.st_b;
            char *hf_d = base + h.slice0 + (size_t)k * h.slice + h.hf;
            cudaError_t e = h0 ? cudaMemcpyAsync(hf_d, (const char *)h0 + (size_t)c.b0 * h.st_b, n,
                                                 cudaMemcpyHostToDevice, st)
                               : cudaMemsetAsync(hf_d, 0, n, st);
            if (e == cudaSuccess)
                e = cudaMemcpyAsync((char *)h_final + (size_t)c.b0 * h.st_b, hf_d, n, cudaMemcpyDeviceToHost, st);
            if (e != cudaSuccess) return SSD_ERR_CUDA;
        }
        return SSD_OK;
    }
    std::lock_guard<std::mutex> lock(host_mutex());
    HostStreams *hs = host_streams();
    if (!hs) return SSD_ERR_CUDA;
    float *A_d = (float *)(base + h.a), *D_d = (float *)(base + h.d);
    void *ws = base + h.ws;
    auto H2D = [&](void *dst, const void *src, size_t n) {
        return n == 0 || cudaMemcpyAsync(dst, src, n, cudaMemcpyHostToDevice, hs->in) == cudaSuccess;
    };
    auto D2H = [&](void *dst, const void *src, size_t n) {
        return n == 0 || cudaMemcpyAsync(dst, src, n, cudaMemcpyDeviceToHost, hs->out) == cudaSuccess;
    };
    // the copy streams start after everything enqueued on the caller's stream so far
    if (cudaEventRecord(hs->fork, st) != cudaSuccess || cudaStreamWaitEvent(hs->in, hs->fork, 0) != cudaSuccess ||
        cudaStreamWaitEvent(hs->out, hs->fork, 0) != cudaSuccess)
        return SSD_ERR_CUDA;
    if (!H2D(A_d, A, (size_t)pr.nh * sizeof(float)) || !H2D(D_d, D, (size_t)pr.nh * sizeof(float)))
        return SSD_ERR_CUDA;
    // host offset of token t0 of batch row b0, for an array of `per_token` bytes per (row, token)
    auto hoff = [&](const HostSlice &c, size_t per_token) { return ((size_t)c.b0 * pr.L + c.t0) * per_token; };
    const size_t rows_t = (size_t)(pr.B * pr.L);
    if ((h.m_dt && !H2D(base + h.dt_all, dt, rows_t * h.dt_t)) ||
        (h.m_bc && (!H2D(base + h.b_all, Bm, rows_t * h.bc_t) || !H2D(base + h.c_all, Cm, rows_t * h.bc_t))) ||
        (h.m_h0 && h0 && !H2D(base + h.h0_all, h0, (size_t)pr.B * h.st_b)))
        return SSD_ERR_CUDA;
    // device addresses of slice k's inputs: its own regions, or its part of a whole copy
    auto dt_of = [&](const HostSlice &c, char *r) { return h.m_dt ? base + h.dt_all + hoff(c, h.dt_t) : r + h.dt; };
    auto b_of = [&](const HostSlice &c, char *r) { return h.m_bc ? base + h.b_all + hoff(c, h.bc_t) : r + h.bm; };
    auto c_of = [&](const HostSlice &c, char *r) { return h.m_bc ? base + h.c_all + hoff(c, h.bc_t) : r + h.cm; };
    auto h0_of = [&](const HostSlice &c, char *r) {
        return h.m_h0 ? base + h.h0_all + (size_t)c.b0 * h.st_b : r + h.h0;
    };
    for (int64_t k = 0; k < h.parts; ++k) {
        const HostSlice c = host_slice(h, pr, k);
        char *r = base + h.slice0 + (size_t)k * h.slice;
        const size_t nt = (size_t)(c.nb * c.nt);
        if (!H2D(r + h.x, (const char *)x + hoff(c, h.x_t), nt * h.x_t) ||
            (!h.m_dt && !H2D(r + h.dt, (const char *)dt + hoff(c, h.dt_t), nt * h.dt_t)) ||
            (!h.m_bc && (!H2D(r + h.bm, (const char *)Bm + hoff(c, h.bc_t), nt * h.bc_t) ||
                         !H2D(r + h.cm, (const char *)Cm + hoff(c, h.bc_t), nt * h.bc_t))) ||
            (h0 && !h.m_h0 && c.t0 == 0 &&
             !H2D(r + h.h0, (const char *)h0 + (size_t)c.b0 * h.st_b, (size_t)c.nb * h.st_b)) ||
            cudaEventRecord(hs->landed[k], hs->in) != cudaSuccess)
            return SSD_ERR_CUDA;
    }
    for (int64_t k = 0; k < h.parts; ++k) {
        const HostSlice c = host_slice(h, pr, k);
        char *r = base + h.slice0 + (size_t)k * h.slice;
        const size_t nt = (size_t)(c.nb * c.nt);
        const bool row_end = c.t0 + c.nt == pr.L;
        // a range after the first of its row enters from the state the range before it left
        const float *h0_d = c.t0 > 0 ? (const float *)(base + h.slice0 + (size_t)(k - 1) * h.slice + h.hf)
                                     : (h0 ? (const float *)h0_of(c, r) : nullptr);
        float *hf_d = (h_final || !row_end) ? (float *)(r + h.hf) : nullptr;
        ssd_desc sub = *desc;
        sub.batch = c.nb;
        sub.seqlen = c.nt;
        if (cudaStreamWaitEvent(st, hs->landed[k], 0) != cudaSuccess) return SSD_ERR_CUDA;
        s = fwd_impl(&sub, r + h.x, dt_of(c, r), A_d, b_of(c, r), c_of(c, r), D_d, h0_d, r + h.y, hf_d, ws, h.ws_bytes,
                     st, nullptr);
        if (s != SSD_OK) return s;
        // keep this slice's error word: the next slice clears the workspace's
        if (cudaMemcpyAsync(errs + k, ws, sizeof(int), cudaMemcpyDeviceToDevice, st) != cudaSuccess ||
            cudaEventRecord(hs->done[k], st) != cudaSuccess)
            return SSD_ERR_CUDA;
        if (cudaStreamWaitEvent(hs->out, hs->done[k], 0) != cudaSuccess ||
            !D2H((char *)y + hoff(c, h.y_t), r + h.y, nt * h.y_t) ||
            (h_final && row_end &&
             !D2H((char *)h_final + (size_t)c.b0 * h.st_b, r + h.hf, (size_t)c.nb * h.st_b)))
            return SSD_ERR_CUDA;
    }
    // the caller's stream continues once the outputs are back in host memory
    if (cudaEventRecord(hs->join, hs->out) != cudaSuccess || cudaStreamWaitEvent(st, hs->join, 0) != cudaSuccess)
        return SSD_ERR_CUDA;
    return SSD_OK;
}

ssd_status ssd_fwd_host_check(const void *device_buffer, ssd_stream_t stream)
{
    if (!device_buffer || !aligned(device_buffer, kWsAlign)) return SSD_ERR_INVALID_ARG;
    int words[kHostParts] = {0};
    if (cudaMemcpyAsync(words, device_buffer, sizeof(words), cudaMemcpyDeviceToHost, (cudaStream_t)stream) !=
            cudaSuccess ||
        cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess)
        return SSD_ERR_CUDA;
    for (int w : words)
        if (w) return SSD_ERR_TIMEOUT;
    return SSD_OK;
}

ssd_status ssd_fwd_check(const void *workspace, ssd_stream_t stream)
{
    if (!workspace || !aligned(workspace, kWsAlign)) return SSD_ERR_INVALID_ARG;
    int word = 0;
    if (cudaMemcpyAsync(&word, workspace, sizeof(int), cudaMemcpyDeviceToHost, (cudaStream_t)stream) != cudaSuccess ||
        cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess)
        return SSD_ERR_CUDA;
    return word ? SSD_ERR_TIMEOUT : SSD_OK;
}

ssd_status ssd_step(const ssd_desc *desc, const void *x, const void *dt, const float *A,
                    const void *Bm, const void *Cm, const float *D, float *h, void *y,
                    ssd_stream_t stream)
{
    Problem pr;
    ssd_status s = check_desc(desc, &pr, false);
    if (s != SSD_OK) return s;
    if (pr.dt_f32) return SSD_ERR_UNSUPPORTED;
    if (pr.B == 0 || pr.nh == 0) return SSD_OK;
    if (!x || !dt || !A || !Bm || !Cm || !D || !h || !y) return SSD_ERR_INVALID_ARG;
    if (!aligned(x, 4) || !aligned(dt, 2) || !aligned(Bm, 2) || !aligned(Cm, 2) || !aligned(y, 2) ||
        !aligned(h, 4) || !aligned(A, 4) || !aligned(D, 4))
        return SSD_ERR_INVALID_ARG;
    return cuda_status(ssd::launch_ssd_step(pr, x, dt, A, Bm, Cm, D, h, y, (cudaStream_t)stream));
}

ssd_status ssd_chunk_cumsum(const ssd_desc *desc, const void *dt, const float *A, float *G,
                            ssd_stream_t stream)
{
    Problem pr;
    ssd_status s = check_desc(desc, &pr, true);
    if (s != SSD_OK) return s;
    if (!nonempty(pr)) return SSD_OK;
    if (!dt || !A || !G || !aligned(G, 4) || !aligned(A, 4)) return SSD_ERR_INVALID_ARG;
    return cuda_status(ssd::launch_chunk_cumsum(pr, dt, A, G, nullptr, 0, 0, (cudaStream_t)stream));
}

ssd_status ssd_chunk_state(const ssd_desc *desc, const void *x, const void *dt, const void *Bm,
                           const float *G, float *s_local, ssd_stream_t stream)
{
    Problem pr;
    ssd_status s = check_desc(desc, &pr, true);
    if (s != SSD_OK) return s;
    if (pr.dt_f32) return SSD_ERR_UNSUPPORTED;
    if (!nonempty(pr)) return SSD_OK;
    if (!x || !dt || !Bm || !G || !s_local) return SSD_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(dt, 16) || !aligned(Bm, 16) || !aligned(G, 16) || !aligned(s_local, 16))
        return SSD_ERR_INVALID_ARG;
    const int nc = (int)pr.nc;
    // every chunk's state, the last one included: the tensor-core kernel takes whole chunks only
    cudaError_t e = use_tensor_cores(desc, pr) && pr.L % pr.T == 0
                        ? ssd::launch_chunk_state_tc(pr, ssd::SeqRange{0, pr.B * pr.nh}, x, dt, nullptr, Bm, G, s_local,
                                                     1, nc, nc, nullptr, (cudaStream_t)stream)
                        : ssd::launch_chunk_state_simt(pr, x, dt, Bm, G, s_local, (cudaStream_t)stream);
    return cuda_status(e);
}

ssd_status ssd_state_passing(const ssd_desc *desc, const float *G, const float *s_local,
                             const float *h0, float *h_start, float *h_final, ssd_stream_t stream)
{
    Problem pr;
    ssd_status s = check_desc(desc, &pr, true);
    if (s != SSD_OK) return s;
    if (!nonempty(pr)) return SSD_OK;
    if (!G || !s_local || !h_start) return SSD_ERR_INVALID_ARG;
    if (!aligned(G, 4) || !aligned(s_local, 4) || !aligned(h_start, 4) ||
        (h0 && !aligned(h0, 4)) || (h_final && !aligned(h_final, 4)))
        return SSD_ERR_INVALID_ARG;
    const size_t states = (size_t)(pr.B * pr.nh * pr.nc * pr.H * pr.S);
    if (overlaps(s_local, states * 4, h_start, states * 4)) return SSD_ERR_INVALID_ARG;
    const int nc = (int)pr.nc;
    return cuda_status(ssd::launch_state_passing(pr, ssd::SeqRange{0, pr.B * pr.nh}, G, s_local, h0, h_start, h_final,
                                                 1, nc, nc, (cudaStream_t)stream));
}

ssd_status ssd_chunk_scan(const ssd_desc *desc, const void *x, const void *dt, const void *Bm,
                          const void *Cm, const float *D, const float *G, const float *h_start,
                          void *y, ssd_stream_t stream)
{
    Problem pr;
    ssd_status s = check_desc(desc, &pr, true);
    if (s != SSD_OK) return s;
    if (pr.dt_f32) return SSD_ERR_UNSUPPORTED;
    if (!nonempty(pr)) return SSD_OK;
    if (!x || !dt || !Bm || !Cm || !D || !G || !h_start || !y) return SSD_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(dt, 16) || !aligned(Bm, 16) || !aligned(Cm, 16) || !aligned(G, 16) ||
        !aligned(h_start, 16) || !aligned(y, 16) || !aligned(D, 4))
        return SSD_ERR_INVALID_ARG;
    // one chunk per scan unit: chunk k starts from h_start[k] (chunk 0 included)
    const int nc = (int)pr.nc;
    cudaError_t e;
    if (use_tensor_cores(desc, pr)) {
        const ssd::ScanSplit sp{pr.B * pr.nh, 1, nc, 1, nc, 0, 0};
        e = ssd::launch_chunk_scan_tc(pr, x, dt, Bm, Cm, D, G, nullptr, h_start, nullptr, y, sp, nullptr,
                                      (cudaStream_t)stream);
    } else {
        e = ssd::launch_chunk_scan_simt(pr, x, dt, Bm, Cm, D, G, h_start, y, (cudaStream_t)stream);
    }
    return cuda_status(e);
}

ssd_status ssd_bwd_workspace_size(const ssd_desc *desc, size_t *bytes)
{
    Problem pr;
    if (!bytes) return SSD_ERR_INVALID_ARG;
    ssd_status s = check_desc(desc, &pr, true);
    if (s != SSD_OK) return s;
    if (pr.dt_f32 || !ssd::bwd_supported(pr)) return SSD_ERR_UNSUPPORTED;
    *bytes = nonempty(pr) ? ssd::bwd_workspace(pr, nullptr, nullptr) : 0;
    return SSD_OK;
}

ssd_status ssd_bwd(const ssd_desc *desc, const void *x, const void *dt, const float *A,
                   const void *Bm, const void *Cm, const float *D, const float *h0,
                   const void *dy, const float *dh_final, void *dx, void *ddt, float *dA,
                   void *dB, void *dC, float *dD, float *dh0, void *workspace, size_t ws_bytes,
                   ssd_stream_t stream)
{
    Problem pr;
    ssd_status s = check_desc(desc, &pr, true);
    if (s != SSD_OK) return s;
    if (pr.dt_f32 || !ssd::bwd_supported(pr)) return SSD_ERR_UNSUPPORTED;
    cudaStream_t st = (cudaStream_t)stream;
    const size_t es = esize(pr.in_dt);
    const size_t nstate = (size_t)(pr.B * pr.nh * pr.H * pr.S);
    if ((dA && !aligned(dA, 4)) || (dD && !aligned(dD, 4)) || (h0 && !aligned(h0, 4)) ||
        (dh_final && !aligned(dh_final, 4)) || (dh0 && !aligned(dh0, 4)))
        return SSD_ERR_INVALID_ARG;
    if (pr.nh > 0 && (!dA || !dD)) return SSD_ERR_INVALID_ARG;
    if (!nonempty(pr)) {
        // no tokens: h_final = h0, so dh0 = dh_final; dA and dD are empty sums
        if (pr.nh > 0 && (cudaMemsetAsync(dA, 0, pr.nh * sizeof(float), st) != cudaSuccess ||
                          cudaMemsetAsync(dD, 0, pr.nh * sizeof(float), st) != cudaSuccess))
            return SSD_ERR_CUDA;
        if (dh0 && nstate) {
            cudaError_t e = dh_final ? cudaMemcpyAsync(dh0, dh_final, nstate * sizeof(float), cudaMemcpyDeviceToDevice, st)
                                     : cudaMemsetAsync(dh0, 0, nstate * sizeof(float), st);
            return cuda_status(e);
        }
        return SSD_OK;
    }
    if (!x || !dt || !A || !Bm || !Cm || !D || !dy || !dx || !ddt || !dB || !dC) return SSD_ERR_INVALID_ARG;
    if (!aligned(x, es) || !aligned(dt, es) || !aligned(Bm, es) || !aligned(Cm, es) || !aligned(dy, es) ||
        !aligned(dx, es) || !aligned(ddt, es) || !aligned(dB, es) || !aligned(dC, es) || !aligned(A, 4) ||
        !aligned(D, 4))
        return SSD_ERR_INVALID_ARG;
    const size_t nx = (size_t)(pr.B * pr.L * pr.nh * pr.H) * es;
    const size_t ndt = (size_t)(pr.B * pr.L * pr.nh) * es;
    const size_t nbc = (size_t)(pr.B * pr.L * pr.G * pr.S) * es;
    const void *ins[] = {x, dt, Bm, Cm, dy, h0, dh_final, A, D};
    const size_t in_sz[] = {nx, ndt, nbc, nbc, nx, h0 ? nstate * 4 : 0, dh_final ? nstate * 4 : 0,
                            (size_t)pr.nh * 4, (size_t)pr.nh * 4};
    const void *outs[] = {dx, ddt, dB, dC, dA, dD, dh0};
    const size_t out_sz[] = {nx, ndt, nbc, nbc, (size_t)pr.nh * 4, (size_t)pr.nh * 4, dh0 ? nstate * 4 : 0};
    for (int o = 0; o < 7; ++o) {
        for (int i = 0; i < 9; ++i)
            if (overlaps(outs[o], out_sz[o], ins[i], in_sz[i])) return SSD_ERR_INVALID_ARG;
        for (int o2 = o + 1; o2 < 7; ++o2)
            if (overlaps(outs[o], out_sz[o], outs[o2], out_sz[o2])) return SSD_ERR_INVALID_ARG;
    }
    ssd::BwdWork w;
    const size_t need = ssd::bwd_workspace(pr, workspace, &w);
    if (!workspace || !aligned(workspace, kWsAlign) || ws_bytes < need) return SSD_ERR_WORKSPACE;
    const ssd::BwdArgs a{x, dt, Bm, Cm, dy, A, D, h0, dh_final, dx, ddt, dB, dC, dA, dD, dh0};
    return cuda_status(ssd::launch_bwd(pr, a, w, st));
}

ssd_status ssd_s6_fwd(const ssd_s6_desc *desc, const void *x, const void *delta, const float *A, const void *Bm,
                  const void *Cm, const float *D, const float *h0, void *y, float *h_final, ssd_stream_t stream)
{
    if (!desc) return SSD_ERR_INVALID_ARG;
    if (desc->batch < 0 || desc->seqlen < 0 || desc->dim < 0 || desc->dstate < 1 || desc->ngroups < 1 ||
        desc->dim % desc->ngroups != 0 || desc->flags != 0 || desc->reserved != 0)
        return SSD_ERR_INVALID_ARG;
    if ((desc->in_dtype != SSD_F32 && desc->in_dtype != SSD_BF16) ||
        (desc->out_dtype != SSD_F32 && desc->out_dtype != SSD_BF16))
        return SSD_ERR_INVALID_ARG;
    if (desc->dstate > 32 || desc->batch > 65535 || desc->dim > 0x7fffffffLL) return SSD_ERR_UNSUPPORTED;
    // the offsets the kernel forms are 64-bit: arrays of 2^62 bytes or more are refused
    if (16.0 * (double)desc->batch * (double)desc->dim * (double)desc->seqlen * (double)desc->dstate >=
        4611686018427387904.0)
        return SSD_ERR_UNSUPPORTED;
    const ssd::S6Problem p{desc->batch, desc->seqlen, desc->dim, desc->dstate, desc->ngroups, desc->in_dtype,
                           desc->out_dtype};
    cudaStream_t st = (cudaStream_t)stream;
    const size_t nstate = (size_t)(p.B * p.dim * p.N);
    if ((h0 && !aligned(h0, 4)) || (h_final && !aligned(h_final, 4))) return SSD_ERR_INVALID_ARG;
    if (p.B == 0 || p.dim == 0) return SSD_OK;
    if (p.L == 0) {
        if (h_final) {
            cudaError_t e = h0 ? cudaMemcpyAsync(h_final, h0, nstate * sizeof(float), cudaMemcpyDeviceToDevice, st)
                               : cudaMemsetAsync(h_final, 0, nstate * sizeof(float), st);
            return cuda_status(e);
        }
        return SSD_OK;
    }
    if (!x || !delta || !A || !Bm || !Cm || !y) return SSD_ERR_INVALID_ARG;
    const size_t ei = esize(p.in_dt), eo = esize(p.out_dt);
    if (!aligned(x, ei) || !aligned(delta, ei) || !aligned(Bm, ei) || !aligned(Cm, ei) || !aligned(y, eo) ||
        !aligned(A, 4) || (D && !aligned(D, 4)))
        return SSD_ERR_INVALID_ARG;
    const size_t nx = (size_t)(p.B * p.dim * p.L), nbc = (size_t)(p.B * p.G * p.N * p.L);
    if (overlaps(y, nx * eo, x, nx * ei) || overlaps(y, nx * eo, delta, nx * ei) || overlaps(y, nx * eo, Bm, nbc * ei) ||
        overlaps(y, nx * eo, Cm, nbc * ei) || (h_final && overlaps(h_final, nstate * 4, y, nx * eo)))
        return SSD_ERR_INVALID_ARG;
    return cuda_status(ssd::launch_s6_scan(p, x, delta, A, Bm, Cm, D, h0, y, h_final, st));
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Forward pass without a caller-provided workspace (ssd_fwd_noalloc).
//
// For callers that cannot allocate device memory when they run the forward
// pass (graph capture in progress, allocator-less runtimes, plug-ins whose host
// owns all allocations): the scratch lives in this file-scope device array,
// which every GPU that loads libssd.so keeps for the life of the process.
// Host code must not hand the array's name to a kernel -- on the host it is only a
// stand-in symbol -- so its device address is looked up with cudaGetSymbolAddress while
// the device is current, and cached per CUDA context (the address belongs to the context
// the module is loaded in, so a context created later -- after cudaDeviceReset, or a
// host application's own context -- gets its own lookup).
// ---------------------------------------------------------------------------
static __device__ __align__(256) unsigned char g_noalloc_scratch[SSD_NOALLOC_SCRATCH_BYTES];

namespace {
constexpr int kMaxContexts = 64;
std::mutex g_noalloc_mutex;
struct NoallocEntry {
    CUcontext ctx;
    void *addr;
};
NoallocEntry g_noalloc[kMaxContexts];
int g_noalloc_used = 0;

// cuCtxGetCurrent through the runtime's driver entry-point query (the library does not link
// the driver API directly, so it loads where no driver is installed).
CUresult current_context(CUcontext *ctx)
{
    using Fn = CUresult (*)(CUcontext *);
    static Fn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (Fn)p;
    });
    return fn ? fn(ctx) : CUDA_ERROR_NOT_INITIALIZED;
}

// Device address of the scratch array in the current context (nullptr on error).  The
// lookup itself makes the device's primary context current when no context is.
void *noalloc_scratch_address()
{
    CUcontext ctx = nullptr;
    if (current_context(&ctx) == CUDA_SUCCESS && ctx) {
        std::lock_guard<std::mutex> lock(g_noalloc_mutex);
        for (int i = 0; i < g_noalloc_used; ++i)
            if (g_noalloc[i].ctx == ctx) return g_noalloc[i].addr;
    }
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return nullptr;
    if (current_context(&ctx) != CUDA_SUCCESS || !ctx) return p;
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    for (int i = 0; i < g_noalloc_used; ++i)
        if (g_noalloc[i].ctx == ctx) return g_noalloc[i].addr;
    const int slot = g_noalloc_used < kMaxContexts ? g_noalloc_used++ : kMaxContexts - 1;
    g_noalloc[slot] = NoallocEntry{ctx, p};
    return p;
}
}  // namespace

extern "C" ssd_status ssd_fwd_noalloc(const ssd_desc *desc, const void *x, const void *dt, const float *A,
                                      const void *Bm, const void *Cm, const float *D, const float *h0,
                                      void *y, float *h_final, ssd_stream_t stream)
{
    Problem pr;
    ssd_status s = check_desc(desc, &pr, true);
    if (s != SSD_OK) return s;
    const size_t need = nonempty(pr) ? carve(pr, nullptr).bytes : 0;
    if (need > SSD_NOALLOC_SCRATCH_BYTES) return SSD_ERR_TOO_LARGE;
    void *scratch = noalloc_scratch_address();
    if (!scratch) return SSD_ERR_CUDA;
    return fwd_impl(desc, x, dt, A, Bm, Cm, D, h0, y, h_final, scratch, SSD_NOALLOC_SCRATCH_BYTES,
                    (cudaStream_t)stream, nullptr);
}

extern "C" ssd_status ssd_fwd_noalloc_check(ssd_stream_t stream)
{
    void *scratch = noalloc_scratch_address();
    if (!scratch) return SSD_ERR_CUDA;
    return ssd_fwd_check(scratch, stream);
}
