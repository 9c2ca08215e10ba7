// ssd_bwd.cu -- gradients of the chunked SSD forward pass, on the CUDA cores (float32).
//
// Reverse mode of the recurrence h_t = exp(A dt_t) h_{t-1} + dt_t B_t x_t^T,
// y_t = c_t^T h_t + D x_t (NVIDIA developer blog "Accelerating Mamba-2 with
// High-Performance Forward Pass Kernels in NVIDIA CUDA Tile", section "Mamba-2
// architecture"), taken chunk by chunk.  "Sasha Rush: Mamba: The Hard Way",
// Part 3, shows the pattern: the adjoint state is the same scan run backwards,
// and each coefficient's gradient pairs a forward quantity with a backward one.
//
// Per (batch, head) and chunk k, with the in-chunk cumsum G (stored x log2 e),
// the state h_in entering the chunk and the gradient Lam of the state leaving it:
//   u_k        = sum_i exp(G_i) dy_i C_i^T                        (k_bwd_dstate)
//   Lam_{k-1}  = exp(G_last,k) Lam_k + u_k,  Lam_{nc-1} = dh_final,
//   dh0        = exp(G_last,0) Lam_0 + u_0                        (k_bwd_state_passing)
//   Dec[i,j]   = exp(G_i - G_j) for i >= j, else 0;  el_j = exp(G_last - G_j)
//   v_j        = sum_i Dec (C_i.B_j) dy_i + el_j Lam B_j,    dx_j = dt_j v_j + D dy_j
//   dB_j      += dt_j (sum_i Dec (dy_i.x_j) C_i + el_j Lam^T x_j)   (k_bwd_chunk_cols)
//   dC_i      += exp(G_i) h_in^T dy_i + sum_j Dec dt_j (dy_i.x_j) B_j  (k_bwd_chunk_rows)
//   M[i,j]     = Dec (C_i.B_j) dt_j (dy_i.x_j),   N_j = el_j dt_j x_j.(Lam B_j)
//   dG_i       = exp(G_i) dy_i.(h_in C_i) + sum_j M[i,j] - sum_i' M[i',i] - N_i
//                + [i last] (exp(G_last) <Lam, h_in> + sum_j N_j)
//   da_t       = sum_{i >= t} dG_i,  ddt_t = x_t.v_t + A da_t,  dA = sum dt_t da_t   (k_bwd_finalize)
//
// Every sum over heads (dB, dC), over tokens and batch (dA, dD) is taken in a fixed
// order: the result does not depend on scheduling.
#include <string.h>

#include <algorithm>

#include "ssd_common.cuh"
#include "ssd_tc.cuh"

namespace ssd {
namespace {

constexpr int kTok = 32;        // tokens per tile (rows of the column / row kernels)
constexpr int kTilePad = 33;    // padded row of a 32 x 32 tile

template <typename T>
__device__ __forceinline__ void load_rows(float *dst, int ld, const T *src, int64_t stride, int valid, int width)
{
    // rows r < 32 of width `width` from src + r * stride; rows >= valid are zero.
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int r = warp; r < kTok; r += 8) {
        const T *row = src + (int64_t)(r < valid ? r : 0) * stride;
        for (int c = lane; c < width; c += 32) dst[r * ld + c] = r < valid ? to_f32(row[c]) : 0.f;
    }
}

__device__ __forceinline__ float dot_rows(const float *a, const float *b, int n)
{
    float acc = 0.f;
    for (int e = 0; e < n; ++e) acc = fmaf(a[e], b[e], acc);
    return acc;
}

__device__ __forceinline__ float sum8(float v)   // sum over the 8 lanes that share tid >> 3
{
    v += __shfl_xor_sync(0xffffffffu, v, 1);
    v += __shfl_xor_sync(0xffffffffu, v, 2);
    v += __shfl_xor_sync(0xffffffffu, v, 4);
    return v;
}

__device__ __forceinline__ float sum32(float v)
{
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}

// ---------------------------------------------------------------------------
// u_k[p][s] = sum_{i in chunk k} exp2(G_i) dy_i[p] C_i[s]: the gradient that chunk k's
// outputs send to the state entering it.  One block per (chunk, head x 32-row p tile x
// 64-column s tile, batch), like the forward chunk_state on CUDA cores.
// ---------------------------------------------------------------------------
template <typename Tio>
__global__ void __launch_bounds__(256)
k_bwd_dstate(const Tio *__restrict__ dy, const Tio *__restrict__ Cm, const float *__restrict__ G,
             float *__restrict__ u, Problem pr, int ptiles, int stiles)
{
    __shared__ float yw[kTok][33];   // [token][p]  exp2(G_t) dy[t][p]
    __shared__ float ct[kTok][64];   // [token][s]
    __shared__ float w[kTok];
    const int k = blockIdx.x, b = blockIdx.z;
    const int h = blockIdx.y / (ptiles * stiles);
    const int tile = blockIdx.y % (ptiles * stiles);
    const int p0 = (tile / stiles) * 32, s0 = (tile % stiles) * 64;
    const int g = (int)(h / pr.hpg);
    const int64_t t0 = (int64_t)k * pr.T;
    const int n = (int)(pr.T < pr.L - t0 ? pr.T : pr.L - t0);
    const float *Gh = G + ((int64_t)b * pr.nh + h) * pr.L + t0;
    const int tx = threadIdx.x & 63, ty = threadIdx.x >> 6;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.f;
    for (int seg = 0; seg < n; seg += kTok) {
        if (threadIdx.x < kTok) {
            const int t = seg + threadIdx.x;
            w[threadIdx.x] = t < n ? exp2f(Gh[t]) : 0.f;
        }
        __syncthreads();
        for (int r = warp; r < kTok; r += 8) {
            const int t = seg + r, p = p0 + lane;
            float v = 0.f;
            if (t < n && p < pr.H) v = w[r] * to_f32(dy[(((int64_t)b * pr.L + t0 + t) * pr.nh + h) * pr.H + p]);
            yw[r][lane] = v;
            for (int c = lane; c < 64; c += 32) {
                const int s = s0 + c;
                float q = 0.f;
                if (t < n && s < pr.S) q = to_f32(Cm[(((int64_t)b * pr.L + t0 + t) * pr.G + g) * pr.S + s]);
                ct[r][c] = q;
            }
        }
        __syncthreads();
#pragma unroll 8
        for (int r = 0; r < kTok; ++r) {
            const float cv = ct[r][tx];
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[i] = fmaf(yw[r][ty * 8 + i], cv, acc[i]);
        }
        __syncthreads();
    }
    const int s = s0 + tx;
    if (s < pr.S) {
        float *dst = u + ((((int64_t)b * pr.nh + h) * pr.nc + k) * pr.H) * pr.S;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int p = p0 + ty * 8 + i;
            if (p < pr.H) dst[(int64_t)p * pr.S + s] = acc[i];
        }
    }
}

// The same contraction with register blocking, for H = 64 or 128 and S = 128 or 256:
// one block per (chunk, 64-row p tile, batch x head), each thread 4 rows p x 8 columns s
// (the columns 4 (c + 32 k) + e of 128-wide halves), 32 tokens per step staged in shared
// memory as exp2(G_t) dy[t][p] and C[t][s].
template <typename Tio, int S>
__global__ void __launch_bounds__(256)
k_bwd_dstate_fast(const Tio *__restrict__ dy, const Tio *__restrict__ Cm, const float *__restrict__ G,
                  float *__restrict__ u, Problem pr)
{
    constexpr int SQ = S / 128;                   // 4-column chunks per thread
    __shared__ __align__(16) float yw[kTok][64];  // [token][p]  exp2(G_t) dy[t][p0 + p]
    __shared__ __align__(16) float ct[kTok][S];   // [token][s]
    const int k = blockIdx.x, p0 = blockIdx.y * 64;
    const int64_t bh = blockIdx.z;
    const int b = (int)(bh / pr.nh), h = (int)(bh % pr.nh);
    const int g = (int)(h / pr.hpg);
    const int64_t t0 = (int64_t)k * pr.T;
    const int n = (int)(pr.T < pr.L - t0 ? pr.T : pr.L - t0);
    const float *Gh = G + bh * pr.L + t0;
    const int tid = threadIdx.x;
    const int pr4 = (tid >> 4) * 4;               // rows p0 + pr4 .. + 3
    const int cc = tid & 15;                      // columns 4 (cc + 16 k) + e... within S
    float acc[4][4 * 2 * SQ];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 8 * SQ; ++j) acc[i][j] = 0.f;
    for (int seg = 0; seg < n; seg += kTok) {
        __syncthreads();
        for (int e = tid; e < kTok * 64; e += 256) {
            const int r = e >> 6, p = e & 63, t = seg + r;
            float v = 0.f;
            if (t < n) v = exp2f(Gh[t]) * to_f32(dy[(((int64_t)b * pr.L + t0 + t) * pr.nh + h) * pr.H + p0 + p]);
            yw[r][p] = v;
        }
        for (int e = tid; e < kTok * S; e += 256) {
            const int r = e / S, s = e % S, t = seg + r;
            ct[r][s] = t < n ? to_f32(Cm[(((int64_t)b * pr.L + t0 + t) * pr.G + g) * pr.S + s]) : 0.f;
        }
        __syncthreads();
#pragma unroll 4
        for (int r = 0; r < kTok; ++r) {
            const float4 a = *reinterpret_cast<const float4 *>(&yw[r][pr4]);
            const float av[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
            for (int q = 0; q < 2 * SQ; ++q) {
                const float4 cv = *reinterpret_cast<const float4 *>(&ct[r][4 * (cc + 16 * q)]);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    acc[i][4 * q] = fmaf(av[i], cv.x, acc[i][4 * q]);
                    acc[i][4 * q + 1] = fmaf(av[i], cv.y, acc[i][4 * q + 1]);
                    acc[i][4 * q + 2] = fmaf(av[i], cv.z, acc[i][4 * q + 2]);
                    acc[i][4 * q + 3] = fmaf(av[i], cv.w, acc[i][4 * q + 3]);
                }
            }
        }
    }
    float *dst = u + (((bh * pr.nc + k) * pr.H) + p0 + pr4) * pr.S;
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int q = 0; q < 2 * SQ; ++q)
            *reinterpret_cast<float4 *>(dst + (int64_t)i * pr.S + 4 * (cc + 16 * q)) =
                make_float4(acc[i][4 * q], acc[i][4 * q + 1], acc[i][4 * q + 2], acc[i][4 * q + 3]);
}

// ---------------------------------------------------------------------------
// Backwards over chunks, in place: on entry lam[k] holds u_k, on exit the gradient
// Lam_k of the state leaving chunk k.  One thread per state element of one sequence;
// dh0 (nullable) receives exp2(G_last,0) Lam_0 + u_0.  The u loads of kBatch chunks are
// issued together (they do not depend on the running value).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256)
k_bwd_state_passing(const float *__restrict__ G, float *__restrict__ lam, const float *__restrict__ dh_final,
                    float *__restrict__ dh0, Problem pr)
{
    constexpr int kBatch = 8;
    const int64_t HS = pr.H * pr.S;
    const int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= HS) return;
    for (int64_t bh = blockIdx.y; bh < pr.B * pr.nh; bh += gridDim.y) {
        const float *Gh = G + bh * pr.L;
        float *base = lam + bh * pr.nc * HS + e;
        float run = dh_final ? dh_final[bh * HS + e] : 0.f;
        for (int64_t k1 = pr.nc; k1 > 0; k1 -= kBatch) {
            const int cnt = (int)(k1 < kBatch ? k1 : kBatch);
            float uv[kBatch], dec[kBatch];
#pragma unroll
            for (int i = 0; i < kBatch; ++i) {
                if (i < cnt) {
                    const int64_t k = k1 - 1 - i;
                    uv[i] = base[k * HS];
                    dec[i] = exp2f(Gh[min(pr.L, (k + 1) * pr.T) - 1]);
                }
            }
#pragma unroll
            for (int i = 0; i < kBatch; ++i) {
                if (i < cnt) {
                    base[(k1 - 1 - i) * HS] = run;
                    run = fmaf(dec[i], run, uv[i]);
                }
            }
        }
        if (dh0) dh0[bh * HS + e] = run;
    }
}

// ---------------------------------------------------------------------------
// Column side of one chunk: for a tile J of 32 tokens j and each head h of a slice of
// the group's heads, sums over the rows i >= j of the chunk:
//   dx_j, q_j = x_j.v_j, N_j, colM_j = sum_i M[i,j], dy_j.x_j   (per head, per token)
//   dB_j                                                         (summed over the slice)
// Block: 256 threads.  Tile builds: lane = j, warp w takes rows i = w, w+8, w+16, w+24.
// Accumulation: thread (r = tid >> 3, c = tid & 7) owns row j = j0 + r, columns
// c, c + 8, ... (HQ of p, SQ of s).
// ---------------------------------------------------------------------------
template <typename Tio, int HQ, int SQ>
__global__ void __launch_bounds__(256)
k_bwd_chunk_cols(const Tio *__restrict__ x, const Tio *__restrict__ dt, const Tio *__restrict__ Bm,
                 const Tio *__restrict__ Cm, const Tio *__restrict__ dy, const float *__restrict__ D,
                 const float *__restrict__ G, const float *__restrict__ lam, Tio *__restrict__ dx,
                 float *__restrict__ Qd, float *__restrict__ Nd, float *__restrict__ Cmd, float *__restrict__ Dd,
                 float *__restrict__ dBp, Problem pr, int nT, int nslice, int hps)
{
    extern __shared__ float sm[];
    const int H = (int)pr.H, S = (int)pr.S, SP = S + 1, HP = H + 1;
    float *Bj = sm;                              // [32][SP]  B rows of J
    float *Ci = Bj + kTok * SP;                  // [32][SP]  C rows of I
    float *Xj = Ci + kTok * SP;                  // [32][HP]  x rows of J (current head)
    float *Yi = Xj + kTok * HP;                  // [32][HP]  dy rows of I (current head)
    float *CBc = Yi + kTok * HP;                 // [nT][32][33]  C_i . B_j for the tiles I >= J
    float *Pc = CBc + nT * kTok * kTilePad;      // [32][33]  Dec (C_i . B_j)
    float *Py = Pc + kTok * kTilePad;            // [32][33]  Dec dt_j (dy_i . x_j)
    float *Gt = Py + kTok * kTilePad;            // [T]       G of the chunk (current head)
    float *red = Gt + pr.T;                      // [8][32]   per-warp column partials
    float *dtj = red + 8 * kTok;                 // [32]
    float *diag = dtj + kTok;                    // [32]      dy_j . x_j
    float *Ls = diag + kTok;                     // staging of Lam: [H][33] or [8][S]

    const int k = blockIdx.x / nT, jb = blockIdx.x % nT;
    const int g = blockIdx.y / nslice, sl = blockIdx.y % nslice;
    const int b = blockIdx.z;
    const int64_t t0 = (int64_t)k * pr.T;
    const int n = (int)(pr.T < pr.L - t0 ? pr.T : pr.L - t0);
    const int j0 = jb * kTok;
    if (j0 >= n) return;
    const int h_lo = g * (int)pr.hpg + sl * hps;
    const int h_hi = min(h_lo + hps, (g + 1) * (int)pr.hpg);
    const int nvT = (n + kTok - 1) / kTok;
    const int rows_j = min(kTok, n - j0);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int r = tid >> 3, c = tid & 7;
    const int64_t xs = pr.nh * pr.H, bs = pr.G * pr.S;     // token strides of x / dy and of B / C

    load_rows(Bj, SP, Bm + (((int64_t)b * pr.L + t0 + j0) * pr.G + g) * pr.S, bs, rows_j, S);
    for (int ib = jb; ib < nvT; ++ib) {
        const int i0 = ib * kTok;
        __syncthreads();
        load_rows(Ci, SP, Cm + (((int64_t)b * pr.L + t0 + i0) * pr.G + g) * pr.S, bs, min(kTok, n - i0), S);
        __syncthreads();
        float *cb = CBc + (ib - jb) * kTok * kTilePad;
        for (int m = 0; m < 4; ++m) {
            const int ii = warp + 8 * m;
            cb[ii * kTilePad + lane] = dot_rows(Ci + ii * SP, Bj + lane * SP, S);
        }
    }

    float accB[SQ];
#pragma unroll
    for (int q = 0; q < SQ; ++q) accB[q] = 0.f;

    for (int h = h_lo; h < h_hi; ++h) {
        const int64_t bh = (int64_t)b * pr.nh + h;
        __syncthreads();
        load_rows(Xj, HP, x + (((int64_t)b * pr.L + t0 + j0) * pr.nh + h) * pr.H, xs, rows_j, H);
        for (int t = tid; t < n; t += blockDim.x) Gt[t] = G[bh * pr.L + t0 + t];
        if (tid < kTok) dtj[tid] = tid < rows_j ? to_f32(dt[((int64_t)b * pr.L + t0 + j0 + tid) * pr.nh + h]) : 0.f;
        float accV[HQ];
#pragma unroll
        for (int q = 0; q < HQ; ++q) accV[q] = 0.f;
        float colp = 0.f;
        for (int ib = jb; ib < nvT; ++ib) {
            const int i0 = ib * kTok;
            const int rows_i = min(kTok, n - i0);
            __syncthreads();
            load_rows(Yi, HP, dy + (((int64_t)b * pr.L + t0 + i0) * pr.nh + h) * pr.H, xs, rows_i, H);
            load_rows(Ci, SP, Cm + (((int64_t)b * pr.L + t0 + i0) * pr.G + g) * pr.S, bs, rows_i, S);
            __syncthreads();
            const float *cb = CBc + (ib - jb) * kTok * kTilePad;
            const int j = j0 + lane;
            for (int m = 0; m < 4; ++m) {
                const int ii = warp + 8 * m, i = i0 + ii;
                const float yx = dot_rows(Yi + ii * HP, Xj + lane * HP, H);
                const bool on = i < n && j < n && i >= j;            // select, never multiply, the mask
                const float dec = on ? exp2f(Gt[on ? i : 0] - Gt[on ? j : 0]) : 0.f;
                const float pc = dec * cb[ii * kTilePad + lane];
                Pc[ii * kTilePad + lane] = pc;
                Py[ii * kTilePad + lane] = dec * yx * dtj[lane];
                colp = fmaf(pc, yx, colp);
                if (ib == jb && ii == lane) diag[lane] = yx;
            }
            __syncthreads();
#pragma unroll 4
            for (int ii = 0; ii < kTok; ++ii) {
                const float pcv = Pc[ii * kTilePad + r], pyv = Py[ii * kTilePad + r];
#pragma unroll
                for (int q = 0; q < HQ; ++q)
                    if (c + 8 * q < H) accV[q] = fmaf(pcv, Yi[ii * HP + c + 8 * q], accV[q]);
#pragma unroll
                for (int q = 0; q < SQ; ++q)
                    if (c + 8 * q < S) accB[q] = fmaf(pyv, Ci[ii * SP + c + 8 * q], accB[q]);
            }
        }
        // Lam B_j (p = c + 8q) and Lam^T x_j (s = c + 8q), Lam streamed through shared memory
        const float *Lk = lam + ((bh * pr.nc + k) * pr.H) * pr.S;
        float accLB[HQ], accLX[SQ];
#pragma unroll
        for (int q = 0; q < HQ; ++q) accLB[q] = 0.f;
#pragma unroll
        for (int q = 0; q < SQ; ++q) accLX[q] = 0.f;
        for (int s0 = 0; s0 < S; s0 += 32) {
            __syncthreads();
            for (int p = warp; p < H; p += 8) Ls[p * 33 + lane] = s0 + lane < S ? Lk[(int64_t)p * S + s0 + lane] : 0.f;
            __syncthreads();
            const int send = min(32, S - s0);
            for (int ss = 0; ss < send; ++ss) {
                const float bv = Bj[r * SP + s0 + ss];
#pragma unroll
                for (int q = 0; q < HQ; ++q)
                    if (c + 8 * q < H) accLB[q] = fmaf(bv, Ls[(c + 8 * q) * 33 + ss], accLB[q]);
            }
        }
        for (int p0 = 0; p0 < H; p0 += 8) {
            __syncthreads();
            for (int e = tid; e < 8 * S; e += blockDim.x) {
                const int pp = e / S, s = e - pp * S;
                Ls[e] = p0 + pp < H ? Lk[(int64_t)(p0 + pp) * S + s] : 0.f;
            }
            __syncthreads();
            const int pend = min(8, H - p0);
            for (int pp = 0; pp < pend; ++pp) {
                const float xv = Xj[r * HP + p0 + pp];
#pragma unroll
                for (int q = 0; q < SQ; ++q)
                    if (c + 8 * q < S) accLX[q] = fmaf(xv, Ls[pp * S + c + 8 * q], accLX[q]);
            }
        }
        red[warp * kTok + lane] = colp;
        __syncthreads();
        // outputs of row j = j0 + r
        const int j = j0 + r;
        const bool valid = r < rows_j;
        const float el = exp2f(Gt[n - 1] - Gt[valid ? j : 0]);
        const float dtv = dtj[r];
        const float dh = D[h];
        const Tio *dyj = dy + (((int64_t)b * pr.L + t0 + (valid ? j : 0)) * pr.nh + h) * pr.H;
        Tio *dxj = dx + (((int64_t)b * pr.L + t0 + (valid ? j : 0)) * pr.nh + h) * pr.H;
        float qpart = 0.f, npart = 0.f;
#pragma unroll
        for (int q = 0; q < HQ; ++q) {
            const int p = c + 8 * q;
            if (p < H) {
                const float v = fmaf(el, accLB[q], accV[q]);
                const float xv = Xj[r * HP + p];
                qpart = fmaf(xv, v, qpart);
                npart = fmaf(xv, accLB[q], npart);
                if (valid) dxj[p] = from_f32<Tio>(fmaf(dtv, v, dh * to_f32(dyj[p])));
            }
        }
        qpart = sum8(qpart);
        npart = sum8(npart);
#pragma unroll
        for (int q = 0; q < SQ; ++q) accB[q] = fmaf(dtv * el, accLX[q], accB[q]);
        if (c == 0 && valid) {
            float cm = 0.f;
            for (int w2 = 0; w2 < 8; ++w2) cm += red[w2 * kTok + r];
            const int64_t o = bh * pr.L + t0 + j;
            Qd[o] = qpart;
            Nd[o] = el * dtv * npart;
            Cmd[o] = dtv * cm;
            Dd[o] = diag[r];
        }
    }
    if (r < rows_j) {
        float *dst = dBp + ((((int64_t)sl * pr.B + b) * pr.L + t0 + j0 + r) * pr.G + g) * pr.S;
#pragma unroll
        for (int q = 0; q < SQ; ++q)
            if (c + 8 * q < S) dst[c + 8 * q] = accB[q];
    }
}

// ---------------------------------------------------------------------------
// Row side of one chunk: for a tile I of 32 tokens i and each head h of a slice, sums
// over the columns j <= i:
//   R_i = exp(G_i) dy_i.(h_in C_i) + sum_j M[i,j]                 (per head, per token)
//   dC_i = exp(G_i) h_in^T dy_i + sum_j Dec dt_j (dy_i.x_j) B_j    (summed over the slice)
// Same thread layout as the column kernel, with rows i in place of j.
// ---------------------------------------------------------------------------
template <typename Tio, int SQ>
__global__ void __launch_bounds__(256)
k_bwd_chunk_rows(const Tio *__restrict__ x, const Tio *__restrict__ dt, const Tio *__restrict__ Bm,
                 const Tio *__restrict__ Cm, const Tio *__restrict__ dy, const float *__restrict__ G,
                 const float *__restrict__ h_start, float *__restrict__ Rw, float *__restrict__ dCp,
                 Problem pr, int nT, int nslice, int hps)
{
    extern __shared__ float sm[];
    const int H = (int)pr.H, S = (int)pr.S, SP = S + 1, HP = H + 1;
    float *Ci = sm;                              // [32][SP]  C rows of I
    float *Bj = Ci + kTok * SP;                  // [32][SP]  B rows of J
    float *Xj = Bj + kTok * SP;                  // [32][HP]  x rows of J (current head)
    float *Yi = Xj + kTok * HP;                  // [32][HP]  dy rows of I (current head)
    float *CBc = Yi + kTok * HP;                 // [nT][32][33]  C_i . B_j for the tiles J <= I
    float *Pd = CBc + nT * kTok * kTilePad;      // [32][33]  Dec dt_j (dy_i . x_j)
    float *Gt = Pd + kTok * kTilePad;            // [T]
    float *dtj = Gt + pr.T;                      // [32]
    float *rowM = dtj + kTok;                    // [32]
    float *Hs = rowM + kTok;                     // staging of h_in: [8][S]

    const int k = blockIdx.x / nT, ib = blockIdx.x % nT;
    const int g = blockIdx.y / nslice, sl = blockIdx.y % nslice;
    const int b = blockIdx.z;
    const int64_t t0 = (int64_t)k * pr.T;
    const int n = (int)(pr.T < pr.L - t0 ? pr.T : pr.L - t0);
    const int i0 = ib * kTok;
    if (i0 >= n) return;
    const int h_lo = g * (int)pr.hpg + sl * hps;
    const int h_hi = min(h_lo + hps, (g + 1) * (int)pr.hpg);
    const int rows_i = min(kTok, n - i0);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int r = tid >> 3, c = tid & 7;
    const int64_t xs = pr.nh * pr.H, bs = pr.G * pr.S;

    load_rows(Ci, SP, Cm + (((int64_t)b * pr.L + t0 + i0) * pr.G + g) * pr.S, bs, rows_i, S);
    for (int jb = 0; jb <= ib; ++jb) {
        const int jj0 = jb * kTok;
        __syncthreads();
        load_rows(Bj, SP, Bm + (((int64_t)b * pr.L + t0 + jj0) * pr.G + g) * pr.S, bs, min(kTok, n - jj0), S);
        __syncthreads();
        float *cb = CBc + jb * kTok * kTilePad;
        for (int m = 0; m < 4; ++m) {
            const int ii = warp + 8 * m;
            cb[ii * kTilePad + lane] = dot_rows(Ci + ii * SP, Bj + lane * SP, S);
        }
    }

    float accC[SQ];
#pragma unroll
    for (int q = 0; q < SQ; ++q) accC[q] = 0.f;

    for (int h = h_lo; h < h_hi; ++h) {
        const int64_t bh = (int64_t)b * pr.nh + h;
        __syncthreads();
        load_rows(Yi, HP, dy + (((int64_t)b * pr.L + t0 + i0) * pr.nh + h) * pr.H, xs, rows_i, H);
        for (int t = tid; t < n; t += blockDim.x) Gt[t] = G[bh * pr.L + t0 + t];
        float rowp[4] = {0.f, 0.f, 0.f, 0.f};
        for (int jb = 0; jb <= ib; ++jb) {
            const int jj0 = jb * kTok;
            const int rows_j = min(kTok, n - jj0);
            __syncthreads();
            load_rows(Xj, HP, x + (((int64_t)b * pr.L + t0 + jj0) * pr.nh + h) * pr.H, xs, rows_j, H);
            load_rows(Bj, SP, Bm + (((int64_t)b * pr.L + t0 + jj0) * pr.G + g) * pr.S, bs, rows_j, S);
            if (tid < kTok) dtj[tid] = tid < rows_j ? to_f32(dt[((int64_t)b * pr.L + t0 + jj0 + tid) * pr.nh + h]) : 0.f;
            __syncthreads();
            const float *cb = CBc + jb * kTok * kTilePad;
            const int j = jj0 + lane;
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const int ii = warp + 8 * m, i = i0 + ii;
                const float yx = dot_rows(Yi + ii * HP, Xj + lane * HP, H);
                const bool on = i < n && j < n && i >= j;
                const float dec = on ? exp2f(Gt[on ? i : 0] - Gt[on ? j : 0]) : 0.f;
                const float pd = dec * dtj[lane] * yx;
                Pd[ii * kTilePad + lane] = pd;
                rowp[m] = fmaf(pd, cb[ii * kTilePad + lane], rowp[m]);
            }
            __syncthreads();
#pragma unroll 4
            for (int jj = 0; jj < kTok; ++jj) {
                const float pv = Pd[r * kTilePad + jj];
#pragma unroll
                for (int q = 0; q < SQ; ++q)
                    if (c + 8 * q < S) accC[q] = fmaf(pv, Bj[jj * SP + c + 8 * q], accC[q]);
            }
        }
        // carried term: w_i = h_in^T dy_i, streamed 8 rows of h_in at a time
        const float *Hk = h_start + ((bh * pr.nc + k) * pr.H) * pr.S;
        float accW[SQ];
#pragma unroll
        for (int q = 0; q < SQ; ++q) accW[q] = 0.f;
        for (int p0 = 0; p0 < H; p0 += 8) {
            __syncthreads();
            for (int e = tid; e < 8 * S; e += blockDim.x) {
                const int pp = e / S, s = e - pp * S;
                Hs[e] = p0 + pp < H ? Hk[(int64_t)(p0 + pp) * S + s] : 0.f;
            }
            __syncthreads();
            const int pend = min(8, H - p0);
            for (int pp = 0; pp < pend; ++pp) {
                const float yv = Yi[r * HP + p0 + pp];
#pragma unroll
                for (int q = 0; q < SQ; ++q)
                    if (c + 8 * q < S) accW[q] = fmaf(yv, Hs[pp * S + c + 8 * q], accW[q]);
            }
        }
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            const float v = sum32(rowp[m]);
            if (lane == 0) rowM[warp + 8 * m] = v;
        }
        __syncthreads();
        const bool valid = r < rows_i;
        const float eg = exp2f(Gt[valid ? i0 + r : 0]);
        float ypart = 0.f;
#pragma unroll
        for (int q = 0; q < SQ; ++q) {
            if (c + 8 * q < S) {
                ypart = fmaf(accW[q], Ci[r * SP + c + 8 * q], ypart);
                accC[q] = fmaf(eg, accW[q], accC[q]);
            }
        }
        ypart = sum8(ypart);
        if (c == 0 && valid) Rw[bh * pr.L + t0 + i0 + r] = fmaf(eg, ypart, rowM[r]);
    }
    if (r < rows_i) {
        float *dst = dCp + ((((int64_t)sl * pr.B + b) * pr.L + t0 + i0 + r) * pr.G + g) * pr.S;
#pragma unroll
        for (int q = 0; q < SQ; ++q)
            if (c + 8 * q < S) dst[c + 8 * q] = accC[q];
    }
}

// ---------------------------------------------------------------------------
// Fast column and row kernels for H in {64, 128} and S in {128, 256} (16-byte aligned
// rows).  Same sums as k_bwd_chunk_cols / k_bwd_chunk_rows, organised for the load/store
// unit and for latency:
//  * 32 x 32 tile products (C.B, dy.x) read the broadcast row from a 16-byte-aligned
//    buffer and the per-lane row with stride K + 4, both by 128-bit loads (5 loads per
//    16 FMA, conflict-free per quarter warp);
//  * in the accumulations thread (r, c) owns the column chunks 4 (c + 8k): the 8 lanes
//    of a quarter warp read 128 contiguous bytes;
//  * the next tile's rows are loaded into registers (16-byte vectors) while the current
//    tile is computed;
//  * one pass over Lam (or h_in) per head, in slabs of 32 rows.
// ---------------------------------------------------------------------------
template <typename Tio, int W>
struct RowTile {                                   // 32 rows of W elements, 16-byte vectors
    static constexpr int kPer = 16 / (int)sizeof(Tio);
    static constexpr int kVecRow = W / kPer;
    static constexpr int kVec = 32 * kVecRow / 256;
    static_assert(kVec >= 1 && (32 * kVecRow) % 256 == 0, "tile");
    uint4 r[kVec];
    __device__ __forceinline__ void load(const Tio *base, int64_t stride, int valid)
    {
#pragma unroll
        for (int i = 0; i < kVec; ++i) {
            const int v = i * 256 + (int)threadIdx.x, row = v / kVecRow, col = v % kVecRow;
            r[i] = make_uint4(0u, 0u, 0u, 0u);
            if (row < valid) r[i] = *reinterpret_cast<const uint4 *>(base + (int64_t)row * stride + col * kPer);
        }
    }
    __device__ __forceinline__ void store(float *dst, int ld) const
    {
#pragma unroll
        for (int i = 0; i < kVec; ++i) {
            const int v = i * 256 + (int)threadIdx.x, row = v / kVecRow, col = v % kVecRow;
            float *d = dst + row * ld + col * kPer;
            if constexpr (sizeof(Tio) == 2) {
                const uint32_t w[4] = {r[i].x, r[i].y, r[i].z, r[i].w};
                float f[8];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    f[2 * e] = __uint_as_float(w[e] << 16);
                    f[2 * e + 1] = __uint_as_float(w[e] & 0xffff0000u);
                }
                *reinterpret_cast<float4 *>(d) = make_float4(f[0], f[1], f[2], f[3]);
                *reinterpret_cast<float4 *>(d + 4) = make_float4(f[4], f[5], f[6], f[7]);
            } else {
                *reinterpret_cast<float4 *>(d) = make_float4(__uint_as_float(r[i].x), __uint_as_float(r[i].y),
                                                             __uint_as_float(r[i].z), __uint_as_float(r[i].w));
            }
        }
    }
};

__device__ __forceinline__ float4 ld4(const float *p) { return *reinterpret_cast<const float4 *>(p); }

// acc[m] += dot(rows[m] (broadcast, stride lda), lane row (stride ldb)) over K, m < 4
template <int K>
__device__ __forceinline__ void dots4(float acc[4], const float *a0, int lda, const float *bl)
{
#pragma unroll 4
    for (int k = 0; k < K; k += 4) {
        const float4 b = ld4(bl + k);
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            const float4 a = ld4(a0 + m * 8 * lda + k);
            acc[m] = fmaf(a.x, b.x, fmaf(a.y, b.y, fmaf(a.z, b.z, fmaf(a.w, b.w, acc[m]))));
        }
    }
}

template <typename Tio, int H, int S>
struct FastCfg {
    static constexpr int BS = S + 4, XS = H + 4;   // strides of the per-lane-row tiles
    static constexpr int HV = H / 8, SV = S / 8;   // columns per thread (chunks of 4)
    static size_t cols_floats(int T, int nT)
    {
        const int region = 32 * H + 32 * S;        // dy tile + C tile; later the Lam slab and Lam B
        return (size_t)32 * BS + 32 * XS + region + (size_t)nT * kTok * kTilePad + 2 * kTok * kTilePad + T + 8 * kTok +
               2 * kTok;
    }
    static size_t rows_floats(int T, int nT)
    {
        return (size_t)32 * S + 32 * H + 32 * BS + 32 * XS + (size_t)nT * kTok * kTilePad + kTok * kTilePad + T +
               2 * kTok;
    }
};

template <typename Tio, int H, int S>
__global__ void __launch_bounds__(256)
k_bwd_cols_fast(const Tio *__restrict__ x, const Tio *__restrict__ dt, const Tio *__restrict__ Bm,
                const Tio *__restrict__ Cm, const Tio *__restrict__ dy, const float *__restrict__ D,
                const float *__restrict__ G, const float *__restrict__ lam, Tio *__restrict__ dx,
                float *__restrict__ Qd, float *__restrict__ Nd, float *__restrict__ Cmd, float *__restrict__ Dd,
                float *__restrict__ dBp, Problem pr, int nT, int nslice, int hps)
{
    using Cfg = FastCfg<Tio, H, S>;
    constexpr int BS = Cfg::BS, XS = Cfg::XS, HV = Cfg::HV, SV = Cfg::SV;
    extern __shared__ float4 smv[];
    float *Bj = reinterpret_cast<float *>(smv);  // [32][BS]  B rows of J
    float *Xj = Bj + 32 * BS;                    // [32][XS]  x rows of J (current head)
    float *Yi = Xj + 32 * XS;                    // [32][H]   dy rows of I (current head)
    float *Ci = Yi + 32 * H;                     // [32][S]   C rows of I
    float *Ls = Yi;                              // [32][BS]  a slab of 32 Lam rows (over Yi and Ci)
    float *LB = Yi;                              // [32][H]   Lam B_j, after the slabs
    float *CBc = Ci + 32 * S;                    // [nT][32][33]
    float *Pc = CBc + nT * kTok * kTilePad;      // [32][33]  Dec (C_i . B_j)
    float *Py = Pc + kTok * kTilePad;            // [32][33]  Dec dt_j (dy_i . x_j)
    float *Gt = Py + kTok * kTilePad;            // [T]
    float *red = Gt + pr.T;                      // [8][32]
    float *dtj = red + 8 * kTok;                 // [32]
    float *diag = dtj + kTok;                    // [32]

    const int k = blockIdx.x / nT, jb = blockIdx.x % nT;
    const int g = blockIdx.y / nslice, sl = blockIdx.y % nslice;
    const int b = blockIdx.z;
    const int64_t t0 = (int64_t)k * pr.T;
    const int n = (int)(pr.T < pr.L - t0 ? pr.T : pr.L - t0);
    const int j0 = jb * kTok;
    if (j0 >= n) return;
    const int h_lo = g * (int)pr.hpg + sl * hps;
    const int h_hi = min(h_lo + hps, (g + 1) * (int)pr.hpg);
    const int nvT = (n + kTok - 1) / kTok;
    const int rows_j = min(kTok, n - j0);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int r = tid >> 3, c = tid & 7;
    const int64_t xs = pr.nh * pr.H, bs = pr.G * pr.S;
    const Tio *Brow = Bm + (((int64_t)b * pr.L + t0) * pr.G + g) * pr.S;   // token 0 of the chunk
    const Tio *Crow = Cm + (((int64_t)b * pr.L + t0) * pr.G + g) * pr.S;

    RowTile<Tio, S> tb, tc;
    RowTile<Tio, H> ty, tx;
    tb.load(Brow + (int64_t)j0 * bs, bs, rows_j);
    tb.store(Bj, BS);
    // C_i . B_j for every tile I >= J, shared by the heads of the block
    for (int ib = jb; ib < nvT; ++ib) {
        tc.load(Crow + (int64_t)ib * kTok * bs, bs, min(kTok, n - ib * kTok));
        __syncthreads();
        tc.store(Ci, S);
        __syncthreads();
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        dots4<S>(acc, Ci + warp * S, S, Bj + lane * BS);
        float *cb = CBc + (ib - jb) * kTok * kTilePad;
#pragma unroll
        for (int m = 0; m < 4; ++m) cb[(warp + 8 * m) * kTilePad + lane] = acc[m];
    }

    float accB[SV];
#pragma unroll
    for (int q = 0; q < SV; ++q) accB[q] = 0.f;

    for (int h = h_lo; h < h_hi; ++h) {
        const int64_t bh = (int64_t)b * pr.nh + h;
        const Tio *xh = x + (((int64_t)b * pr.L + t0) * pr.nh + h) * pr.H;   // token 0 of the chunk
        const Tio *dyh = dy + (((int64_t)b * pr.L + t0) * pr.nh + h) * pr.H;
        tx.load(xh + (int64_t)j0 * xs, xs, rows_j);
        ty.load(dyh + (int64_t)j0 * xs, xs, rows_j);
        tc.load(Crow + (int64_t)j0 * bs, bs, rows_j);
        __syncthreads();                          // the previous head's readers are done
        tx.store(Xj, XS);
        ty.store(Yi, H);
        tc.store(Ci, S);
        for (int t = tid; t < n; t += blockDim.x) Gt[t] = G[bh * pr.L + t0 + t];
        if (tid < kTok) dtj[tid] = tid < rows_j ? to_f32(dt[((int64_t)b * pr.L + t0 + j0 + tid) * pr.nh + h]) : 0.f;
        __syncthreads();
        float accV[HV];
#pragma unroll
        for (int q = 0; q < HV; ++q) accV[q] = 0.f;
        float colp = 0.f;
        for (int ib = jb; ib < nvT; ++ib) {
            const int i0 = ib * kTok;
            const bool more = ib + 1 < nvT;
            if (more) {
                const int nxt = min(kTok, n - i0 - kTok);
                ty.load(dyh + (int64_t)(i0 + kTok) * xs, xs, nxt);
                tc.load(Crow + (int64_t)(i0 + kTok) * bs, bs, nxt);
            }
            float yx[4] = {0.f, 0.f, 0.f, 0.f};
            dots4<H>(yx, Yi + warp * H, H, Xj + lane * XS);
            const float *cb = CBc + (ib - jb) * kTok * kTilePad;
            const int j = j0 + lane;
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const int ii = warp + 8 * m, i = i0 + ii;
                const bool on = i < n && j < n && i >= j;            // select, never multiply, the mask
                const float dec = on ? exp2f(Gt[on ? i : 0] - Gt[on ? j : 0]) : 0.f;
                const float pc = dec * cb[ii * kTilePad + lane];
                Pc[ii * kTilePad + lane] = pc;
                Py[ii * kTilePad + lane] = dec * yx[m] * dtj[lane];
                colp = fmaf(pc, yx[m], colp);
                if (ib == jb && ii == lane) diag[lane] = yx[m];
            }
            __syncthreads();
#pragma unroll 2
            for (int ii = 0; ii < kTok; ++ii) {
                const float pcv = Pc[ii * kTilePad + r], pyv = Py[ii * kTilePad + r];
#pragma unroll
                for (int q = 0; q < HV / 4; ++q) {
                    const float4 v = ld4(Yi + ii * H + 4 * (c + 8 * q));
                    accV[4 * q] = fmaf(pcv, v.x, accV[4 * q]);
                    accV[4 * q + 1] = fmaf(pcv, v.y, accV[4 * q + 1]);
                    accV[4 * q + 2] = fmaf(pcv, v.z, accV[4 * q + 2]);
                    accV[4 * q + 3] = fmaf(pcv, v.w, accV[4 * q + 3]);
                }
#pragma unroll
                for (int q = 0; q < SV / 4; ++q) {
                    const float4 v = ld4(Ci + ii * S + 4 * (c + 8 * q));
                    accB[4 * q] = fmaf(pyv, v.x, accB[4 * q]);
                    accB[4 * q + 1] = fmaf(pyv, v.y, accB[4 * q + 1]);
                    accB[4 * q + 2] = fmaf(pyv, v.z, accB[4 * q + 2]);
                    accB[4 * q + 3] = fmaf(pyv, v.w, accB[4 * q + 3]);
                }
            }
            __syncthreads();
            if (more) {
                ty.store(Yi, H);
                tc.store(Ci, S);
                __syncthreads();
            }
        }
        // Lam, 32 rows p at a time: Lam B_j (thread rows p = c + 8k' of the slab) and
        // Lam^T x_j (thread columns s = 4 (c + 8q) + e)
        const float *Lk = lam + ((bh * pr.nc + k) * pr.H) * pr.S;
        float accLB[HV], accLX[SV];
#pragma unroll
        for (int q = 0; q < SV; ++q) accLX[q] = 0.f;
#pragma unroll
        for (int p0 = 0; p0 < H; p0 += 32) {
            __syncthreads();                      // the previous slab (or tile) is no longer read
#pragma unroll
            for (int i = 0; i < S / 32; ++i) {    // 32 x S floats, 16-byte vectors
                const int v = i * 256 + tid, row = v / (S / 4), col = v % (S / 4);
                *reinterpret_cast<float4 *>(Ls + row * BS + 4 * col) =
                    *reinterpret_cast<const float4 *>(Lk + (int64_t)(p0 + row) * S + 4 * col);
            }
            __syncthreads();
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const float *lrow = Ls + (c + 8 * kk) * BS, *brow = Bj + r * BS;
                float acc = 0.f;
#pragma unroll 8
                for (int s4 = 0; s4 < S; s4 += 4) {
                    const float4 u = ld4(brow + s4), w = ld4(lrow + s4);
                    acc = fmaf(u.x, w.x, fmaf(u.y, w.y, fmaf(u.z, w.z, fmaf(u.w, w.w, acc))));
                }
                accLB[p0 / 8 + kk] = acc;
            }
#pragma unroll 4
            for (int pp = 0; pp < 32; ++pp) {
                const float xv = Xj[r * XS + p0 + pp];
#pragma unroll
                for (int q = 0; q < SV / 4; ++q) {
                    const float4 v = ld4(Ls + pp * BS + 4 * (c + 8 * q));
                    accLX[4 * q] = fmaf(xv, v.x, accLX[4 * q]);
                    accLX[4 * q + 1] = fmaf(xv, v.y, accLX[4 * q + 1]);
                    accLX[4 * q + 2] = fmaf(xv, v.z, accLX[4 * q + 2]);
                    accLX[4 * q + 3] = fmaf(xv, v.w, accLX[4 * q + 3]);
                }
            }
        }
        __syncthreads();                          // the last slab is no longer read
#pragma unroll
        for (int p0 = 0; p0 < H; p0 += 32)
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) LB[r * H + p0 + c + 8 * kk] = accLB[p0 / 8 + kk];
        red[warp * kTok + lane] = colp;
        __syncthreads();
        // outputs of row j = j0 + r
        const int j = j0 + r;
        const bool valid = r < rows_j;
        const float el = exp2f(Gt[n - 1] - Gt[valid ? j : 0]);
        const float dtv = dtj[r];
        const float dh = D[h];
        const Tio *dyj = dyh + (int64_t)(valid ? j : 0) * xs;
        Tio *dxj = dx + (((int64_t)b * pr.L + t0 + (valid ? j : 0)) * pr.nh + h) * pr.H;
        float qpart = 0.f, npart = 0.f;
#pragma unroll
        for (int q = 0; q < HV / 4; ++q) {
            const int p = 4 * (c + 8 * q);
            const float4 lb = ld4(LB + r * H + p), xv = ld4(Xj + r * XS + p);
            const float lbv[4] = {lb.x, lb.y, lb.z, lb.w}, xvv[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float v = fmaf(el, lbv[e], accV[4 * q + e]);
                qpart = fmaf(xvv[e], v, qpart);
                npart = fmaf(xvv[e], lbv[e], npart);
                if (valid) dxj[p + e] = from_f32<Tio>(fmaf(dtv, v, dh * to_f32(dyj[p + e])));
            }
        }
        qpart = sum8(qpart);
        npart = sum8(npart);
#pragma unroll
        for (int q = 0; q < SV; ++q) accB[q] = fmaf(dtv * el, accLX[q], accB[q]);
        if (c == 0 && valid) {
            float cm = 0.f;
            for (int w2 = 0; w2 < 8; ++w2) cm += red[w2 * kTok + r];
            const int64_t o = bh * pr.L + t0 + j;
            Qd[o] = qpart;
            Nd[o] = el * dtv * npart;
            Cmd[o] = dtv * cm;
            Dd[o] = diag[r];
        }
    }
    if (r < rows_j) {
        float *dst = dBp + ((((int64_t)sl * pr.B + b) * pr.L + t0 + j0 + r) * pr.G + g) * pr.S;
#pragma unroll
        for (int q = 0; q < SV / 4; ++q)
            *reinterpret_cast<float4 *>(dst + 4 * (c + 8 * q)) =
                make_float4(accB[4 * q], accB[4 * q + 1], accB[4 * q + 2], accB[4 * q + 3]);
    }
}

template <typename Tio, int H, int S>
__global__ void __launch_bounds__(256)
k_bwd_rows_fast(const Tio *__restrict__ x, const Tio *__restrict__ dt, const Tio *__restrict__ Bm,
                const Tio *__restrict__ Cm, const Tio *__restrict__ dy, const float *__restrict__ G,
                const float *__restrict__ h_start, float *__restrict__ Rw, float *__restrict__ dCp,
                Problem pr, int nT, int nslice, int hps)
{
    using Cfg = FastCfg<Tio, H, S>;
    constexpr int BS = Cfg::BS, XS = Cfg::XS, SV = Cfg::SV;
    extern __shared__ float4 smv[];
    float *Ci = reinterpret_cast<float *>(smv);  // [32][S]   C rows of I
    float *Yi = Ci + 32 * S;                     // [32][H]   dy rows of I (current head)
    float *Bj = Yi + 32 * H;                     // [32][BS]  B rows of J
    float *Xj = Bj + 32 * BS;                    // [32][XS]  x rows of J (current head)
    float *Hs = Bj;                              // [32][S]   a slab of 32 rows of h_in (over Bj and Xj)
    float *CBc = Xj + 32 * XS;                   // [nT][32][33]
    float *Pd = CBc + nT * kTok * kTilePad;      // [32][33]  Dec dt_j (dy_i . x_j)
    float *Gt = Pd + kTok * kTilePad;            // [T]
    float *dtj = Gt + pr.T;                      // [32]
    float *rowM = dtj + kTok;                    // [32]

    const int k = blockIdx.x / nT, ib = blockIdx.x % nT;
    const int g = blockIdx.y / nslice, sl = blockIdx.y % nslice;
    const int b = blockIdx.z;
    const int64_t t0 = (int64_t)k * pr.T;
    const int n = (int)(pr.T < pr.L - t0 ? pr.T : pr.L - t0);
    const int i0 = ib * kTok;
    if (i0 >= n) return;
    const int h_lo = g * (int)pr.hpg + sl * hps;
    const int h_hi = min(h_lo + hps, (g + 1) * (int)pr.hpg);
    const int rows_i = min(kTok, n - i0);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int r = tid >> 3, c = tid & 7;
    const int64_t xs = pr.nh * pr.H, bs = pr.G * pr.S;
    const Tio *Brow = Bm + (((int64_t)b * pr.L + t0) * pr.G + g) * pr.S;
    const Tio *Crow = Cm + (((int64_t)b * pr.L + t0) * pr.G + g) * pr.S;

    RowTile<Tio, S> tb, tc;
    RowTile<Tio, H> ty, tx;
    tc.load(Crow + (int64_t)i0 * bs, bs, rows_i);
    tc.store(Ci, S);
    for (int jb = 0; jb <= ib; ++jb) {
        tb.load(Brow + (int64_t)jb * kTok * bs, bs, min(kTok, n - jb * kTok));
        __syncthreads();
        tb.store(Bj, BS);
        __syncthreads();
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        dots4<S>(acc, Ci + warp * S, S, Bj + lane * BS);
        float *cb = CBc + jb * kTok * kTilePad;
#pragma unroll
        for (int m = 0; m < 4; ++m) cb[(warp + 8 * m) * kTilePad + lane] = acc[m];
    }

    float accC[SV];
#pragma unroll
    for (int q = 0; q < SV; ++q) accC[q] = 0.f;

    for (int h = h_lo; h < h_hi; ++h) {
        const int64_t bh = (int64_t)b * pr.nh + h;
        const Tio *xh = x + (((int64_t)b * pr.L + t0) * pr.nh + h) * pr.H;
        const Tio *dyh = dy + (((int64_t)b * pr.L + t0) * pr.nh + h) * pr.H;
        ty.load(dyh + (int64_t)i0 * xs, xs, rows_i);
        tx.load(xh, xs, min(kTok, n));
        tb.load(Brow, bs, min(kTok, n));
        __syncthreads();                          // the previous head's readers are done
        ty.store(Yi, H);
        tx.store(Xj, XS);
        tb.store(Bj, BS);
        for (int t = tid; t < n; t += blockDim.x) Gt[t] = G[bh * pr.L + t0 + t];
        if (tid < kTok) dtj[tid] = tid < min(kTok, n) ? to_f32(dt[((int64_t)b * pr.L + t0 + tid) * pr.nh + h]) : 0.f;
        __syncthreads();
        float rowp[4] = {0.f, 0.f, 0.f, 0.f};
        for (int jb = 0; jb <= ib; ++jb) {
            const int jj0 = jb * kTok;
            const bool more = jb < ib;
            if (more) {
                const int nxt = min(kTok, n - jj0 - kTok);
                tx.load(xh + (int64_t)(jj0 + kTok) * xs, xs, nxt);
                tb.load(Brow + (int64_t)(jj0 + kTok) * bs, bs, nxt);
            }
            float yx[4] = {0.f, 0.f, 0.f, 0.f};
            dots4<H>(yx, Yi + warp * H, H, Xj + lane * XS);
            const float *cb = CBc + jb * kTok * kTilePad;
            const int j = jj0 + lane;
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const int ii = warp + 8 * m, i = i0 + ii;
                const bool on = i < n && j < n && i >= j;
                const float dec = on ? exp2f(Gt[on ? i : 0] - Gt[on ? j : 0]) : 0.f;
                const float pd = dec * dtj[lane] * yx[m];
                Pd[ii * kTilePad + lane] = pd;
                rowp[m] = fmaf(pd, cb[ii * kTilePad + lane], rowp[m]);
            }
            __syncthreads();
#pragma unroll 2
            for (int jj = 0; jj < kTok; ++jj) {
                const float pv = Pd[r * kTilePad + jj];
#pragma unroll
                for (int q = 0; q < SV / 4; ++q) {
                    const float4 v = ld4(Bj + jj * BS + 4 * (c + 8 * q));
                    accC[4 * q] = fmaf(pv, v.x, accC[4 * q]);
                    accC[4 * q + 1] = fmaf(pv, v.y, accC[4 * q + 1]);
                    accC[4 * q + 2] = fmaf(pv, v.z, accC[4 * q + 2]);
                    accC[4 * q + 3] = fmaf(pv, v.w, accC[4 * q + 3]);
                }
            }
            __syncthreads();
            if (more) {
                tx.store(Xj, XS);
                tb.store(Bj, BS);
                if (tid < kTok) {
                    const int jn = jj0 + kTok + tid;
                    dtj[tid] = jn < n ? to_f32(dt[((int64_t)b * pr.L + t0 + jn) * pr.nh + h]) : 0.f;
                }
                __syncthreads();
            }
        }
        // carried term: w_i = h_in^T dy_i, 32 rows of h_in at a time
        const float *Hk = h_start + ((bh * pr.nc + k) * pr.H) * pr.S;
        float accW[SV];
#pragma unroll
        for (int q = 0; q < SV; ++q) accW[q] = 0.f;
#pragma unroll
        for (int p0 = 0; p0 < H; p0 += 32) {
            if (p0 > 0) __syncthreads();          // the previous slab is no longer read
#pragma unroll
            for (int i = 0; i < S / 32; ++i) {
                const int v = i * 256 + tid, row = v / (S / 4), col = v % (S / 4);
                *reinterpret_cast<float4 *>(Hs + row * S + 4 * col) =
                    *reinterpret_cast<const float4 *>(Hk + (int64_t)(p0 + row) * S + 4 * col);
            }
            __syncthreads();
#pragma unroll 4
            for (int pp = 0; pp < 32; ++pp) {
                const float yv = Yi[r * H + p0 + pp];
#pragma unroll
                for (int q = 0; q < SV / 4; ++q) {
                    const float4 v = ld4(Hs + pp * S + 4 * (c + 8 * q));
                    accW[4 * q] = fmaf(yv, v.x, accW[4 * q]);
                    accW[4 * q + 1] = fmaf(yv, v.y, accW[4 * q + 1]);
                    accW[4 * q + 2] = fmaf(yv, v.z, accW[4 * q + 2]);
                    accW[4 * q + 3] = fmaf(yv, v.w, accW[4 * q + 3]);
                }
            }
        }
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            const float v = sum32(rowp[m]);
            if (lane == 0) rowM[warp + 8 * m] = v;
        }
        __syncthreads();
        const bool valid = r < rows_i;
        const float eg = exp2f(Gt[valid ? i0 + r : 0]);
        float ypart = 0.f;
#pragma unroll
        for (int q = 0; q < SV / 4; ++q) {
            const float4 cv = ld4(Ci + r * S + 4 * (c + 8 * q));
            const float cvv[4] = {cv.x, cv.y, cv.z, cv.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                ypart = fmaf(accW[4 * q + e], cvv[e], ypart);
                accC[4 * q + e] = fmaf(eg, accW[4 * q + e], accC[4 * q + e]);
            }
        }
        ypart = sum8(ypart);
        if (c == 0 && valid) Rw[bh * pr.L + t0 + i0 + r] = fmaf(eg, ypart, rowM[r]);
    }
    if (r < rows_i) {
        float *dst = dCp + ((((int64_t)sl * pr.B + b) * pr.L + t0 + i0 + r) * pr.G + g) * pr.S;
#pragma unroll
        for (int q = 0; q < SV / 4; ++q)
            *reinterpret_cast<float4 *>(dst + 4 * (c + 8 * q)) =
                make_float4(accC[4 * q], accC[4 * q + 1], accC[4 * q + 2], accC[4 * q + 3]);
    }
}

// ---------------------------------------------------------------------------
// Per (chunk, head, batch): dG, its reverse cumsum da, ddt and dt da (for dA).
// Block of 256 threads, one token each (chunk <= 256).
// ---------------------------------------------------------------------------
template <typename Tio>
__global__ void __launch_bounds__(256)
k_bwd_finalize(const Tio *__restrict__ dt, const float *__restrict__ A, const float *__restrict__ G,
               const float *__restrict__ lam, const float *__restrict__ h_start, const float *__restrict__ Qd,
               const float *__restrict__ Nd, const float *__restrict__ Cmd, const float *__restrict__ Rw,
               Tio *__restrict__ ddt, float *__restrict__ Ad, Problem pr)
{
    __shared__ float wsum[8];
    __shared__ float bcast[2];
    __shared__ float dgs[256];                                // dG of each token of the chunk
    const int k = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t bh = (int64_t)b * pr.nh + h;
    const int64_t t0 = (int64_t)k * pr.T;
    const int n = (int)(pr.T < pr.L - t0 ? pr.T : pr.L - t0);
    const int64_t HS = pr.H * pr.S;
    // <Lam_k, h_in,k>
    const float *Lk = lam + (bh * pr.nc + k) * HS, *Hk = h_start + (bh * pr.nc + k) * HS;
    float e = 0.f;
    for (int64_t i = tid; i < HS; i += blockDim.x) e = fmaf(Lk[i], Hk[i], e);
    e = sum32(e);
    if (lane == 0) wsum[warp] = e;
    const int64_t o = bh * pr.L + t0 + tid;
    const bool on = tid < n;
    const float nv = on ? Nd[o] : 0.f;
    __syncthreads();
    if (tid == 0) {
        float s = 0.f;
        for (int w = 0; w < 8; ++w) s += wsum[w];
        bcast[0] = s;
    }
    __syncthreads();
    const float E = bcast[0];
    float ns = sum32(nv);
    __syncthreads();
    if (lane == 0) wsum[warp] = ns;
    __syncthreads();
    if (tid == 0) {
        float s = 0.f;
        for (int w = 0; w < 8; ++w) s += wsum[w];
        bcast[1] = s;
    }
    __syncthreads();
    const float glast = G[bh * pr.L + t0 + n - 1];
    float dg = on ? Rw[o] - Cmd[o] - nv : 0.f;
    if (tid == n - 1) dg += exp2f(glast) * E + bcast[1];
    // da_t = sum_{i >= t} dG_i: inclusive scan over the reversed token order
    const int rt = n - 1 - tid;                              // token whose dG this thread scans
    dgs[tid] = dg;
    __syncthreads();
    float v = tid < n ? dgs[rt] : 0.f;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const float u = __shfl_up_sync(0xffffffffu, v, off);
        if (lane >= off) v += u;
    }
    __syncthreads();
    if (lane == 31) wsum[warp] = v;
    __syncthreads();
    float pre = 0.f;
    for (int w = 0; w < warp; ++w) pre += wsum[w];
    v += pre;                                                 // da of token rt
    if (tid < n) {
        const int64_t ot = bh * pr.L + t0 + rt;
        const float dtv = to_f32(dt[((int64_t)b * pr.L + t0 + rt) * pr.nh + h]);
        ddt[((int64_t)b * pr.L + t0 + rt) * pr.nh + h] = from_f32<Tio>(fmaf(A[h], v, Qd[ot]));
        Ad[ot] = dtv * v;
    }
}

// dA[h] = sum_{b, t} dt da, dD[h] = sum_{b, t} dy.x: one block per head, fixed order.
__global__ void __launch_bounds__(256)
k_bwd_reduce_heads(const float *__restrict__ Ad, const float *__restrict__ Dd, float *__restrict__ dA,
                   float *__restrict__ dD, Problem pr)
{
    __shared__ float sa[8], sd[8];
    const int h = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    float a = 0.f, d = 0.f;
    for (int64_t b = 0; b < pr.B; ++b) {
        const int64_t base = (b * pr.nh + h) * pr.L;
        for (int64_t t = tid; t < pr.L; t += blockDim.x) {
            a += Ad[base + t];
            d += Dd[base + t];
        }
    }
    a = sum32(a);
    d = sum32(d);
    if (lane == 0) { sa[warp] = a; sd[warp] = d; }
    __syncthreads();
    if (tid == 0) {
        float ta = 0.f, td = 0.f;
        for (int w = 0; w < 8; ++w) { ta += sa[w]; td += sd[w]; }
        dA[h] = ta;
        dD[h] = td;
    }
}

// dB, dC: the slices' partial sums added in slice order, cast to the gradient dtype.
template <typename Tio>
__global__ void __launch_bounds__(256)
k_bwd_combine(const float *__restrict__ dBp, const float *__restrict__ dCp, Tio *__restrict__ dB,
              Tio *__restrict__ dC, int64_t count, int nslice)
{
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < count; e += (int64_t)gridDim.x * blockDim.x) {
        float sb = 0.f, sc = 0.f;
        for (int s = 0; s < nslice; ++s) {
            sb += dBp[s * count + e];
            sc += dCp[s * count + e];
        }
        dB[e] = from_f32<Tio>(sb);
        dC[e] = from_f32<Tio>(sc);
    }
}

size_t cols_smem(const Problem &pr, int nT)
{
    const size_t SP = pr.S + 1, HP = pr.H + 1;
    const size_t stage = std::max<size_t>((size_t)pr.H * 33, 8 * (size_t)pr.S);
    return sizeof(float) * (2 * kTok * SP + 2 * kTok * HP + (size_t)nT * kTok * kTilePad + 2 * kTok * kTilePad +
                            (size_t)pr.T + 8 * kTok + 2 * kTok + stage);
}

size_t rows_smem(const Problem &pr, int nT)
{
    const size_t SP = pr.S + 1, HP = pr.H + 1;
    return sizeof(float) * (2 * kTok * SP + 2 * kTok * HP + (size_t)nT * kTok * kTilePad + kTok * kTilePad +
                            (size_t)pr.T + 2 * kTok + 8 * (size_t)pr.S);
}

bool bwd_fast_shape(const Problem &pr) { return (pr.H == 64 || pr.H == 128) && (pr.S == 128 || pr.S == 256); }

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

template <typename Tio, int H, int S>
cudaError_t launch_sides_fast(const Problem &pr, const BwdArgs &a, const BwdWork &w, int nT, cudaStream_t st)
{
    using Cfg = FastCfg<Tio, H, S>;
    dim3 grid((unsigned)(pr.nc * nT), (unsigned)(pr.G * w.nslice), (unsigned)pr.B);
    const size_t sc = sizeof(float) * Cfg::cols_floats((int)pr.T, nT), sr = sizeof(float) * Cfg::rows_floats((int)pr.T, nT);
    auto kc = k_bwd_cols_fast<Tio, H, S>;
    auto kr = k_bwd_rows_fast<Tio, H, S>;
    cudaError_t e;
    if ((e = cudaFuncSetAttribute(kc, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sc)) != cudaSuccess) return e;
    if ((e = cudaFuncSetAttribute(kr, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sr)) != cudaSuccess) return e;
    kc<<<grid, 256, sc, st>>>((const Tio *)a.x, (const Tio *)a.dt, (const Tio *)a.Bm, (const Tio *)a.Cm,
                              (const Tio *)a.dy, a.D, w.G, w.lam, (Tio *)a.dx, w.Qd, w.Nd, w.Cmd, w.Dd, w.dBp, pr, nT,
                              w.nslice, w.hps);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    kr<<<grid, 256, sr, st>>>((const Tio *)a.x, (const Tio *)a.dt, (const Tio *)a.Bm, (const Tio *)a.Cm,
                              (const Tio *)a.dy, w.G, w.h_start, w.Rw, w.dCp, pr, nT, w.nslice, w.hps);
    return cudaGetLastError();
}

template <typename Tio, int HQ, int SQ>
cudaError_t launch_bwd_t(const Problem &pr, const BwdArgs &a, const BwdWork &w, cudaStream_t st)
{
    cudaError_t e;
    const int nT = (int)((pr.T + kTok - 1) / kTok);
    // forward recompute: G, the local chunk states (in w.lam) and the entering states
    if ((e = launch_chunk_cumsum(pr, a.dt, a.A, w.G, nullptr, 0, 0, st)) != cudaSuccess) return e;
    const int nc = (int)pr.nc;
    // the local chunk states on tensor cores where that kernel takes the shape (whole chunks, 16-byte rows)
    const bool tc_state = tc_supported(pr) && pr.L % pr.T == 0 && aligned16(a.x) && aligned16(a.dt) && aligned16(a.Bm);
    e = tc_state ? launch_chunk_state_tc(pr, SeqRange{0, pr.B * pr.nh}, a.x, a.dt, nullptr, a.Bm, w.G, w.lam, 1, nc, nc,
                                         nullptr, st)
                 : launch_chunk_state_simt(pr, a.x, a.dt, a.Bm, w.G, w.lam, st);
    if (e != cudaSuccess) return e;
    if ((e = launch_state_passing(pr, SeqRange{0, pr.B * pr.nh}, w.G, w.lam, a.h0, w.h_start, nullptr, 1, nc, nc,
                                  st)) != cudaSuccess)
        return e;
    // entering-state gradients, then backwards over chunks
    {
        const int ptiles = (int)((pr.H + 31) / 32), stiles = (int)((pr.S + 63) / 64);
        dim3 grid((unsigned)pr.nc, (unsigned)(pr.nh * ptiles * stiles), (unsigned)pr.B);
        if (bwd_fast_shape(pr) && pr.B * pr.nh <= 65535) {
            dim3 gf((unsigned)pr.nc, (unsigned)(pr.H / 64), (unsigned)(pr.B * pr.nh));
            if (pr.S == 128)
                k_bwd_dstate_fast<Tio, 128><<<gf, 256, 0, st>>>((const Tio *)a.dy, (const Tio *)a.Cm, w.G, w.lam, pr);
            else
                k_bwd_dstate_fast<Tio, 256><<<gf, 256, 0, st>>>((const Tio *)a.dy, (const Tio *)a.Cm, w.G, w.lam, pr);
        } else {
            k_bwd_dstate<Tio><<<grid, 256, 0, st>>>((const Tio *)a.dy, (const Tio *)a.Cm, w.G, w.lam, pr, ptiles, stiles);
        }
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        const int64_t seqs = pr.B * pr.nh;
        dim3 g2((unsigned)((pr.H * pr.S + 255) / 256), (unsigned)(seqs < 65535 ? seqs : 65535));
        k_bwd_state_passing<<<g2, 256, 0, st>>>(w.G, w.lam, a.dh_final, a.dh0, pr);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    // per-chunk column and row sides
    if (bwd_fast_shape(pr) && aligned16(a.x) && aligned16(a.dy) && aligned16(a.Bm) && aligned16(a.Cm)) {
        e = pr.H == 64 ? (pr.S == 128 ? launch_sides_fast<Tio, 64, 128>(pr, a, w, nT, st)
                                      : launch_sides_fast<Tio, 64, 256>(pr, a, w, nT, st))
                       : (pr.S == 128 ? launch_sides_fast<Tio, 128, 128>(pr, a, w, nT, st)
                                      : launch_sides_fast<Tio, 128, 256>(pr, a, w, nT, st));
        if (e != cudaSuccess) return e;
    } else {
        dim3 grid((unsigned)(pr.nc * nT), (unsigned)(pr.G * w.nslice), (unsigned)pr.B);
        const size_t sc = cols_smem(pr, nT), sr = rows_smem(pr, nT);
        auto kc = k_bwd_chunk_cols<Tio, HQ, SQ>;
        auto kr = k_bwd_chunk_rows<Tio, SQ>;
        if ((e = cudaFuncSetAttribute(kc, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sc)) != cudaSuccess) return e;
        if ((e = cudaFuncSetAttribute(kr, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sr)) != cudaSuccess) return e;
        kc<<<grid, 256, sc, st>>>((const Tio *)a.x, (const Tio *)a.dt, (const Tio *)a.Bm, (const Tio *)a.Cm,
                                  (const Tio *)a.dy, a.D, w.G, w.lam, (Tio *)a.dx, w.Qd, w.Nd, w.Cmd, w.Dd, w.dBp, pr,
                                  nT, w.nslice, w.hps);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        kr<<<grid, 256, sr, st>>>((const Tio *)a.x, (const Tio *)a.dt, (const Tio *)a.Bm, (const Tio *)a.Cm,
                                  (const Tio *)a.dy, w.G, w.h_start, w.Rw, w.dCp, pr, nT, w.nslice, w.hps);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    {
        dim3 grid((unsigned)pr.nc, (unsigned)pr.nh, (unsigned)pr.B);
        k_bwd_finalize<Tio><<<grid, 256, 0, st>>>((const Tio *)a.dt, a.A, w.G, w.lam, w.h_start, w.Qd, w.Nd, w.Cmd,
                                                  w.Rw, (Tio *)a.ddt, w.Ad, pr);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        k_bwd_reduce_heads<<<(unsigned)pr.nh, 256, 0, st>>>(w.Ad, w.Dd, a.dA, a.dD, pr);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        const int64_t count = pr.B * pr.L * pr.G * pr.S;
        const int64_t blocks = std::min<int64_t>((count + 255) / 256, 8192);
        k_bwd_combine<Tio><<<(unsigned)blocks, 256, 0, st>>>(w.dBp, w.dCp, (Tio *)a.dB, (Tio *)a.dC, count, w.nslice);
        return cudaGetLastError();
    }
}

}  // namespace

bool bwd_supported(const Problem &pr)
{
    return pr.in_dt == pr.out_dt && pr.H <= 128 && pr.S <= 256 && pr.T <= 256;
}

size_t bwd_workspace(const Problem &pr, void *base, BwdWork *w)
{
    constexpr size_t kAlign = 256;
    auto up = [](size_t v) { return (v + kAlign - 1) / kAlign * kAlign; };
    const int64_t nT = (pr.T + kTok - 1) / kTok;
    const int64_t tiles = pr.B * pr.G * pr.nc * nT;
    // slices of a group's heads: enough blocks to fill the GPU when there are few tiles
    int64_t nslice = tiles > 0 ? (1024 + tiles - 1) / tiles : 1;
    nslice = std::max<int64_t>(1, std::min<int64_t>(nslice, pr.hpg));
    const int64_t hps = (pr.hpg + nslice - 1) / nslice;
    nslice = (pr.hpg + hps - 1) / hps;                         // every slice holds at least one head
    const size_t tok = up(sizeof(float) * (size_t)(pr.B * pr.nh * pr.L));
    const size_t states = up(sizeof(float) * (size_t)(pr.B * pr.nh * pr.nc * pr.H * pr.S));
    const size_t part = up(sizeof(float) * (size_t)(nslice * pr.B * pr.L * pr.G * pr.S));
    char *p = (char *)base;
    size_t off = 0;
    auto take = [&](size_t n) { float *q = (float *)(p ? p + off : nullptr); off += n; return q; };
    BwdWork v;
    v.G = take(tok);
    v.h_start = take(states);
    v.lam = take(states);
    v.Qd = take(tok);
    v.Nd = take(tok);
    v.Cmd = take(tok);
    v.Dd = take(tok);
    v.Rw = take(tok);
    v.Ad = take(tok);
    v.dBp = take(part);
    v.dCp = take(part);
    v.nslice = (int)nslice;
    v.hps = (int)hps;
    if (w) *w = v;
    return off;
}

cudaError_t launch_bwd(const Problem &pr, const BwdArgs &a, const BwdWork &w, cudaStream_t st)
{
    const bool small = pr.H <= 64 && pr.S <= 128;
    if (pr.in_dt == SSD_BF16)
        return small ? launch_bwd_t<__nv_bfloat16, 8, 16>(pr, a, w, st) : launch_bwd_t<__nv_bfloat16, 16, 32>(pr, a, w, st);
    return small ? launch_bwd_t<float, 8, 16>(pr, a, w, st) : launch_bwd_t<float, 16, 32>(pr, a, w, st);
}

}  // namespace ssd
