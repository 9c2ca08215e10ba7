// ssd_simt.cu -- CUDA-core kernels for the four SSD stages and the decode step.
//
// These kernels handle every supported shape (any L, any chunk up to 1024,
// S up to 256, any H) in float32 arithmetic on the CUDA cores.  The
// tensor-core kernels in ssd_tc.cu take over the chunk_state and chunk_scan
// stages for the shapes they are built for.
//
// Method: NVIDIA developer blog "Accelerating Mamba-2 with High-Performance
// Forward Pass Kernels in NVIDIA CUDA Tile", sections "Mamba-2 architecture"
// and "Kernel 1" .. "Kernel 3".
#include <string.h>

#include <type_traits>

#include "ssd_common.cuh"

namespace ssd {
namespace {

// ---------------------------------------------------------------------------
// Stage 1 -- chunk_cumsum (blog section "Kernel 1: cumulative sum").
// G[b][h][t] = log2(e) * sum_{s in chunk(t), s <= t} A[h] dt[b][s][h].
// One block per (chunk, 32-head tile, batch).  Lane = head, so every dt row of 32
// heads is one coalesced load.  Warp w takes runs of 32 consecutive tokens: each lane
// loads its run (independent loads), forms the running sum in registers, and records
// the run total; after one barrier, one thread per (run, head) sums the totals of the
// runs before it into an offset table, and after a second barrier G is written
// transposed, [head][token], coalesced, with the offset of its run added on the way out.
// ---------------------------------------------------------------------------
template <typename Tin>
__global__ void __launch_bounds__(256)
k_chunk_cumsum(const Tin *__restrict__ dt, const float *__restrict__ A, float *__restrict__ G,
               float *__restrict__ dtT, int64_t dtT_lo, int64_t dtT_hi, int64_t L, int nh, int T,
               unsigned *count, __nv_bfloat16 *__restrict__ dt16)
{
    extern __shared__ float tile[];   // [T][33] in-run cumsum, then (dtT only) [T][33] dt
    __shared__ float run_sum[32][33]; // [run][head] run totals (T <= 1024: at most 32 runs)
    __shared__ float run_off[32][33]; // [run][head] sum of the totals of the runs before
    pdl_trigger();                    // the next kernel may launch; it waits for this one's G
    const int k = blockIdx.x, hbase = blockIdx.y * 32, b = blockIdx.z;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t t0 = (int64_t)k * T;
    const int n = (int)((int64_t)T < L - t0 ? (int64_t)T : L - t0);
    const int runs = (n + 31) / 32;
    const int h = hbase + lane;
    // lanes past the last head load head 0 (a valid address) with a = 0; their rows are never written out
    const float a = h < nh ? __ldg(A + h) : 0.f;
    for (int r = warp; r < runs; r += 8) {
        float v[32];
        const Tin *src = dt + ((int64_t)b * L + t0 + 32 * r) * nh + (h < nh ? h : 0);
        float *trow = tile + (32 * r) * 33 + lane;
        float acc = 0.f;
        if (32 * r + 32 <= n) {                // whole run inside the chunk: no per-token checks
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = to_f32(__ldg(src + (int64_t)i * nh));
            if (dt16 && h < nh) {
                __nv_bfloat16 *d16 = dt16 + ((int64_t)b * L + t0 + 32 * r) * nh + h;
#pragma unroll
                for (int i = 0; i < 32; ++i) d16[(int64_t)i * nh] = __float2bfloat16_rn(v[i]);
            }
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                acc += a * v[i];
                trow[i * 33] = acc;
            }
            if (dtT) {
#pragma unroll
                for (int i = 0; i < 32; ++i) trow[(T + i) * 33] = v[i];
            }
        } else {                               // the chunk ends inside this run
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = (32 * r + i < n) ? to_f32(__ldg(src + (int64_t)i * nh)) : 0.f;
            if (dt16 && h < nh) {
                __nv_bfloat16 *d16 = dt16 + ((int64_t)b * L + t0 + 32 * r) * nh + h;
                for (int i = 0; i < 32 && 32 * r + i < n; ++i) d16[(int64_t)i * nh] = __float2bfloat16_rn(v[i]);
            }
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                acc += a * v[i];
                if (32 * r + i < n) {
                    trow[i * 33] = acc;
                    if (dtT) trow[(T + i) * 33] = v[i];
                }
            }
        }
        run_sum[r][lane] = acc;
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < 32 * runs; idx += blockDim.x) {
        const int r = idx >> 5, j = idx & 31;
        float off = 0.f;
        for (int rr = 0; rr < r; ++rr) off += run_sum[rr][j];
        run_off[r][j] = off;
    }
    __syncthreads();
    for (int j = warp; j < 32; j += 8) {
        const int hh = hbase + j;
        if (hh >= nh) continue;
        float *dst = G + ((int64_t)b * nh + hh) * L + t0;
        for (int t = lane; t < n; t += 32) dst[t] = (tile[t * 33 + j] + run_off[t >> 5][j]) * kLog2e;
        const int64_t bh = (int64_t)b * nh + hh;
        if (dtT && bh >= dtT_lo && bh < dtT_hi) {
            float *dd = dtT + bh * L + t0;
            for (int t = lane; t < n; t += 32) dd[t] = tile[(T + t) * 33 + j];
        }
    }
    if (count) {
        // this CTA's G is written: make it visible device-wide, then count the CTA
        __threadfence();
        __syncthreads();
        if (threadIdx.x == 0) atomicAdd(count, 1u);
    }
}

// ---------------------------------------------------------------------------
// Stage 2 -- chunk_state on CUDA cores (blog section "Kernel 2: fwd_pass_state",
// the contraction x_tile^T (b dt exp2(d_last - d))).
// s_local[b][h][k][p][s] = sum_t w_t x[t][p] B[t][s],  w_t = dt_t exp2(G_last - G_t).
// One block per (chunk, head x 32-row p tile x 64-column s tile, batch).
// ---------------------------------------------------------------------------
template <typename Tin>
__global__ void __launch_bounds__(256)
k_chunk_state_simt(const Tin *__restrict__ x, const Tin *__restrict__ dt,
                   const Tin *__restrict__ Bm, const float *__restrict__ G,
                   float *__restrict__ s_local, Problem pr, int ptiles, int stiles)
{
    __shared__ float xw[32][33];   // [token][p]  w_t x[t][p]
    __shared__ float bt[32][64];   // [token][s]
    __shared__ float w[32];
    const int k = blockIdx.x, b = blockIdx.z;
    const int h = blockIdx.y / (ptiles * stiles);
    const int tile = blockIdx.y % (ptiles * stiles);
    const int p0 = (tile / stiles) * 32, s0 = (tile % stiles) * 64;
    const int g = (int)(h / pr.hpg);
    const int64_t t0 = (int64_t)k * pr.T;
    const int n = (int)(pr.T < pr.L - t0 ? pr.T : pr.L - t0);
    const float *Gh = G + ((int64_t)b * pr.nh + h) * pr.L;
    const float glast = Gh[t0 + n - 1];
    const int tx = threadIdx.x & 63, ty = threadIdx.x >> 6;   // s column, p group of 8
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.f;
    for (int seg = 0; seg < n; seg += 32) {
        if (threadIdx.x < 32) {
            const int t = seg + threadIdx.x;
            float v = 0.f;
            if (t < n) v = to_f32(dt[((int64_t)b * pr.L + t0 + t) * pr.nh + h]) * exp2f(glast - Gh[t0 + t]);
            w[threadIdx.x] = v;
        }
        __syncthreads();
        for (int r = warp; r < 32; r += 8) {
            const int t = seg + r, p = p0 + lane;
            float v = 0.f;
            if (t < n && p < pr.H) v = w[r] * to_f32(x[(((int64_t)b * pr.L + t0 + t) * pr.nh + h) * pr.H + p]);
            xw[r][lane] = v;
            for (int c = lane; c < 64; c += 32) {
                const int s = s0 + c;
                float u = 0.f;
                if (t < n && s < pr.S) u = to_f32(Bm[(((int64_t)b * pr.L + t0 + t) * pr.G + g) * pr.S + s]);
                bt[r][c] = u;
            }
        }
        __syncthreads();
#pragma unroll 8
        for (int r = 0; r < 32; ++r) {
            const float bv = bt[r][tx];
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[i] = fmaf(xw[r][ty * 8 + i], bv, acc[i]);
        }
        __syncthreads();
    }
    const int s = s0 + tx;
    if (s < pr.S) {
        float *dst = s_local + ((((int64_t)b * pr.nh + h) * pr.nc + k) * pr.H) * pr.S;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int p = p0 + ty * 8 + i;
            if (p < pr.H) dst[(int64_t)p * pr.S + s] = acc[i];
        }
    }
}

// ---------------------------------------------------------------------------
// Stage 3 -- state_passing (blog section "Kernel 2: fwd_pass_state", the
// sequential loop over chunks), generalised to super-chunks of R chunks:
//   h_start[m] = h_m,  h_{m+1} = exp2(sum_{k in m} G_last,k) h_m + s_local[m],
// for m = 0 .. nsup-1 starting from h0 (NULL: zeros); s_local is read for m < nm
// only and h_final = h_nm is written when nm == nsup (and h_final is not NULL).
// With R = 1 this is the blog's per-chunk loop.  VEC consecutive state elements
// per thread (float4 when H*S allows), consecutive threads on consecutive
// elements: every step is a coalesced 128-bit stream.  Blocks of 1024 threads: the
// work is a few dependent load rounds per sequence, so a few large CTAs finish as
// soon as many small ones, and hold fewer SMs that the scan's CTAs could start on.
// ---------------------------------------------------------------------------
constexpr int kPassThreads = 1024;

template <int VEC>
__global__ void __launch_bounds__(kPassThreads)
k_state_passing(const float *__restrict__ G, const float *__restrict__ s_local,
                const float *__restrict__ h0, float *__restrict__ h_start,
                float *__restrict__ h_final, Problem pr, SeqRange seqs, int R, int nsup, int nm)
{
    using V = typename std::conditional<VEC == 4, float4, float>::type;
    constexpr int kBatch = 8;                     // states loaded together (independent loads)
    constexpr int kWin = 1024;                    // super-chunks whose decays are staged at once
    constexpr int kTile = kPassThreads;           // chunk-end G values loaded together (= block size)
    __shared__ float sdec[kWin];                  // exp2 of each super-chunk's total log2 decay
    __shared__ float sdl[kWin];                   // the total log2 decays, summed tile by tile
    __shared__ float sgl[kTile];                  // G at the end of each chunk of the tile
    pdl_trigger();
    pdl_wait();                                   // G and s_local come from the kernels before
    const int64_t HS = pr.H * pr.S;
    const int64_t e = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * VEC;
    const bool active = e < HS;
    // one sequence at a time (a grid row may serve several when there are more than 65535)
    for (int64_t rel = blockIdx.y; rel < seqs.n; rel += gridDim.y) {
        const int64_t bh = seqs.lo + rel;
        const float *Gh = G + bh * pr.L;
        float st[VEC];
#pragma unroll
        for (int i = 0; i < VEC; ++i) st[i] = 0.f;
        if (active && h0) {
            const V v = *reinterpret_cast<const V *>(h0 + bh * HS + e);
            memcpy(st, &v, sizeof(V));
        }
        const int64_t base = rel * nsup * HS + e;
        for (int w0 = 0; w0 < nsup; w0 += kWin) {
            const int w1 = min(nsup, w0 + kWin);
            // each super-chunk's log2 decay is the sum of its chunks' last G values, added in
            // chunk order; the chunk values are loaded a tile at a time by the whole block
            __syncthreads();                          // the previous window's decays are no longer read
            const int wm = min(w1, nm);
            for (int m = w0 + threadIdx.x; m < wm; m += blockDim.x) sdl[m - w0] = 0.f;
            const int64_t c_end = min((int64_t)pr.nc, (int64_t)wm * R);
            for (int64_t c0 = (int64_t)w0 * R; c0 < c_end; c0 += kTile) {
                __syncthreads();
                const int64_t c = c0 + threadIdx.x;
                sgl[threadIdx.x] = c < c_end ? Gh[min(pr.L, (c + 1) * pr.T) - 1] : 0.f;
                __syncthreads();
                for (int m = w0 + threadIdx.x; m < wm; m += blockDim.x) {
                    const int64_t k_lo = max((int64_t)m * R, c0);
                    const int64_t k_hi = min(min((int64_t)(m + 1) * R, c0 + kTile), c_end);
                    float acc = sdl[m - w0];
                    for (int64_t k = k_lo; k < k_hi; ++k) acc += sgl[k - c0];
                    sdl[m - w0] = acc;
                }
            }
            __syncthreads();
            for (int m = w0 + threadIdx.x; m < wm; m += blockDim.x) sdec[m - w0] = exp2f(sdl[m - w0]);
            __syncthreads();
            if (!active) continue;
            for (int m0 = w0; m0 < w1; m0 += kBatch) {
                V sv[kBatch];
#pragma unroll
                for (int i = 0; i < kBatch; ++i)
                    if (m0 + i < min(w1, nm)) sv[i] = *reinterpret_cast<const V *>(s_local + base + (int64_t)(m0 + i) * HS);
#pragma unroll
                for (int i = 0; i < kBatch; ++i) {
                    const int m = m0 + i;
                    if (m >= w1) break;
                    V out;
                    memcpy(&out, st, sizeof(V));
                    *reinterpret_cast<V *>(h_start + base + (int64_t)m * HS) = out;
                    if (m >= nm) continue;
                    const float a = sdec[m - w0];
                    float sa[VEC];
                    memcpy(sa, &sv[i], sizeof(V));
#pragma unroll
                    for (int j = 0; j < VEC; ++j) st[j] = fmaf(a, st[j], sa[j]);
                }
            }
        }
        if (active && h_final && nm == nsup) {
            V out;
            memcpy(&out, st, sizeof(V));
            *reinterpret_cast<V *>(h_final + bh * HS + e) = out;
        }
    }
}

// ---------------------------------------------------------------------------
// Stage 4 -- chunk_scan on CUDA cores (blog section "Kernel 3: compute_out").
// For 32 rows i of one chunk and a 64-wide slice of p:
//   y[i][p] = exp2(G_i) sum_s C[i][s] h_k[p][s]
//           + sum_{j <= i} (C_i . B_j) exp2(G_i - G_j) dt_j x[j][p]      (select, never multiply, the mask)
//           + D x[i][p]
// ---------------------------------------------------------------------------
constexpr int kScanRows = 32, kScanCols = 64;

template <typename Tin, typename Tout>
__global__ void __launch_bounds__(256)
k_chunk_scan_simt(const Tin *__restrict__ x, const Tin *__restrict__ dt,
                  const Tin *__restrict__ Bm, const Tin *__restrict__ Cm,
                  const float *__restrict__ D, const float *__restrict__ G,
                  const float *__restrict__ h_start, Tout *__restrict__ y, Problem pr,
                  int rtiles, int ptiles)
{
    extern __shared__ float smem[];
    const int SP = (int)pr.S + 1;                 // padded row stride
    float *Ct = smem;                             // [32][SP]   C rows i
    float *Bs = Ct + kScanRows * SP;              // [32][SP]   B rows j
    float *Xs = Bs + kScanRows * SP;              // [32][65]   dt_j x[j][p]
    float *Pm = Xs + kScanRows * (kScanCols + 1); // [32][33]   masked, decayed C B^T
    float *Hs = Pm + kScanRows * 33;              // [64][33]   h_k[p][s-slice]
    float *Gi = Hs + kScanCols * 33;              // [32]
    float *Gj = Gi + kScanRows;                   // [32]

    const int k = blockIdx.x / rtiles, rt = blockIdx.x % rtiles;
    const int h = blockIdx.y / ptiles, pt = blockIdx.y % ptiles;
    const int b = blockIdx.z;
    const int g = (int)(h / pr.hpg);
    const int64_t t0 = (int64_t)k * pr.T;
    const int n = (int)(pr.T < pr.L - t0 ? pr.T : pr.L - t0);
    const int i0 = rt * kScanRows, p0 = pt * kScanCols;
    if (i0 >= n) return;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int r = tid >> 3, c = tid & 7;           // output row, p lane (p = c + 8q)
    const float *Gh = G + ((int64_t)b * pr.nh + h) * pr.L + t0;
    auto bc_row = [&](const Tin *M, int t) { return M + (((int64_t)b * pr.L + t0 + t) * pr.G + g) * pr.S; };

    for (int rr = warp; rr < kScanRows; rr += 8) {
        const int i = i0 + rr;
        const Tin *src = bc_row(Cm, i < n ? i : 0);
        for (int s = lane; s < pr.S; s += 32) Ct[rr * SP + s] = (i < n) ? to_f32(src[s]) : 0.f;
    }
    if (tid < kScanRows) Gi[tid] = (i0 + tid < n) ? Gh[i0 + tid] : 0.f;

    float acc[8], sacc[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) { acc[q] = 0.f; sacc[q] = 0.f; }

    const int jend = min(n, i0 + kScanRows);
    for (int js = 0; js < jend; js += kScanRows) {
        __syncthreads();
        for (int rr = warp; rr < kScanRows; rr += 8) {
            const int j = js + rr;
            const Tin *src = bc_row(Bm, j < n ? j : 0);
            for (int s = lane; s < pr.S; s += 32) Bs[rr * SP + s] = (j < n) ? to_f32(src[s]) : 0.f;
            const float dtj = (j < n) ? to_f32(dt[((int64_t)b * pr.L + t0 + j) * pr.nh + h]) : 0.f;
            for (int pp = lane; pp < kScanCols; pp += 32) {
                const int p = p0 + pp;
                float v = 0.f;
                if (j < n && p < pr.H) v = dtj * to_f32(x[(((int64_t)b * pr.L + t0 + j) * pr.nh + h) * pr.H + p]);
                Xs[rr * (kScanCols + 1) + pp] = v;
            }
        }
        if (tid < kScanRows) Gj[tid] = (js + tid < n) ? Gh[js + tid] : 0.f;
        __syncthreads();
        // masked, decayed C B^T for rows i0.., columns js..
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int jj = c + 8 * q;
            const int i = i0 + r, j = js + jj;
            float v = 0.f;
            if (j <= i && i < n && j < n) {
                float cb = 0.f;
                const float *ci = Ct + r * SP, *bj = Bs + jj * SP;
                for (int s = 0; s < pr.S; ++s) cb = fmaf(ci[s], bj[s], cb);
                v = cb * exp2f(Gi[r] - Gj[jj]);
            }
            Pm[r * 33 + jj] = v;
        }
        __syncthreads();
#pragma unroll 4
        for (int jj = 0; jj < kScanRows; ++jj) {
            const float pv = Pm[r * 33 + jj];
#pragma unroll
            for (int q = 0; q < 8; ++q) acc[q] = fmaf(pv, Xs[jj * (kScanCols + 1) + c + 8 * q], acc[q]);
        }
    }
    // carried-state term: C_i . h_k[p]
    const float *hk = h_start + ((((int64_t)b * pr.nh + h) * pr.nc + k) * pr.H) * pr.S;
    for (int ss = 0; ss < pr.S; ss += 32) {
        __syncthreads();
        for (int pp = warp; pp < kScanCols; pp += 8) {
            const int p = p0 + pp, s = ss + lane;
            Hs[pp * 33 + lane] = (p < pr.H && s < pr.S) ? hk[(int64_t)p * pr.S + s] : 0.f;
        }
        __syncthreads();
        const int send = min(32, (int)pr.S - ss);
        for (int s2 = 0; s2 < send; ++s2) {
            const float cv = Ct[r * SP + ss + s2];
#pragma unroll
            for (int q = 0; q < 8; ++q) sacc[q] = fmaf(cv, Hs[(c + 8 * q) * 33 + s2], sacc[q]);
        }
    }
    const int i = i0 + r;
    if (i < n) {
        const float eg = exp2f(Gi[r]);
        const float dh = D[h];
        const int64_t row = (((int64_t)b * pr.L + t0 + i) * pr.nh + h) * pr.H;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const int p = p0 + c + 8 * q;
            if (p < pr.H) {
                const float xv = to_f32(x[row + p]);
                y[row + p] = from_f32<Tout>(fmaf(eg, sacc[q], acc[q]) + dh * xv);
            }
        }
    }
}

// ---------------------------------------------------------------------------
// Decode step (blog section "Mamba-2 architecture", the recurrent form).
// h[p][s] = exp(A dt) h[p][s] + dt x[p] B[s],  y[p] = sum_s C[s] h[p][s] + D x[p].
// The state is read and written once: the kernel is bound by HBM.  One block per
// (batch, head); warp w takes rows p = w, w + 8, ...; each lane holds a run of S/32
// consecutive s, so a row is one 16-byte access per lane per 128 floats, and B, C are
// loaded once per block.  Rows are processed kRows at a time with every state load
// issued before the first use, to keep enough bytes in flight.
// ---------------------------------------------------------------------------
template <typename Tin, typename Tout, int SV>   // SV: float4 per lane per row (S = 128 SV)
__global__ void __launch_bounds__(256)
k_ssd_step(const Tin *__restrict__ x, const Tin *__restrict__ dt, const float *__restrict__ A,
           const Tin *__restrict__ Bm, const Tin *__restrict__ Cm, const float *__restrict__ D,
           float *__restrict__ hst, Tout *__restrict__ y, Problem pr)
{
    constexpr int kRows = 4;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int hh = blockIdx.x, b = blockIdx.y;
    const int g = (int)(hh / pr.hpg);
    const int64_t bh = (int64_t)b * pr.nh + hh;
    const float dtv = to_f32(dt[bh]);
    const float alpha = exp2f(A[hh] * dtv * kLog2e);
    const float dh = D[hh];
    const Tin *Bv = Bm + ((int64_t)b * pr.G + g) * pr.S;
    const Tin *Cv = Cm + ((int64_t)b * pr.G + g) * pr.S;
    float bv[4 * SV], cv[4 * SV];
#pragma unroll
    for (int k = 0; k < SV; ++k)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int s = 128 * k + 4 * lane + e;
            bv[4 * k + e] = to_f32(Bv[s]);
            cv[4 * k + e] = to_f32(Cv[s]);
        }
    float4 *hrow = reinterpret_cast<float4 *>(hst + bh * pr.H * pr.S);
    const int rows_per_warp = (int)((pr.H + 7) / 8);
    for (int r0 = 0; r0 < rows_per_warp; r0 += kRows) {
        float4 hv[kRows][SV];
        float xp[kRows];
#pragma unroll
        for (int i = 0; i < kRows; ++i) {
            const int p = warp + 8 * (r0 + i);
            const bool valid = r0 + i < rows_per_warp && p < pr.H;
            xp[i] = valid ? to_f32(x[bh * pr.H + p]) : 0.f;
#pragma unroll
            for (int k = 0; k < SV; ++k)
                hv[i][k] = valid ? hrow[(int64_t)p * (pr.S / 4) + 32 * k + lane] : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int i = 0; i < kRows; ++i) {
            const int p = warp + 8 * (r0 + i);
            const bool valid = r0 + i < rows_per_warp && p < pr.H;
            const float u = dtv * xp[i];
            float acc = 0.f;
#pragma unroll
            for (int k = 0; k < SV; ++k) {
                float4 v = hv[i][k];
                v.x = fmaf(alpha, v.x, u * bv[4 * k + 0]);
                v.y = fmaf(alpha, v.y, u * bv[4 * k + 1]);
                v.z = fmaf(alpha, v.z, u * bv[4 * k + 2]);
                v.w = fmaf(alpha, v.w, u * bv[4 * k + 3]);
                if (valid) hrow[(int64_t)p * (pr.S / 4) + 32 * k + lane] = v;
                acc = fmaf(cv[4 * k + 0], v.x, acc);
                acc = fmaf(cv[4 * k + 1], v.y, acc);
                acc = fmaf(cv[4 * k + 2], v.z, acc);
                acc = fmaf(cv[4 * k + 3], v.w, acc);
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
            if (valid && lane == 0) y[bh * pr.H + p] = from_f32<Tout>(fmaf(dh, xp[i], acc));
        }
    }
}

// Any S: one warp per state row (b, h, p), lanes striding over s.
template <typename Tin, typename Tout>
__global__ void __launch_bounds__(256)
k_ssd_step_any(const Tin *__restrict__ x, const Tin *__restrict__ dt, const float *__restrict__ A,
               const Tin *__restrict__ Bm, const Tin *__restrict__ Cm, const float *__restrict__ D,
               float *__restrict__ hst, Tout *__restrict__ y, Problem pr)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t p = (int64_t)blockIdx.x * 8 + warp;
    const int hh = blockIdx.y, b = blockIdx.z;
    if (p >= pr.H) return;
    const int g = (int)(hh / pr.hpg);
    const int64_t bh = (int64_t)b * pr.nh + hh;
    const float dtv = to_f32(dt[bh]);
    const float alpha = exp2f(A[hh] * dtv * kLog2e);
    const float xp = to_f32(x[bh * pr.H + p]);
    const Tin *Bv = Bm + ((int64_t)b * pr.G + g) * pr.S;
    const Tin *Cv = Cm + ((int64_t)b * pr.G + g) * pr.S;
    float *row = hst + (bh * pr.H + p) * pr.S;
    const float u = dtv * xp;
    float acc = 0.f;
    for (int64_t s = lane; s < pr.S; s += 32) {
        const float v = fmaf(alpha, row[s], u * to_f32(Bv[s]));
        row[s] = v;
        acc = fmaf(to_f32(Cv[s]), v, acc);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (lane == 0) y[bh * pr.H + p] = from_f32<Tout>(fmaf(D[hh], xp, acc));
}

size_t scan_smem_bytes(const Problem &pr)
{
    const size_t SP = (size_t)pr.S + 1;
    return sizeof(float) * (2 * kScanRows * SP + kScanRows * (kScanCols + 1) + kScanRows * 33 +
                            kScanCols * 33 + 2 * kScanRows);
}

}  // namespace

unsigned cumsum_ctas(const Problem &pr)
{
    return (unsigned)(pr.nc * ((pr.nh + 31) / 32) * pr.B);
}

cudaError_t launch_chunk_cumsum(const Problem &pr, const void *dt, const float *A, float *G,
                                float *dtT, int64_t dtT_lo, int64_t dtT_hi, cudaStream_t st, unsigned *count,
                                __nv_bfloat16 *dt16)
{
    dim3 grid((unsigned)pr.nc, (unsigned)((pr.nh + 31) / 32), (unsigned)pr.B);
    const size_t smem = sizeof(float) * 33 * (size_t)pr.T * (dtT ? 2 : 1);
    cudaError_t e;
    if (pr.in_dt == SSD_BF16 && !pr.dt_f32) {
        auto kern = k_chunk_cumsum<__nv_bfloat16>;
        if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) != cudaSuccess) return e;
        kern<<<grid, 256, smem, st>>>((const __nv_bfloat16 *)dt, A, G, dtT, dtT_lo, dtT_hi, pr.L, (int)pr.nh, (int)pr.T,
                                      count, nullptr);
    } else {
        auto kern = k_chunk_cumsum<float>;
        if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) != cudaSuccess) return e;
        kern<<<grid, 256, smem, st>>>((const float *)dt, A, G, dtT, dtT_lo, dtT_hi, pr.L, (int)pr.nh, (int)pr.T,
                                      count, dt16);
    }
    return cudaGetLastError();
}

cudaError_t launch_chunk_state_simt(const Problem &pr, const void *x, const void *dt,
                                    const void *Bm, const float *G, float *s_local,
                                    cudaStream_t st)
{
    const int ptiles = (int)((pr.H + 31) / 32), stiles = (int)((pr.S + 63) / 64);
    dim3 grid((unsigned)pr.nc, (unsigned)(pr.nh * ptiles * stiles), (unsigned)pr.B);
    if (pr.in_dt == SSD_BF16)
        k_chunk_state_simt<__nv_bfloat16><<<grid, 256, 0, st>>>(
            (const __nv_bfloat16 *)x, (const __nv_bfloat16 *)dt, (const __nv_bfloat16 *)Bm, G, s_local, pr, ptiles, stiles);
    else
        k_chunk_state_simt<float><<<grid, 256, 0, st>>>(
            (const float *)x, (const float *)dt, (const float *)Bm, G, s_local, pr, ptiles, stiles);
    return cudaGetLastError();
}

cudaError_t launch_state_passing(const Problem &pr, SeqRange seqs, const float *G, const float *s_local,
                                 const float *h0, float *h_start, float *h_final, int R, int nsup, int nm,
                                 cudaStream_t st)
{
    if (seqs.n <= 0) return cudaSuccess;
    const int64_t HS = pr.H * pr.S;
    const bool v4 = (HS % 4 == 0) && ((uintptr_t)s_local % 16 == 0) && ((uintptr_t)h_start % 16 == 0) &&
                    (!h0 || (uintptr_t)h0 % 16 == 0) && (!h_final || (uintptr_t)h_final % 16 == 0);
    const int vec = v4 ? 4 : 1;
    dim3 grid((unsigned)((HS / vec + kPassThreads - 1) / kPassThreads), (unsigned)(seqs.n < 65535 ? seqs.n : 65535));
    if (v4)
        return launch_pdl(k_state_passing<4>, grid, dim3(kPassThreads), 0, st, G, s_local, h0, h_start, h_final, pr,
                          seqs, R, nsup, nm);
    return launch_pdl(k_state_passing<1>, grid, dim3(kPassThreads), 0, st, G, s_local, h0, h_start, h_final, pr, seqs,
                      R, nsup, nm);
}

template <typename Tin, typename Tout>
static cudaError_t scan_launch(const Problem &pr, const void *x, const void *dt, const void *Bm,
                               const void *Cm, const float *D, const float *G, const float *h_start,
                               void *y, cudaStream_t st)
{
    const int rtiles = (int)((pr.T + kScanRows - 1) / kScanRows);
    const int ptiles = (int)((pr.H + kScanCols - 1) / kScanCols);
    const size_t smem = scan_smem_bytes(pr);
    auto kern = k_chunk_scan_simt<Tin, Tout>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)(pr.nc * rtiles), (unsigned)(pr.nh * ptiles), (unsigned)pr.B);
    kern<<<grid, 256, smem, st>>>((const Tin *)x, (const Tin *)dt, (const Tin *)Bm, (const Tin *)Cm, D, G,
                                  h_start, (Tout *)y, pr, rtiles, ptiles);
    return cudaGetLastError();
}

cudaError_t launch_chunk_scan_simt(const Problem &pr, const void *x, const void *dt,
                                   const void *Bm, const void *Cm, const float *D, const float *G,
                                   const float *h_start, void *y, cudaStream_t st)
{
    const bool ib = pr.in_dt == SSD_BF16, ob = pr.out_dt == SSD_BF16;
    if (ib && ob) return scan_launch<__nv_bfloat16, __nv_bfloat16>(pr, x, dt, Bm, Cm, D, G, h_start, y, st);
    if (ib) return scan_launch<__nv_bfloat16, float>(pr, x, dt, Bm, Cm, D, G, h_start, y, st);
    if (ob) return scan_launch<float, __nv_bfloat16>(pr, x, dt, Bm, Cm, D, G, h_start, y, st);
    return scan_launch<float, float>(pr, x, dt, Bm, Cm, D, G, h_start, y, st);
}

template <typename Tin, typename Tout>
static cudaError_t step_launch(const Problem &pr, const void *x, const void *dt, const float *A,
                               const void *Bm, const void *Cm, const float *D, float *h, void *y,
                               cudaStream_t st)
{
    // S a multiple of 128 (and h 16-byte aligned): the vectorised kernel; any other S: one warp per row
    if (pr.S % 128 == 0 && pr.S <= 512 && (reinterpret_cast<uintptr_t>(h) & 15) == 0 && pr.nh <= 65535 && pr.B <= 65535) {
        dim3 grid((unsigned)pr.nh, (unsigned)pr.B);
        const Tin *xi = (const Tin *)x, *di = (const Tin *)dt, *bi = (const Tin *)Bm, *ci = (const Tin *)Cm;
        switch (pr.S / 128) {
            case 1: k_ssd_step<Tin, Tout, 1><<<grid, 256, 0, st>>>(xi, di, A, bi, ci, D, h, (Tout *)y, pr); break;
            case 2: k_ssd_step<Tin, Tout, 2><<<grid, 256, 0, st>>>(xi, di, A, bi, ci, D, h, (Tout *)y, pr); break;
            case 3: k_ssd_step<Tin, Tout, 3><<<grid, 256, 0, st>>>(xi, di, A, bi, ci, D, h, (Tout *)y, pr); break;
            default: k_ssd_step<Tin, Tout, 4><<<grid, 256, 0, st>>>(xi, di, A, bi, ci, D, h, (Tout *)y, pr); break;
        }
        return cudaGetLastError();
    }
    dim3 grid((unsigned)((pr.H + 7) / 8), (unsigned)pr.nh, (unsigned)pr.B);
    k_ssd_step_any<Tin, Tout><<<grid, 256, 0, st>>>((const Tin *)x, (const Tin *)dt, A, (const Tin *)Bm,
                                                    (const Tin *)Cm, D, h, (Tout *)y, pr);
    return cudaGetLastError();
}

cudaError_t launch_ssd_step(const Problem &pr, const void *x, const void *dt, const float *A,
                            const void *Bm, const void *Cm, const float *D, float *h, void *y,
                            cudaStream_t st)
{
    const bool ib = pr.in_dt == SSD_BF16, ob = pr.out_dt == SSD_BF16;
    if (ib && ob) return step_launch<__nv_bfloat16, __nv_bfloat16>(pr, x, dt, A, Bm, Cm, D, h, y, st);
    if (ib) return step_launch<__nv_bfloat16, float>(pr, x, dt, A, Bm, Cm, D, h, y, st);
    if (ob) return step_launch<float, __nv_bfloat16>(pr, x, dt, A, Bm, Cm, D, h, y, st);
    return step_launch<float, float>(pr, x, dt, A, Bm, Cm, D, h, y, st);
}

}  // namespace ssd
