// s6_scan.cu -- Mamba-1 selective scan (S6), forward, on the CUDA cores.
//
// "Sasha Rush: Mamba: The Hard Way", Part 5: per channel d and state n the step
// is discretised, abar = exp(delta_t A[d][n]), bbar = delta_t B_t[n], and the
// vector recurrence h[n] = abar h[n] + bbar x_t, y_t = sum_n C_t[n] h[n] runs
// over the tokens (plus D[d] x_t when D is given).
//
// Each channel's N states are split over kSplit adjacent lanes (NS states each);
// a block holds kCh = 128 / kSplit channels of one B/C group of one batch row.
// Tiles of kTT tokens are staged through shared memory: rows of x and delta are
// contiguous in time, so consecutive threads load consecutive tokens; B and C rows
// of the group are shared by all channels of the block.  The next tile is loaded
// into registers while the current one is scanned.  Tokens go kU at a time: every
// shared-memory read of the group is issued first, then the recurrences run (two
// states per paired float32 instruction when a lane holds an even number of them),
// then each lane records its partial sums of C h in shared memory.  (Interleaving
// those stores with the next token's reads would keep the reads behind them.)  The
// output pass adds the kSplit partials and D x and writes y coalesced, so the token
// loop carries no shuffle.  The scan is bound by the special-function unit (one exp2
// per channel, state and token) once N >= 8.
#include "ssd_common.cuh"

namespace ssd {
namespace {

constexpr int kSplit = 4;              // lanes per channel
constexpr int kThreads = 128;
constexpr int kCh = kThreads / kSplit; // channels per block
constexpr int kTT = 64;                // tokens per tile
constexpr int kXP = kTT + 1;           // padded row of a channel tile
constexpr int kLx = kCh * kTT / kThreads;   // x (and delta) elements per thread per tile

__device__ __forceinline__ float fast_exp2(float v)
{
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(v));
    return r;
}

// Shared memory of one block (dynamic): the channel tile as (x, delta) pairs, the group's
// B and C per state, each lane's partial sum of C h per channel and token (the four lanes of a
// channel write four different banks), and D of the block's channels.  With an even number of
// states per lane, B and C are stored per pair of states as (B_n, B_n+1, C_n, C_n+1), one
// 16-byte read for two states; with one state per lane, as (B_n, C_n).
template <int NS>
struct S6Smem {
    static constexpr int NP = NS * kSplit;     // padded state count
    static constexpr size_t xd = (size_t)kCh * kXP;            // float2
    static constexpr size_t bc = (size_t)NP * kXP;             // float2
    static constexpr size_t yp = (size_t)kSplit * kCh * kXP;   // float
    static constexpr size_t bytes = 8 * (xd + bc) + 4 * (yp + kCh);
};

template <typename Tin, typename Tout, int NS>
__global__ void __launch_bounds__(kThreads)
k_s6_scan(const Tin *__restrict__ x, const Tin *__restrict__ delta, const float *__restrict__ A,
          const Tin *__restrict__ Bm, const Tin *__restrict__ Cm, const float *__restrict__ D,
          const float *__restrict__ h0, Tout *__restrict__ y, float *__restrict__ h_final,
          int64_t L, int dim, int N, int G, int blocks_per_group)
{
    using Sm = S6Smem<NS>;
    constexpr int NP = Sm::NP;
    constexpr bool kPair = NS % 2 == 0;                         // states taken two at a time
    constexpr int NQ = kPair ? NS / 2 : NS;                     // (pairs of) states per lane
    constexpr int kU = NS >= 8 ? 4 : 8;                         // tokens whose reads are issued together
    constexpr int kLb = (NP * kTT + kThreads - 1) / kThreads;   // B (and C) elements per thread per tile
    extern __shared__ float4 s6_smem[];
    float2 *xd = reinterpret_cast<float2 *>(s6_smem);          // [kCh][kXP]  (x, delta)
    float2 *bc = xd + Sm::xd;                                   // [NP][kXP] (B, C), or [NP/2][kXP] float4 pairs
    float *yp = reinterpret_cast<float *>(bc + Sm::bc);         // [kCh][kSplit][kXP]
    float *dsk = yp + Sm::yp;                                   // [kCh]  D of the block's channels
    const int tid = threadIdx.x;
    const int g = blockIdx.x / blocks_per_group;
    const int cpg = dim / G;
    const int c0 = (blockIdx.x % blocks_per_group) * kCh;      // first channel of the block inside the group
    const int b = blockIdx.y;
    const int nch = min(kCh, cpg - c0);                        // channels of this block
    const int64_t row0 = (int64_t)b * dim + (int64_t)g * cpg + c0;   // (b, d) row of the first channel
    const Tin *Bg = Bm + ((int64_t)b * G + g) * N * L;
    const Tin *Cg = Cm + ((int64_t)b * G + g) * N * L;

    // this thread's channel and states; with kPair, element q holds states 2q and 2q + 1
    const int ch = tid / kSplit, slice = tid % kSplit;
    const bool active = ch < nch;
    const int d = g * cpg + c0 + (active ? ch : 0);
    float h[NS], a2[NS];
#pragma unroll
    for (int s = 0; s < NS; ++s) {
        const int n = slice * NS + s;
        const bool on = active && n < N;
        a2[s] = on ? A[(int64_t)d * N + n] * kLog2e : 0.f;
        h[s] = (on && h0) ? h0[((int64_t)b * dim + d) * N + n] : 0.f;
    }
    float2 hp[kPair ? NQ : 1], ap[kPair ? NQ : 1];
    if constexpr (kPair) {
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
            hp[q] = make_float2(h[2 * q], h[2 * q + 1]);
            ap[q] = make_float2(a2[2 * q], a2[2 * q + 1]);
        }
    }
    // global -> registers for the tile starting at t0, kept in the input dtype: nothing consumes the
    // loads until stage() converts them, after the current tile's scan
    const Tin zero = from_f32<Tin>(0.f);
    Tin rx[kLx], rd[kLx], rb[kLb], rc[kLb];
    auto fetch = [&](int64_t t0) {
#pragma unroll
        for (int i = 0; i < kLx; ++i) {
            const int e = i * kThreads + tid, r = e / kTT, t = e % kTT;
            const bool on = r < nch && t0 + t < L;
            const int64_t o = (row0 + r) * L + t0 + t;
            rx[i] = zero;
            rd[i] = zero;
            if (on) {
                rx[i] = x[o];
                rd[i] = delta[o];
            }
        }
#pragma unroll
        for (int i = 0; i < kLb; ++i) {
            const int e = i * kThreads + tid, n = e / kTT, t = e % kTT;
            const bool on = n < N && e < NP * kTT && t0 + t < L;
            const int64_t o = (int64_t)n * L + t0 + t;
            rb[i] = zero;
            rc[i] = zero;
            if (on) {
                rb[i] = Bg[o];
                rc[i] = Cg[o];
            }
        }
    };
    auto stage = [&]() {
#pragma unroll
        for (int i = 0; i < kLx; ++i) {
            const int e = i * kThreads + tid, r = e / kTT, t = e % kTT;
            xd[r * kXP + t] = make_float2(to_f32(rx[i]), to_f32(rd[i]));
        }
#pragma unroll
        for (int i = 0; i < kLb; ++i) {
            const int e = i * kThreads + tid, n = e / kTT, t = e % kTT;
            if (e < NP * kTT) {
                if constexpr (kPair) {
                    float *cell = reinterpret_cast<float *>(bc) + ((n >> 1) * kXP + t) * 4 + (n & 1);
                    cell[0] = to_f32(rb[i]);
                    cell[2] = to_f32(rc[i]);
                } else {
                    bc[n * kXP + t] = make_float2(to_f32(rb[i]), to_f32(rc[i]));
                }
            }
        }
    };
    const float2 *xr = xd + ch * kXP;
    const float2 *bcr = bc + (slice * NS) * kXP;                                         // (B, C) rows
    const float4 *bc4r = reinterpret_cast<const float4 *>(bc) + (slice * NQ) * kXP;      // pair rows
    float *ypr = yp + (ch * kSplit + slice) * kXP;
    // one token: update this lane's states and return its partial sum of C h
    auto step = [&](float2 v, const float4 *q4, const float2 *q2) {
        const float dx = v.y * v.x;
        if constexpr (kPair) {
            float2 acc = make_float2(0.f, 0.f);
#pragma unroll
            for (int q = 0; q < NQ; ++q) {
                const float2 e = __fmul2_rn(make_float2(v.y, v.y), ap[q]);
                const float2 abar = make_float2(fast_exp2(e.x), fast_exp2(e.y));
                hp[q] = __ffma2_rn(abar, hp[q], __fmul2_rn(make_float2(dx, dx), make_float2(q4[q].x, q4[q].y)));
                acc = __ffma2_rn(make_float2(q4[q].z, q4[q].w), hp[q], acc);
            }
            return acc.x + acc.y;
        } else {
            float acc = 0.f;
#pragma unroll
            for (int s = 0; s < NS; ++s) {
                const float abar = fast_exp2(v.y * a2[s]);
                h[s] = fmaf(abar, h[s], dx * q2[s].x);
                acc = fmaf(q2[s].y, h[s], acc);
            }
            return acc;
        }
    };
    // kU tokens from t: every shared-memory read first, then the recurrences, then the partial
    // sums
    auto tokens = [&](int t) {
        float2 v[kU];
        float4 q4[kPair ? kU : 1][kPair ? NQ : 1];
        float2 q2[kPair ? 1 : kU][kPair ? 1 : NS];
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            v[u] = xr[t + u];
#pragma unroll
            for (int q = 0; q < NQ; ++q) {
                if constexpr (kPair) q4[u][q] = bc4r[q * kXP + t + u];
                else q2[u][q] = bcr[q * kXP + t + u];
            }
        }
        float acc[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u) acc[u] = step(v[u], q4[kPair ? u : 0], q2[kPair ? 0 : u]);
#pragma unroll
        for (int u = 0; u < kU; ++u) ypr[t + u] = acc[u];
    };
    auto token = [&](int t) {
        float4 q4[kPair ? NQ : 1];
        float2 q2[kPair ? 1 : NS];
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
            if constexpr (kPair) q4[q] = bc4r[q * kXP + t];
            else q2[q] = bcr[q * kXP + t];
        }
        ypr[t] = step(xr[t], q4, q2);
    };
    const int64_t ntiles = (L + kTT - 1) / kTT;
    if (tid < kCh) dsk[tid] = (D && tid < nch) ? D[g * cpg + c0 + tid] : 0.f;
    fetch(0);
    stage();
    __syncthreads();
    for (int64_t k = 0; k < ntiles; ++k) {
        const int64_t t0 = k * kTT;
        if (k + 1 < ntiles) fetch(t0 + kTT);
        const int tn = (int)min((int64_t)kTT, L - t0);
        if (tn == kTT) {
#pragma unroll 1
            for (int t = 0; t < kTT; t += kU) tokens(t);
        } else {
            for (int t = 0; t < tn; ++t) token(t);
        }
        __syncthreads();
        // y = D x + the kSplit partial sums, written back coalesced
#pragma unroll
        for (int i = 0; i < kLx; ++i) {
            const int e = i * kThreads + tid, r = e / kTT, t = e % kTT;
            if (r < nch && t0 + t < L) {
                float acc = dsk[r] * xd[r * kXP + t].x;
#pragma unroll
                for (int sl = 0; sl < kSplit; ++sl) acc += yp[(r * kSplit + sl) * kXP + t];
                y[(row0 + r) * L + t0 + t] = from_f32<Tout>(acc);
            }
        }
        __syncthreads();
        if (k + 1 < ntiles) {
            stage();
            __syncthreads();
        }
    }
    if (active && h_final) {
#pragma unroll
        for (int s = 0; s < NS; ++s) {
            const int n = slice * NS + s;
            const float hv = kPair ? ((s & 1) ? hp[s >> 1].y : hp[s >> 1].x) : h[s];
            if (n < N) h_final[((int64_t)b * dim + d) * N + n] = hv;
        }
    }
}

template <typename Tin, typename Tout, int NS>
cudaError_t s6_launch_t(const S6Problem &p, const void *x, const void *delta, const float *A, const void *Bm,
                        const void *Cm, const float *D, const float *h0, void *y, float *h_final, cudaStream_t st)
{
    const int cpg = (int)(p.dim / p.G);
    const int bpg = (cpg + kCh - 1) / kCh;
    dim3 grid((unsigned)(bpg * p.G), (unsigned)p.B);
    auto kern = k_s6_scan<Tin, Tout, NS>;
    const size_t smem = S6Smem<NS>::bytes;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<grid, kThreads, smem, st>>>((const Tin *)x, (const Tin *)delta, A, (const Tin *)Bm,
                                                        (const Tin *)Cm, D, h0, (Tout *)y, h_final, p.L, (int)p.dim,
                                                        (int)p.N, (int)p.G, bpg);
    return cudaGetLastError();
}

template <typename Tin, typename Tout>
cudaError_t s6_launch_io(const S6Problem &p, const void *x, const void *delta, const float *A, const void *Bm,
                         const void *Cm, const float *D, const float *h0, void *y, float *h_final, cudaStream_t st)
{
    const int64_t ns = (p.N + kSplit - 1) / kSplit;
    if (ns <= 1) return s6_launch_t<Tin, Tout, 1>(p, x, delta, A, Bm, Cm, D, h0, y, h_final, st);
    if (ns <= 2) return s6_launch_t<Tin, Tout, 2>(p, x, delta, A, Bm, Cm, D, h0, y, h_final, st);
    if (ns <= 4) return s6_launch_t<Tin, Tout, 4>(p, x, delta, A, Bm, Cm, D, h0, y, h_final, st);
    return s6_launch_t<Tin, Tout, 8>(p, x, delta, A, Bm, Cm, D, h0, y, h_final, st);   // N <= 32
}

}  // namespace

cudaError_t launch_s6_scan(const S6Problem &p, const void *x, const void *delta, const float *A, const void *Bm,
                           const void *Cm, const float *D, const float *h0, void *y, float *h_final, cudaStream_t st)
{
    const bool ib = p.in_dt == SSD_BF16, ob = p.out_dt == SSD_BF16;
    if (ib && ob) return s6_launch_io<__nv_bfloat16, __nv_bfloat16>(p, x, delta, A, Bm, Cm, D, h0, y, h_final, st);
    if (ib) return s6_launch_io<__nv_bfloat16, float>(p, x, delta, A, Bm, Cm, D, h0, y, h_final, st);
    if (ob) return s6_launch_io<float, __nv_bfloat16>(p, x, delta, A, Bm, Cm, D, h0, y, h_final, st);
    return s6_launch_io<float, float>(p, x, delta, A, Bm, Cm, D, h0, y, h_final, st);
}

}  // namespace ssd
