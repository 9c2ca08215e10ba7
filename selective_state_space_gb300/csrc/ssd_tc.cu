// ssd_tc.cu -- tensor-core kernels (tcgen05 MMA, TMEM accumulators, TMA staging) for
// the chunk_state and chunk_scan stages of the chunked SSD forward pass.
//
// Method: NVIDIA developer blog "Accelerating Mamba-2 with High-Performance Forward
// Pass Kernels in NVIDIA CUDA Tile", section "Mamba-2 architecture" (the log-space
// chunk jump and the chunk output) and sections "Kernel 2" and "Kernel 3".
//
// Design (GB300-first, not the blog's kernel structure):
//  * Every tensor-core contraction runs on 128-row tiles ("sub-chunks" of Q = 128
//    tokens); a chunk of T = 128 or 256 tokens is one or two sub-chunks.  The result is
//    the same chunked algorithm: inside a chunk the state handed from one sub-chunk to
//    the next is exact (it is the chunk jump applied to the first Q tokens).
//  * The sequence of each (batch, head) is cut into "super-chunks" of R chunks.
//    chunk_state computes the state each super-chunk produces from a zero start,
//    state_passing chains those states, and the scan kernel walks the chunks of one
//    super-chunk sequentially, carrying the state on chip (TMEM, float32) and writing
//    y.  With R = 1 this is exactly the blog's three-stage pipeline; larger R removes
//    the per-chunk state round trips through HBM.
//  * Operands are staged by TMA with 128-byte swizzle.  Scaled operands (dt o X,
//    w o X, the decayed and masked C B^T, the bf16 state) are written by CUDA-core
//    warps straight into the swizzled layout the MMA reads.
//  * One elected thread issues all MMAs; accumulators live in TMEM and are drained
//    with tcgen05.ld.  Every wait is bounded; on expiry the kernel records an error
//    bit in the workspace and winds down.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "sm100_ptx.cuh"
#include "ssd_tc.cuh"

namespace ssd {
namespace {

using namespace ptx;

constexpr int kQ = 128;                       // tokens per tensor-core sub-chunk (MMA M)
constexpr int kPB = 64;                       // p-columns per scan unit (one swizzle atom)
constexpr uint32_t kAtom = kQ * 128;          // bytes of one 128-row x 128-byte swizzled region
constexpr uint64_t kWaitNs = 2000000000ull;   // bound on every wait: 2 s

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

__device__ __forceinline__ float2 unpack_bf16x2(uint32_t u)
{
    __nv_bfloat162 v = *reinterpret_cast<__nv_bfloat162 *>(&u);
    return __bfloat1622float2(v);
}

// Byte offset of 16-byte chunk c of row r inside a 1024-byte-aligned region of
// 128-byte rows with the 128-byte swizzle (the layout TMA writes and the MMA reads).
__device__ __forceinline__ uint32_t sw128(uint32_t r, uint32_t c) { return r * 128u + (((c ^ (r & 7u)) & 7u) << 4); }

__device__ __forceinline__ void named_bar(uint32_t id, uint32_t nthreads)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

__device__ __forceinline__ void set_error(int *err, int bit)
{
    if (err) atomicOr(err, bit);
}

// ===========================================================================
// chunk_state on tensor cores: the state one super-chunk produces from a zero start.
//   s^T[s][p] = sum_{t in super-chunk m} w_t B_t[s] x_t[p],
//   w_t = dt_t exp2(decay from t to the end of the super-chunk)
//       = dt_t exp2((G_last(k) - G_t) + sum_{k' > k in m} G_last(k')).
// MMA: D[s][p] (TMEM lanes s, columns p) += B^T (A: M = s, K = t, MN-major, from the TMA
// tile of B) x (w o X) (B operand: K = t, N = p, MN-major, x tile scaled in place).
// One CTA per (batch, head, super-chunk); warp 0 issues TMA, warp 1 issues MMAs,
// warps 2..5 scale x and drain the accumulator.
// ===========================================================================
template <int S, int H>
struct StateCfg {
    static constexpr int kStages = 2;
    static constexpr uint32_t kBBytes = (S / 64) * kAtom;
    static constexpr uint32_t kXBytes = (H / 64) * kAtom;
    static constexpr uint32_t kStage = kBBytes + kXBytes;
    static constexpr int kMaxR = 256;
    static constexpr uint32_t kSmem = kStages * kStage + kMaxR * 4 + 256 + 1024;
    static constexpr uint32_t kTmemCols = (S / 128) * H <= 32 ? 32 : ((S / 128) * H <= 64 ? 64 : ((S / 128) * H <= 128 ? 128 : 256));
};

template <int S, int H>
__global__ void __launch_bounds__(192, 1)
k_chunk_state_tc(const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmX,
                 const float *__restrict__ G, const __nv_bfloat16 *__restrict__ dt, float *__restrict__ s_out,
                 Problem pr, int R, int nsup, int nm, int *err)
{
    using Cfg = StateCfg<S, H>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    float *sGl = (float *)(smem + Cfg::kStages * Cfg::kStage);                    // G_last of each chunk
    uint64_t *bars = (uint64_t *)(smem + Cfg::kStages * Cfg::kStage + Cfg::kMaxR * 4);
    uint32_t *tmem_slot = (uint32_t *)(bars + 8);
    // bars: [0,1] full, [2,3] free, [4,5] x_ready (per stage), [6] done
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // unit = (b, m, h) for m < nm, h fastest so heads sharing B tiles run together
    int u = blockIdx.x;
    const int h = u % pr.nh; u /= pr.nh;
    const int m = u % nm;
    const int b = u / nm;
    const int g = (int)(h / pr.hpg);
    const int k_begin = m * R;
    const int k_end = min((int)pr.nc, k_begin + R);
    const int nk = k_end - k_begin;
    const int qpc = (int)(pr.T / kQ);                    // sub-chunks per chunk
    const int nq = nk * qpc;
    const int64_t t_begin = (int64_t)k_begin * pr.T;
    const float *Gh = G + ((int64_t)b * pr.nh + h) * pr.L;

    if (threadIdx.x == 0) {
        for (int i = 0; i < 7; ++i) mbar_init(smem_u32(&bars[i]), (i >= 4 && i < 6) ? 128 : 1);
        fence_mbar_init();
    }
    if (warp == 1) { tmem_alloc(smem_u32(tmem_slot), Cfg::kTmemCols); tmem_relinquish(); }
    for (int i = threadIdx.x; i < nk; i += blockDim.x) sGl[i] = Gh[(int64_t)(k_begin + i) * pr.T + pr.T - 1];
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    bool ok = true;

    if (warp == 0) {
        if (lane == 0) {
            prefetch_tmap(&tmB);
            prefetch_tmap(&tmX);
            for (int q = 0; q < nq && ok; ++q) {
                const int st = q % Cfg::kStages;
                if (q >= Cfg::kStages && !mbar_wait(smem_u32(&bars[2 + st]), ((q / Cfg::kStages) - 1) & 1, kWaitNs)) {
                    ok = false; set_error(err, 1); break;
                }
                uint8_t *base = smem + st * Cfg::kStage;
                const uint32_t full = smem_u32(&bars[st]);
                mbar_arrive_expect_tx(full, Cfg::kStage);
                const int t0 = (int)(t_begin + (int64_t)q * kQ);
                for (int a = 0; a < S / 64; ++a) tma_load_4d(smem_u32(base + a * kAtom), &tmB, full, 64 * a, g, t0, b);
                for (int a = 0; a < H / 64; ++a)
                    tma_load_4d(smem_u32(base + Cfg::kBBytes + a * kAtom), &tmX, full, 64 * a, h, t0, b);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16_f32(128, H, 1, 1);
            for (int q = 0; q < nq && ok; ++q) {
                const int st = q % Cfg::kStages;
                if (!mbar_wait(smem_u32(&bars[4 + st]), (q / Cfg::kStages) & 1, kWaitNs)) { ok = false; set_error(err, 1); break; }
                tc_fence_after();
                const uint32_t bbase = smem_u32(smem + st * Cfg::kStage);
                const uint32_t xbase = bbase + Cfg::kBBytes;
#pragma unroll
                for (int lb = 0; lb < S / 128; ++lb) {
#pragma unroll
                    for (int kk = 0; kk < kQ / 16; ++kk) {
                        const uint64_t ad = smem_desc(bbase + lb * 2 * kAtom + kk * 2048, kAtom, 1024);
                        const uint64_t bd = smem_desc(xbase + kk * 2048, kAtom, 1024);
                        mma_bf16(tmem + lb * H, ad, bd, idesc, (q > 0 || kk > 0) ? 1u : 0u);
                    }
                }
                mma_commit(smem_u32(&bars[2 + st]));
            }
            if (ok) mma_commit(smem_u32(&bars[6]));
        }
        __syncwarp();
    } else {
        // warps 2..5: scale x rows in place, then drain the accumulator
        const int r = 32 * (warp & 3) + lane;       // token row of the tile / TMEM lane
        for (int q = 0; q < nq && ok; ++q) {
            const int st = q % Cfg::kStages;
            if (!mbar_wait(smem_u32(&bars[st]), (q / Cfg::kStages) & 1, kWaitNs)) { ok = false; set_error(err, 1); break; }
            const int kl = q / qpc;                          // chunk index inside the super-chunk
            float suffix = 0.f;
            for (int kk = kl + 1; kk < nk; ++kk) suffix += sGl[kk];
            const int64_t t = t_begin + (int64_t)q * kQ + r;
            const float wr = __bfloat162float(dt[((int64_t)b * pr.L + t) * pr.nh + h]) *
                             exp2f((sGl[kl] - Gh[t]) + suffix);
            uint8_t *xt = smem + st * Cfg::kStage + Cfg::kBBytes;
#pragma unroll
            for (int a = 0; a < H / 64; ++a) {
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    uint4 *p = (uint4 *)(xt + a * kAtom + sw128(r, c));
                    uint4 v = *p;
                    float2 f0 = unpack_bf16x2(v.x), f1 = unpack_bf16x2(v.y), f2 = unpack_bf16x2(v.z), f3 = unpack_bf16x2(v.w);
                    v.x = pack_bf16x2(f0.x * wr, f0.y * wr);
                    v.y = pack_bf16x2(f1.x * wr, f1.y * wr);
                    v.z = pack_bf16x2(f2.x * wr, f2.y * wr);
                    v.w = pack_bf16x2(f3.x * wr, f3.y * wr);
                    *p = v;
                }
            }
            fence_proxy_async_smem();
            mbar_arrive(smem_u32(&bars[4 + st]));
        }
        if (ok && !mbar_wait(smem_u32(&bars[6]), 0, kWaitNs)) { ok = false; set_error(err, 1); }
        if (ok) {
            tc_fence_after();
            const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
            float *dst = s_out + (((int64_t)b * pr.nh + h) * nsup + m) * (int64_t)(H * S);
#pragma unroll
            for (int lb = 0; lb < S / 128; ++lb) {
                const int s = lb * 128 + r;
#pragma unroll
                for (int c0 = 0; c0 < H; c0 += 16) {
                    uint32_t v[16];
                    tmem_ld16(tmem + lane_base + lb * H + c0, v);
                    tmem_ld_wait();
#pragma unroll
                    for (int j = 0; j < 16; ++j) dst[(int64_t)(c0 + j) * S + s] = __uint_as_float(v[j]);
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) tmem_dealloc(tmem, Cfg::kTmemCols);
}

// ===========================================================================
// chunk_scan on tensor cores: walk the chunks of one super-chunk for one
// (batch, head, 64-column p block), 128 tokens at a time, carrying the state.
// For a sub-chunk with rows i, j (tokens) and entering state h (H x S):
//   CB      = C B^T                                   (TMEM, fp32; M = i, N = j, K = s)
//   P[i][j] = CB[i][j] exp2(G_i - G_j) if j <= i else 0  (CUDA cores, bf16, swizzled)
//   Ys      = C h^T                                   (M = i, N = p, K = s)
//   Yi      = P (dt o X)                              (M = i, N = p, K = j)
//   y_i     = exp2(G_i - G_base) Ys_i + Yi_i + D x_i
//   h'^T    = exp2(G_last - G_base) h^T + B^T (w o X),  w_t = dt_t exp2(G_last - G_t)
// The state lives in TMEM as h^T (lanes s, columns p); a bf16 copy [s][p] in shared
// memory is the B operand of Ys.  G is the chunk-relative log2 cumsum; G_base is G
// at the token before the sub-chunk (0 at a chunk start).
// Warp 0: TMA.  Warp 1: MMA issue and TMEM allocation.  Warps 2..: CUDA-core work,
// 4*NW warps, NW per TMEM lane quarter, splitting columns.
// ===========================================================================
template <int S>
struct ScanCfg {
    static constexpr int kStages = (S <= 128) ? 2 : 1;
    static constexpr uint32_t kCBytes = (S / 64) * kAtom;    // C tile [i][s], K-major
    static constexpr uint32_t kBBytes = (S / 64) * kAtom;    // B tile [j][s]
    static constexpr uint32_t kXBytes = kAtom;               // x tile [t][p], 64 p
    static constexpr uint32_t kStage = kCBytes + kBBytes + kXBytes;
    static constexpr uint32_t kXw = kStages * kStage;        // w o x   [t][p]
    static constexpr uint32_t kP = kXw + kAtom;              // P       [i][j], 2 K-atoms
    static constexpr uint32_t kH = kP + 2 * kAtom;           // h bf16  [s][p], S rows
    static constexpr uint32_t kSmall = kH + S * 128;         // sG[128], sdt[128]
    static constexpr uint32_t kBars = kSmall + 2 * kQ * 4;
    static constexpr uint32_t kSmem = kBars + 256 + 1024;
    // TMEM columns
    static constexpr uint32_t kTcb = 0, kTys = 128, kTyi = 192, kTds = 256;
    static constexpr uint32_t kTmemCols = 512;
};

// kGroup: barrier among the CUDA-core warps only (an mbarrier, so its wait is bounded)
enum ScanBar { kFull0 = 0, kFree0 = 2, kCb = 4, kHReady, kXReady, kPReady, kIntra, kUpdate, kEpi, kGroup, kNumScanBars };

template <int S, int NW>
__global__ void __launch_bounds__(64 + 128 * NW, 1)
k_chunk_scan_tc(const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmB,
                const __grid_constant__ CUtensorMap tmX, const float *__restrict__ G,
                const __nv_bfloat16 *__restrict__ dt, const float *__restrict__ Dp,
                const float *__restrict__ h0, const float *__restrict__ h_start, float *__restrict__ h_final,
                __nv_bfloat16 *__restrict__ y, Problem pr, int R, int nsup, int hs_from, int *err)
{
    using Cfg = ScanCfg<S>;
    constexpr int kSimt = 128 * NW;
    constexpr int kCols = kPB / NW;                  // p columns per CUDA-core thread
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    float *sG = (float *)(smem + Cfg::kSmall);
    float *sdt = sG + kQ;
    uint64_t *bars = (uint64_t *)(smem + Cfg::kBars);
    uint32_t *tmem_slot = (uint32_t *)(bars + kNumScanBars);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    const int npb = (int)(pr.H / kPB);
    int u = blockIdx.x;
    const int pb = u % npb; u /= npb;
    const int h = u % pr.nh; u /= pr.nh;
    const int m = u % nsup;
    const int b = u / nsup;
    const int g = (int)(h / pr.hpg);
    const int k_begin = m * R;
    const int k_end = min((int)pr.nc, k_begin + R);
    const int qpc = (int)(pr.T / kQ);
    const int nq = (k_end - k_begin) * qpc;
    const int64_t t_begin = (int64_t)k_begin * pr.T;
    const int64_t bh = (int64_t)b * pr.nh + h;
    const float *Gh = G + bh * pr.L;
    const bool write_final = (m == nsup - 1) && h_final;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kNumScanBars; ++i) {
            uint32_t cnt = 1;
            if (i == kHReady || i == kXReady || i == kPReady || i == kEpi || i == kGroup) cnt = kSimt;
            mbar_init(smem_u32(&bars[i]), cnt);
        }
        fence_mbar_init();
    }
    if (warp == 1) { tmem_alloc(smem_u32(tmem_slot), Cfg::kTmemCols); tmem_relinquish(); }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    bool ok = true;

    if (warp == 0) {
        if (lane == 0) {
            prefetch_tmap(&tmC);
            prefetch_tmap(&tmB);
            prefetch_tmap(&tmX);
            for (int q = 0; q < nq && ok; ++q) {
                const int st = q % Cfg::kStages;
                if (q >= Cfg::kStages &&
                    !mbar_wait(smem_u32(&bars[kFree0 + st]), ((q / Cfg::kStages) - 1) & 1, kWaitNs)) {
                    ok = false; set_error(err, 1); break;
                }
                uint8_t *base = smem + st * Cfg::kStage;
                const uint32_t full = smem_u32(&bars[kFull0 + st]);
                mbar_arrive_expect_tx(full, Cfg::kStage);
                const int t0 = (int)(t_begin + (int64_t)q * kQ);
                for (int a = 0; a < S / 64; ++a) {
                    tma_load_4d(smem_u32(base + a * kAtom), &tmC, full, 64 * a, g, t0, b);
                    tma_load_4d(smem_u32(base + Cfg::kCBytes + a * kAtom), &tmB, full, 64 * a, g, t0, b);
                }
                tma_load_4d(smem_u32(base + Cfg::kCBytes + Cfg::kBBytes), &tmX, full, pb * kPB, h, t0, b);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t id_cb = idesc_bf16_f32(128, 128, 0, 0);
            constexpr uint32_t id_ys = idesc_bf16_f32(128, kPB, 0, 1);
            constexpr uint32_t id_yi = idesc_bf16_f32(128, kPB, 0, 1);
            constexpr uint32_t id_up = idesc_bf16_f32(128, kPB, 1, 1);
            const uint32_t hbase = smem_u32(smem + Cfg::kH);
            const uint32_t pbase = smem_u32(smem + Cfg::kP);
            const uint32_t xwbase = smem_u32(smem + Cfg::kXw);
            for (int q = 0; q < nq; ++q) {
                const int st = q % Cfg::kStages;
                const uint32_t cbase = smem_u32(smem + st * Cfg::kStage);
                const uint32_t bbase = cbase + Cfg::kCBytes;
                const uint32_t xbase = bbase + Cfg::kBBytes;
                if (!mbar_wait(smem_u32(&bars[kFull0 + st]), (q / Cfg::kStages) & 1, kWaitNs)) { ok = false; break; }
                tc_fence_after();
                // CB = C B^T (K = s)
#pragma unroll
                for (int kk = 0; kk < S / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * kAtom + (kk & 3) * 32;
                    mma_bf16(tmem + Cfg::kTcb, smem_desc(cbase + off, 16, 1024), smem_desc(bbase + off, 16, 1024),
                             id_cb, kk > 0 ? 1u : 0u);
                }
                mma_commit(smem_u32(&bars[kCb]));
                // Ys = C h^T (K = s), once the state copy is ready and the last epilogue drained Ys/Yi
                if (!mbar_wait(smem_u32(&bars[kHReady]), q & 1, kWaitNs)) { ok = false; break; }
                if (q > 0 && !mbar_wait(smem_u32(&bars[kEpi]), (q - 1) & 1, kWaitNs)) { ok = false; break; }
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < S / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * kAtom + (kk & 3) * 32;
                    mma_bf16(tmem + Cfg::kTys, smem_desc(cbase + off, 16, 1024), smem_desc(hbase + kk * 2048, kAtom, 1024),
                             id_ys, kk > 0 ? 1u : 0u);
                }
                // Yi = P (dt o X) (K = j)
                if (!mbar_wait(smem_u32(&bars[kPReady]), q & 1, kWaitNs)) { ok = false; break; }
                if (!mbar_wait(smem_u32(&bars[kXReady]), q & 1, kWaitNs)) { ok = false; break; }
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < kQ / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * kAtom + (kk & 3) * 32;
                    mma_bf16(tmem + Cfg::kTyi, smem_desc(pbase + off, 16, 1024), smem_desc(xbase + kk * 2048, kAtom, 1024),
                             id_yi, kk > 0 ? 1u : 0u);
                }
                mma_commit(smem_u32(&bars[kIntra]));
                // state update h^T += B^T (w o X) (K = t), on the state pre-scaled by the CUDA-core warps
                if (q + 1 < nq || write_final) {
#pragma unroll
                    for (int lb = 0; lb < S / 128; ++lb) {
#pragma unroll
                        for (int kk = 0; kk < kQ / 16; ++kk)
                            mma_bf16(tmem + Cfg::kTds + lb * kPB, smem_desc(bbase + lb * 2 * kAtom + kk * 2048, kAtom, 1024),
                                     smem_desc(xwbase + kk * 2048, kAtom, 1024), id_up, 1u);
                    }
                    mma_commit(smem_u32(&bars[kUpdate]));
                }
                mma_commit(smem_u32(&bars[kFree0 + st]));
            }
            if (!ok) set_error(err, 1);
        }
        __syncwarp();
    } else {
        // ---- CUDA-core warps --------------------------------------------------------
        const int sw = warp - 2;
        const int gw = sw >> 2;                        // column group
        const int r = 32 * (warp & 3) + lane;          // TMEM lane = tile row
        const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
        const float dh = Dp[h];
        uint8_t *xw = smem + Cfg::kXw;
        uint8_t *pt = smem + Cfg::kP;
        uint8_t *ht = smem + Cfg::kH;
        uint32_t xr[kCols / 2];                        // this thread's row of x (raw bf16 pairs)
        uint32_t grp_phase = 0;
        auto group_sync = [&]() -> bool {              // all CUDA-core threads; bounded
            mbar_arrive(smem_u32(&bars[kGroup]));
            const bool done = mbar_wait(smem_u32(&bars[kGroup]), grp_phase, kWaitNs);
            grp_phase ^= 1u;
            return done;
        };
        for (int q = 0; q < nq && ok; ++q) {
            const int st = q % Cfg::kStages;
            const int qin = q % qpc;                   // sub-chunk index inside its chunk
            const int64_t t0 = t_begin + (int64_t)q * kQ;
            const float gbase = (qin == 0) ? 0.f : Gh[t0 - 1];
            const float glast = Gh[t0 + kQ - 1];
            if (gw == 0) {
                sG[r] = Gh[t0 + r];
                sdt[r] = __bfloat162float(dt[((int64_t)b * pr.L + t0 + r) * pr.nh + h]);
            }
            if (!group_sync()) { ok = false; set_error(err, 1); break; }
            const float gr = sG[r], dtr = sdt[r];

            // (C) state hand-off: h (fp32) -> bf16 copy [s][p] for Ys, and h * exp2(glast - gbase) -> TMEM
            {
                const float dec = exp2f(glast - gbase);
                if (q > 0) {
                    if (!mbar_wait(smem_u32(&bars[kUpdate]), (q - 1) & 1, kWaitNs)) { ok = false; set_error(err, 1); break; }
                    tc_fence_after();
                }
#pragma unroll
                for (int lb = 0; lb < S / 128; ++lb) {
                    const int s = lb * 128 + r;
#pragma unroll
                    for (int c0 = 0; c0 < kCols; c0 += 16) {
                        const int p0 = gw * kCols + c0;
                        uint32_t v[16];
                        if (q == 0) {
                            // entering state: h0 (zeros if absent) for super-chunks m < hs_from, else h_start[m]
                            const float *src = (m < hs_from) ? (h0 ? h0 + bh * (int64_t)(pr.H * S) : nullptr)
                                                             : h_start + (bh * nsup + m) * (int64_t)(pr.H * S);
                            if (src) {
                                src += (int64_t)(pb * kPB + p0) * S + s;
#pragma unroll
                                for (int j = 0; j < 16; ++j) v[j] = __float_as_uint(src[(int64_t)j * S]);
                            } else {
#pragma unroll
                                for (int j = 0; j < 16; ++j) v[j] = 0u;
                            }
                        } else {
                            tmem_ld16(tmem + lane_base + Cfg::kTds + lb * kPB + p0, v);
                            tmem_ld_wait();
                        }
                        uint4 lo, hi;
                        lo.x = pack_bf16x2(__uint_as_float(v[0]), __uint_as_float(v[1]));
                        lo.y = pack_bf16x2(__uint_as_float(v[2]), __uint_as_float(v[3]));
                        lo.z = pack_bf16x2(__uint_as_float(v[4]), __uint_as_float(v[5]));
                        lo.w = pack_bf16x2(__uint_as_float(v[6]), __uint_as_float(v[7]));
                        hi.x = pack_bf16x2(__uint_as_float(v[8]), __uint_as_float(v[9]));
                        hi.y = pack_bf16x2(__uint_as_float(v[10]), __uint_as_float(v[11]));
                        hi.z = pack_bf16x2(__uint_as_float(v[12]), __uint_as_float(v[13]));
                        hi.w = pack_bf16x2(__uint_as_float(v[14]), __uint_as_float(v[15]));
                        *(uint4 *)(ht + sw128(s, p0 >> 3)) = lo;
                        *(uint4 *)(ht + sw128(s, (p0 >> 3) + 1)) = hi;
#pragma unroll
                        for (int j = 0; j < 16; ++j) v[j] = __float_as_uint(__uint_as_float(v[j]) * dec);
                        tmem_st16(tmem + lane_base + Cfg::kTds + lb * kPB + p0, v);
                    }
                }
                tmem_st_wait();
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(smem_u32(&bars[kHReady]));
            }

            // (A) x tile: keep raw row, write dt o x in place and w o x to the Xw tile
            {
                if (!mbar_wait(smem_u32(&bars[kFull0 + st]), (q / Cfg::kStages) & 1, kWaitNs)) { ok = false; set_error(err, 1); break; }
                uint8_t *xt = smem + st * Cfg::kStage + Cfg::kCBytes + Cfg::kBBytes;
                const float wr = dtr * exp2f(glast - gr);
#pragma unroll
                for (int cc = 0; cc < kCols / 8; ++cc) {
                    const int c = gw * (kCols / 8) + cc;
                    const uint32_t off = sw128(r, c);
                    uint4 v = *(uint4 *)(xt + off);
                    xr[4 * cc + 0] = v.x; xr[4 * cc + 1] = v.y; xr[4 * cc + 2] = v.z; xr[4 * cc + 3] = v.w;
                    const uint32_t in[4] = {v.x, v.y, v.z, v.w};
                    uint32_t os[4], ow[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 f = unpack_bf16x2(in[e]);
                        os[e] = pack_bf16x2(f.x * dtr, f.y * dtr);
                        ow[e] = pack_bf16x2(f.x * wr, f.y * wr);
                    }
                    *(uint4 *)(xt + off) = make_uint4(os[0], os[1], os[2], os[3]);
                    *(uint4 *)(xw + off) = make_uint4(ow[0], ow[1], ow[2], ow[3]);
                }
                fence_proxy_async_smem();
                mbar_arrive(smem_u32(&bars[kXReady]));
            }

            // (B) P = CB o exp2(G_i - G_j) o [j <= i], bf16, K-major swizzled [i][j]
            {
                if (!mbar_wait(smem_u32(&bars[kCb]), q & 1, kWaitNs)) { ok = false; set_error(err, 1); break; }
                tc_fence_after();
                const int wrow_hi = 32 * (warp & 3) + 31;   // largest row of this warp
                for (int jb = gw; jb < kQ / 16; jb += NW) {
                    const int j0 = jb * 16;
                    uint32_t pk[8];
                    if (j0 > wrow_hi) {                    // whole block above the diagonal: zeros
#pragma unroll
                        for (int e = 0; e < 8; ++e) pk[e] = 0u;
                    } else {
                        uint32_t v[16];
                        tmem_ld16(tmem + lane_base + Cfg::kTcb + j0, v);
                        tmem_ld_wait();
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            const int j = j0 + 2 * e;
                            const float a0 = (j <= r) ? __uint_as_float(v[2 * e]) * exp2f(gr - sG[j]) : 0.f;
                            const float a1 = (j + 1 <= r) ? __uint_as_float(v[2 * e + 1]) * exp2f(gr - sG[j + 1]) : 0.f;
                            pk[e] = pack_bf16x2(a0, a1);
                        }
                    }
                    const int a = j0 >> 6, c = (j0 & 63) >> 3;
                    *(uint4 *)(pt + a * kAtom + sw128(r, c)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                    *(uint4 *)(pt + a * kAtom + sw128(r, c + 1)) = make_uint4(pk[4], pk[5], pk[6], pk[7]);
                }
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(smem_u32(&bars[kPReady]));
            }

            // (D) epilogue: y = exp2(G_i - G_base) Ys + Yi + D x
            {
                if (!mbar_wait(smem_u32(&bars[kIntra]), q & 1, kWaitNs)) { ok = false; set_error(err, 1); break; }
                tc_fence_after();
                const float eg = exp2f(gr - gbase);
                __nv_bfloat16 *yrow = y + ((((int64_t)b * pr.L + t0 + r) * pr.nh + h) * pr.H + pb * kPB);
#pragma unroll
                for (int c0 = 0; c0 < kCols; c0 += 16) {
                    const int p0 = gw * kCols + c0;
                    uint32_t vs[16], vi[16];
                    tmem_ld16(tmem + lane_base + Cfg::kTys + p0, vs);
                    tmem_ld16(tmem + lane_base + Cfg::kTyi + p0, vi);
                    tmem_ld_wait();
                    uint32_t o[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const float2 xv = unpack_bf16x2(xr[(c0 >> 1) + e]);
                        const float y0 = fmaf(eg, __uint_as_float(vs[2 * e]), __uint_as_float(vi[2 * e])) + dh * xv.x;
                        const float y1 = fmaf(eg, __uint_as_float(vs[2 * e + 1]), __uint_as_float(vi[2 * e + 1])) + dh * xv.y;
                        o[e] = pack_bf16x2(y0, y1);
                    }
                    *(uint4 *)(yrow + p0) = make_uint4(o[0], o[1], o[2], o[3]);
                    *(uint4 *)(yrow + p0 + 8) = make_uint4(o[4], o[5], o[6], o[7]);
                }
                tc_fence_before();
                mbar_arrive(smem_u32(&bars[kEpi]));
            }
            // sG / sdt are rewritten by the next sub-chunk
            if (!group_sync()) { ok = false; set_error(err, 1); break; }
        }
        // final state of the sequence, from the last unit of each (batch, head)
        if (ok && write_final) {
            if (!mbar_wait(smem_u32(&bars[kUpdate]), (nq - 1) & 1, kWaitNs)) { ok = false; set_error(err, 1); }
            if (ok) {
                tc_fence_after();
#pragma unroll
                for (int lb = 0; lb < S / 128; ++lb) {
                    const int s = lb * 128 + r;
#pragma unroll
                    for (int c0 = 0; c0 < kCols; c0 += 16) {
                        const int p0 = gw * kCols + c0;
                        uint32_t v[16];
                        tmem_ld16(tmem + lane_base + Cfg::kTds + lb * kPB + p0, v);
                        tmem_ld_wait();
                        float *dst = h_final + bh * (int64_t)(pr.H * S) + (int64_t)(pb * kPB + p0) * S + s;
#pragma unroll
                        for (int j = 0; j < 16; ++j) dst[(int64_t)j * S] = __uint_as_float(v[j]);
                    }
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) tmem_dealloc(tmem, Cfg::kTmemCols);
}

// ---- host side ---------------------------------------------------------------------

PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (PFN_cuTensorMapEncodeTiled_v12000)p;
    });
    return fn;
}

// 4-D bf16 tensor [d3][d2][d1][d0] (d0 contiguous), box {64, 1, rows, 1}, 128-byte swizzle.
bool make_map_4d(CUtensorMap *map, const void *ptr, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t d3, uint32_t rows)
{
    auto enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[4] = {d0, d1, d2, d3};
    cuuint64_t strides[3] = {d0 * 2, d0 * d1 * 2, d0 * d1 * d2 * 2};
    cuuint32_t box[4] = {64, 1, rows, 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(ptr), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int S, int H>
cudaError_t state_launch(const Problem &pr, const void *x, const void *dt, const void *Bm, const float *G, float *s_out,
                         int R, int nsup, int nm, int *err, cudaStream_t st)
{
    CUtensorMap mB, mX;
    if (!make_map_4d(&mB, Bm, pr.S, pr.G, pr.L, pr.B, kQ) || !make_map_4d(&mX, x, pr.H, pr.nh, pr.L, pr.B, kQ))
        return cudaErrorInvalidValue;
    using Cfg = StateCfg<S, H>;
    auto kern = k_chunk_state_tc<S, H>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Cfg::kSmem);
    if (e != cudaSuccess) return e;
    const unsigned grid = (unsigned)(pr.B * nm * pr.nh);
    if (grid == 0) return cudaSuccess;
    kern<<<grid, 192, Cfg::kSmem, st>>>(mB, mX, G, (const __nv_bfloat16 *)dt, s_out, pr, R, nsup, nm, err);
    return cudaGetLastError();
}

template <int S, int NW>
cudaError_t scan_launch(const Problem &pr, const void *x, const void *dt, const void *Bm, const void *Cm, const float *D,
                        const float *G, const float *h0, const float *h_start, float *h_final, void *y, int R, int nsup,
                        int hs_from, int *err, cudaStream_t st)
{
    CUtensorMap mC, mB, mX;
    if (!make_map_4d(&mC, Cm, pr.S, pr.G, pr.L, pr.B, kQ) || !make_map_4d(&mB, Bm, pr.S, pr.G, pr.L, pr.B, kQ) ||
        !make_map_4d(&mX, x, pr.H, pr.nh, pr.L, pr.B, kQ))
        return cudaErrorInvalidValue;
    using Cfg = ScanCfg<S>;
    auto kern = k_chunk_scan_tc<S, NW>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Cfg::kSmem);
    if (e != cudaSuccess) return e;
    const unsigned grid = (unsigned)(pr.B * nsup * pr.nh * (pr.H / kPB));
    kern<<<grid, 64 + 128 * NW, Cfg::kSmem, st>>>(mC, mB, mX, G, (const __nv_bfloat16 *)dt, D, h0, h_start, h_final,
                                                  (__nv_bfloat16 *)y, pr, R, nsup, hs_from, err);
    return cudaGetLastError();
}

}  // namespace

bool tc_supported(const Problem &pr)
{
    if (pr.in_dt != SSD_BF16 || pr.out_dt != SSD_BF16) return false;
    if (pr.S != 128 && pr.S != 256) return false;
    if (pr.H != 64 && pr.H != 128) return false;
    if (pr.T % kQ != 0 || pr.T > 256) return false;
    if (pr.L % pr.T != 0) return false;
    if (pr.L > 0x7fffffffLL || pr.B > 65535) return false;
    return true;
}

cudaError_t launch_chunk_state_tc(const Problem &pr, const void *x, const void *dt, const void *Bm, const float *G,
                                  float *s_out, int R, int nsup, int nm, int *err, cudaStream_t st)
{
    if (R < 1 || R > StateCfg<128, 64>::kMaxR) return cudaErrorInvalidValue;
    if (pr.S == 128 && pr.H == 64) return state_launch<128, 64>(pr, x, dt, Bm, G, s_out, R, nsup, nm, err, st);
    if (pr.S == 128 && pr.H == 128) return state_launch<128, 128>(pr, x, dt, Bm, G, s_out, R, nsup, nm, err, st);
    if (pr.S == 256 && pr.H == 64) return state_launch<256, 64>(pr, x, dt, Bm, G, s_out, R, nsup, nm, err, st);
    if (pr.S == 256 && pr.H == 128) return state_launch<256, 128>(pr, x, dt, Bm, G, s_out, R, nsup, nm, err, st);
    return cudaErrorNotSupported;
}

cudaError_t launch_chunk_scan_tc(const Problem &pr, const void *x, const void *dt, const void *Bm, const void *Cm,
                                 const float *D, const float *G, const float *h0, const float *h_start, float *h_final,
                                 void *y, int R, int nsup, int hs_from, int *err, cudaStream_t st)
{
    if (pr.S == 128) return scan_launch<128, 2>(pr, x, dt, Bm, Cm, D, G, h0, h_start, h_final, y, R, nsup, hs_from, err, st);
    if (pr.S == 256) return scan_launch<256, 2>(pr, x, dt, Bm, Cm, D, G, h0, h_start, h_final, y, R, nsup, hs_from, err, st);
    return cudaErrorNotSupported;
}

}  // namespace ssd
