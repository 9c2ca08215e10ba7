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
//    bit in the workspace and winds down: each role stops, the loaders wait for the
//    copies they issued to land, the MMA thread for its MMAs to complete and the
//    storer for its bulk stores to finish reading, and only then is TMEM released and
//    the CTA retired.  A warp enters every wait converged (after a named barrier, an
//    arrive by all its lanes or a __syncwarp), so its lanes poll the barrier and read the
//    clock together and agree on the answer: the warp-collective TMEM instructions and the
//    named barriers after a wait always see whole warps.
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
// Bound on every wait: 250 ms (legitimate waits take microseconds).  Each kernel also has an
// instantiation for the test hook of the timeout path (kExpire, chosen when Problem::wait_ns
// is 0) in which every wait for another warp's work tests its barrier once and expires if the
// phase is not complete; the waits for hardware the CTA itself started (a TMA load, an MMA),
// which always end, keep the full bound there too.
constexpr uint64_t kRetireNs = 250000000ull;

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

// Two bf16 products (the low and high halves of u times w), rounded to bf16.
__device__ __forceinline__ uint32_t mul_bf16x2(uint32_t u, __nv_bfloat162 w)
{
    __nv_bfloat162 v = __hmul2(*reinterpret_cast<__nv_bfloat162 *>(&u), w);
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

// Hardware barrier among `nthreads` threads (named barrier `id`).  Callers keep their
// control flow uniform -- every participating thread reaches every call, errors or
// not -- so this never waits on a thread that left.
__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t nthreads)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

__device__ __forceinline__ void set_error(int *err, int bit)
{
    if (err) atomicOr(err, bit);
}

// (The two retire helpers run once, at the end of a role; they are kept out of line so that
// the kernels' hot loops keep their register allocation and code layout.)
// Wait for the loads a loader issued into a ring of `stages` slots to land: load i (of
// `issued`) went to slot i % stages, whose barrier bars[first + i % stages] completes phase
// (i / stages) & 1 when it lands.  A loader re-arms a slot only once the slot's consumers
// are done with it, which they are only after its previous load landed, so only the last
// `stages` loads can still be in flight.
__device__ __noinline__ void retire_loads(uint64_t *bars, int first, int stages, int issued, int *err)
{
    for (int i = issued > stages ? issued - stages : 0; i < issued; ++i)
        if (!mbar_wait(smem_u32(&bars[first + i % stages]), (uint32_t)(i / stages) & 1u, kRetireNs)) set_error(err, 1);
}

// Thread 0 of a CTA: wait until *count reaches target; false once about limit_ns has passed
// (0: one test).  The acquire load orders the CTA's later reads (after a barrier) behind the
// writes the count stands for.
__device__ __noinline__ bool wait_count(const unsigned *count, unsigned target, uint64_t limit_ns)
{
    auto ready = [&]() {
        unsigned v;
        asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(count) : "memory");
        return v >= target;
    };
    if (ready()) return true;
    if (limit_ns == 0) return false;
    const long long c0 = clock64(), limit = (long long)(limit_ns * 5 / 2);
    while (!ready()) {
        if (clock64() - c0 > limit) return false;
        __nanosleep(64);
    }
    return true;
}

// The MMA thread: wait until every MMA it issued has completed (a commit to `bar`, used for
// nothing else, arrives once they all have).
__device__ __noinline__ void retire_mmas(uint32_t bar, int *err)
{
    mma_commit(bar);
    if (!mbar_wait(bar, 0, kRetireNs)) set_error(err, 1);
}

// Token index t clamped to the sequence, and whether t holds a token: only a kernel built for
// a ragged last chunk (kRagged) pays for the checks; with whole chunks every t is inside.
template <bool kRagged> __device__ __forceinline__ int64_t clamp_t(int64_t t, int64_t L)
{
    return kRagged ? (t < L ? t : L - 1) : t;
}
template <bool kRagged> __device__ __forceinline__ bool in_seq(int64_t t, int64_t L) { return !kRagged || t < L; }

// ===========================================================================
// chunk_state on tensor cores: the state one super-chunk produces from a zero start.
//   s^T[s][p] = sum_{t in super-chunk m} w_t B_t[s] x_t[p],
//   w_t = dt_t exp2(decay from t to the end of the super-chunk)
//       = dt_t exp2((G_last(k) - G_t) + sum_{k' > k in m} G_last(k')).
// Work unit = (batch, super-chunk m, HG consecutive heads of one B/C group): the heads
// share the B tile, and their scaled x tiles sit side by side as one N = HG*H operand.
// The kernel is persistent: the units' 64-token stages are laid end to end and each
// CTA takes an equal contiguous slice of them, so every SM streams the same number of
// bytes through a 4..8-deep TMA ring.  A slice covers pieces of one or more units; a
// unit cut by a slice boundary is finished by two CTAs that each add their part of the
// sum into s_out (zeroed by the host beforehand), a unit inside one slice is stored.
// MMA: D[s][hh*H + p] (TMEM lanes s) += B^T (A: M = s, K = t, MN-major, the TMA tile of
// B) x (w o X) (B operand: K = t, N = HG*H, MN-major, x tiles scaled in place).
// Warp 0 issues TMA, warp 1 issues MMAs, warps 2..5 scale x and drain the accumulator.
// ===========================================================================
template <int S, int H, int HG>
struct StateCfg {
    static constexpr int kTok = 64;                        // tokens per stage (MMA K per stage)
    static constexpr uint32_t kAtomT = kTok * 128;         // one 64-row x 128-byte swizzled region
    static constexpr int kN = HG * H;                      // MMA N: all heads' p columns
    static constexpr uint32_t kBBytes = (S / 64) * kAtomT;
    static constexpr uint32_t kXBytes = (kN / 64) * kAtomT;
    // G and dt rows of the stage, [2][HG][kTok] f32 (kSideLoad bytes), in a region padded to
    // keep stages 1024-byte aligned
    static constexpr uint32_t kSideLoad = 2 * HG * kTok * 4;
    static constexpr uint32_t kSideBytes = (kSideLoad + 1023) / 1024 * 1024;
    static constexpr uint32_t kStage = kBBytes + kXBytes + kSideBytes;   // a multiple of 1024
    static constexpr int kStages = (204 * 1024) / kStage < 8 ? (204 * 1024) / kStage : 8;
    static constexpr int kMaxR = 256;
    // per chunk k of the unit: sum of G_last over chunks k..R-1, [2 pieces][HG][kMaxR], and a
    // staging copy of the G_last values themselves, [HG][kMaxR]
    static constexpr uint32_t kGl = kStages * kStage;
    static constexpr uint32_t kGraw = kGl + 2 * HG * kMaxR * 4;
    static constexpr uint32_t kBars = kGraw + HG * kMaxR * 4;
    // barriers: full[kStages], free[kStages], x_ready[kStages], done, drained, retire; then the
    // TMEM slot
    static constexpr int kNumBars = 3 * kStages + 3;
    static constexpr uint32_t kSmem = kBars + kNumBars * 8 + 8 + 1024;
    static constexpr uint32_t kCols = (S / 128) * kN;
    static constexpr uint32_t kTmemCols = kCols <= 32 ? 32 : (kCols <= 64 ? 64 : (kCols <= 128 ? 128 : (kCols <= 256 ? 256 : 512)));
    static_assert(kStages >= 4, "TMA ring too shallow");
    static_assert(kStage % 1024 == 0, "stages must keep the 1024-byte swizzle alignment");
};

// (batch, super-chunk, first head) of a chunk_state unit, and the unit's first sequence
// relative to the run being processed.  A unit is HG heads of one group over one
// super-chunk; the run's head groups vary fastest.
struct StateUnit {
    int b, m, h0;
    int64_t rel;         // (b * nh + h0) - first sequence of the run
};

__device__ __forceinline__ StateUnit state_unit(int64_t u, int64_t bhg_lo, int64_t nbhg, int nhq, int HG)
{
    StateUnit r;
    const int64_t rel_g = u % nbhg, bhg = bhg_lo + rel_g;
    r.m = (int)(u / nbhg);
    r.b = (int)(bhg / nhq);
    r.h0 = (int)(bhg % nhq) * HG;
    r.rel = rel_g * HG;
    return r;
}

template <int S, int H, int HG, bool kExpire>
__global__ void __launch_bounds__(192, 1)
k_chunk_state_tc(const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmX,
                 const float *__restrict__ G, const __nv_bfloat16 *__restrict__ dt, const float *__restrict__ dtT,
                 float *__restrict__ s_out, Problem pr, int64_t bhg_lo, int64_t nbhg, int R, int nsup, int nm,
                 int *err)
{
    using Cfg = StateCfg<S, H, HG>;
    constexpr int kN = Cfg::kN, kS = Cfg::kStages, kTok = Cfg::kTok;
    constexpr uint64_t kWait = kExpire ? 0ull : kRetireNs;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    float *sGl = (float *)(smem + Cfg::kGl);
    float *sGraw = (float *)(smem + Cfg::kGraw);
    uint64_t *bars = (uint64_t *)(smem + Cfg::kBars);
    uint32_t *tmem_slot = (uint32_t *)(bars + Cfg::kNumBars);
    constexpr int kFullB = 0, kFreeB = kS, kReadyB = 2 * kS, kDoneB = 3 * kS, kDrainedB = 3 * kS + 1;
    constexpr int kRetireB = 3 * kS + 2;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    const int nhq = (int)(pr.nh / HG);
    const int qpc = (int)(pr.T / kTok);                      // stages per chunk
    const int64_t nq_u = (int64_t)R * qpc;                   // stages per unit (every unit holds R chunks)
    const int64_t total = nbhg * nm * nq_u;
    const int64_t q_lo = total * blockIdx.x / gridDim.x;
    const int64_t q_hi = total * (blockIdx.x + 1) / gridDim.x;
    // staged: the TMA thread also copies each stage's G and dt rows (dt from the float32
    // [b][h][L] copy) into the stage; otherwise every thread loads its row one stage ahead
    const bool staged = dtT != nullptr;

    if (threadIdx.x == 0) {
        for (int i = 0; i < Cfg::kNumBars; ++i)
            mbar_init(smem_u32(&bars[i]), ((i >= kReadyB && i < kDoneB) || i == kDrainedB) ? 128 : 1);
        fence_mbar_init();
    }
    if (warp == 1) { tmem_alloc(smem_u32(tmem_slot), Cfg::kTmemCols); tmem_relinquish(); }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    bool ok = true;
    // the next kernel may launch now; this one reads G (and the states) of the kernels before
    pdl_trigger();
    pdl_wait();

    if (warp == 0) {
        if (lane == 0) {
            prefetch_tmap(&tmB);
            prefetch_tmap(&tmX);
            int issued = 0;
            for (int64_t gq = q_lo; gq < q_hi; ++gq) {
                const int i = (int)(gq - q_lo), st = i % kS;
                // (the MMAs that free a stage wait for its load: free implies landed)
                if (i >= kS && !mbar_wait(smem_u32(&bars[kFreeB + st]), ((i / kS) - 1) & 1, kWait)) {
                    ok = false; set_error(err, 1); break;
                }
                const StateUnit un = state_unit(gq / nq_u, bhg_lo, nbhg, nhq, HG);
                const int g = (int)(un.h0 / pr.hpg);
                const int t0 = (int)((int64_t)un.m * R * pr.T + (gq % nq_u) * kTok);
                uint8_t *base = smem + st * Cfg::kStage;
                const uint32_t full = smem_u32(&bars[kFullB + st]);
                mbar_arrive_expect_tx(full, Cfg::kBBytes + Cfg::kXBytes + (staged ? Cfg::kSideLoad : 0u));
                if (staged) {
                    uint8_t *side = base + Cfg::kBBytes + Cfg::kXBytes;
                    for (int hh = 0; hh < HG; ++hh) {
                        const int64_t row = ((int64_t)un.b * pr.nh + un.h0 + hh) * pr.L + t0;
                        bulk_load(smem_u32(side + hh * kTok * 4), G + row, kTok * 4, full);
                        bulk_load(smem_u32(side + (HG + hh) * kTok * 4), dtT + row, kTok * 4, full);
                    }
                }
                for (int a = 0; a < S / 64; ++a)
                    tma_load_4d(smem_u32(base + a * Cfg::kAtomT), &tmB, full, 64 * a, g, t0, un.b);
                for (int a = 0; a < kN / 64; ++a)   // atom a: head h0 + a / (H/64), columns 64 * (a % (H/64))
                    tma_load_4d(smem_u32(base + Cfg::kBBytes + a * Cfg::kAtomT), &tmX, full, 64 * (a % (H / 64)),
                                un.h0 + a / (H / 64), t0, un.b);
                ++issued;
            }
            retire_loads(bars, kFullB, kS, issued, err);
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16_f32(128, kN, 1, 1);
            int piece = 0;
            for (int64_t gq = q_lo; gq < q_hi; ++gq) {
                const int i = (int)(gq - q_lo), st = i % kS;
                const bool first = gq == q_lo || gq % nq_u == 0;
                const bool last = gq + 1 == q_hi || (gq + 1) % nq_u == 0;
                // a new piece overwrites the accumulator: the previous one must be drained
                if (first && piece > 0 && !mbar_wait(smem_u32(&bars[kDrainedB]), (piece - 1) & 1, kWait)) {
                    ok = false; set_error(err, 1); break;
                }
                if (!mbar_wait(smem_u32(&bars[kReadyB + st]), (i / kS) & 1, kWait)) { ok = false; set_error(err, 1); break; }
                tc_fence_after();
                const uint32_t bbase = smem_u32(smem + st * Cfg::kStage);
                const uint32_t xbase = bbase + Cfg::kBBytes;
                const uint64_t ad0 = smem_desc(bbase, Cfg::kAtomT, 1024), bd0 = smem_desc(xbase, Cfg::kAtomT, 1024);
#pragma unroll
                for (int lb = 0; lb < S / 128; ++lb) {
#pragma unroll
                    for (int kk = 0; kk < kTok / 16; ++kk)
                        mma_bf16(tmem + lb * kN, ad0 + (uint64_t)((lb * 2 * Cfg::kAtomT + kk * 2048) >> 4),
                                 bd0 + (uint64_t)((kk * 2048) >> 4), idesc, (!first || kk > 0) ? 1u : 0u);
                }
                mma_commit(smem_u32(&bars[kFreeB + st]));
                if (last) { mma_commit(smem_u32(&bars[kDoneB])); ++piece; }
            }
            retire_mmas(smem_u32(&bars[kRetireB]), err);
        }
        __syncwarp();
    } else {
        // warps 2..5: scale x rows in place (each head by its own w), then drain the accumulator.
        // All 128 threads walk the same pieces and stages (work is skipped after an error), so
        // the named barrier below is always reached by all of them.
        const int tid = threadIdx.x - 64;
        const int r = 32 * (warp & 3) + lane;       // TMEM lane (state row s in the epilogue)
        const int xr = r & (kTok - 1);              // token row of the stage this thread scales
        const int xc0 = (r / kTok) * 4;             // first of its four 16-byte chunks per row
        const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
        // this row's dt and G for every head, loaded one stage ahead
        float n_dt[HG], n_g[HG];
        auto load_row = [&](int64_t gq) {
            const StateUnit un = state_unit(gq / nq_u, bhg_lo, nbhg, nhq, HG);
            const int64_t t = (int64_t)un.m * R * pr.T + (gq % nq_u) * kTok + xr;
#pragma unroll
            for (int hh = 0; hh < HG; ++hh) {
                n_dt[hh] = __bfloat162float(dt[((int64_t)un.b * pr.L + t) * pr.nh + un.h0 + hh]);
                n_g[hh] = G[((int64_t)un.b * pr.nh + un.h0 + hh) * pr.L + t];
            }
        };
        if (!staged && q_lo < q_hi) load_row(q_lo);
        int piece = 0;
        for (int64_t gq = q_lo; gq < q_hi; ++piece) {
            const int64_t u = gq / nq_u;
            const int64_t p_begin = gq, p_end = q_hi < (u + 1) * nq_u ? q_hi : (u + 1) * nq_u;
            const StateUnit un = state_unit(u, bhg_lo, nbhg, nhq, HG);
            // log2 decay from the end of chunk k to the end of the super-chunk, plus chunk k's own
            // G_last: gl[hh][k] = sum_{k' >= k} G_last(k'), per head (double-buffered by piece)
            float *gl = sGl + (piece & 1) * (HG * Cfg::kMaxR);
            for (int idx = tid; idx < HG * R; idx += 128) {
                const int hh = idx / R, kk = idx % R;
                sGraw[hh * Cfg::kMaxR + kk] =
                    G[((int64_t)un.b * pr.nh + un.h0 + hh) * pr.L + ((int64_t)un.m * R + kk) * pr.T + pr.T - 1];
            }
            named_bar_sync(1, 128);
            for (int idx = tid; idx < HG * R; idx += 128) {
                const int hh = idx / R, kk = idx % R;
                float acc = 0.f;
                for (int k2 = R - 1; k2 >= kk; --k2) acc += sGraw[hh * Cfg::kMaxR + k2];
                gl[hh * Cfg::kMaxR + kk] = acc;
            }
            named_bar_sync(1, 128);
            for (; gq < p_end; ++gq) {
                const int i = (int)(gq - q_lo), st = i % kS;
                float dtr[HG], gr[HG];
                if (!staged) {
#pragma unroll
                    for (int hh = 0; hh < HG; ++hh) { dtr[hh] = n_dt[hh]; gr[hh] = n_g[hh]; }
                    if (gq + 1 < q_hi) load_row(gq + 1);
                }
                const int kl = (int)((gq % nq_u) / qpc);           // chunk index inside the super-chunk
                float lw[HG];                                       // log2 of w / dt, without this row's G
#pragma unroll
                for (int hh = 0; hh < HG; ++hh) lw[hh] = gl[hh * Cfg::kMaxR + kl];
                if (ok && !mbar_wait(smem_u32(&bars[kFullB + st]), (i / kS) & 1, kWait)) { ok = false; set_error(err, 1); }
                if (ok) {
                    if (staged) {
                        const float *side = (const float *)(smem + st * Cfg::kStage + Cfg::kBBytes + Cfg::kXBytes);
#pragma unroll
                        for (int hh = 0; hh < HG; ++hh) { gr[hh] = side[hh * kTok + xr]; dtr[hh] = side[(HG + hh) * kTok + xr]; }
                    }
                    float wr[HG];
#pragma unroll
                    for (int hh = 0; hh < HG; ++hh) wr[hh] = dtr[hh] * exp2f(lw[hh] - gr[hh]);
                    uint8_t *xt = smem + st * Cfg::kStage + Cfg::kBBytes;
                    // w rounded to bf16 and the products taken in bf16 pairs (they are MMA operands,
                    // rounded to bf16 either way)
#pragma unroll
                    for (int a = 0; a < kN / 64; ++a) {
                        const __nv_bfloat162 w2 = __float2bfloat162_rn(wr[a / (H / 64)]);
                        uint4 v[4];
#pragma unroll
                        for (int c = 0; c < 4; ++c) v[c] = *(const uint4 *)(xt + a * Cfg::kAtomT + sw128(xr, xc0 + c));
#pragma unroll
                        for (int c = 0; c < 4; ++c) {
                            uint4 o;
                            o.x = mul_bf16x2(v[c].x, w2);
                            o.y = mul_bf16x2(v[c].y, w2);
                            o.z = mul_bf16x2(v[c].z, w2);
                            o.w = mul_bf16x2(v[c].w, w2);
                            *(uint4 *)(xt + a * Cfg::kAtomT + sw128(xr, xc0 + c)) = o;
                        }
                    }
                    fence_proxy_async_smem();
                    mbar_arrive(smem_u32(&bars[kReadyB + st]));
                }
            }
            // drain the piece: a whole unit is stored, a part of one is added
            const bool whole = p_begin % nq_u == 0 && p_end % nq_u == 0;
            if (ok && !mbar_wait(smem_u32(&bars[kDoneB]), piece & 1, kWait)) { ok = false; set_error(err, 1); }
            if (ok) {
                tc_fence_after();
#pragma unroll
                for (int lb = 0; lb < S / 128; ++lb) {
                    const int s = lb * 128 + r;
#pragma unroll 4
                    for (int c0 = 0; c0 < kN; c0 += 16) {
                        const int hh = c0 / H, p0 = c0 % H;
                        float *dst = s_out + ((un.rel + hh) * nsup + un.m) * (int64_t)(H * S) + s;
                        uint32_t v[16];
                        tmem_ld16(tmem + lane_base + lb * kN + c0, v);
                        tmem_ld_wait();
                        if (whole) {
#pragma unroll
                            for (int j = 0; j < 16; ++j) dst[(int64_t)(p0 + j) * S] = __uint_as_float(v[j]);
                        } else {
#pragma unroll
                            for (int j = 0; j < 16; ++j) atomicAdd(dst + (int64_t)(p0 + j) * S, __uint_as_float(v[j]));
                        }
                    }
                }
                tc_fence_before();
                mbar_arrive(smem_u32(&bars[kDrainedB]));
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
//   P[i][j] = CB[i][j] exp2(G_i - G_j) if j <= i else 0  (CUDA cores; bf16, back into TMEM)
//   Ys      = C h^T                                   (M = i, N = p, K = s)
//   Yi      = P (dt o X)                              (M = i, N = p, K = j; A operand from TMEM)
//   y_i     = exp2(G_i - G_base) Ys_i + Yi_i + D x_i
//   h'^T    = exp2(G_last - G_base) h^T + B^T (w o X),  w_t = dt_t exp2(G_last - G_t)
// The state lives in TMEM as h^T (lanes s, columns p); a bf16 copy [s][p] in shared
// memory is the B operand of Ys.  G is the chunk-relative log2 cumsum; G_base is G
// at the token before the sub-chunk (0 at a chunk start).
//
// Warp roles: warp 0 issues TMA, warp 1 issues every MMA (and owns TMEM).
// Warps 2..5 ("state group") hand the state over between sub-chunks and scale the
// x tile (dt o x in place, w o x into its own tile).  Warps 6..13 ("output group", two warps per TMEM lane quarter
// splitting the columns) build P and write y.  MMA
// issue order per sub-chunk: Ys, state update, Yi, next CB; the state chain therefore
// never waits for P, and the tensor pipe runs Ys and the update while P is built.
// Buffers: C/B tiles in a 2-stage ring (1 stage for S = 256), x tiles in a 4-stage ring
// (3 for S = 256) whose slots also stage y for its bulk tensor store, Ys (S = 128) and
// Yi double-buffered in TMEM so one sub-chunk's epilogue overlaps the next sub-chunk's
// MMAs.  The tensor cores read shared memory at 128 B per clock, the same port TMA and
// the CUDA cores use; P lives in TMEM (the A operand of Yi), which keeps it off that
// port.  y goes through shared memory because a bulk store writes whole lines of it;
// stores from the row-per-lane TMEM layout would touch 32 rows per instruction.
// ===========================================================================
template <int S>
struct ScanCfg {
    static constexpr int kCBStages = (S <= 128) ? 2 : 1;     // C and B tiles
    static constexpr int kXStages = (S <= 128) ? 4 : 3;       // x tiles, then y staging
    static constexpr int kYsBufs = (S <= 128) ? 2 : 1;
    static constexpr uint32_t kCBytes = (S / 64) * kAtom;     // C tile [i][s], K-major
    static constexpr uint32_t kBBytes = (S / 64) * kAtom;     // B tile [j][s]
    static constexpr uint32_t kCBStage = kCBytes + kBBytes;
    static constexpr uint32_t kX = kCBStages * kCBStage;      // x ring: [t][p], 64 p per tile
    static constexpr uint32_t kXw = kX + kXStages * kAtom;    // w o x   [t][p]
    static constexpr uint32_t kH = kXw + kAtom;               // h bf16  [s][p], S rows
    // output group, per column j of the sub-chunk: G_j and 2^(G_blockend - G_j)
    static constexpr uint32_t kSmall = kH + S * 128;
    static constexpr uint32_t kBars = kSmall + 2 * kQ * 4;
    static constexpr uint32_t kSmem = kBars + 256 + 1024;
    // TMEM columns: CB, P (bf16 pairs), Ys buffers, two Yi buffers, state (S/128 blocks of 64)
    static constexpr uint32_t kTcb = 0, kTp = 128, kTys = 192, kTyi = kTys + 64 * kYsBufs, kTds = kTyi + 128;
    static constexpr uint32_t kTmemCols = 512;
    static_assert(kTds + (S / 128) * kPB <= kTmemCols, "TMEM columns");
    static_assert(kSmem <= 227 * 1024, "shared memory");
    static_assert(kXStages <= 4, "x-slot barriers");
};

// kFull/kFree: the C and B tiles of a C/B stage; kIntra0/1: the Yi MMAs into Yi buffer 0/1
// are done; kXFull: an x tile; kYSt: the y staged in an x slot has been read by its bulk
// store (the slot may be reloaded); kRetire: every MMA issued has completed.
enum ScanBar {
    kFull0 = 0, kFree0 = 2, kCb = 4, kHReady, kXReady, kPReady, kIntra0, kIntra1, kUpdate, kEpi0, kEpi1,
    kXFull0, kYSt0 = kXFull0 + 4, kRetire = kYSt0 + 4, kNumScanBars
};

template <int S, bool kRagged, bool kExpire>
__global__ void __launch_bounds__(448, 1)
k_chunk_scan_tc(const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmB,
                const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmY,
                const float *__restrict__ G, const __nv_bfloat16 *__restrict__ dt, const float *__restrict__ Dp,
                const float *__restrict__ h0,
                const float *__restrict__ h_start, float *__restrict__ h_final,
                __nv_bfloat16 *__restrict__ y, Problem pr, ScanSplit sp, int *err)
{
    using Cfg = ScanCfg<S>;
    constexpr int kCBS = Cfg::kCBStages, kXS = Cfg::kXStages;
    constexpr uint64_t kWait = kExpire ? 0ull : kRetireNs;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    float *sG = (float *)(smem + Cfg::kSmall);
    uint64_t *bars = (uint64_t *)(smem + Cfg::kBars);
    uint32_t *tmem_slot = (uint32_t *)(bars + kNumScanBars);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // CTA -> (part, super-chunk m, sequence bh, 64-column block pb), column blocks fastest,
    // then the part's sequences, then m
    // (32-bit: the launcher checks that the CTA count fits)
    const int npb = (int)(pr.H / kPB);
    const int units0 = (int)sp.split * sp.nsup0 * npb;
    const bool part1 = (int)blockIdx.x >= units0;
    int u = part1 ? (int)blockIdx.x - units0 : (int)blockIdx.x;
    const int seq_lo = part1 ? (int)sp.split : 0;
    const int nseq = part1 ? (int)(pr.B * pr.nh - sp.split) : (int)sp.split;
    const int R = part1 ? sp.R1 : sp.R0, nsup = part1 ? sp.nsup1 : sp.nsup0;
    const int pb = u % npb; u /= npb;
    const int bhi = seq_lo + u % nseq;
    const int m = u / nseq;
    const int b = bhi / (int)pr.nh, h = bhi % (int)pr.nh;
    const int g = (int)(h / pr.hpg);
    const int k_begin = m * R;
    const int k_end = min((int)pr.nc, k_begin + R);
    const int qpc = (int)(pr.T / kQ);
    // sub-chunks of this super-chunk that hold tokens (the last chunk of a sequence may be short;
    // its tokens past L are zero-filled by TMA, hold the state (dt = 0) and are not stored)
    const int nq = kRagged ? (int)((min(pr.L, (int64_t)k_end * pr.T) - (int64_t)k_begin * pr.T + kQ - 1) / kQ)
                           : (k_end - k_begin) * qpc;
    const int64_t t_begin = (int64_t)k_begin * pr.T;
    const int64_t bh = bhi;
    const float *Gh = G + bh * pr.L;
    const bool write_final = (m == nsup - 1) && h_final;
    // h_start index of this super-chunk's entering state (used when m >= hs_from)
    const int64_t hs_idx = (part1 ? sp.base1 : 0) + (int64_t)(bhi - seq_lo) * nsup + m;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kNumScanBars; ++i) {
            uint32_t cnt = 1;
            if (i == kHReady || i == kXReady) cnt = 128;                 // state group
            if (i == kPReady || i == kEpi0 || i == kEpi1) cnt = 256;     // output group
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
    // the next kernel may launch now.  A CTA that enters from h0 reads only G of the kernels
    // before, so it waits for the cumsum's CTAs alone (when the launcher passed their count);
    // the others wait for every kernel before (their entering states come last).  G is then
    // read through L2 (__ldcg): it may be written while this grid runs.
    pdl_trigger();
    if (sp.g_count && m < sp.hs_from) {
        if (threadIdx.x == 0 && !wait_count(sp.g_count, sp.g_target, kWait)) set_error(err, 1);
        __syncthreads();
    } else {
        pdl_wait();
    }

    if (warp == 0) {
        // ---- TMA producer ---------------------------------------------------------------
        if (lane == 0) {
            prefetch_tmap(&tmC);
            prefetch_tmap(&tmB);
            prefetch_tmap(&tmX);
            int issued_cb = 0, issued_x = 0;
            for (int q = 0; q < nq && ok; ++q) {
                const int t0 = (int)(t_begin + (int64_t)q * kQ);
                // C and B tiles: free once the MMAs reading them (CB, Ys, state update) are done
                // (those MMAs wait for the tiles: free implies landed)
                const int cs = q % kCBS;
                if (q >= kCBS && !mbar_wait(smem_u32(&bars[kFree0 + cs]), ((q / kCBS) - 1) & 1, kWait)) {
                    ok = false; set_error(err, 1); break;
                }
                uint8_t *base = smem + cs * Cfg::kCBStage;
                const uint32_t full = smem_u32(&bars[kFull0 + cs]);
                mbar_arrive_expect_tx(full, Cfg::kCBStage);
                for (int a = 0; a < S / 64; ++a) {
                    tma_load_4d(smem_u32(base + a * kAtom), &tmC, full, 64 * a, g, t0, b);
                    tma_load_4d(smem_u32(base + Cfg::kCBytes + a * kAtom), &tmB, full, 64 * a, g, t0, b);
                }
                ++issued_cb;
                // x tile: its slot is free once the y staged there kXS sub-chunks ago is stored
                const int xs = q % kXS;
                if (q >= kXS && !mbar_wait(smem_u32(&bars[kYSt0 + xs]), ((q / kXS) - 1) & 1, kWait)) {
                    ok = false; set_error(err, 1); break;
                }
                const uint32_t xfull = smem_u32(&bars[kXFull0 + xs]);
                mbar_arrive_expect_tx(xfull, kAtom);
                tma_load_4d(smem_u32(smem + Cfg::kX + xs * kAtom), &tmX, xfull, pb * kPB, h, t0, b);
                ++issued_x;
            }
            retire_loads(bars, kFull0, kCBS, issued_cb, err);
            retire_loads(bars, kXFull0, kXS, issued_x, err);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ---- MMA issuer -----------------------------------------------------------------
        if (lane == 0) {
            constexpr uint32_t id_cb = idesc_bf16_f32(128, 128, 0, 0);
            constexpr uint32_t id_y = idesc_bf16_f32(128, kPB, 0, 1);
            constexpr uint32_t id_up = idesc_bf16_f32(128, kPB, 1, 1);
            // Descriptors are built once; they advance by byte offsets added to the
            // start-address field (all shared addresses stay below 256 KB).
            auto adv = [](uint64_t d, uint32_t bytes) -> uint64_t { return d + (uint64_t)(bytes >> 4); };
            const uint32_t s0 = smem_u32(smem);
            const uint64_t dC0 = smem_desc(s0, 16, 1024);                          // C [i][s], K-major
            const uint64_t dBk0 = smem_desc(s0 + Cfg::kCBytes, 16, 1024);          // B [j][s], K-major
            const uint64_t dBm0 = smem_desc(s0 + Cfg::kCBytes, kAtom, 1024);       // B^T [s][t], MN-major
            const uint64_t dX0 = smem_desc(s0 + Cfg::kX, kAtom, 1024);             // dt o x [t][p], MN-major
            const uint64_t dH = smem_desc(s0 + Cfg::kH, kAtom, 1024);              // h bf16 [s][p], MN-major
            const uint64_t dXw = smem_desc(s0 + Cfg::kXw, kAtom, 1024);            // w o x [t][p], MN-major
            auto issue_cb = [&](int q) {
                const uint32_t so = (uint32_t)(q % kCBS) * Cfg::kCBStage;
#pragma unroll
                for (int kk = 0; kk < S / 16; ++kk) {
                    const uint32_t off = so + (kk >> 2) * kAtom + (kk & 3) * 32;
                    mma_bf16(tmem + Cfg::kTcb, adv(dC0, off), adv(dBk0, off), id_cb, kk > 0 ? 1u : 0u);
                }
                mma_commit(smem_u32(&bars[kCb]));
            };
            do {
                if (nq == 0) break;
                if (!mbar_wait(smem_u32(&bars[kFull0]), 0, kWait)) { ok = false; break; }
                tc_fence_after();
                issue_cb(0);
                for (int q = 0; q < nq; ++q) {
                    const int cs = q % kCBS, xs = q % kXS;
                    const uint32_t so = (uint32_t)cs * Cfg::kCBStage;
                    const uint32_t ys = Cfg::kTys + (uint32_t)(q % Cfg::kYsBufs) * kPB;
                    const uint32_t yi = Cfg::kTyi + (uint32_t)(q & 1) * kPB;
                    // Ys = C h^T (K = s): needs the state copy and a drained Ys buffer; the state group
                    // arrives kHReady after both (one wait here instead of two)
                    if (!mbar_wait(smem_u32(&bars[kHReady]), q & 1, kWait)) { ok = false; break; }
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < S / 16; ++kk) {
                        const uint32_t off = so + (kk >> 2) * kAtom + (kk & 3) * 32;
                        mma_bf16(tmem + ys, adv(dC0, off), adv(dH, kk * 2048), id_y, kk > 0 ? 1u : 0u);
                    }
                    // state update h^T += B^T (w o X) (K = t) on the state pre-scaled by the state group
                    if (!mbar_wait(smem_u32(&bars[kXReady]), q & 1, kWait)) { ok = false; break; }
                    tc_fence_after();
                    if (q + 1 < nq || write_final) {
#pragma unroll
                        for (int lb = 0; lb < S / 128; ++lb) {
#pragma unroll
                            for (int kk = 0; kk < kQ / 16; ++kk)
                                mma_bf16(tmem + Cfg::kTds + lb * kPB, adv(dBm0, so + lb * 2 * kAtom + kk * 2048),
                                         adv(dXw, kk * 2048), id_up, 1u);
                        }
                        mma_commit(smem_u32(&bars[kUpdate]));
                    }
                    mma_commit(smem_u32(&bars[kFree0 + cs]));     // CB, Ys and the update have read C and B
                    // Yi = D x + P (dt o X) (K = j), P from TMEM: the state group stored D x in the accumulator
                    if (!mbar_wait(smem_u32(&bars[kPReady]), q & 1, kWait)) { ok = false; break; }
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < kQ / 16; ++kk)
                        mma_bf16_ts(tmem + yi, tmem + Cfg::kTp + 8 * kk, adv(dX0, xs * kAtom + kk * 2048), id_y, 1u);
                    mma_commit(smem_u32(&bars[kIntra0 + (q & 1)]));
                    // next CB: the output group has read this one (P is built); with two C/B stages it
                    // arrived kPReady only after the next sub-chunk's C and B tiles had landed.  With
                    // one stage those tiles load only after this sub-chunk's update, which waits on the
                    // epilogue the output group runs after kPReady, so this thread waits for them.
                    if (q + 1 < nq) {
                        if (kCBS == 1) {
                            if (!mbar_wait(smem_u32(&bars[kFull0]), (q + 1) & 1, kWait)) { ok = false; break; }
                            tc_fence_after();
                        }
                        issue_cb(q + 1);
                    }
                }
            } while (0);
            if (!ok) set_error(err, 1);
            retire_mmas(smem_u32(&bars[kRetire]), err);
        }
        __syncwarp();
    } else if (warp < 6) {
        // ---- state group: state hand-off and x scaling ------------------------------------
        const float dh = Dp[h];
        const int r = 32 * (warp & 3) + lane;          // TMEM lane = tile row / state row
        const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
        uint8_t *xw = smem + Cfg::kXw;
        uint8_t *ht = smem + Cfg::kH;
        // per-sub-chunk scalars, loaded one sub-chunk ahead
        float n_gr = 0.f, n_dt = 0.f, n_glast = 0.f, n_gbase = 0.f;
        auto load_scalars = [&](int q) {
            const int64_t t0 = t_begin + (int64_t)q * kQ;
            const int64_t tr = clamp_t<kRagged>(t0 + r, pr.L), tl = clamp_t<kRagged>(t0 + kQ - 1, pr.L);
            n_gr = __ldcg(Gh + tr);
            n_dt = in_seq<kRagged>(t0 + r, pr.L) ? __bfloat162float(dt[((int64_t)b * pr.L + t0 + r) * pr.nh + h]) : 0.f;
            n_glast = __ldcg(Gh + tl);
            n_gbase = (q % qpc == 0) ? 0.f : __ldcg(Gh + t0 - 1);
        };
        if (nq > 0) load_scalars(0);
        for (int q = 0; q < nq && ok; ++q) {
            const int xs = q % kXS;
            const float gr = n_gr, dtr = n_dt, glast = n_glast, gbase = n_gbase;
            if (q + 1 < nq) load_scalars(q + 1);

            // h (fp32) -> bf16 copy [s][p] for Ys, and h * exp2(glast - gbase) back to TMEM
            {
                const float dec = exp2f(glast - gbase);
                if (q > 0) {
                    if (!mbar_wait(smem_u32(&bars[kUpdate]), (q - 1) & 1, kWait)) { ok = false; set_error(err, 1); break; }
                    tc_fence_after();
                }
#pragma unroll
                for (int lb = 0; lb < S / 128; ++lb) {
                    const int s = lb * 128 + r;
                    uint32_t v[64];
                    if (q == 0) {
                        // entering state: h0 (zeros if absent) for super-chunks m < hs_from, else h_start
                        const float *src = (m < sp.hs_from) ? (h0 ? h0 + bh * (int64_t)(pr.H * S) : nullptr)
                                                            : h_start + hs_idx * (int64_t)(pr.H * S);
                        if (src) {
                            src += (int64_t)(pb * kPB) * S + s;
#pragma unroll
                            for (int j = 0; j < 64; ++j) v[j] = __float_as_uint(src[(int64_t)j * S]);
                        } else {
#pragma unroll
                            for (int j = 0; j < 64; ++j) v[j] = 0u;
                        }
                    } else {
                        const uint32_t ta = tmem + lane_base + Cfg::kTds + lb * kPB;
                        tmem_ld16(ta + 0, *reinterpret_cast<uint32_t(*)[16]>(&v[0]));
                        tmem_ld16(ta + 16, *reinterpret_cast<uint32_t(*)[16]>(&v[16]));
                        tmem_ld16(ta + 32, *reinterpret_cast<uint32_t(*)[16]>(&v[32]));
                        tmem_ld16(ta + 48, *reinterpret_cast<uint32_t(*)[16]>(&v[48]));
                        tmem_ld_wait();
                    }
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        uint4 o;
                        o.x = pack_bf16x2(__uint_as_float(v[8 * c + 0]), __uint_as_float(v[8 * c + 1]));
                        o.y = pack_bf16x2(__uint_as_float(v[8 * c + 2]), __uint_as_float(v[8 * c + 3]));
                        o.z = pack_bf16x2(__uint_as_float(v[8 * c + 4]), __uint_as_float(v[8 * c + 5]));
                        o.w = pack_bf16x2(__uint_as_float(v[8 * c + 6]), __uint_as_float(v[8 * c + 7]));
                        *(uint4 *)(ht + sw128(s, c)) = o;
                    }
#pragma unroll
                    for (int j = 0; j < 64; ++j) v[j] = __float_as_uint(__uint_as_float(v[j]) * dec);
                    const uint32_t ta = tmem + lane_base + Cfg::kTds + lb * kPB;
                    tmem_st16(ta + 0, *reinterpret_cast<uint32_t(*)[16]>(&v[0]));
                    tmem_st16(ta + 16, *reinterpret_cast<uint32_t(*)[16]>(&v[16]));
                    tmem_st16(ta + 32, *reinterpret_cast<uint32_t(*)[16]>(&v[32]));
                    tmem_st16(ta + 48, *reinterpret_cast<uint32_t(*)[16]>(&v[48]));
                }
                tmem_st_wait();
                fence_proxy_async_smem();
                // the Ys buffer this sub-chunk writes is drained once the epilogue of sub-chunk
                // q - kYsBufs has read it (and, kYsBufs <= 2, so is the Yi buffer of sub-chunk q:
                // the epilogues arrive in order)
                if (q >= Cfg::kYsBufs) {
                    const int e = q - Cfg::kYsBufs;
                    if (!mbar_wait(smem_u32(&bars[kEpi0 + (e & 1)]), (e >> 1) & 1, kWait)) {
                        ok = false; set_error(err, 1); break;
                    }
                }
                tc_fence_before();
                mbar_arrive(smem_u32(&bars[kHReady]));
            }
            // x tile: dt o x in place (Yi operand), w o x into the Xw tile (state-update operand),
            // and D x into this sub-chunk's Yi accumulator (the Yi MMAs accumulate on top of it)
            {
                if (!mbar_wait(smem_u32(&bars[kXFull0 + xs]), (q / kXS) & 1, kWait)) { ok = false; set_error(err, 1); break; }
                // (the Yi buffer of this sub-chunk was drained before kHReady, above)
                tc_fence_after();
                uint8_t *xt = smem + Cfg::kX + xs * kAtom;
                const float wr = dtr * exp2f(glast - gr);
                const uint32_t tyi = tmem + lane_base + Cfg::kTyi + (uint32_t)(q & 1) * kPB;
#pragma unroll
                for (int cp = 0; cp < 4; ++cp) {
                    uint32_t dx[16];
#pragma unroll
                    for (int ch = 0; ch < 2; ++ch) {
                        const int c = 2 * cp + ch;
                        const uint32_t off = sw128(r, c);
                        const uint4 v = *(const uint4 *)(xt + off);
                        const uint32_t in[4] = {v.x, v.y, v.z, v.w};
                        uint32_t os[4], ow[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float2 f = unpack_bf16x2(in[e]);
                            os[e] = pack_bf16x2(f.x * dtr, f.y * dtr);
                            ow[e] = pack_bf16x2(f.x * wr, f.y * wr);
                            dx[8 * ch + 2 * e] = __float_as_uint(dh * f.x);
                            dx[8 * ch + 2 * e + 1] = __float_as_uint(dh * f.y);
                        }
                        *(uint4 *)(xt + off) = make_uint4(os[0], os[1], os[2], os[3]);
                        *(uint4 *)(xw + off) = make_uint4(ow[0], ow[1], ow[2], ow[3]);
                    }
                    tmem_st16(tyi + 16 * cp, dx);
                }
                tmem_st_wait();
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(smem_u32(&bars[kXReady]));
            }
        }
        // final state of the sequence, from the last super-chunk of each (batch, head)
        if (ok && write_final && nq > 0) {
            if (!mbar_wait(smem_u32(&bars[kUpdate]), (nq - 1) & 1, kWait)) { ok = false; set_error(err, 1); }
            if (ok) {
                tc_fence_after();
#pragma unroll
                for (int lb = 0; lb < S / 128; ++lb) {
                    const int s = lb * 128 + r;
                    float *dst = h_final + bh * (int64_t)(pr.H * S) + (int64_t)(pb * kPB) * S + s;
#pragma unroll
                    for (int c0 = 0; c0 < kPB; c0 += 16) {
                        uint32_t v[16];
                        tmem_ld16(tmem + lane_base + Cfg::kTds + lb * kPB + c0, v);
                        tmem_ld_wait();
#pragma unroll
                        for (int j = 0; j < 16; ++j) dst[(int64_t)(c0 + j) * S] = __uint_as_float(v[j]);
                    }
                }
            }
        }
    } else {
        // ---- output group: P and y (8 warps: two per TMEM lane quarter, splitting columns) --------
        const int half = (warp - 6) >> 2;              // 0 or 1: which half of the columns
        const int r = 32 * (warp & 3) + lane;          // TMEM lane = tile row i
        const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
        const int wrow_lo = 32 * (warp & 3), wrow_hi = wrow_lo + 31;   // rows of this warp
        const bool storer = warp == 6 && lane == 0;    // issues the bulk stores of y
        // column arrays of the current sub-chunk
        float *cG = sG, *cF = cG + kQ;
        // the 256 output-group threads run every iteration (work is skipped after an error),
        // so the named barrier below is always reached by all of them
        auto group_sync = [&]() { named_bar_sync(1, 256); };
        float n_gr = 0.f, n_gend = 0.f, n_gbase = 0.f;
        auto load_scalars = [&](int q) {
            const int64_t t0 = t_begin + (int64_t)q * kQ;
            n_gr = __ldcg(Gh + clamp_t<kRagged>(t0 + r, pr.L));
            n_gend = __ldcg(Gh + clamp_t<kRagged>(t0 + (r | 15), pr.L));  // G at the end of row r's 16-token block
            n_gbase = (q % qpc == 0) ? 0.f : __ldcg(Gh + t0 - 1);
        };
        // Software-pipelined by one sub-chunk: iteration q builds P of sub-chunk q + 1, then
        // writes y of sub-chunk q.  The MMAs of q + 1 wait on that P, while the y of q waits
        // only on the Yi MMAs of q, which run meanwhile.
        float gr_y = 0.f, gbase_y = 0.f;               // scalars of the sub-chunk whose y is next
        if (nq > 0) load_scalars(0);
        for (int q = -1; q < nq; ++q) {
            float gr_p = gr_y, gbase_p = gbase_y;
            if (q + 1 < nq) {
                const int qp = q + 1;                      // the sub-chunk whose P is built
                const float gr = n_gr, gend = n_gend;
                gr_p = n_gr;
                gbase_p = n_gbase;
                if (half == 0) {
                    cG[r] = gr;
                    cF[r] = ex2_approx(gend - gr);          // 2^(G_blockend - G_j) <= 1 for A dt >= 0
                }
                group_sync();
                if (qp + 1 < nq) load_scalars(qp + 1);

                // P[i][j] = CB[i][j] 2^(G_i - G_j) for j <= i, else 0, as bf16 pairs in TMEM (the
                // A operand of Yi).  Blocks of 16 columns entirely left of this warp's rows use the
                // factored form 2^(G_i - G_e) 2^(G_e - G_j) (G_e = G at the block's last column; both
                // factors <= 1); blocks that meet the diagonal evaluate 2^(G_i - G_j) per element.
                // (the CB of qp is issued after the Yi of q, the last reader of the single P buffer)
                if (ok && !mbar_wait(smem_u32(&bars[kCb]), qp & 1, kWait)) { ok = false; set_error(err, 1); }
                if (ok) {
                    tc_fence_after();
                    const int jh = 64 * half;
                    const uint32_t ta = tmem + lane_base + Cfg::kTcb + jh;
                    const uint32_t tp = tmem + lane_base + Cfg::kTp + 32 * half;
                    // one 16-column block per iteration (a compact loop body: the four warp roles
                    // share each sub-partition's instruction cache)
#pragma unroll 1
                    for (int blk = 0; blk < 4; ++blk) {
                        const int j0 = jh + 16 * blk;
                        uint32_t pk[8];
                        if (j0 > wrow_hi) {                           // above the diagonal for the whole warp
#pragma unroll
                            for (int e = 0; e < 8; ++e) pk[e] = 0u;
                        } else {
                            uint32_t v[16];
                            tmem_ld16(ta + 16 * blk, v);
                            tmem_ld_wait();
                            float f[16];
                            if (j0 + 15 < wrow_lo) {                  // left of every row of the warp: factored
                                const float ei = ex2_approx(gr - cG[j0 + 15]);
                                const float4 *f4 = reinterpret_cast<const float4 *>(cF + j0);
#pragma unroll
                                for (int e4 = 0; e4 < 4; ++e4) {
                                    const float4 fj = f4[e4];
                                    f[4 * e4 + 0] = __uint_as_float(v[4 * e4 + 0]) * ei * fj.x;
                                    f[4 * e4 + 1] = __uint_as_float(v[4 * e4 + 1]) * ei * fj.y;
                                    f[4 * e4 + 2] = __uint_as_float(v[4 * e4 + 2]) * ei * fj.z;
                                    f[4 * e4 + 3] = __uint_as_float(v[4 * e4 + 3]) * ei * fj.w;
                                }
                            } else {                                  // meets the diagonal: exact, selected
                                const float4 *g4 = reinterpret_cast<const float4 *>(cG + j0);
#pragma unroll
                                for (int e4 = 0; e4 < 4; ++e4) {
                                    const float4 gj = g4[e4];
                                    const float gjs[4] = {gj.x, gj.y, gj.z, gj.w};
#pragma unroll
                                    for (int c = 0; c < 4; ++c) {
                                        const int e = 4 * e4 + c, j = j0 + e;
                                        const float val = __uint_as_float(v[e]) * ex2_approx(gr - gjs[c]);
                                        f[e] = (j <= r) ? val : 0.f;
                                    }
                                }
                            }
#pragma unroll
                            for (int e = 0; e < 8; ++e) pk[e] = pack_bf16x2(f[2 * e], f[2 * e + 1]);
                        }
                        tmem_st8(tp + 8 * blk, pk);
                    }
                    tmem_st_wait();
                    // the MMA warp issues the next CB right after kPReady: one warp checks that its
                    // C and B tiles have landed (the stage cannot be reloaded before this arrival)
                    if (kCBS > 1 && warp == 6 && qp + 1 < nq &&
                        !mbar_wait(smem_u32(&bars[kFull0 + (qp + 1) % kCBS]), ((qp + 1) / kCBS) & 1, kWait)) {
                        ok = false; set_error(err, 1);
                    }
                    tc_fence_before();
                    mbar_arrive(smem_u32(&bars[kPReady]));
                }
            }
            // y = 2^(G_i - G_base) Ys + Yi   (Yi already holds D x; this thread: 32 columns).
            // y is staged in this sub-chunk's x slot (its last reader, the Yi MMA, has completed)
            // in the same swizzled [t][p] layout, then written by one bulk tensor store.
            const int64_t t0 = t_begin + (int64_t)q * kQ;
            const int xs = (q + kXS) % kXS;
            const float gr = gr_y, gbase = gbase_y;
            uint8_t *ystage = smem + Cfg::kX + xs * kAtom;
            if (q >= 0 && ok && !mbar_wait(smem_u32(&bars[kIntra0 + (q & 1)]), (q >> 1) & 1, kWait)) {
                ok = false; set_error(err, 1);
            }
            if (q >= 0 && ok) {
                tc_fence_after();
                const float eg = ex2_approx(gr - gbase);
                const uint32_t c0 = 32 * half;
                const uint32_t ys = Cfg::kTys + (uint32_t)(q % Cfg::kYsBufs) * kPB + c0;
                const uint32_t yi = Cfg::kTyi + (uint32_t)(q & 1) * kPB + c0;
                // 16 columns per iteration (compact loop body, as above)
#pragma unroll 1
                for (int c16 = 0; c16 < 32; c16 += 16) {
                    uint32_t vs[16], vi[16];
                    tmem_ld16(tmem + lane_base + ys + c16, vs);
                    tmem_ld16(tmem + lane_base + yi + c16, vi);
                    tmem_ld_wait();
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        uint32_t o[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int k = 8 * c + 2 * e;
                            o[e] = pack_bf16x2(fmaf(eg, __uint_as_float(vs[k]), __uint_as_float(vi[k])),
                                               fmaf(eg, __uint_as_float(vs[k + 1]), __uint_as_float(vi[k + 1])));
                        }
                        *(uint4 *)(ystage + sw128(r, 4 * half + (c16 >> 3) + c)) = make_uint4(o[0], o[1], o[2], o[3]);
                    }
                }
                tc_fence_before();
                mbar_arrive(smem_u32(&bars[kEpi0 + (q & 1)]));
                fence_proxy_async_smem();
            }
            // all rows staged (and the column arrays free for the next sub-chunk)
            group_sync();
            if (storer && q >= 0 && ok) {
                // the store of sub-chunk q stays in flight; the slot of sub-chunk q - 1 is
                // released once its store has read it.  After an error no slot is released:
                // its load may still be in flight, and the loader, whose wait then expires,
                // must not re-arm it
                tma_store_4d(&tmY, smem_u32(ystage), pb * kPB, h, (int)t0, b);
                bulk_commit();
                bulk_wait_read_1();
                if (q > 0) mbar_arrive(smem_u32(&bars[kYSt0 + (q - 1) % kXS]));
            }
            gr_y = gr_p;
            gbase_y = gbase_p;
        }
        if (storer) {
            bulk_wait_all();
            if (nq > 0 && ok) mbar_arrive(smem_u32(&bars[kYSt0 + (nq - 1) % kXS]));
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) tmem_dealloc(tmem, Cfg::kTmemCols);
}

// ===========================================================================
// chunk_scan on tensor cores, two heads of one B/C group per CTA (S = 128, H = 64).
// Same arithmetic as k_chunk_scan_tc; the two heads share every C and B tile, one
// C B^T product, and the N = 128 MMAs of the state product and the state update:
//   CB        = C B^T                                   (M = i, N = j, K = s; shared)
//   P_h[i][j] = CB[i][j] exp2(G_h,i - G_h,j) dt_h,j  if j <= i, else 0
//             (built by the CUDA cores over CB in place: block k of 16 columns
//              holds P_A of that block in its first 8 columns, P_B in the last 8)
//   Y         = C [h_A^T | h_B^T]                       (M = i, N = 2 x 64 p, K = s)
//   Y_h,i    <- exp2(G_h,i - G_h,base) Y_h,i              (CUDA cores, in TMEM)
//   Y_h      += P_h x_h                                 (M = i, N = 64, K = j; A from TMEM)
//   y_h       = Y_h + D_h x_h (bf16)
//   [h_A^T | h_B^T] <- decayed state + B^T [w_A o x_A | w_B o x_B]   (M = s, N = 128, K = t)
// Folding dt_j into P leaves the raw x tile as the B operand of P x, so the CUDA cores
// write one scaled copy of x (w o x, for the update); the epilogue reads the raw tile
// once more for D x.  The CUDA-core arithmetic runs on pairs (bf16x2 for w o x,
// float32x2 elsewhere): it is the bulk of the issued instructions.  Scaling C h^T in place before P x
// accumulates onto it lets one accumulator per sub-chunk hold y, so two of them fit in
// TMEM and the next sub-chunk's C h^T never waits for this one's epilogue.
// MMA issue order per sub-chunk: C h^T, update, P x, next CB.  The state chain (update ->
// hand-off -> w o x -> update) waits on nothing else, and the C/B stage is free for the
// next tiles once the update has read it.
// TMEM (512 columns): CB / P 0..127, Y buffers 128..255 and 256..383 (sub-chunk q in
// buffer q % 2; head A then head B), state 384..511 (h_A^T then h_B^T; lanes = s).
// Shared memory: one C/B stage, x in a 3-slot ring (the slots also stage y for its bulk
// stores), w o x, the bf16 state copy.
// Warps: 0 loads C and B, 14 loads x, 1 issues MMAs, 2..5 hand the state over and write
// w o x, 6..13 build P and scale C h^T (two warps per TMEM lane quarter, one per 64
// columns / head), 15..18 write y and issue its bulk stores.
// ===========================================================================
struct PairCfg {
    static constexpr int kXStages = 3;
    static constexpr uint32_t kCBytes = 2 * kAtom;             // C tile [i][s], K-major (2 atoms of 64 s)
    static constexpr uint32_t kCBStage = 4 * kAtom;            // C then B [j][s]
    static constexpr uint32_t kX = kCBStage;                   // x ring: per slot [head][t][p]
    static constexpr uint32_t kXSlot = 2 * kAtom;
    static constexpr uint32_t kWx = kX + kXStages * kXSlot;    // w o x, [head][t][p]
    static constexpr uint32_t kHc = kWx + 2 * kAtom;           // bf16 state copy, [head][s][p]
    // per head, for the columns j of the sub-chunk being built: Gd_j = G_j - log2 dt_j,
    // F_j = 2^(G_e - G_j) dt_j (G_e: G at the end of j's 16-column block) and the 8
    // block-end values G_e
    static constexpr uint32_t kArrHead = (2 * kQ + 8) * 4;
    static constexpr uint32_t kArr = kHc + 2 * kAtom;
    static constexpr uint32_t kBars = kArr + 2 * kArrHead;
    static constexpr int kNumBars = 19;
    static constexpr uint32_t kSmem = kBars + kNumBars * 8 + 8;
    static constexpr uint32_t kTcb = 0, kTy = 128, kTst = 384, kTmemCols = 512;
    static constexpr int kThreads = 608;
    static_assert(kSmem <= 227 * 1024, "shared memory");
};

// pFull/pFree: the C/B stage (loaded / read by CB, the update and C h^T); pYs: C h^T of
// the sub-chunk done; pIntra0/1: P x into Y buffer 0/1 done; pEpi0/1: Y buffer 0/1
// drained; pXFull/pYSt: x slots (loaded / the y store has read the slot); pRetire: every
// MMA issued has completed.  Every barrier a role waits on by parity is one its own
// progress keeps within one phase of the wait.
enum PairBar {
    pFull = 0, pFree, pCb, pYs, pHReady, pXReady, pPReady, pIntra0, pIntra1, pUpdate, pEpi0, pEpi1,
    pXFull0, pYSt0 = pXFull0 + 3, pRetire = pYSt0 + 3
};
static_assert(pRetire + 1 == PairCfg::kNumBars, "pair barriers");

template <bool kRagged, bool kExpire>
__global__ void __launch_bounds__(PairCfg::kThreads, 1)
k_chunk_scan_pair(const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmB,
                  const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmY,
                  const float *__restrict__ G, const __nv_bfloat16 *__restrict__ dt, const float *__restrict__ Dp,
                  const float *__restrict__ h0, const float *__restrict__ h_start, float *__restrict__ h_final,
                  Problem pr, ScanSplit sp, int *err)
{
    using Cfg = PairCfg;
    constexpr int S = 128, kXS = Cfg::kXStages;
    constexpr uint64_t kWait = kExpire ? 0ull : kRetireNs;
    // the swizzled tiles need a 1024-byte aligned base; the whole budget is used, so the
    // base is not re-aligned here: a misaligned base is reported and nothing runs
    extern __shared__ __align__(1024) uint8_t smem[];
    if (smem_u32(smem) & 1023u) {
        if (threadIdx.x == 0) set_error(err, 4);
        return;
    }
    uint64_t *bars = (uint64_t *)(smem + Cfg::kBars);
    uint32_t *tmem_slot = (uint32_t *)(bars + Cfg::kNumBars);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // CTA -> (part, super-chunk m, head pair), pairs fastest
    const int64_t nseq_all = pr.B * pr.nh;
    const int units0 = (int)(sp.split / 2) * sp.nsup0;
    const bool part1 = (int)blockIdx.x >= units0;
    const int u = part1 ? (int)blockIdx.x - units0 : (int)blockIdx.x;
    const int seq_lo = part1 ? (int)sp.split : 0;
    const int npair = part1 ? (int)((nseq_all - sp.split) / 2) : (int)(sp.split / 2);
    const int nsup = part1 ? sp.nsup1 : sp.nsup0, R = part1 ? sp.R1 : sp.R0;
    const int bhA = seq_lo + 2 * (u % npair);
    const int m = u / npair;
    const int b = bhA / (int)pr.nh, hA = bhA % (int)pr.nh;
    const int g = (int)(hA / pr.hpg);
    const int k_begin = m * R;
    const int k_end = min((int)pr.nc, k_begin + R);
    const int qpc = (int)(pr.T / kQ);
    // sub-chunks of this super-chunk that hold tokens (the last chunk of a sequence may be short;
    // its tokens past L are zero-filled by TMA, hold the state (dt = 0) and are not stored)
    const int nq = kRagged ? (int)((min(pr.L, (int64_t)k_end * pr.T) - (int64_t)k_begin * pr.T + kQ - 1) / kQ)
                           : (k_end - k_begin) * qpc;
    const int64_t t_begin = (int64_t)k_begin * pr.T;
    const float *GA = G + (int64_t)bhA * pr.L, *GB = GA + pr.L;
    const bool write_final = (m == nsup - 1) && h_final;
    const int64_t hs_idx = (part1 ? sp.base1 : 0) + (int64_t)(bhA - seq_lo) * nsup + m;   // head A; head B: + nsup

    if (threadIdx.x == 0) {
        for (int i = 0; i < Cfg::kNumBars; ++i) {
            uint32_t cnt = 1;
            if (i == pHReady || i == pXReady) cnt = 128;
            if (i == pEpi0 || i == pEpi1) cnt = 128;
            if (i == pPReady) cnt = 256;
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
    // the next kernel may launch now.  A CTA that enters from h0 reads only G of the kernels
    // before, so it waits for the cumsum's CTAs alone (when the launcher passed their count);
    // the others wait for every kernel before (their entering states come last).  G is then
    // read through L2 (__ldcg): it may be written while this grid runs.
    pdl_trigger();
    if (sp.g_count && m < sp.hs_from) {
        if (threadIdx.x == 0 && !wait_count(sp.g_count, sp.g_target, kWait)) set_error(err, 1);
        __syncthreads();
    } else {
        pdl_wait();
    }

    if (warp == 0) {
        // ---- C and B tiles (one stage: free once CB, the update and C h^T have read it) -------
        if (lane == 0) {
            prefetch_tmap(&tmC);
            prefetch_tmap(&tmB);
            int issued = 0;
            for (int q = 0; q < nq; ++q) {
                const int t0 = (int)(t_begin + (int64_t)q * kQ);
                // (the MMAs that free the stage wait for its load: free implies landed)
                if (q >= 1 && !mbar_wait(smem_u32(&bars[pFree]), (q - 1) & 1, kWait)) {
                    set_error(err, 1); break;
                }
                const uint32_t full = smem_u32(&bars[pFull]);
                mbar_arrive_expect_tx(full, Cfg::kCBStage);
                for (int a = 0; a < 2; ++a) {
                    tma_load_4d(smem_u32(smem + a * kAtom), &tmC, full, 64 * a, g, t0, b);
                    tma_load_4d(smem_u32(smem + Cfg::kCBytes + a * kAtom), &tmB, full, 64 * a, g, t0, b);
                }
                // the tiles two sub-chunks ahead into L2: the single stage reloads right after the
                // update and C h^T have read it, so its load latency is on the critical path
                if (q + 2 < nq) {
                    for (int a = 0; a < 2; ++a) {
                        tma_prefetch_4d(&tmC, 64 * a, g, t0 + 2 * kQ, b);
                        tma_prefetch_4d(&tmB, 64 * a, g, t0 + 2 * kQ, b);
                    }
                }
                ++issued;
            }
            retire_loads(bars, pFull, 1, issued, err);
        }
        __syncwarp();
    } else if (warp == 14) {
        // ---- x tiles of both heads (slot of sub-chunk q: free once y of q - 3 is stored) ------
        if (lane == 0) {
            // the entering states of both heads into L2 first: the first hand-off reads them
            // with strided loads, one head after the other
            for (int hh = 0; hh < 2; ++hh) {
                const float *src = (m < sp.hs_from) ? (h0 ? h0 + (int64_t)(bhA + hh) * (pr.H * S) : nullptr)
                                                    : h_start + (hs_idx + hh * nsup) * (int64_t)(pr.H * S);
                // (h0 need only be 4-byte aligned; a bulk prefetch needs 16)
                if (src && nq > 0 && ((uintptr_t)src & 15u) == 0)
                    bulk_prefetch_l2(src, (uint32_t)(pr.H * S * sizeof(float)));
            }
            prefetch_tmap(&tmX);
            int issued = 0;
            for (int q = 0; q < nq; ++q) {
                const int t0 = (int)(t_begin + (int64_t)q * kQ);
                const int xs = q % kXS;
                if (q >= kXS && !mbar_wait(smem_u32(&bars[pYSt0 + xs]), ((q / kXS) - 1) & 1, kWait)) {
                    set_error(err, 1); break;
                }
                const uint32_t xfull = smem_u32(&bars[pXFull0 + xs]);
                mbar_arrive_expect_tx(xfull, Cfg::kXSlot);
                for (int hh = 0; hh < 2; ++hh)
                    tma_load_4d(smem_u32(smem + Cfg::kX + xs * Cfg::kXSlot + hh * kAtom), &tmX, xfull, 0, hA + hh,
                                t0, b);
                ++issued;
            }
            retire_loads(bars, pXFull0, kXS, issued, err);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ---- MMA issuer -----------------------------------------------------------------
        if (lane == 0) {
            constexpr uint32_t id_cb = idesc_bf16_f32(128, 128, 0, 0);
            constexpr uint32_t id_ys = idesc_bf16_f32(128, 128, 0, 1);
            constexpr uint32_t id_up = idesc_bf16_f32(128, 128, 1, 1);
            constexpr uint32_t id_yi = idesc_bf16_f32(128, 64, 0, 1);
            auto adv = [](uint64_t d, uint32_t bytes) -> uint64_t { return d + (uint64_t)(bytes >> 4); };
            const uint32_t s0 = smem_u32(smem);
            const uint64_t dC = smem_desc(s0, 16, 1024);                        // C [i][s], K-major
            const uint64_t dBk = smem_desc(s0 + Cfg::kCBytes, 16, 1024);        // B [j][s], K-major
            const uint64_t dBm = smem_desc(s0 + Cfg::kCBytes, kAtom, 1024);     // B^T [s][t], MN-major
            const uint64_t dX = smem_desc(s0 + Cfg::kX, kAtom, 1024);           // x [t][p], MN-major
            const uint64_t dHc = smem_desc(s0 + Cfg::kHc, kAtom, 1024);         // h bf16 [s][p], 2 atoms along N
            const uint64_t dWx = smem_desc(s0 + Cfg::kWx, kAtom, 1024);         // w o x [t][p], 2 atoms along N
            auto issue_cb = [&]() {
#pragma unroll
                for (int kk = 0; kk < S / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * kAtom + (kk & 3) * 32;
                    mma_bf16(tmem + Cfg::kTcb, adv(dC, off), adv(dBk, off), id_cb, kk > 0 ? 1u : 0u);
                }
                mma_commit(smem_u32(&bars[pCb]));
            };
            do {
                if (nq == 0) break;
                if (!mbar_wait(smem_u32(&bars[pFull]), 0, kWait)) { ok = false; break; }
                tc_fence_after();
                issue_cb();
                for (int q = 0; q < nq; ++q) {
                    const int xs = q % kXS;
                    const uint32_t ty = tmem + Cfg::kTy + (uint32_t)(q & 1) * 128;
                    // C [h_A^T | h_B^T] into Y buffer q % 2 (drained by the epilogue of q - 2), from the
                    // bf16 state copy of the hand-off
                    if (!mbar_wait(smem_u32(&bars[pHReady]), q & 1, kWait) ||
                        (q >= 2 && !mbar_wait(smem_u32(&bars[pEpi0 + (q & 1)]), ((q - 2) >> 1) & 1, kWait))) {
                        ok = false; break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < S / 16; ++kk) {
                        const uint32_t off = (kk >> 2) * kAtom + (kk & 3) * 32;
                        mma_bf16(ty, adv(dC, off), adv(dHc, kk * 2048), id_ys, kk > 0 ? 1u : 0u);
                    }
                    mma_commit(smem_u32(&bars[pYs]));
                    // update on the state the state warps decayed, with their w o x
                    if (!mbar_wait(smem_u32(&bars[pXReady]), q & 1, kWait)) { ok = false; break; }
                    tc_fence_after();
                    if (q + 1 < nq || write_final) {
#pragma unroll
                        for (int kk = 0; kk < kQ / 16; ++kk)
                            mma_bf16(tmem + Cfg::kTst, adv(dBm, kk * 2048), adv(dWx, kk * 2048), id_up, 1u);
                        mma_commit(smem_u32(&bars[pUpdate]));
                    }
                    mma_commit(smem_u32(&bars[pFree]));      // CB, C h^T and the update have read C and B
                    // Y_h += P_h x_h (P from TMEM) once P is built and C h^T scaled
                    if (!mbar_wait(smem_u32(&bars[pPReady]), q & 1, kWait)) { ok = false; break; }
                    tc_fence_after();
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
#pragma unroll
                        for (int kk = 0; kk < kQ / 16; ++kk)
                            mma_bf16_ts(ty + 64 * hh, tmem + Cfg::kTcb + 16 * kk + 8 * hh,
                                        adv(dX, xs * Cfg::kXSlot + hh * kAtom + kk * 2048), id_yi, 1u);
                    }
                    mma_commit(smem_u32(&bars[pIntra0 + (q & 1)]));
                    // next CB over the P just read (in issue order)
                    if (q + 1 < nq) {
                        if (!mbar_wait(smem_u32(&bars[pFull]), (q + 1) & 1, kWait)) { ok = false; break; }
                        tc_fence_after();
                        issue_cb();
                    }
                }
            } while (0);
            if (!ok) set_error(err, 1);
            retire_mmas(smem_u32(&bars[pRetire]), err);
        }
        __syncwarp();
    } else if (warp < 6) {
        // ---- state warps: state hand-off and w o x ----------------------------------------
        const int r = 32 * (warp & 3) + lane;          // TMEM lane = state row s / token row t
        const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
        uint8_t *wx = smem + Cfg::kWx;
        uint8_t *hc = smem + Cfg::kHc;
        float n_g[2] = {0.f, 0.f}, n_gl[2] = {0.f, 0.f}, n_gb[2] = {0.f, 0.f};
        uint32_t n_dt = 0;
        auto load_scalars = [&](int q) {
            const int64_t t0 = t_begin + (int64_t)q * kQ;
            const int64_t tr = clamp_t<kRagged>(t0 + r, pr.L), tl = clamp_t<kRagged>(t0 + kQ - 1, pr.L);
            n_g[0] = __ldcg(GA + tr);
            n_g[1] = __ldcg(GB + tr);
            n_gl[0] = __ldcg(GA + tl);
            n_gl[1] = __ldcg(GB + tl);
            const bool cs = q % qpc == 0;
            n_gb[0] = cs ? 0.f : __ldcg(GA + t0 - 1);
            n_gb[1] = cs ? 0.f : __ldcg(GB + t0 - 1);
            n_dt = in_seq<kRagged>(t0 + r, pr.L)
                       ? *reinterpret_cast<const uint32_t *>(dt + ((int64_t)b * pr.L + t0 + r) * pr.nh + hA)
                       : 0u;
        };
        if (nq > 0) load_scalars(0);
        for (int q = 0; q < nq && ok; ++q) {
            const int xs = q % kXS;
            const float g0 = n_g[0], g1 = n_g[1], gl0 = n_gl[0], gl1 = n_gl[1], gb0 = n_gb[0], gb1 = n_gb[1];
            const float2 dtp = unpack_bf16x2(n_dt);
            if (q + 1 < nq) load_scalars(q + 1);
            // the update of q - 1 has produced the state and read w o x (and C h^T of q - 1,
            // issued before it, has read the bf16 copy)
            if (q > 0) {
                if (!mbar_wait(smem_u32(&bars[pUpdate]), (q - 1) & 1, kWait)) {
                    ok = false; set_error(err, 1); break;
                }
                tc_fence_after();
            }
            // state (float32, TMEM) -> bf16 copy [s][p] for C h^T, and the state times
            // 2^(G_last - G_base) back to TMEM for the update to accumulate on
#pragma unroll 1
            for (int hc32 = 0; hc32 < 4; ++hc32) {             // head hc32 / 2, columns 32 (hc32 % 2) ..
                const int hh = hc32 >> 1, c32 = 32 * (hc32 & 1);
                const float dec = exp2f(hh ? gl1 - gb1 : gl0 - gb0);
                const uint32_t ta = tmem + lane_base + Cfg::kTst + 64 * hh + c32;
                uint32_t v[32];
                if (q == 0) {
                    // entering state: h0 (zeros if absent) for super-chunks m < hs_from, else h_start
                    const float *src = (m < sp.hs_from)
                                           ? (h0 ? h0 + (int64_t)(bhA + hh) * (pr.H * S) : nullptr)
                                           : h_start + (hs_idx + hh * nsup) * (int64_t)(pr.H * S);
                    if (src) {
#pragma unroll
                        for (int j = 0; j < 32; ++j) v[j] = __float_as_uint(src[(int64_t)(c32 + j) * S + r]);
                    } else {
#pragma unroll
                        for (int j = 0; j < 32; ++j) v[j] = 0u;
                    }
                } else {
                    tmem_ld16(ta + 0, *reinterpret_cast<uint32_t(*)[16]>(&v[0]));
                    tmem_ld16(ta + 16, *reinterpret_cast<uint32_t(*)[16]>(&v[16]));
                    tmem_ld_wait();
                }
                uint8_t *hrow = hc + hh * kAtom;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint4 o;
                    o.x = pack_bf16x2(__uint_as_float(v[8 * c + 0]), __uint_as_float(v[8 * c + 1]));
                    o.y = pack_bf16x2(__uint_as_float(v[8 * c + 2]), __uint_as_float(v[8 * c + 3]));
                    o.z = pack_bf16x2(__uint_as_float(v[8 * c + 4]), __uint_as_float(v[8 * c + 5]));
                    o.w = pack_bf16x2(__uint_as_float(v[8 * c + 6]), __uint_as_float(v[8 * c + 7]));
                    *(uint4 *)(hrow + sw128(r, (c32 >> 3) + c)) = o;
                }
#pragma unroll
                for (int j = 0; j < 32; j += 2) {
                    const float2 d2 = __fmul2_rn(make_float2(__uint_as_float(v[j]), __uint_as_float(v[j + 1])),
                                                 make_float2(dec, dec));
                    v[j] = __float_as_uint(d2.x);
                    v[j + 1] = __float_as_uint(d2.y);
                }
                tmem_st16(ta + 0, *reinterpret_cast<uint32_t(*)[16]>(&v[0]));
                tmem_st16(ta + 16, *reinterpret_cast<uint32_t(*)[16]>(&v[16]));
            }
            tmem_st_wait();
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(smem_u32(&bars[pHReady]));

            // x row r of both heads: w o x into the Wx tile (the update of q - 1 has read it)
            if (!mbar_wait(smem_u32(&bars[pXFull0 + xs]), (q / kXS) & 1, kWait)) { ok = false; set_error(err, 1); break; }
            // w_t rounded to bf16 and the product taken in bf16 pairs (the product is an MMA
            // operand, rounded to bf16 either way)
            const float w0 = dtp.x * exp2f(gl0 - g0), w1 = dtp.y * exp2f(gl1 - g1);
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const uint8_t *xt = smem + Cfg::kX + xs * Cfg::kXSlot + hh * kAtom;
                uint8_t *wt = wx + hh * kAtom;
                const __nv_bfloat162 w2 = __float2bfloat162_rn(hh ? w1 : w0);
                uint4 vx[8];
#pragma unroll
                for (int c = 0; c < 8; ++c) vx[c] = *(const uint4 *)(xt + sw128(r, c));
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    uint4 o;
                    o.x = mul_bf16x2(vx[c].x, w2);
                    o.y = mul_bf16x2(vx[c].y, w2);
                    o.z = mul_bf16x2(vx[c].z, w2);
                    o.w = mul_bf16x2(vx[c].w, w2);
                    *(uint4 *)(wt + sw128(r, c)) = o;
                }
            }
            fence_proxy_async_smem();
            mbar_arrive(smem_u32(&bars[pXReady]));
        }
        // final state of the sequence, from the last super-chunk of each (batch, head)
        if (ok && write_final && nq > 0) {
            if (!mbar_wait(smem_u32(&bars[pUpdate]), (nq - 1) & 1, kWait)) { ok = false; set_error(err, 1); }
            if (ok) {
                tc_fence_after();
#pragma unroll 1
                for (int hh = 0; hh < 2; ++hh) {
                    float *dst = h_final + (int64_t)(bhA + hh) * (pr.H * S) + r;
#pragma unroll
                    for (int c0 = 0; c0 < 64; c0 += 16) {
                        uint32_t v[16];
                        tmem_ld16(tmem + lane_base + Cfg::kTst + 64 * hh + c0, v);
                        tmem_ld_wait();
#pragma unroll
                        for (int j = 0; j < 16; ++j) dst[(int64_t)(c0 + j) * S] = __uint_as_float(v[j]);
                    }
                }
            }
        }
    } else if (warp < 14) {
        // ---- P warps: P and the scaled C h^T of sub-chunk q ------------------------------------
        const int half = (warp - 6) >> 2;              // columns 64 half .. 64 half + 63; C h^T of head `half`
        const int r = 32 * (warp & 3) + lane;          // TMEM lane = token row i
        const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
        float *arr = (float *)(smem + Cfg::kArr);
        float *myGd = arr + half * (Cfg::kArrHead / 4);  // the arrays this thread fills (head `half`)
        float *myF = myGd + kQ, *myGe = myF + kQ;
        auto group_sync = [&]() { named_bar_sync(1, 256); };
        // per sub-chunk scalars, loaded one ahead: G of row r for both heads, G_base of head
        // `half`, and for head `half`: dt of row r and G at the end of r's 16-token block
        float n_g[2] = {0.f, 0.f}, n_gb = 0.f, n_gend = 0.f, n_dt = 0.f;
        auto load_scalars = [&](int q) {
            const int64_t t0 = t_begin + (int64_t)q * kQ;
            const int64_t tr = clamp_t<kRagged>(t0 + r, pr.L);
            n_g[0] = __ldcg(GA + tr);
            n_g[1] = __ldcg(GB + tr);
            const float *Gh = half ? GB : GA;
            n_gb = (q % qpc == 0) ? 0.f : __ldcg(Gh + t0 - 1);
            n_gend = __ldcg(Gh + clamp_t<kRagged>(t0 + (r | 15), pr.L));
            n_dt = in_seq<kRagged>(t0 + r, pr.L) ? __bfloat162float(dt[((int64_t)b * pr.L + t0 + r) * pr.nh + hA + half])
                                                 : 0.f;
        };
        if (nq > 0) load_scalars(0);
        for (int q = 0; q < nq; ++q) {
            // every thread is past P of q - 1 (the arrays are free)
            group_sync();
            const float g0 = n_g[0], g1 = n_g[1], gbase = n_gb;
            {
                const float gr = half ? g1 : g0;
                myGd[r] = gr - __log2f(n_dt);                     // dt = 0: +inf, so 2^(G_i - Gd_j) = 0
                myF[r] = ex2_approx(n_gend - gr) * n_dt;          // 2^(G_e - G_j) <= 1 for A dt <= 0
                if ((r & 15) == 15) myGe[r >> 4] = gr;
            }
            if (q + 1 < nq) load_scalars(q + 1);
            group_sync();
            if (ok && !mbar_wait(smem_u32(&bars[pCb]), q & 1, kWait)) { ok = false; set_error(err, 1); }
            if (ok) {
                tc_fence_after();
                const uint32_t tcb = tmem + lane_base + Cfg::kTcb;
                const float *GdA = arr, *FA = arr + kQ, *GeA = arr + 2 * kQ;
                const float *GdB = GdA + Cfg::kArrHead / 4, *FB = FA + Cfg::kArrHead / 4, *GeB = GeA + Cfg::kArrHead / 4;
                // The four 16-column blocks of this half come in two pairs of the same kind
                // (above the diagonal, left of every row of the warp, or meeting the diagonal).
                // Per pair: both blocks' C B^T loaded, one wait, then P_A of each block into its
                // first 8 columns and P_B into its last 8.
                const int wrow_lo = 32 * (warp & 3), wrow_hi = wrow_lo + 31;
#pragma unroll 1
                for (int bp = 0; bp < 2; ++bp) {
                    const int j0 = 64 * half + 32 * bp;
                    if (j0 > wrow_hi) {                            // above the diagonal for the whole warp
                        uint32_t z[16];
#pragma unroll
                        for (int e = 0; e < 16; ++e) z[e] = 0u;
                        tmem_st16(tcb + j0, z);
                        tmem_st16(tcb + j0 + 16, z);
                        continue;
                    }
                    uint32_t v[32];
                    tmem_ld16(tcb + j0, *reinterpret_cast<uint32_t(*)[16]>(&v[0]));
                    tmem_ld16(tcb + j0 + 16, *reinterpret_cast<uint32_t(*)[16]>(&v[16]));
                    tmem_ld_wait();
                    if (j0 + 31 < wrow_lo) {                       // left of every row of the warp: factored
#pragma unroll
                        for (int k2 = 0; k2 < 2; ++k2) {
                            const int jb = j0 + 16 * k2;
                            uint32_t pk[16];
                            const float eA = ex2_approx(g0 - GeA[jb >> 4]);
                            const float eB = ex2_approx(g1 - GeB[jb >> 4]);
                            const float4 *fa = reinterpret_cast<const float4 *>(FA + jb);
                            const float4 *fb = reinterpret_cast<const float4 *>(FB + jb);
#pragma unroll
                            for (int e4 = 0; e4 < 4; ++e4) {
                                const float4 a = fa[e4], c = fb[e4];
                                const float2 v01 = make_float2(__uint_as_float(v[16 * k2 + 4 * e4 + 0]),
                                                               __uint_as_float(v[16 * k2 + 4 * e4 + 1]));
                                const float2 v23 = make_float2(__uint_as_float(v[16 * k2 + 4 * e4 + 2]),
                                                               __uint_as_float(v[16 * k2 + 4 * e4 + 3]));
                                const float2 pA01 = __fmul2_rn(__fmul2_rn(v01, make_float2(eA, eA)), make_float2(a.x, a.y));
                                const float2 pA23 = __fmul2_rn(__fmul2_rn(v23, make_float2(eA, eA)), make_float2(a.z, a.w));
                                const float2 pB01 = __fmul2_rn(__fmul2_rn(v01, make_float2(eB, eB)), make_float2(c.x, c.y));
                                const float2 pB23 = __fmul2_rn(__fmul2_rn(v23, make_float2(eB, eB)), make_float2(c.z, c.w));
                                pk[2 * e4] = pack_bf16x2(pA01.x, pA01.y);
                                pk[2 * e4 + 1] = pack_bf16x2(pA23.x, pA23.y);
                                pk[8 + 2 * e4] = pack_bf16x2(pB01.x, pB01.y);
                                pk[8 + 2 * e4 + 1] = pack_bf16x2(pB23.x, pB23.y);
                            }
                            tmem_st16(tcb + jb, pk);
                        }
                    } else {                                       // meets the diagonal: exact, selected
#pragma unroll
                        for (int k2 = 0; k2 < 2; ++k2) {
                            const int jb = j0 + 16 * k2;
                            uint32_t pk[16];
                            const float4 *da = reinterpret_cast<const float4 *>(GdA + jb);
                            const float4 *db = reinterpret_cast<const float4 *>(GdB + jb);
#pragma unroll
                            for (int e4 = 0; e4 < 4; ++e4) {
                                const float4 a = da[e4], c = db[e4];
                                const float ga[4] = {a.x, a.y, a.z, a.w}, gb[4] = {c.x, c.y, c.z, c.w};
                                float pa[4], pb[4];
#pragma unroll
                                for (int e = 0; e < 4; ++e) {
                                    const int j = jb + 4 * e4 + e;
                                    const float vv = __uint_as_float(v[16 * k2 + 4 * e4 + e]);
                                    const float xa = vv * ex2_approx(g0 - ga[e]);
                                    const float xb = vv * ex2_approx(g1 - gb[e]);
                                    pa[e] = (j <= r) ? xa : 0.f;
                                    pb[e] = (j <= r) ? xb : 0.f;
                                }
                                pk[2 * e4] = pack_bf16x2(pa[0], pa[1]);
                                pk[2 * e4 + 1] = pack_bf16x2(pa[2], pa[3]);
                                pk[8 + 2 * e4] = pack_bf16x2(pb[0], pb[1]);
                                pk[8 + 2 * e4 + 1] = pack_bf16x2(pb[2], pb[3]);
                            }
                            tmem_st16(tcb + jb, pk);
                        }
                    }
                }
                // C h^T of head `half`, row r: Y <- 2^(G_i - G_base) Y before P x accumulates onto it
                if (!mbar_wait(smem_u32(&bars[pYs]), q & 1, kWait)) { ok = false; set_error(err, 1); }
                if (ok) {
                    tc_fence_after();
                    const float eg = ex2_approx((half ? g1 : g0) - gbase);
                    const uint32_t ty = tmem + lane_base + Cfg::kTy + (uint32_t)(q & 1) * 128 + 64 * half;
#pragma unroll 1
                    for (int c32 = 0; c32 < 64; c32 += 32) {
                        uint32_t v[32];
                        tmem_ld16(ty + c32, *reinterpret_cast<uint32_t(*)[16]>(&v[0]));
                        tmem_ld16(ty + c32 + 16, *reinterpret_cast<uint32_t(*)[16]>(&v[16]));
                        tmem_ld_wait();
#pragma unroll
                        for (int j = 0; j < 32; j += 2) {
                            const float2 s2 = __fmul2_rn(make_float2(__uint_as_float(v[j]), __uint_as_float(v[j + 1])),
                                                         make_float2(eg, eg));
                            v[j] = __float_as_uint(s2.x);
                            v[j + 1] = __float_as_uint(s2.y);
                        }
                        tmem_st16(ty + c32, *reinterpret_cast<uint32_t(*)[16]>(&v[0]));
                        tmem_st16(ty + c32 + 16, *reinterpret_cast<uint32_t(*)[16]>(&v[16]));
                    }
                }
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(smem_u32(&bars[pPReady]));
            }
        }
    } else if (warp >= 15) {
        // ---- epilogue warps: y = Y + D x of sub-chunk q, staged over its x tile --------------
        const int r = 32 * (warp & 3) + lane;          // TMEM lane = token row i
        const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
        const bool storer = warp == 15 && lane == 0;
        const float dA = Dp[hA], dB = Dp[hA + 1];
        for (int q = 0; q < nq; ++q) {
            const int xs = q % kXS;
            uint8_t *ystage = smem + Cfg::kX + xs * Cfg::kXSlot;
            if (ok && !mbar_wait(smem_u32(&bars[pIntra0 + (q & 1)]), (q >> 1) & 1, kWait)) {
                ok = false; set_error(err, 1);
            }
            if (ok) {
                tc_fence_after();
#pragma unroll 1
                for (int hh = 0; hh < 2; ++hh) {
                    const uint32_t ty = tmem + lane_base + Cfg::kTy + (uint32_t)(q & 1) * 128 + 64 * hh;
                    uint8_t *yrow = ystage + hh * kAtom;
                    const float dh = hh ? dB : dA;
                    // the x row this y then overwrites (same thread, same row)
#pragma unroll 1
                    for (int c32 = 0; c32 < 64; c32 += 32) {
                        uint32_t v[32];
                        tmem_ld16(ty + c32, *reinterpret_cast<uint32_t(*)[16]>(&v[0]));
                        tmem_ld16(ty + c32 + 16, *reinterpret_cast<uint32_t(*)[16]>(&v[16]));
                        uint4 xv[4];
#pragma unroll
                        for (int c = 0; c < 4; ++c) xv[c] = *(const uint4 *)(yrow + sw128(r, (c32 >> 3) + c));
                        tmem_ld_wait();
#pragma unroll
                        for (int c = 0; c < 4; ++c) {
                            const uint32_t in[4] = {xv[c].x, xv[c].y, xv[c].z, xv[c].w};
                            uint32_t o[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const float2 yv = __ffma2_rn(unpack_bf16x2(in[e]), make_float2(dh, dh),
                                                             make_float2(__uint_as_float(v[8 * c + 2 * e]),
                                                                         __uint_as_float(v[8 * c + 2 * e + 1])));
                                o[e] = pack_bf16x2(yv.x, yv.y);
                            }
                            *(uint4 *)(yrow + sw128(r, (c32 >> 3) + c)) = make_uint4(o[0], o[1], o[2], o[3]);
                        }
                    }
                }
                tc_fence_before();
                mbar_arrive(smem_u32(&bars[pEpi0 + (q & 1)]));
                fence_proxy_async_smem();
            }
            // all rows staged (every epilogue thread reaches this, errors or not)
            named_bar_sync(2, 128);
            if (storer) {
                // the slot goes back to the x loader as soon as the store has read it (the x load
                // for three sub-chunks ahead then has a whole period to land).  After an error
                // the slot is not released: its load may still be in flight, and the loader,
                // whose wait then expires, must not re-arm it
                if (ok) {
                    const int t0 = (int)(t_begin + (int64_t)q * kQ);
                    tma_store_4d(&tmY, smem_u32(ystage), 0, hA, t0, b);
                    tma_store_4d(&tmY, smem_u32(ystage + kAtom), 0, hA + 1, t0, b);
                    bulk_commit();
                    bulk_wait_read();
                    mbar_arrive(smem_u32(&bars[pYSt0 + xs]));
                }
            }
            __syncwarp();
        }
        if (storer) bulk_wait_all();
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

// Whether cutting `total` stages into `grid` equal slices puts a cut inside a unit of
// `nq_u` stages.
bool slices_split_units(int64_t total, int64_t grid, int64_t nq_u)
{
    for (int64_t c = 1; c < grid; ++c)
        if ((total * c / grid) % nq_u != 0) return true;
    return false;
}

int current_sms()
{
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 1;
    return sms > 0 ? sms : 1;
}

// chunk_state CTAs for `total` stages in units of nq_u.  With enough work, one CTA per
// SM, each walking an equal slice (units cut between CTAs are added into a zeroed
// output with atomics, whose cost the long slices amortise); with little work, one
// whole unit per CTA, which needs no zeroing and no atomics.
int64_t state_grid(int64_t total, int64_t nq_u)
{
    const int64_t sms = current_sms();
    if (total < 16 * sms) return total / nq_u;
    return sms;
}

template <int S, int H, int HG>
cudaError_t state_launch(const Problem &pr, SeqRange seqs, const void *x, const void *dt, const float *dtT,
                         const void *Bm, const float *G, float *s_out, int R, int nsup, int nm, int *err,
                         cudaStream_t st)
{
    using Cfg = StateCfg<S, H, HG>;
    if (R > Cfg::kMaxR) return cudaErrorInvalidValue;
    // every unit must hold R whole chunks (a short last super-chunk, and a short last chunk, are
    // left to the scan)
    if ((int64_t)nm * R * pr.T > pr.L) return cudaErrorInvalidValue;
    // units are whole head groups of the run
    if (seqs.lo % HG != 0 || seqs.n % HG != 0) return cudaErrorInvalidValue;
    const int64_t nq_u = (int64_t)R * (pr.T / Cfg::kTok);
    const int64_t total = (seqs.n / HG) * (int64_t)nm * nq_u;
    if (total == 0) return cudaSuccess;
    // the staged path bulk-copies 64-token pieces of G and dtT rows: 16-byte aligned only when L % 4 == 0
    if (dtT && (pr.L % 4 != 0 || ((uintptr_t)G % 16) || ((uintptr_t)dtT % 16))) return cudaErrorInvalidValue;
    CUtensorMap mB, mX;
    if (!make_map_4d(&mB, Bm, pr.S, pr.G, pr.L, pr.B, Cfg::kTok) || !make_map_4d(&mX, x, pr.H, pr.nh, pr.L, pr.B, Cfg::kTok))
        return cudaErrorInvalidValue;
    auto kern = pr.wait_ns ? k_chunk_state_tc<S, H, HG, false> : k_chunk_state_tc<S, H, HG, true>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Cfg::kSmem);
    if (e != cudaSuccess) return e;
    const int64_t grid = state_grid(total, nq_u);
    // a slice boundary inside a unit: both parts add into a zeroed s_out
    if (slices_split_units(total, grid, nq_u)) {
        e = cudaMemsetAsync(s_out, 0, (size_t)(seqs.n * nsup) * (size_t)(pr.H * pr.S) * sizeof(float), st);
        if (e != cudaSuccess) return e;
    }
    return launch_pdl(kern, dim3((unsigned)grid), dim3(192), Cfg::kSmem, st, mB, mX, G, (const __nv_bfloat16 *)dt,
                      dtT, s_out, pr, (int64_t)(seqs.lo / HG), (int64_t)(seqs.n / HG), R, nsup, nm, err);
}

template <int S>
cudaError_t scan_launch(const Problem &pr, const void *x, const void *dt, const void *Bm, const void *Cm, const float *D,
                        const float *G, const float *h0, const float *h_start, float *h_final, void *y,
                        const ScanSplit &sp, int *err, cudaStream_t st)
{
    CUtensorMap mC, mB, mX, mY;
    if (!make_map_4d(&mC, Cm, pr.S, pr.G, pr.L, pr.B, kQ) || !make_map_4d(&mB, Bm, pr.S, pr.G, pr.L, pr.B, kQ) ||
        !make_map_4d(&mX, x, pr.H, pr.nh, pr.L, pr.B, kQ) || !make_map_4d(&mY, y, pr.H, pr.nh, pr.L, pr.B, kQ))
        return cudaErrorInvalidValue;
    using Cfg = ScanCfg<S>;
    auto kern = pr.L % pr.T == 0 ? (pr.wait_ns ? k_chunk_scan_tc<S, false, false> : k_chunk_scan_tc<S, false, true>)
                                 : (pr.wait_ns ? k_chunk_scan_tc<S, true, false> : k_chunk_scan_tc<S, true, true>);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Cfg::kSmem);
    if (e != cudaSuccess) return e;
    const int64_t grid = (sp.split * sp.nsup0 + (pr.B * pr.nh - sp.split) * sp.nsup1) * (pr.H / kPB);
    if (grid == 0) return cudaSuccess;
    if (grid > 0x7fffffffLL) return cudaErrorInvalidValue;
    return launch_pdl(kern, dim3((unsigned)grid), dim3(448), Cfg::kSmem, st, mC, mB, mX, mY, G,
                      (const __nv_bfloat16 *)dt, D, h0, h_start, h_final, (__nv_bfloat16 *)y, pr, sp, err);
}

cudaError_t scan_pair_launch(const Problem &pr, const void *x, const void *dt, const void *Bm, const void *Cm,
                             const float *D, const float *G, const float *h0, const float *h_start, float *h_final,
                             void *y, const ScanSplit &sp, int *err, cudaStream_t st)
{
    // head pairs: the run [0, split) and the rest hold whole pairs
    if ((sp.split & 1) || ((pr.B * pr.nh - sp.split) & 1)) return cudaErrorInvalidValue;
    CUtensorMap mC, mB, mX, mY;
    if (!make_map_4d(&mC, Cm, pr.S, pr.G, pr.L, pr.B, kQ) || !make_map_4d(&mB, Bm, pr.S, pr.G, pr.L, pr.B, kQ) ||
        !make_map_4d(&mX, x, pr.H, pr.nh, pr.L, pr.B, kQ) || !make_map_4d(&mY, y, pr.H, pr.nh, pr.L, pr.B, kQ))
        return cudaErrorInvalidValue;
    auto kern = pr.L % pr.T == 0 ? (pr.wait_ns ? k_chunk_scan_pair<false, false> : k_chunk_scan_pair<false, true>)
                                 : (pr.wait_ns ? k_chunk_scan_pair<true, false> : k_chunk_scan_pair<true, true>);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)PairCfg::kSmem);
    if (e != cudaSuccess) return e;
    const int64_t grid = (sp.split / 2) * sp.nsup0 + ((pr.B * pr.nh - sp.split) / 2) * sp.nsup1;
    if (grid == 0) return cudaSuccess;
    if (grid > 0x7fffffffLL) return cudaErrorInvalidValue;
    return launch_pdl(kern, dim3((unsigned)grid), dim3(PairCfg::kThreads), PairCfg::kSmem, st, mC, mB,
                      mX, mY, G, (const __nv_bfloat16 *)dt, D, h0, h_start, h_final, pr, sp, err);
}

}  // namespace

int scan_seqs_per_cta(const Problem &pr)
{
    return (pr.S == 128 && pr.H == 64 && pr.hpg % 2 == 0) ? 2 : 1;
}

bool tc_supported(const Problem &pr)
{
    if (pr.in_dt != SSD_BF16 || pr.out_dt != SSD_BF16) return false;
    if (pr.S != 128 && pr.S != 256) return false;
    if (pr.H != 64 && pr.H != 128) return false;
    if (pr.T % kQ != 0 || pr.T > 256) return false;
    if (pr.L > 0x7fffffffLL || pr.B > 65535) return false;
    return true;
}

// Heads per chunk_state CTA: as many heads of one group as fit N = HG * H <= 256 (S = 128).
int state_heads_per_cta(const Problem &pr)
{
    const int hpg = (int)pr.hpg;
    if (pr.S == 128 && pr.H == 64) return hpg % 4 == 0 ? 4 : (hpg % 2 == 0 ? 2 : 1);
    if (pr.S == 128 && pr.H == 128) return hpg % 2 == 0 ? 2 : 1;
    return 1;
}

// Heads per chunk_state CTA for a launch over `seqs` with nm super-chunks of R chunks:
// the most that share B tiles; for a small launch (one whole unit per CTA, see
// state_grid), halved while the units still fit in one wave of CTAs, since such a
// launch is latency-bound and more, smaller units finish sooner -- but a second wave
// costs a whole unit's latency again.
int state_launch_heads(const Problem &pr, SeqRange seqs, int R, int nm)
{
    int hg = state_heads_per_cta(pr);
    const int64_t sms = current_sms(), nq_u = (int64_t)R * (pr.T / 64);
    while (hg > 1) {
        const int64_t units = (seqs.n / hg) * nm;
        if (units * nq_u >= 16 * sms || 2 * units > sms) break;
        hg /= 2;
    }
    return hg;
}

bool chunk_state_tc_memsets(const Problem &pr, SeqRange seqs, int R, int nm)
{
    const int64_t nq_u = (int64_t)R * (pr.T / 64);
    const int64_t total = (seqs.n / state_launch_heads(pr, seqs, R, nm)) * (int64_t)nm * nq_u;
    if (total == 0) return false;
    return slices_split_units(total, state_grid(total, nq_u), nq_u);
}

cudaError_t launch_chunk_state_tc(const Problem &pr, SeqRange seqs, const void *x, const void *dt, const float *dtT,
                                  const void *Bm, const float *G, float *s_out, int R, int nsup, int nm, int *err,
                                  cudaStream_t st)
{
    if (R < 1 || R > 256) return cudaErrorInvalidValue;
    const int hg = state_launch_heads(pr, seqs, R, nm);
    if (pr.S == 128 && pr.H == 64) {
        if (hg == 4) return state_launch<128, 64, 4>(pr, seqs, x, dt, dtT, Bm, G, s_out, R, nsup, nm, err, st);
        if (hg == 2) return state_launch<128, 64, 2>(pr, seqs, x, dt, dtT, Bm, G, s_out, R, nsup, nm, err, st);
        return state_launch<128, 64, 1>(pr, seqs, x, dt, dtT, Bm, G, s_out, R, nsup, nm, err, st);
    }
    if (pr.S == 128 && pr.H == 128) {
        if (hg == 2) return state_launch<128, 128, 2>(pr, seqs, x, dt, dtT, Bm, G, s_out, R, nsup, nm, err, st);
        return state_launch<128, 128, 1>(pr, seqs, x, dt, dtT, Bm, G, s_out, R, nsup, nm, err, st);
    }
    if (pr.S == 256 && pr.H == 64) return state_launch<256, 64, 1>(pr, seqs, x, dt, dtT, Bm, G, s_out, R, nsup, nm, err, st);
    if (pr.S == 256 && pr.H == 128) return state_launch<256, 128, 1>(pr, seqs, x, dt, dtT, Bm, G, s_out, R, nsup, nm, err, st);
    return cudaErrorNotSupported;
}

cudaError_t launch_chunk_scan_tc(const Problem &pr, const void *x, const void *dt, const void *Bm, const void *Cm,
                                 const float *D, const float *G, const float *h0, const float *h_start, float *h_final,
                                 void *y, const ScanSplit &sp, int *err, cudaStream_t st)
{
    if (scan_seqs_per_cta(pr) == 2)
        return scan_pair_launch(pr, x, dt, Bm, Cm, D, G, h0, h_start, h_final, y, sp, err, st);
    if (pr.S == 128) return scan_launch<128>(pr, x, dt, Bm, Cm, D, G, h0, h_start, h_final, y, sp, err, st);
    if (pr.S == 256) return scan_launch<256>(pr, x, dt, Bm, Cm, D, G, h0, h_start, h_final, y, sp, err, st);
    return cudaErrorNotSupported;
}

}  // namespace ssd
