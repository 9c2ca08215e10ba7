// ssd_fused.cu -- the chunked SSD forward pass as ONE persistent tensor-core kernel, for two
// heads of one B/C group per work item (S = 128, H = 64, an even number of heads per group).
//
// Method: NVIDIA developer blog "Accelerating Mamba-2 with High-Performance Forward Pass
// Kernels in NVIDIA CUDA Tile", section "Mamba-2 architecture" (the in-chunk cumsum, the
// chunk jump and the chunk output) and sections "Kernel 1" .. "Kernel 3" (the stages).
//
// What is fused, and why.  The blog runs three kernels in sequence (cumsum, state pass,
// output).  Here every stage runs inside one kernel launch, one CTA per SM:
//  * The cumsum is taken per 128-token sub-chunk, in registers, from dt and A: every
//    exponent the path needs is a difference of cumsums within one sub-chunk (the
//    decay of the carried state across the sub-chunk, the weights exp2(G_last - G_t),
//    the mask exp2(G_i - G_j), and exp2(G_i - G_start) for C h^T), so no G array is
//    written or read.  Values are log2(e) multiples, as in the blog's Kernel 1.
//  * Work items come from an atomic ticket in dependency order (fused_plan.cuh): STATE
//    items (the state a super-chunk produces from a zero start: the chunk_state stage,
//    run over a whole super-chunk with the state carried in TMEM), PASS items (the
//    sequential chunk loop of the blog's Kernel 2, one slice of state columns each) and
//    SCAN items (the chunk output walk with the state on chip).  A CTA takes the next
//    ticket when its loader is about to need it, so every SM stays busy to the end and
//    the next item's loads overlap the current item's last sub-chunks.
//  * A wait on another CTA (PASS on STATE, SCAN on PASS) is only ever on a lower ticket,
//    which a running CTA has taken: it ends without any assumption about which CTAs are
//    resident.  Every wait is bounded (wait_ns); on expiry the kernel sets the error word
//    and winds down, still retiring the copies and MMAs it has issued.
//
// Per sub-chunk of a SCAN item (rows i, j = tokens; states h_A, h_B, each H x S), the same
// arithmetic as the blog's output kernel, arranged for the tensor cores:
//   CB        = C B^T                                   (M = i, N = j, K = s; shared)
//   P_h[i][j] = CB[i][j] exp2(G_h,i - G_h,j) dt_h,j  if j <= i, else 0
//             (built by the CUDA cores over CB in place: block k of 16 columns
//              holds P_A of that block in its first 8 columns, P_B in the last 8)
//   Y         = C [h_A^T | h_B^T]                       (M = i, N = 2 x 64 p, K = s)
//   Y_h,i    <- exp2(G_h,i) Y_h,i                        (CUDA cores, in TMEM)
//   Y_h      += P_h x_h                                 (M = i, N = 64, K = j; A from TMEM)
//   y_h       = Y_h + D_h x_h (bf16)
//   [h_A^T | h_B^T] <- exp2(G_last) state + B^T [w_A o x_A | w_B o x_B]   (M = s, N = 128, K = t)
// with G the cumsum from the sub-chunk start and w_t = dt_t exp2(G_last - G_t).  A STATE
// sub-chunk runs only the last line.
//
// TMEM (512 columns): CB / P 0..127, Y buffers 128..255 and 256..383 (SCAN sub-chunk q in
// buffer q % 2; head A then head B), state 384..511 (h_A^T then h_B^T; lanes = s).
// Shared memory: one C/B stage, x in a 3-slot ring (the slots also stage y for its bulk
// stores), w o x, the bf16 state copy, the P warps' column arrays, the item ring.
// Warps: 0 takes tickets and loads C and B, 14 loads x, 1 issues MMAs, 2..5 ("state
// warps") hand the state over, write w o x and run PASS items, 6..13 ("P warps") build P
// and scale C h^T, 15..18 ("epilogue warps") write y and issue its bulk stores.
#include "fused_plan.cuh"
#include "ssd_tc.cuh"
#include "tc_common.cuh"

namespace ssd {
namespace {

using namespace ptx;
using tc::kAtom;
using tc::kQ;

struct FusedCfg {
    static constexpr int kXStages = 3;
    static constexpr int kRing = 4;                            // item ring slots
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
    // per-warp cumsum totals of a sub-chunk, float2 (both heads): state warps [2 buffers][4],
    // P warps [2 halves][4]
    static constexpr uint32_t kTot = kArr + 2 * kArrHead;
    // item ring [kRing], group broadcasts [3][2], abort flag
    static constexpr uint32_t kMisc = kTot + 128;
    static constexpr uint32_t kBars = kMisc + 64;
    static constexpr int kNumBars = 22 + 2 * kRing;
    static constexpr uint32_t kSmem = kBars + kNumBars * 8 + 8;
    static constexpr uint32_t kTcb = 0, kTy = 128, kTst = 384, kTmemCols = 512;
    static constexpr int kThreads = 608;
    static constexpr int kSlices = 16;                         // PASS slices per cut pair
    static constexpr int kPassBatch = 16;                      // chained states staged per PASS copy (a power of 2)
    static_assert(2 * kPassBatch == 32, "one decay per lane of a warp");
    static_assert(2 * kPassBatch * (64 * 128 / kSlices) * 4 == 4 * kAtom, "PASS staging = w o x + bf16 state");
    static_assert(kSmem <= 227 * 1024, "shared memory");
};

// fFull0/1, fFree0/1: the two halves of the C/B stage (loaded / read by their last MMA): a
// SCAN sub-chunk loads C into half 0 and B into half 1, a STATE sub-chunk loads only B, into
// the halves in turn, so that one STATE sub-chunk's B loads while the previous one's update
// reads the other half; fCb: C B^T done; fYs: C h^T done; fHReady: bf16 state copy written
// and the decayed state back in TMEM (SCAN); fXReady: w o x written; fPReady: P built and
// C h^T scaled; fIntra0/1: P x into Y buffer 0/1 done; fUpdate: the state update (or, when it
// is skipped, every MMA before it) done; fEpi0/1: Y buffer 0/1 drained; fStage: a bulk copy
// of the state warps into the w o x and bf16-state buffers landed (PASS items); fXFull/fYSt:
// x slots (loaded / free again); fRingFull/fRingEmpty: item ring slots; fDone: every MMA of
// the CTA done (before TMEM is freed).  Every barrier a role waits on by parity is one its
// own progress keeps within one phase of the wait.
enum FusedBar {
    fFull0 = 0, fFull1, fFree0, fFree1, fCb, fYs, fHReady, fXReady, fPReady, fIntra0, fIntra1, fUpdate, fEpi0,
    fEpi1, fStage, fXFull0, fYSt0 = fXFull0 + 3, fRingFull0 = fYSt0 + 3, fRingEmpty0 = fRingFull0 + FusedCfg::kRing,
    fDone = fRingEmpty0 + FusedCfg::kRing, fNumBars
};
static_assert(fNumBars == FusedCfg::kNumBars, "fused barriers");

// Named barriers: 1 = P warps (256), 2 = epilogue warps (128), 3 = state warps (128).
constexpr uint32_t kBarP = 1, kBarEpi = 2, kBarState = 3;

// Items the ring holds: a ticket, -1 at the end of the list, -2 after an error.
struct Ring {
    uint64_t *bars;
    volatile int *slot;
    uint64_t wait_ns;

    // One consumer's take of item n (each consumer takes every item once, in order).
    __device__ __forceinline__ int take(int n, bool &ok) const
    {
        const int s = n % FusedCfg::kRing;
        if (!mbar_wait(smem_u32(&bars[fRingFull0 + s]), (n / FusedCfg::kRing) & 1, wait_ns)) {
            ok = false;
            return -2;
        }
        const int t = slot[s];
        mbar_arrive(smem_u32(&bars[fRingEmpty0 + s]));
        return t;
    }

    // The take of a group of threads: its leader takes the item and broadcasts it; the
    // named barrier makes the broadcast and the decision to stop (any thread's error, or
    // the end of the list) the same in every thread of the group.
    __device__ __forceinline__ int group_take(int n, bool leader, uint32_t bar_id, uint32_t nthreads,
                                              volatile int *bcast, bool &ok, int *err) const
    {
        if (leader) {
            bool lok = true;
            int t = take(n, lok);
            if (!lok) { t = -2; tc::set_error(err, tc::kErrTimeout); }
            bcast[n & 1] = t;
        }
        const bool fail = tc::named_bar_or(bar_id, nthreads, !ok);
        const int t = bcast[n & 1];
        return fail ? -2 : t;
    }
};

// Inclusive cumsum of v over the 32 lanes of a warp (both heads at once).
__device__ __forceinline__ float2 warp_cumsum2(float2 v, int lane)
{
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float a = __shfl_up_sync(0xffffffffu, v.x, o);
        const float b = __shfl_up_sync(0xffffffffu, v.y, o);
        if (lane >= o) { v.x += a; v.y += b; }
    }
    return v;
}

// The cumsum of a sub-chunk from the per-warp totals (4 warps of 32 rows): row r's value
// is its warp's inclusive cumsum `pre` plus the totals of the warps before it.  The state
// warps and the P warps both call this with the same inputs, in the same order, so their
// results agree to the bit.
__device__ __forceinline__ void cumsum_from_totals(const float2 *tot, int w4, float2 pre, float2 &g, float2 &total)
{
    float2 off = make_float2(0.f, 0.f), all = make_float2(0.f, 0.f);
#pragma unroll
    for (int w = 0; w < 4; ++w) {
        const float2 t = tot[w];
        if (w < w4) { off.x += t.x; off.y += t.y; }
        all.x += t.x;
        all.y += t.y;
    }
    g = make_float2(off.x + pre.x, off.y + pre.y);
    total = all;
}

// The work item of ticket t (one out-of-line copy for every role: item boundaries are rare,
// and the decoder's divisions would otherwise sit in each role's instruction stream).
__device__ __noinline__ FusedItem item_of(const FusedPlan &pl, int t) { return fused_item(pl, t); }

// Bounded wait until *p >= target (acquire: writes released before the increment are
// visible to this thread afterwards).
__device__ __noinline__ bool wait_count(const int *p, int target, uint64_t wait_ns)
{
    const long long c0 = clock64();
    const long long limit = (long long)(wait_ns * 5 / 2);
    while (true) {
        int v;
        asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
        if (v >= target) return true;
        if (clock64() - c0 > limit) return false;
        __nanosleep(200);
    }
}

// dt of both heads of a pair at token t (bf16 pair; 0 past the end of the sequence).
template <bool kRagged>
__device__ __forceinline__ uint32_t load_dt2(const __nv_bfloat16 *dt, const Problem &pr, int b, int hA, int64_t t)
{
    if (kRagged && t >= pr.L) return 0u;
    return __ldg(reinterpret_cast<const unsigned int *>(dt + ((int64_t)b * pr.L + t) * pr.nh + hA));
}

// A PASS item, run by the 128 state warps (thread r; `leader` is r == 0):
// h_start(m + 1) = 2^(log2 decay of m) h_start(m) + s_local(m), h_start(0) = h0 (or 0), for one
// slice of the state elements of both heads of the pair, once every STATE item of the pair is
// done.  kPassBatch chained states at a time are staged by bulk copies into the w o x and
// bf16-state buffers (free once the MMAs of the items before are done): stage[head][k][slice].
// One out-of-line copy: PASS items are rare, and their code stays out of the state warps'
// per-sub-chunk instruction stream.
__device__ __noinline__ void run_pass(const FusedItem &it, uint8_t *smem, uint64_t *bars, int r, int lane, bool leader,
                                      int bhA, const float *__restrict__ h0, const float *s_loc, const float *sdec,
                                      float *h_st, int *cnt, int npair, int qc, uint64_t wait_ns, int *err, bool &ok,
                                      int &nstage, int &pass_issued)
{
    using Cfg = FusedCfg;
    constexpr int64_t HS = 64 * 128;
    constexpr int kPer = (int)(HS / Cfg::kSlices);
    bool fail = false;
    if (leader) {
        if (!wait_count(cnt + it.pair, it.nsup - 1, wait_ns)) fail = true;
        if (qc > 0 && !mbar_wait(smem_u32(&bars[fUpdate]), (qc - 1) & 1, wait_ns)) fail = true;
    }
    if (tc::named_bar_or(kBarState, 128, fail)) { ok = false; tc::set_error(err, tc::kErrTimeout); }
    float *stage = (float *)(smem + Cfg::kWx);
    const int64_t e = (int64_t)it.slice * kPer + 4 * r;   // this thread's 4 elements
    float4 h[2];
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
        h[hh] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (h0) {   // (h0 need only be 4-byte aligned)
            const float *p0 = h0 + (int64_t)(bhA + hh) * HS + e;
            h[hh] = make_float4(__ldcg(p0), __ldcg(p0 + 1), __ldcg(p0 + 2), __ldcg(p0 + 3));
        }
    }
#pragma unroll 1
    for (int m0 = 0; m0 < it.nsup - 1; m0 += Cfg::kPassBatch) {
        const int nb = min(Cfg::kPassBatch, it.nsup - 1 - m0);
        if (leader && ok) {
            // the generic-proxy reads of the previous batch come before these async writes
            fence_proxy_async_smem();
            mbar_arrive_expect_tx(smem_u32(&bars[fStage]), (uint32_t)(2 * nb * kPer * 4));
            for (int hh = 0; hh < 2; ++hh)
                for (int k = 0; k < nb; ++k)
                    bulk_load(smem_u32(stage + (hh * Cfg::kPassBatch + k) * kPer),
                              s_loc + (it.slot + (int64_t)hh * it.nsup + m0 + k) * HS + (int64_t)it.slice * kPer,
                              (uint32_t)(kPer * 4), smem_u32(&bars[fStage]));
            ++pass_issued;
        }
        if (ok && !mbar_wait(smem_u32(&bars[fStage]), nstage & 1, wait_ns)) {
            ok = false;
            tc::set_error(err, tc::kErrTimeout);
        }
        ++nstage;
        if (ok) {
            // the batch's decays, one per lane (head 0 in lanes 0..15, head 1 in 16..31), loaded
            // together and handed out by shuffles
            const int kl = lane & (Cfg::kPassBatch - 1), hl = lane / Cfg::kPassBatch;
            float dl = 1.f;
            if (kl < nb) dl = exp2f(__ldcg(sdec + it.slot + (int64_t)hl * it.nsup + m0 + kl));
#pragma unroll 1
            for (int k = 0; k < nb; ++k) {
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const int64_t sl = it.slot + (int64_t)hh * it.nsup + m0 + k;
                    const float d = __shfl_sync(0xffffffffu, dl, hh * Cfg::kPassBatch + k);
                    const float4 sv = *reinterpret_cast<const float4 *>(stage + (hh * Cfg::kPassBatch + k) * kPer + 4 * r);
                    h[hh].x = fmaf(d, h[hh].x, sv.x);
                    h[hh].y = fmaf(d, h[hh].y, sv.y);
                    h[hh].z = fmaf(d, h[hh].z, sv.z);
                    h[hh].w = fmaf(d, h[hh].w, sv.w);
                    *reinterpret_cast<float4 *>(h_st + (sl + 1) * HS + e) = h[hh];
                }
            }
        }
        // every thread is done with the batch before the next one overwrites it
        tc::named_bar_sync(kBarState, 128);
    }
    __threadfence();
    tc::named_bar_sync(kBarState, 128);
    if (leader) atomicAdd(cnt + npair + it.pair, 1);
}

template <bool kRagged>
__global__ void __launch_bounds__(FusedCfg::kThreads, 1)
k_ssd_fwd_fused(const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmB,
                const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmY,
                const __nv_bfloat16 *__restrict__ dt, const float *__restrict__ Ap, const float *__restrict__ Dp,
                const float *__restrict__ h0, float *__restrict__ h_final, float *s_loc, float *h_st, float *sdec,
                int *hdr, int *cnt, Problem pr, const __grid_constant__ FusedPlan pl, unsigned long long wait_ns)
{
    using Cfg = FusedCfg;
    constexpr int S = 128, kXS = Cfg::kXStages;
    constexpr int64_t HS = 64 * 128;
    extern __shared__ __align__(1024) uint8_t smem[];
    int *err = hdr;
    if (smem_u32(smem) & 1023u) {
        if (threadIdx.x == 0) tc::set_error(err, tc::kErrSmemAlign);
        return;
    }
    uint64_t *bars = (uint64_t *)(smem + Cfg::kBars);
    uint32_t *tmem_slot = (uint32_t *)(bars + Cfg::kNumBars);
    volatile int *misc = (volatile int *)(smem + Cfg::kMisc);
    volatile int *ring_slot = misc;                 // [kRing]
    volatile int *bcast_state = misc + 4, *bcast_p = misc + 6, *bcast_epi = misc + 8;
    volatile int *abort_flag = misc + 10;
    const Ring ring{bars, ring_slot, wait_ns};
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < Cfg::kNumBars; ++i) {
            uint32_t c = 1;
            if (i == fHReady || i == fXReady || i == fEpi0 || i == fEpi1) c = 128;
            if (i == fPReady) c = 256;
            if (i >= fRingEmpty0 && i < fRingEmpty0 + Cfg::kRing) c = 5;   // x loader, MMA, three group leaders
            mbar_init(smem_u32(&bars[i]), c);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) { tmem_alloc(smem_u32(tmem_slot), Cfg::kTmemCols); tmem_relinquish(); }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    bool ok = true;

    if (warp == 0) {
        // ---- tickets, and the C and B tiles (one stage: free once its last MMA has read it) -------
        if (lane == 0) {
            prefetch_tmap(&tmC);
            prefetch_tmap(&tmB);
            int uses0 = 0, uses1 = 0;                   // loads into each half of the C/B stage so far
            int sh = 0;                                 // the half the next STATE sub-chunk loads into
            // expect and load a C or B tile (two 64-column atoms) into half hv of the stage
            auto load_half = [&](int hv, const CUtensorMap *map, int g, int t0, int b) {
                const uint32_t full = smem_u32(&bars[fFull0 + hv]);
                mbar_arrive_expect_tx(full, 2 * kAtom);
                for (int a = 0; a < 2; ++a)
                    tma_load_4d(smem_u32(smem + hv * Cfg::kCBytes + a * kAtom), map, full, 64 * a, g, t0, b);
            };
            for (int n = 0;; ++n) {
                const int s = n % Cfg::kRing;
                if (n >= Cfg::kRing &&
                    !mbar_wait(smem_u32(&bars[fRingEmpty0 + s]), ((n / Cfg::kRing) - 1) & 1, wait_ns)) {
                    ok = false;
                    break;
                }
                int t = -1;
                if (!*abort_flag) {
                    t = atomicAdd(&hdr[1], 1);
                    if (t >= pl.n_items) t = -1;
                }
                ring_slot[s] = t;
                mbar_arrive(smem_u32(&bars[fRingFull0 + s]));
                if (t < 0) break;
                const FusedItem it = item_of(pl, t);
                if (it.kind == kItemPass) continue;
                const int b = (int)((2 * it.pair) / pr.nh), g = (int)(((2 * it.pair) % pr.nh) / pr.hpg);
                const bool scan = it.kind == kItemScan;
#pragma unroll 1
                for (int q = 0; q < it.nq; ++q) {
                    const int t0 = (it.sub_begin + q) * kQ;
                    if (scan) {
                        // C into half 0, B into half 1
                        if ((uses0 >= 1 && !mbar_wait(smem_u32(&bars[fFree0]), (uses0 - 1) & 1, wait_ns)) ||
                            (uses1 >= 1 && !mbar_wait(smem_u32(&bars[fFree1]), (uses1 - 1) & 1, wait_ns))) {
                            ok = false;
                            break;
                        }
                        load_half(0, &tmC, g, t0, b);
                        load_half(1, &tmB, g, t0, b);
                        ++uses0;
                        ++uses1;
                    } else {
                        // B into the halves in turn
                        const int hv = sh, u = hv ? uses1 : uses0;
                        sh ^= 1;
                        if (u >= 1 && !mbar_wait(smem_u32(&bars[fFree0 + hv]), (u - 1) & 1, wait_ns)) { ok = false; break; }
                        load_half(hv, &tmB, g, t0, b);
                        if (hv) ++uses1; else ++uses0;
                    }
                    // the tiles two sub-chunks ahead into L2: a half reloads right after its last MMA
                    // has read it, so the load latency is on the critical path
                    if (q + 2 < it.nq) {
                        for (int a = 0; a < 2; ++a) {
                            if (scan) tma_prefetch_4d(&tmC, 64 * a, g, t0 + 2 * kQ, b);
                            tma_prefetch_4d(&tmB, 64 * a, g, t0 + 2 * kQ, b);
                        }
                    }
                }
                if (!ok) break;
            }
            if (!ok) { tc::set_error(err, tc::kErrTimeout); *abort_flag = 1; }
            // retire: the last load into each half must have landed before the CTA may exit
            if (uses0 > 0) mbar_wait(smem_u32(&bars[fFull0]), (uses0 - 1) & 1, tc::kWaitNs);
            if (uses1 > 0) mbar_wait(smem_u32(&bars[fFull1]), (uses1 - 1) & 1, tc::kWaitNs);
        }
        __syncwarp();
    } else if (warp == 14) {
        // ---- x tiles of both heads (slot of sub-chunk qc: free once its last reader is done) --
        if (lane == 0) {
            prefetch_tmap(&tmX);
            int qc = 0;
            for (int n = 0;; ++n) {
                const int t = ring.take(n, ok);
                if (t < 0) break;
                const FusedItem it = item_of(pl, t);
                if (it.kind == kItemPass) continue;
                const int bhA = 2 * it.pair, b = (int)(bhA / pr.nh), hA = (int)(bhA % pr.nh);
                if (it.kind == kItemScan && it.m == 0 && h0) {
                    // the entering states of both heads into L2 first: the first hand-off reads them
                    // with strided loads (h0 need only be 4-byte aligned; a bulk prefetch needs 16)
                    for (int hh = 0; hh < 2; ++hh) {
                        const float *src = h0 + (int64_t)(bhA + hh) * HS;
                        if (((uintptr_t)src & 15u) == 0) bulk_prefetch_l2(src, (uint32_t)(HS * sizeof(float)));
                    }
                }
                for (int q = 0; q < it.nq; ++q, ++qc) {
                    const int t0 = (it.sub_begin + q) * kQ;
                    const int xs = qc % kXS;
                    if (qc >= kXS && !mbar_wait(smem_u32(&bars[fYSt0 + xs]), ((qc / kXS) - 1) & 1, wait_ns)) {
                        ok = false;
                        break;
                    }
                    const uint32_t xfull = smem_u32(&bars[fXFull0 + xs]);
                    mbar_arrive_expect_tx(xfull, Cfg::kXSlot);
                    for (int hh = 0; hh < 2; ++hh)
                        tma_load_4d(smem_u32(smem + Cfg::kX + xs * Cfg::kXSlot + hh * kAtom), &tmX, xfull, 0,
                                    hA + hh, t0, b);
                }
                if (!ok) break;
            }
            if (!ok) { tc::set_error(err, tc::kErrTimeout); *abort_flag = 1; }
            // retire: the last load of every slot must have landed
            for (int k = qc - 1; k >= 0 && k >= qc - kXS; --k)
                mbar_wait(smem_u32(&bars[fXFull0 + k % kXS]), (k / kXS) & 1, tc::kWaitNs);
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
            const uint64_t dBm0 = smem_desc(s0, kAtom, 1024);                   // B^T [s][t], MN-major, half 0
            const uint64_t dBm = smem_desc(s0 + Cfg::kCBytes, kAtom, 1024);     // B^T [s][t], MN-major, half 1
            const uint64_t dX = smem_desc(s0 + Cfg::kX, kAtom, 1024);           // x [t][p], MN-major
            const uint64_t dHc = smem_desc(s0 + Cfg::kHc, kAtom, 1024);         // h bf16 [s][p], 2 atoms along N
            const uint64_t dWx = smem_desc(s0 + Cfg::kWx, kAtom, 1024);         // w o x [t][p], 2 atoms along N
            auto issue_cb = [&]() {
#pragma unroll
                for (int kk = 0; kk < S / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * kAtom + (kk & 3) * 32;
                    mma_bf16(tmem + Cfg::kTcb, adv(dC, off), adv(dBk, off), id_cb, kk > 0 ? 1u : 0u);
                }
                mma_commit(smem_u32(&bars[fCb]));
            };
            int n = 0, qc = 0, qs = 0;
            int uses0 = 0, uses1 = 0;                  // loads into each half of the C/B stage consumed so far
            int sh = 0;                                // the half of the next STATE sub-chunk
            bool cb_issued = false;                    // C B^T of the next SCAN sub-chunk already issued
            int pending = -3;                          // an item taken ahead (-3: none)
            auto wait_cb_tiles = [&]() -> bool {       // C (half 0) and B (half 1) of the next SCAN sub-chunk
                return mbar_wait(smem_u32(&bars[fFull0]), uses0 & 1, wait_ns) &&
                       mbar_wait(smem_u32(&bars[fFull1]), uses1 & 1, wait_ns);
            };
            while (ok) {
                int t;
                if (pending != -3) { t = pending; pending = -3; }
                else t = ring.take(n++, ok);
                if (t < 0) break;
                const FusedItem it = item_of(pl, t);
                if (it.kind == kItemPass) continue;
                if (it.kind == kItemState) {
#pragma unroll
                    for (int q = 0; q < it.nq; ++q, ++qc) {
                        const int hv = sh;
                        sh ^= 1;
                        // B landed and w o x written (the state warps have also read the x slot)
                        if (!mbar_wait(smem_u32(&bars[fFull0 + hv]), (hv ? uses1 : uses0) & 1, wait_ns) ||
                            !mbar_wait(smem_u32(&bars[fXReady]), qc & 1, wait_ns)) { ok = false; break; }
                        tc_fence_after();
                        const uint64_t dB = hv ? dBm : dBm0;
#pragma unroll
                        for (int kk = 0; kk < kQ / 16; ++kk)
                            mma_bf16(tmem + Cfg::kTst, adv(dB, kk * 2048), adv(dWx, kk * 2048), id_up, 1u);
                        mma_commit(smem_u32(&bars[fUpdate]));
                        mma_commit(smem_u32(&bars[fFree0 + hv]));
                        if (hv) ++uses1; else ++uses0;
                        mbar_arrive(smem_u32(&bars[fYSt0 + qc % kXS]));   // the x slot is free again
                    }
                    continue;
                }
                const bool final = it.m == it.nsup - 1 && h_final;
#pragma unroll
                for (int q = 0; q < it.nq; ++q, ++qc, ++qs) {
                    const int xs = qc % kXS;
                    const uint32_t ty = tmem + Cfg::kTy + (uint32_t)(qs & 1) * 128;
                    if (!cb_issued) {
                        if (!wait_cb_tiles()) { ok = false; break; }
                        tc_fence_after();
                        issue_cb();
                    }
                    cb_issued = false;
                    // C [h_A^T | h_B^T] into Y buffer qs % 2 (drained by the epilogue of qs - 2), from
                    // the bf16 state copy of the hand-off
                    if (!mbar_wait(smem_u32(&bars[fHReady]), qs & 1, wait_ns) ||
                        (qs >= 2 && !mbar_wait(smem_u32(&bars[fEpi0 + (qs & 1)]), ((qs - 2) >> 1) & 1, wait_ns))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < S / 16; ++kk) {
                        const uint32_t off = (kk >> 2) * kAtom + (kk & 3) * 32;
                        mma_bf16(ty, adv(dC, off), adv(dHc, kk * 2048), id_ys, kk > 0 ? 1u : 0u);
                    }
                    mma_commit(smem_u32(&bars[fYs]));
                    // update on the state the state warps decayed, with their w o x (the state after the
                    // last sub-chunk is needed only for h_final)
                    if (!mbar_wait(smem_u32(&bars[fXReady]), qc & 1, wait_ns)) { ok = false; break; }
                    tc_fence_after();
                    if (q + 1 < it.nq || final) {
#pragma unroll
                        for (int kk = 0; kk < kQ / 16; ++kk)
                            mma_bf16(tmem + Cfg::kTst, adv(dBm, kk * 2048), adv(dWx, kk * 2048), id_up, 1u);
                    }
                    mma_commit(smem_u32(&bars[fUpdate]));
                    mma_commit(smem_u32(&bars[fFree0]));     // CB and C h^T have read C,
                    mma_commit(smem_u32(&bars[fFree1]));     // CB and the update have read B
                    ++uses0;
                    ++uses1;
                    // Y_h += P_h x_h (P from TMEM) once P is built and C h^T scaled
                    if (!mbar_wait(smem_u32(&bars[fPReady]), qs & 1, wait_ns)) { ok = false; break; }
                    tc_fence_after();
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
#pragma unroll
                        for (int kk = 0; kk < kQ / 16; ++kk)
                            mma_bf16_ts(ty + 64 * hh, tmem + Cfg::kTcb + 16 * kk + 8 * hh,
                                        adv(dX, xs * Cfg::kXSlot + hh * kAtom + kk * 2048), id_yi, 1u);
                    }
                    mma_commit(smem_u32(&bars[fIntra0 + (qs & 1)]));
                    // C B^T of the next sub-chunk of the item over the P just read (in issue order): the P
                    // warps start on it while this one finishes
                    if (q + 1 < it.nq) {
                        if (!wait_cb_tiles()) { ok = false; break; }
                        tc_fence_after();
                        issue_cb();
                        cb_issued = true;
                    }
                }
                if (!ok) break;
                // the same for the first sub-chunk of the next item, when that item is a SCAN one
                while (pending == -3) {
                    const int t2 = ring.take(n++, ok);
                    if (t2 >= 0 && item_of(pl, t2).kind == kItemPass) continue;
                    pending = t2;
                }
                if (ok && pending >= 0 && item_of(pl, pending).kind == kItemScan) {
                    if (!wait_cb_tiles()) { ok = false; break; }
                    tc_fence_after();
                    issue_cb();
                    cb_issued = true;
                }
            }
            if (!ok) { tc::set_error(err, tc::kErrTimeout); *abort_flag = 1; }
            // retire: every MMA issued must be complete before TMEM is freed
            mma_commit(smem_u32(&bars[fDone]));
            mbar_wait(smem_u32(&bars[fDone]), 0, tc::kWaitNs);
        }
        __syncwarp();
    } else if (warp < 6) {
        // ---- state warps: cumsum, state hand-off, w o x; PASS items --------------------------
        const int r = 32 * (warp & 3) + lane;          // TMEM lane = state row s / token row t
        const int w4 = warp & 3;
        const uint32_t lane_base = (uint32_t)(32 * w4) << 16;
        const bool leader = r == 0;
        uint8_t *wx = smem + Cfg::kWx;
        uint8_t *hc = smem + Cfg::kHc;
        float2 *tot = (float2 *)(smem + Cfg::kTot);    // [2 buffers][4 warps]
        int qc = 0;
        int nstage = 0, pass_issued = 0;               // bulk copies into the staging buffers: waited, issued
        for (int n = 0;; ++n) {
            const int t = ring.group_take(n, leader, kBarState, 128, bcast_state, ok, err);
            if (t < 0) break;
            const FusedItem it = item_of(pl, t);
            const int bhA = 2 * it.pair, b = (int)(bhA / pr.nh), hA = (int)(bhA % pr.nh);
            if (it.kind == kItemPass) {
                run_pass(it, smem, bars, r, lane, leader, bhA, h0, s_loc, sdec, h_st, cnt, pl.npair, qc, wait_ns, err, ok,
                         nstage, pass_issued);
                continue;
            }
            const bool scan = it.kind == kItemScan;
            const float2 a2 = make_float2(Ap[hA] * kLog2e, Ap[hA + 1] * kLog2e);
            // entering state of both heads (SCAN): h0 (zeros if absent) for super-chunk 0, else the
            // state the PASS items wrote; a STATE item starts from zero
            const float *srcA = nullptr;
            int64_t hstride = HS;
            if (scan && it.m == 0 && h0) srcA = h0 + (int64_t)bhA * HS;
            if (scan && it.m > 0) {
                bool fail = false;
                if (leader && !wait_count(cnt + pl.npair + it.pair, Cfg::kSlices, wait_ns)) fail = true;
                if (tc::named_bar_or(kBarState, 128, fail)) { ok = false; tc::set_error(err, tc::kErrTimeout); }
                srcA = h_st + it.slot * HS;
                hstride = (int64_t)it.nsup * HS;
            }
            float2 dsum = make_float2(0.f, 0.f);        // log2 decay of the whole item (STATE)
            uint32_t n_dt = load_dt2<kRagged>(dt, pr, b, hA, (int64_t)it.sub_begin * kQ + r);
            // The entering state, as it is, into the state columns of TMEM before the sub-chunk loop
            // (which then always starts from TMEM), once the MMAs of the items before are done with
            // them: from memory with 16-byte alignment by two bulk copies into the w o x and
            // bf16-state buffers ([head][p][s] float32), else by plain loads, or zeros.
            {
                const bool staged = srcA && ((uintptr_t)srcA & 15u) == 0 && ((hstride * 4) & 15) == 0;
                if (qc > 0 && ok && !mbar_wait(smem_u32(&bars[fUpdate]), (qc - 1) & 1, wait_ns)) {
                    ok = false;
                    tc::set_error(err, tc::kErrTimeout);
                }
                if (staged) {
                    if (leader && ok) {
                        fence_proxy_async_smem();
                        mbar_arrive_expect_tx(smem_u32(&bars[fStage]), (uint32_t)(2 * HS * 4));
                        for (int hh = 0; hh < 2; ++hh)
                            bulk_load(smem_u32(smem + Cfg::kWx + hh * HS * 4), srcA + hh * hstride,
                                      (uint32_t)(HS * 4), smem_u32(&bars[fStage]));
                        ++pass_issued;
                    }
                    if (ok && !mbar_wait(smem_u32(&bars[fStage]), nstage & 1, wait_ns)) {
                        ok = false;
                        tc::set_error(err, tc::kErrTimeout);
                    }
                    ++nstage;
                }
                if (ok) {
                    const float *stg = (const float *)(smem + Cfg::kWx) + r;
#pragma unroll 1
                    for (int hc32 = 0; hc32 < 4; ++hc32) {
                        const int hh = hc32 >> 1, c32 = 32 * (hc32 & 1);
                        uint32_t v[32];
                        if (staged) {
#pragma unroll
                            for (int j = 0; j < 32; ++j) v[j] = __float_as_uint(stg[(hh * 64 + c32 + j) * S]);
                        } else if (srcA) {
                            const float *src = srcA + hh * hstride + r;
#pragma unroll
                            for (int j = 0; j < 32; ++j) v[j] = __float_as_uint(__ldcg(src + (int64_t)(c32 + j) * S));
                        } else {
#pragma unroll
                            for (int j = 0; j < 32; ++j) v[j] = 0u;
                        }
                        const uint32_t ta = tmem + lane_base + Cfg::kTst + 64 * hh + c32;
                        tmem_st16(ta + 0, *reinterpret_cast<uint32_t(*)[16]>(&v[0]));
                        tmem_st16(ta + 16, *reinterpret_cast<uint32_t(*)[16]>(&v[16]));
                    }
                    tmem_st_wait();
                }
                // every thread has read the staging buffers before the hand-off writes the bf16 copy
                // over them
                if (staged) tc::named_bar_sync(kBarState, 128);
            }
            for (int q = 0; q < it.nq; ++q, ++qc) {
                const int xs = qc % kXS;
                const float2 dtp = tc::unpack_bf16x2(n_dt);
                if (q + 1 < it.nq) n_dt = load_dt2<kRagged>(dt, pr, b, hA, (int64_t)(it.sub_begin + q + 1) * kQ + r);
                // cumsum of A dt over the sub-chunk (log2 units): this row's value and the total
                const float2 pre = warp_cumsum2(make_float2(a2.x * dtp.x, a2.y * dtp.y), lane);
                float2 *tq = tot + (qc & 1) * 4;
                if (lane == 31) tq[w4] = pre;
                tc::named_bar_sync(kBarState, 128);
                float2 gr, gl;
                cumsum_from_totals(tq, w4, pre, gr, gl);
                dsum.x += gl.x;
                dsum.y += gl.y;
                // the update of qc - 1 has produced the state and read w o x (and C h^T of the same
                // sub-chunk, issued before it, has read the bf16 copy)
                if (q > 0 && ok && !mbar_wait(smem_u32(&bars[fUpdate]), (qc - 1) & 1, wait_ns)) {
                    ok = false;
                    tc::set_error(err, tc::kErrTimeout);
                }
                if (ok) {
                    tc_fence_after();
                    // state (float32, TMEM) -> bf16 copy [s][p] for C h^T (SCAN), and the state times
                    // 2^(G_last) back to TMEM for the update to accumulate on
#pragma unroll 1
                    for (int hc32 = 0; hc32 < 4; ++hc32) {          // head hc32 / 2, columns 32 (hc32 % 2) ..
                        const int hh = hc32 >> 1, c32 = 32 * (hc32 & 1);
                        const float dec = exp2f(hh ? gl.y : gl.x);
                        const uint32_t ta = tmem + lane_base + Cfg::kTst + 64 * hh + c32;
                        uint32_t v[32];
                        tmem_ld16(ta + 0, *reinterpret_cast<uint32_t(*)[16]>(&v[0]));
                        tmem_ld16(ta + 16, *reinterpret_cast<uint32_t(*)[16]>(&v[16]));
                        tmem_ld_wait();
                        if (scan) {
                            uint8_t *hrow = hc + hh * kAtom;
#pragma unroll
                            for (int c = 0; c < 4; ++c) {
                                uint4 o;
                                o.x = tc::pack_bf16x2(__uint_as_float(v[8 * c + 0]), __uint_as_float(v[8 * c + 1]));
                                o.y = tc::pack_bf16x2(__uint_as_float(v[8 * c + 2]), __uint_as_float(v[8 * c + 3]));
                                o.z = tc::pack_bf16x2(__uint_as_float(v[8 * c + 4]), __uint_as_float(v[8 * c + 5]));
                                o.w = tc::pack_bf16x2(__uint_as_float(v[8 * c + 6]), __uint_as_float(v[8 * c + 7]));
                                *(uint4 *)(hrow + tc::sw128(r, (c32 >> 3) + c)) = o;
                            }
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
                    if (scan) mbar_arrive(smem_u32(&bars[fHReady]));
                }
                // x row r of both heads: w o x into the Wx tile (the update of qc - 1 has read it)
                if (ok && !mbar_wait(smem_u32(&bars[fXFull0 + xs]), (qc / kXS) & 1, wait_ns)) {
                    ok = false;
                    tc::set_error(err, tc::kErrTimeout);
                }
                if (ok) {
                    // w_t rounded to bf16 and the product taken in bf16 pairs (the product is an MMA
                    // operand, rounded to bf16 either way)
                    const float w0 = dtp.x * exp2f(gl.x - gr.x), w1 = dtp.y * exp2f(gl.y - gr.y);
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        const uint8_t *xt = smem + Cfg::kX + xs * Cfg::kXSlot + hh * kAtom;
                        uint8_t *wt = wx + hh * kAtom;
                        const __nv_bfloat162 w2 = __float2bfloat162_rn(hh ? w1 : w0);
                        uint4 vx[8];
#pragma unroll
                        for (int c = 0; c < 8; ++c) vx[c] = *(const uint4 *)(xt + tc::sw128(r, c));
#pragma unroll
                        for (int c = 0; c < 8; ++c) {
                            uint4 o;
                            o.x = tc::mul_bf16x2(vx[c].x, w2);
                            o.y = tc::mul_bf16x2(vx[c].y, w2);
                            o.z = tc::mul_bf16x2(vx[c].z, w2);
                            o.w = tc::mul_bf16x2(vx[c].w, w2);
                            *(uint4 *)(wt + tc::sw128(r, c)) = o;
                        }
                    }
                    fence_proxy_async_smem();
                    mbar_arrive(smem_u32(&bars[fXReady]));
                }
            }
            // the state after the item: h_final (the last super-chunk of a sequence) or the state a
            // STATE item's super-chunk produces from zero, with its log2 decay
            const bool final = scan && it.m == it.nsup - 1 && h_final;
            if (final || !scan) {
                if (ok && !mbar_wait(smem_u32(&bars[fUpdate]), (qc - 1) & 1, wait_ns)) {
                    ok = false;
                    tc::set_error(err, tc::kErrTimeout);
                }
                if (ok) {
                    tc_fence_after();
#pragma unroll 1
                    for (int hh = 0; hh < 2; ++hh) {
                        float *dst = scan ? h_final + (int64_t)(bhA + hh) * HS + r
                                          : s_loc + (it.slot + (int64_t)hh * it.nsup) * HS + r;
#pragma unroll 1
                        for (int c0 = 0; c0 < 64; c0 += 16) {
                            uint32_t v[16];
                            tmem_ld16(tmem + lane_base + Cfg::kTst + 64 * hh + c0, v);
                            tmem_ld_wait();
#pragma unroll
                            for (int j = 0; j < 16; ++j) dst[(int64_t)(c0 + j) * S] = __uint_as_float(v[j]);
                        }
                    }
                    if (!scan && leader) {
                        sdec[it.slot] = dsum.x;
                        sdec[it.slot + it.nsup] = dsum.y;
                    }
                }
                if (!scan) {
                    // publish: every thread's stores, then one count per finished STATE item
                    __threadfence();
                    tc::named_bar_sync(kBarState, 128);
                    if (leader) atomicAdd(cnt + it.pair, 1);
                }
            }
        }
        if (!ok) *abort_flag = 1;
        // retire: a staging copy whose wait expired must land before the CTA may exit
        if (leader && pass_issued > 0) mbar_wait(smem_u32(&bars[fStage]), (pass_issued - 1) & 1, tc::kWaitNs);
    } else if (warp < 14) {
        // ---- P warps: P and the scaled C h^T of each SCAN sub-chunk ---------------------------
        const int half = (warp - 6) >> 2;              // columns 64 half .. 64 half + 63; C h^T of head `half`
        const int w4 = warp & 3;
        const int r = 32 * w4 + lane;                  // TMEM lane = token row i
        const uint32_t lane_base = (uint32_t)(32 * w4) << 16;
        const bool leader = warp == 6 && lane == 0;
        float *arr = (float *)(smem + Cfg::kArr);
        float *myGd = arr + half * (Cfg::kArrHead / 4);  // the arrays this thread fills (head `half`)
        float *myF = myGd + kQ, *myGe = myF + kQ;
        float2 *tot = (float2 *)(smem + Cfg::kTot) + 8 + 4 * half;   // this half's per-warp totals
        auto group_sync = [&]() { tc::named_bar_sync(kBarP, 256); };
        int qs = 0;
        for (int n = 0;; ++n) {
            const int t = ring.group_take(n, leader, kBarP, 256, bcast_p, ok, err);
            if (t < 0) break;
            const FusedItem it = item_of(pl, t);
            if (it.kind != kItemScan) continue;
            const int bhA = 2 * it.pair, b = (int)(bhA / pr.nh), hA = (int)(bhA % pr.nh);
            const float2 a2 = make_float2(Ap[hA] * kLog2e, Ap[hA + 1] * kLog2e);
            uint32_t n_dt = load_dt2<kRagged>(dt, pr, b, hA, (int64_t)it.sub_begin * kQ + r);
            for (int q = 0; q < it.nq; ++q, ++qs) {
                const float2 dtp = tc::unpack_bf16x2(n_dt);
                if (q + 1 < it.nq) n_dt = load_dt2<kRagged>(dt, pr, b, hA, (int64_t)(it.sub_begin + q + 1) * kQ + r);
                const float2 pre = warp_cumsum2(make_float2(a2.x * dtp.x, a2.y * dtp.y), lane);
                if (lane == 31) tot[w4] = pre;
                // the totals are visible, and every thread is past P of the previous sub-chunk (the
                // column arrays are free)
                group_sync();
                float2 gr, gl;
                cumsum_from_totals(tot, w4, pre, gr, gl);
                const float g0 = gr.x, g1 = gr.y;
                {
                    const float gown = half ? g1 : g0, dto = half ? dtp.y : dtp.x;
                    const float gend = __shfl_sync(0xffffffffu, gown, lane | 15);   // G at the end of r's 16-token block
                    myGd[r] = gown - __log2f(dto);                // dt = 0: +inf, so 2^(G_i - Gd_j) = 0
                    myF[r] = ex2_approx(gend - gown) * dto;       // 2^(G_e - G_j) <= 1 for A dt <= 0
                    if ((r & 15) == 15) myGe[r >> 4] = gown;
                }
                group_sync();
                if (ok && !mbar_wait(smem_u32(&bars[fCb]), qs & 1, wait_ns)) { ok = false; tc::set_error(err, tc::kErrTimeout); }
                if (ok) {
                    tc_fence_after();
                    const uint32_t tcb = tmem + lane_base + Cfg::kTcb;
                    const float *GdA = arr, *FA = arr + kQ, *GeA = arr + 2 * kQ;
                    const float *GdB = GdA + Cfg::kArrHead / 4, *FB = FA + Cfg::kArrHead / 4, *GeB = GeA + Cfg::kArrHead / 4;
                    // The four 16-column blocks of this half come in two pairs of the same kind
                    // (above the diagonal, left of every row of the warp, or meeting the diagonal).
                    // Per pair: both blocks' C B^T loaded, one wait, then P_A of each block into its
                    // first 8 columns and P_B into its last 8.
                    const int wrow_lo = 32 * w4, wrow_hi = wrow_lo + 31;
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
                                    pk[2 * e4] = tc::pack_bf16x2(pA01.x, pA01.y);
                                    pk[2 * e4 + 1] = tc::pack_bf16x2(pA23.x, pA23.y);
                                    pk[8 + 2 * e4] = tc::pack_bf16x2(pB01.x, pB01.y);
                                    pk[8 + 2 * e4 + 1] = tc::pack_bf16x2(pB23.x, pB23.y);
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
                                    pk[2 * e4] = tc::pack_bf16x2(pa[0], pa[1]);
                                    pk[2 * e4 + 1] = tc::pack_bf16x2(pa[2], pa[3]);
                                    pk[8 + 2 * e4] = tc::pack_bf16x2(pb[0], pb[1]);
                                    pk[8 + 2 * e4 + 1] = tc::pack_bf16x2(pb[2], pb[3]);
                                }
                                tmem_st16(tcb + jb, pk);
                            }
                        }
                    }
                    // C h^T of head `half`, row r: Y <- 2^(G_i) Y before P x accumulates onto it
                    if (!mbar_wait(smem_u32(&bars[fYs]), qs & 1, wait_ns)) { ok = false; tc::set_error(err, tc::kErrTimeout); }
                    if (ok) {
                        tc_fence_after();
                        const float eg = ex2_approx(half ? g1 : g0);
                        const uint32_t ty = tmem + lane_base + Cfg::kTy + (uint32_t)(qs & 1) * 128 + 64 * half;
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
                    mbar_arrive(smem_u32(&bars[fPReady]));
                }
            }
        }
        if (!ok) *abort_flag = 1;
    } else if (warp >= 15) {
        // ---- epilogue warps: y = Y + D x of each SCAN sub-chunk, staged over its x tile -------
        const int r = 32 * (warp & 3) + lane;          // TMEM lane = token row i
        const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
        const bool leader = warp == 15 && lane == 0;   // also issues the bulk stores
        int qc = 0, qs = 0;
        for (int n = 0;; ++n) {
            const int t = ring.group_take(n, leader, kBarEpi, 128, bcast_epi, ok, err);
            if (t < 0) break;
            const FusedItem it = item_of(pl, t);
            if (it.kind == kItemPass) continue;
            if (it.kind == kItemState) { qc += it.nq; continue; }
            const int bhA = 2 * it.pair, b = (int)(bhA / pr.nh), hA = (int)(bhA % pr.nh);
            const float dA = Dp[hA], dB = Dp[hA + 1];
            for (int q = 0; q < it.nq; ++q, ++qc, ++qs) {
                const int xs = qc % kXS;
                uint8_t *ystage = smem + Cfg::kX + xs * Cfg::kXSlot;
                if (ok && !mbar_wait(smem_u32(&bars[fIntra0 + (qs & 1)]), (qs >> 1) & 1, wait_ns)) {
                    ok = false;
                    tc::set_error(err, tc::kErrTimeout);
                }
                if (ok) {
                    tc_fence_after();
#pragma unroll 1
                    for (int hh = 0; hh < 2; ++hh) {
                        const uint32_t ty = tmem + lane_base + Cfg::kTy + (uint32_t)(qs & 1) * 128 + 64 * hh;
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
                            for (int c = 0; c < 4; ++c) xv[c] = *(const uint4 *)(yrow + tc::sw128(r, (c32 >> 3) + c));
                            tmem_ld_wait();
#pragma unroll
                            for (int c = 0; c < 4; ++c) {
                                const uint32_t in[4] = {xv[c].x, xv[c].y, xv[c].z, xv[c].w};
                                uint32_t o[4];
#pragma unroll
                                for (int e = 0; e < 4; ++e) {
                                    const float2 yv = __ffma2_rn(tc::unpack_bf16x2(in[e]), make_float2(dh, dh),
                                                                 make_float2(__uint_as_float(v[8 * c + 2 * e]),
                                                                             __uint_as_float(v[8 * c + 2 * e + 1])));
                                    o[e] = tc::pack_bf16x2(yv.x, yv.y);
                                }
                                *(uint4 *)(yrow + tc::sw128(r, (c32 >> 3) + c)) = make_uint4(o[0], o[1], o[2], o[3]);
                            }
                        }
                    }
                    tc_fence_before();
                    mbar_arrive(smem_u32(&bars[fEpi0 + (qs & 1)]));
                    fence_proxy_async_smem();
                }
                // all rows staged (every epilogue thread reaches this, errors or not)
                tc::named_bar_sync(kBarEpi, 128);
                if (leader) {
                    // the slot goes back to the x loader as soon as the store has read it
                    if (ok) {
                        const int t0 = (it.sub_begin + q) * kQ;
                        tma_store_4d(&tmY, smem_u32(ystage), 0, hA, t0, b);
                        tma_store_4d(&tmY, smem_u32(ystage + kAtom), 0, hA + 1, t0, b);
                        bulk_commit();
                    }
                    bulk_wait_read();
                    mbar_arrive(smem_u32(&bars[fYSt0 + xs]));
                }
            }
        }
        if (!ok) *abort_flag = 1;
        if (leader) bulk_wait_all();
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) tmem_dealloc(tmem, Cfg::kTmemCols);
}

}  // namespace

cudaError_t launch_fused_pair(const Problem &pr, const void *x, const void *dt, const float *A, const void *Bm,
                              const void *Cm, const float *D, const float *h0, float *h_final, void *y,
                              const FusedPlan &pl, const FusedWork &w, unsigned long long wait_ns, cudaStream_t st)
{
    if (pl.n_items == 0) return cudaSuccess;
    CUtensorMap mC, mB, mX, mY;
    if (!tc::make_map_4d(&mC, Cm, pr.S, pr.G, pr.L, pr.B, kQ) || !tc::make_map_4d(&mB, Bm, pr.S, pr.G, pr.L, pr.B, kQ) ||
        !tc::make_map_4d(&mX, x, pr.H, pr.nh, pr.L, pr.B, kQ) || !tc::make_map_4d(&mY, y, pr.H, pr.nh, pr.L, pr.B, kQ))
        return cudaErrorInvalidValue;
    auto kern = pr.L % kQ == 0 ? k_ssd_fwd_fused<false> : k_ssd_fwd_fused<true>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)FusedCfg::kSmem);
    if (e != cudaSuccess) return e;

    const int grid = pl.n_items < tc::current_sms() ? pl.n_items : tc::current_sms();
    kern<<<grid, FusedCfg::kThreads, FusedCfg::kSmem, st>>>(mC, mB, mX, mY, (const __nv_bfloat16 *)dt, A, D, h0,
                                                           h_final, w.s_local, w.h_start, w.sdec, w.hdr, w.cnt, pr,
                                                           pl, wait_ns);
    return cudaGetLastError();
}

int fused_pass_slices() { return FusedCfg::kSlices; }

}  // namespace ssd
