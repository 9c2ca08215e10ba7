// ssd_tf32.cu -- the chunked forward pass for float32 inputs on the tensor cores
// (tcgen05 MMAs of kind::tf32, float32 accumulators in TMEM).
//
// Method: NVIDIA developer blog "Accelerating Mamba-2 with High-Performance Forward Pass
// Kernels in NVIDIA CUDA Tile", section "Mamba-2 architecture" (the chunk jump and the
// chunk output) and "Kernel 3: compute_out", whose products take TF32 operands.
//
// Design.  One CTA of 128 threads per (batch, head) walks its whole sequence in sub-chunks
// of 128 tokens and carries the state h^T (S x H, float32) in TMEM.  The in-chunk cumsum is
// taken by the CTA itself, relative to the sub-chunk start (a block scan of A dt log2 e),
// so the pass is one launch: the chunked result does not depend on where the chunks are
// cut, and every exponent it evaluates is <= 0.  Per sub-chunk, in four phases separated by
// barriers (so four shared-memory regions serve every operand in turn):
//   1. C (rows i) and B (rows j) tiles and a copy of the state h [p][s], staged K-major;
//      CB = C B^T (M = i, N = j, K = s) and Ys = C h^T (M = i, N = p, K = s).
//   2. P[i][j] = CB[i][j] 2^(G_i - G_j) dt_j for j <= i (from TMEM, CUDA cores), x^T and
//      (w o x)^T with w_t = dt_t 2^(G_last - G_t), B^T; the state decays by 2^(G_last).
//   3. Yi = P x (M = i, N = p, K = j) and h^T += B^T (w o x) (M = s, N = p, K = t).
//   4. y_i = 2^(G_i) Ys_i + Yi_i + D x_i.
// Every MMA operand is rounded to TF32 (cvt.rna) when it is staged; the accumulators and
// the carried state stay float32.  Operands sit in 128-byte-swizzled K-major panels (32
// floats per row), the layout the MMA descriptors describe; one MMA step is K = 8 (32 bytes
// of a row).  With S = 64 the state update still runs at M = 128: rows s >= S of B^T are
// zero, so those state rows stay zero.
#include "sm100_ptx.cuh"
#include "ssd_tc.cuh"

namespace ssd {
namespace {

using namespace ptx;

constexpr int kTQ = 128;                        // tokens per sub-chunk (MMA M)
constexpr int kTH = 64;                         // head width H
constexpr uint32_t kPan128 = 128u * 128u;       // one 128-row panel (128 bytes per row)
constexpr uint32_t kPan64 = 64u * 128u;         // one 64-row panel
constexpr uint64_t kTf32WaitNs = 250000000ull;  // bound on each wait for the MMAs

// shared memory: four regions reused by the phases, then the small arrays
constexpr uint32_t kR1 = 0;                     // C [i][s], then P [i][j]          (64 KB)
constexpr uint32_t kR2 = 65536;                 // B [j][s], then B^T [s][t]         (64 KB)
constexpr uint32_t kR3 = 131072;                // h [p][s], then x^T [p][j]         (32 KB)
constexpr uint32_t kR4 = 163840;                // (w o x)^T [p][t]                 (32 KB)
constexpr uint32_t kSmallOff = 196608;          // G [128], dt [128], warp sums [4], barrier, TMEM slot
constexpr uint32_t kTf32Smem = kSmallOff + 1024 + 16 + 16 + 1024;   // + alignment slack
// TMEM columns: C B^T 0..127, Ys 128..191, Yi 192..255, the state h^T 256..319
constexpr uint32_t kTcb = 0, kTys = 128, kTyi = 192, kTst = 256, kTcols = 512;

__device__ __forceinline__ uint32_t swz(uint32_t r, uint32_t c) { return r * 128u + (((c ^ (r & 7u)) & 7u) << 4); }

// Byte offset of element (row r, column k) of a K-major float tile in 128-byte-swizzled
// panels of `panel` bytes (panel k / 32 holds columns 32 (k / 32) ..).
__device__ __forceinline__ uint32_t kmaj(uint32_t r, uint32_t k, uint32_t panel)
{
    return (k >> 5) * panel + swz(r, (k & 31u) >> 2) + ((k & 3u) << 2);
}

__device__ __forceinline__ float to_tf32(float v)
{
    uint32_t o;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(o) : "f"(v));
    return __uint_as_float(o);
}

// Instruction descriptor for kind::tf32 with float32 accumulation, both operands K-major:
//   [4,6) D format (1 = f32)  [7,10) A format (2 = tf32)  [10,13) B format (2 = tf32)
//   [17,23) N >> 3  [24,29) M >> 4
__host__ __device__ constexpr uint32_t idesc_tf32(uint32_t M, uint32_t N)
{
    return (1u << 4) | (2u << 7) | (2u << 10) | ((N >> 3) << 17) | ((M >> 4) << 24);
}

__device__ __forceinline__ void mma_tf32(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}"
        ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// D += A B^T over K = 8 k steps of 32 bytes: A rows in panels of pa bytes, B rows in panels of pb.
__device__ __forceinline__ void mma_run(uint32_t d, uint32_t a_base, uint32_t pa, uint32_t b_base, uint32_t pb,
                                        int ksteps, uint32_t idesc, bool first_overwrites)
{
    for (int kk = 0; kk < ksteps; ++kk) {
        const uint32_t oa = (uint32_t)(kk >> 2) * pa + (uint32_t)(kk & 3) * 32u;
        const uint32_t ob = (uint32_t)(kk >> 2) * pb + (uint32_t)(kk & 3) * 32u;
        mma_tf32(d, smem_desc(a_base + oa, 16, 1024), smem_desc(b_base + ob, 16, 1024), idesc,
                 (kk > 0 || !first_overwrites) ? 1u : 0u);
    }
}

template <int S, typename Tout>
__global__ void __launch_bounds__(128, 1)
k_ssd_tf32(const float *__restrict__ x, const float *__restrict__ dt, const float *__restrict__ A,
           const float *__restrict__ Bm, const float *__restrict__ Cm, const float *__restrict__ Dp,
           const float *__restrict__ h0, Tout *__restrict__ y, float *__restrict__ h_final, Problem pr, int *err)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    float *sG = (float *)(smem + kSmallOff);
    float *sDt = sG + kTQ;
    float *sWs = sDt + kTQ;                      // 4 warp totals
    uint64_t *bar = (uint64_t *)(smem + kSmallOff + 1024 + 16);
    uint32_t *slot = (uint32_t *)(bar + 1);
    const int r = threadIdx.x, warp = r >> 5, lane = r & 31;
    const uint32_t lane_base = (uint32_t)(32 * warp) << 16;
    const int64_t bh = blockIdx.x;
    const int b = (int)(bh / pr.nh), h = (int)(bh % pr.nh), g = (int)(h / pr.hpg);
    const float a2 = A[h] * kLog2e, dh = Dp[h];
    const uint32_t s1 = smem_u32(smem + kR1), s2 = smem_u32(smem + kR2), s3 = smem_u32(smem + kR3),
                   s4 = smem_u32(smem + kR4);

    if (r == 0) {
        mbar_init(smem_u32(bar), 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(slot), kTcols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *slot;
    uint32_t phase = 0;
    auto wait_mmas = [&]() {
        if (!mbar_wait(smem_u32(bar), phase, kTf32WaitNs) && err) atomicOr(err, 1);
        phase ^= 1u;
        tc_fence_after();
    };

    // entering state h^T: lane s, column p (lanes s >= S hold zeros)
#pragma unroll 1
    for (int c0 = 0; c0 < kTH; c0 += 16) {
        uint32_t v[16];
#pragma unroll
        for (int j = 0; j < 16; ++j)
            v[j] = __float_as_uint((r < S && h0) ? h0[(bh * kTH + c0 + j) * S + r] : 0.f);
        tmem_st16(tmem + lane_base + kTst + c0, v);
    }
    tmem_st_wait();

#pragma unroll 1
    for (int64_t t0 = 0; t0 < pr.L; t0 += kTQ) {
        const int n = (int)min((int64_t)kTQ, pr.L - t0);
        const bool on = r < n;
        const int64_t tok = (int64_t)b * pr.L + t0 + r;           // (batch, token) row of this thread
        const int64_t tok_c = on ? tok : (int64_t)b * pr.L + t0;   // a valid row for masked loads
        const float dtr = on ? dt[tok * pr.nh + h] : 0.f;
        // this row of x, loaded once (16-byte vectors, all in flight together) for x^T, w o x and D x
        float4 xr[kTH / 4];
        {
            const float4 *xrow4 = reinterpret_cast<const float4 *>(x + (tok_c * pr.nh + h) * kTH);
#pragma unroll
            for (int q = 0; q < kTH / 4; ++q) xr[q] = on ? xrow4[q] : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        // G relative to the sub-chunk start: inclusive block scan of A dt log2 e (rows past n add 0)
        float v = a2 * dtr;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float u = __shfl_up_sync(0xffffffffu, v, o);
            if (lane >= o) v += u;
        }
        if (lane == 31) sWs[warp] = v;
        __syncthreads();
        for (int w = 0; w < warp; ++w) v += sWs[w];
        sG[r] = v;
        sDt[r] = dtr;
        __syncthreads();
        const float gi = v, gl = sG[kTQ - 1];

        // ---- phase 1: C -> R1 [i][s], B -> R2 [j][s], the state h -> R3 [p][s] ----
        {
            const float *crow = Cm + (tok_c * pr.G + g) * S, *brow = Bm + (tok_c * pr.G + g) * S;
#pragma unroll
            for (int k = 0; k < S; k += 4) {
                float4 cv = on ? *reinterpret_cast<const float4 *>(crow + k) : make_float4(0.f, 0.f, 0.f, 0.f);
                float4 bv = on ? *reinterpret_cast<const float4 *>(brow + k) : make_float4(0.f, 0.f, 0.f, 0.f);
                const uint32_t o = (uint32_t)(k >> 5) * kPan128 + swz((uint32_t)r, (uint32_t)(k & 31) >> 2);
                *reinterpret_cast<float4 *>(smem + kR1 + o) =
                    make_float4(to_tf32(cv.x), to_tf32(cv.y), to_tf32(cv.z), to_tf32(cv.w));
                *reinterpret_cast<float4 *>(smem + kR2 + o) =
                    make_float4(to_tf32(bv.x), to_tf32(bv.y), to_tf32(bv.z), to_tf32(bv.w));
            }
#pragma unroll 1
            for (int c0 = 0; c0 < kTH; c0 += 16) {
                uint32_t hv[16];
                tmem_ld16(tmem + lane_base + kTst + c0, hv);
                tmem_ld_wait();
                if (r < S) {
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        *reinterpret_cast<float *>(smem + kR3 + kmaj((uint32_t)(c0 + j), (uint32_t)r, kPan64)) =
                            to_tf32(__uint_as_float(hv[j]));
                }
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        if (r == 0) {
            mma_run(tmem + kTcb, s1, kPan128, s2, kPan128, S / 8, idesc_tf32(128, 128), true);   // C B^T
            mma_run(tmem + kTys, s1, kPan128, s3, kPan64, S / 8, idesc_tf32(128, kTH), true);    // C h^T
            mma_commit(smem_u32(bar));
        }
        wait_mmas();

        // ---- phase 2: P -> R1 [i][j], x^T -> R3 [p][j], (w o x)^T -> R4 [p][t], B^T -> R2 [s][t] ----
#pragma unroll 1
        for (int j0 = 0; j0 < kTQ; j0 += 16) {
            uint32_t cb[16];
            tmem_ld16(tmem + lane_base + kTcb + j0, cb);
            tmem_ld_wait();
            float p[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                const int j = j0 + e;
                // j <= i < n: the causal mask selects, never multiplies (2^(G_i - G_j) <= 1)
                p[e] = (on && j <= r) ? __uint_as_float(cb[e]) * exp2f(gi - sG[j]) * sDt[j] : 0.f;
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const uint32_t o = (uint32_t)(j0 >> 5) * kPan128 + swz((uint32_t)r, (uint32_t)((j0 & 31) >> 2) + q);
                *reinterpret_cast<float4 *>(smem + kR1 + o) = make_float4(
                    to_tf32(p[4 * q]), to_tf32(p[4 * q + 1]), to_tf32(p[4 * q + 2]), to_tf32(p[4 * q + 3]));
            }
        }
        {
            const float wr = dtr * exp2f(gl - gi);          // 0 for rows past n (dt = 0)
#pragma unroll
            for (int q = 0; q < kTH / 4; ++q) {
                const float xv[4] = {xr[q].x, xr[q].y, xr[q].z, xr[q].w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const uint32_t o = kmaj((uint32_t)(4 * q + e), (uint32_t)r, kPan64);
                    *reinterpret_cast<float *>(smem + kR3 + o) = to_tf32(xv[e]);
                    *reinterpret_cast<float *>(smem + kR4 + o) = to_tf32(wr * xv[e]);
                }
            }
            // B^T: this thread's column t = r, rows s < S from its B row (loaded again, L2-resident,
            // all vectors in flight together), rows s >= S zero
            const float4 *brow4 = reinterpret_cast<const float4 *>(Bm + (tok_c * pr.G + g) * S);
            float4 bq[S / 4];
#pragma unroll
            for (int q = 0; q < S / 4; ++q) bq[q] = on ? brow4[q] : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int q = 0; q < S / 4; ++q) {
                const float bv[4] = {bq[q].x, bq[q].y, bq[q].z, bq[q].w};
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    *reinterpret_cast<float *>(smem + kR2 + kmaj((uint32_t)(4 * q + e), (uint32_t)r, kPan128)) =
                        to_tf32(bv[e]);
            }
#pragma unroll 4
            for (int s = S; s < kTQ; ++s)
                *reinterpret_cast<float *>(smem + kR2 + kmaj((uint32_t)s, (uint32_t)r, kPan128)) = 0.f;
        }
        {
            // the state decays over the whole sub-chunk before the update adds this sub-chunk's part
            const float dec = exp2f(gl);
#pragma unroll 1
            for (int c0 = 0; c0 < kTH; c0 += 16) {
                uint32_t hv[16];
                tmem_ld16(tmem + lane_base + kTst + c0, hv);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 16; ++j) hv[j] = __float_as_uint(__uint_as_float(hv[j]) * dec);
                tmem_st16(tmem + lane_base + kTst + c0, hv);
            }
            tmem_st_wait();
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        if (r == 0) {
            mma_run(tmem + kTyi, s1, kPan128, s3, kPan64, kTQ / 8, idesc_tf32(128, kTH), true);    // P x
            mma_run(tmem + kTst, s2, kPan128, s4, kPan64, kTQ / 8, idesc_tf32(128, kTH), false);   // B^T (w o x)
            mma_commit(smem_u32(bar));
        }
        wait_mmas();

        // ---- phase 4: y_i = 2^(G_i) Ys_i + Yi_i + D x_i ----
        {
            const float eg = exp2f(gi);
            Tout *yrow = y + (tok_c * pr.nh + h) * kTH;
#pragma unroll
            for (int c0 = 0; c0 < kTH; c0 += 16) {
                uint32_t ys[16], yi[16];
                tmem_ld16(tmem + lane_base + kTys + c0, ys);
                tmem_ld16(tmem + lane_base + kTyi + c0, yi);
                tmem_ld_wait();
                if (on) {
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const float4 xv = xr[c0 / 4 + q];
                        const float xs[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int j = 4 * q + e;
                            yrow[c0 + j] = from_f32<Tout>(
                                fmaf(eg, __uint_as_float(ys[j]), __uint_as_float(yi[j])) + dh * xs[e]);
                        }
                    }
                }
            }
        }
        tc_fence_before();
        __syncthreads();     // every region and accumulator is free for the next sub-chunk
        tc_fence_after();
    }

    if (h_final) {
#pragma unroll 1
        for (int c0 = 0; c0 < kTH; c0 += 16) {
            uint32_t hv[16];
            tmem_ld16(tmem + lane_base + kTst + c0, hv);
            tmem_ld_wait();
            if (r < S) {
#pragma unroll
                for (int j = 0; j < 16; ++j) h_final[(bh * kTH + c0 + j) * S + r] = __uint_as_float(hv[j]);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem, kTcols);
}

template <int S, typename Tout>
cudaError_t tf32_launch(const Problem &pr, const float *x, const float *dt, const float *A, const float *Bm,
                        const float *Cm, const float *D, const float *h0, void *y, float *h_final, int *err,
                        cudaStream_t st)
{
    auto kern = k_ssd_tf32<S, Tout>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kTf32Smem);
    if (e != cudaSuccess) return e;
    const int64_t grid = pr.B * pr.nh;
    if (grid == 0) return cudaSuccess;
    if (grid > 0x7fffffffLL) return cudaErrorInvalidValue;
    kern<<<dim3((unsigned)grid), dim3(128), kTf32Smem, st>>>(x, dt, A, Bm, Cm, D, h0, (Tout *)y, h_final, pr, err);
    return cudaGetLastError();
}

}  // namespace

// One CTA walks a whole sequence, so long sequences go to the CUDA-core path, which runs
// their chunks in parallel.
bool tf32_supported(const Problem &pr)
{
    return pr.in_dt == SSD_F32 && pr.H == kTH && (pr.S == 64 || pr.S == 128) && pr.L <= 1024;
}

cudaError_t launch_ssd_tf32(const Problem &pr, const void *x, const void *dt, const float *A, const void *Bm,
                            const void *Cm, const float *D, const float *h0, void *y, float *h_final, int *err,
                            cudaStream_t st)
{
    const float *xf = (const float *)x, *dtf = (const float *)dt, *bf = (const float *)Bm, *cf = (const float *)Cm;
    const bool ob = pr.out_dt == SSD_BF16;
    if (pr.S == 64)
        return ob ? tf32_launch<64, __nv_bfloat16>(pr, xf, dtf, A, bf, cf, D, h0, y, h_final, err, st)
                  : tf32_launch<64, float>(pr, xf, dtf, A, bf, cf, D, h0, y, h_final, err, st);
    if (pr.S == 128)
        return ob ? tf32_launch<128, __nv_bfloat16>(pr, xf, dtf, A, bf, cf, D, h0, y, h_final, err, st)
                  : tf32_launch<128, float>(pr, xf, dtf, A, bf, cf, D, h0, y, h_final, err, st);
    return cudaErrorNotSupported;
}

}  // namespace ssd
