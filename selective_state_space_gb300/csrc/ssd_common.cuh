// ssd_common.cuh -- shared definitions for the SSD kernels (GPU side only).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "ssd.h"

namespace ssd {

// G is stored pre-multiplied by log2(e) so that every later stage uses exp2
// (blog section "Kernel 1: cumulative sum": the cumsum is scaled by log2(e)).
constexpr float kLog2e = 1.4426950408889634f;

// Validated problem sizes, passed by value to kernels and launchers.
struct Problem {
    int64_t B, L, nh, H, S, G, T, nc, hpg;
    int in_dt, out_dt;
    int dt_f32;           // 1: dt is float32 while x, B, C are bfloat16 (SSD_DT_FLOAT32)
    // 0 selects the tensor-core kernels built for the test hook of the timeout path (every
    // wait for another warp's work not satisfied at once expires); else 250 ms, the bound
    // the normal kernels have built in
    unsigned long long wait_ns;
};

__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) {
    return __float2bfloat16_rn(v);
}

// Programmatic dependent launch.  The kernels after the cumsum are launched with
// programmatic stream serialisation (launch_pdl): each lets the next kernel of the
// stream start its launch and prologue early (pdl_trigger) and waits for the previous
// kernel's results, with their memory visible, before reading them (pdl_wait).  Both
// instructions are no-ops for a kernel launched without the attribute.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args &&...args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<Args &&>(args)...);
}

// A run of sequences, i.e. (batch, head) pairs in b * nh + h order: [lo, lo + n).
// The chunk_state and state_passing stages work on one run at a time; their
// per-super-chunk states for sequence bh and super-chunk m sit at index
// (bh - lo) * nsup + m of the state arrays they are given.
struct SeqRange {
    int64_t lo, n;
};

// Host-side launchers (one per stage).  Each returns the launch status.
// dtT (nullable): also write dt as float32 in the [b][h][L] layout of G, for the sequences
// (b * nh + h) in [dtT_lo, dtT_hi) only.  count (nullable, zeroed beforehand): each CTA adds 1
// to it once its part of G is written and visible device-wide; there are cumsum_ctas(pr) CTAs.
// dt is float32 when pr.dt_f32 (else in the input dtype); dt16 (nullable): also write dt
// rounded to bfloat16 in its own [b][t][h] layout.
cudaError_t launch_chunk_cumsum(const Problem &pr, const void *dt, const float *A, float *G,
                                float *dtT, int64_t dtT_lo, int64_t dtT_hi, cudaStream_t st,
                                unsigned *count = nullptr, __nv_bfloat16 *dt16 = nullptr);
unsigned cumsum_ctas(const Problem &pr);
cudaError_t launch_chunk_state_simt(const Problem &pr, const void *x, const void *dt,
                                    const void *Bm, const float *G, float *s_local,
                                    cudaStream_t st);
// Super-chunk state passing over the sequences of `seqs`: h_start[m] for m < nsup
// (R chunks per super-chunk); s_local is read for m < nm; h_final (nullable, indexed
// by the absolute sequence) is written when nm == nsup.
cudaError_t launch_state_passing(const Problem &pr, SeqRange seqs, const float *G, const float *s_local,
                                 const float *h0, float *h_start, float *h_final, int R, int nsup, int nm,
                                 cudaStream_t st);
cudaError_t launch_chunk_scan_simt(const Problem &pr, const void *x, const void *dt,
                                   const void *Bm, const void *Cm, const float *D, const float *G,
                                   const float *h_start, void *y, cudaStream_t st);
// Gradients of the forward pass (ssd_bwd.cu).  Pointers as in ssd_bwd of include/ssd.h.
struct BwdArgs {
    const void *x, *dt, *Bm, *Cm, *dy;
    const float *A, *D, *h0, *dh_final;
    void *dx, *ddt, *dB, *dC;
    float *dA, *dD, *dh0;
};
// Workspace of the gradient pass, carved by bwd_workspace: G, the states entering each
// chunk, the gradients of the states leaving them, six per-token float arrays and the
// per-slice partial sums of dB and dC.  nslice slices of hps heads split each group.
struct BwdWork {
    float *G, *h_start, *lam, *Qd, *Nd, *Cmd, *Dd, *Rw, *Ad, *dBp, *dCp;
    int nslice, hps;
};
bool bwd_supported(const Problem &pr);
// Carves `base` (nullptr: sizes only) and returns the bytes needed.
size_t bwd_workspace(const Problem &pr, void *base, BwdWork *w);
cudaError_t launch_bwd(const Problem &pr, const BwdArgs &a, const BwdWork &w, cudaStream_t st);

// Mamba-1 selective scan (s6_scan.cu): validated sizes of an s6_desc.
struct S6Problem {
    int64_t B, L, dim, N, G;
    int in_dt, out_dt;
};
cudaError_t launch_s6_scan(const S6Problem &p, const void *x, const void *delta, const float *A, const void *Bm,
                           const void *Cm, const float *D, const float *h0, void *y, float *h_final, cudaStream_t st);

cudaError_t launch_ssd_step(const Problem &pr, const void *x, const void *dt, const float *A,
                            const void *Bm, const void *Cm, const float *D, float *h, void *y,
                            cudaStream_t st);

}  // namespace ssd
