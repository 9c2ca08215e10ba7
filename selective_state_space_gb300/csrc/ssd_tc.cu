// ssd_tc.cu -- tensor-core kernels (tcgen05 MMA, TMEM accumulators, TMA staging).
#include "ssd_tc.cuh"

namespace ssd {

bool tc_supported(const Problem &) { return false; }

cudaError_t launch_chunk_state_tc(const Problem &, const void *, const void *, const void *,
                                  const float *, float *, cudaStream_t)
{
    return cudaErrorNotSupported;
}

cudaError_t launch_chunk_scan_tc(const Problem &, const void *, const void *, const void *,
                                 const void *, const float *, const float *, const void *, void *,
                                 cudaStream_t)
{
    return cudaErrorNotSupported;
}

}  // namespace ssd
