// ssd_tc.cuh -- tensor-core (tcgen05 / TMEM / TMA) kernels for the chunk_state
// and chunk_scan stages, for the shapes they are specialised for.
#pragma once

#include "ssd_common.cuh"

namespace ssd {

// True when the tensor-core kernels handle this problem shape.
bool tc_supported(const Problem &pr);

cudaError_t launch_chunk_state_tc(const Problem &pr, const void *x, const void *dt, const void *Bm,
                                  const float *G, float *s_local, cudaStream_t st);
cudaError_t launch_chunk_scan_tc(const Problem &pr, const void *x, const void *dt, const void *Bm,
                                 const void *Cm, const float *D, const float *G, const void *h_start,
                                 void *y, cudaStream_t st);

}  // namespace ssd
