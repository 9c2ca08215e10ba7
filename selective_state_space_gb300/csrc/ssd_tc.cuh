// ssd_tc.cuh -- tensor-core (tcgen05 / TMEM / TMA) kernels for the chunk_state
// and chunk_scan stages, for the shapes they are specialised for.
#pragma once

#include "ssd_common.cuh"

namespace ssd {

// True when the tensor-core kernels handle this problem shape.
bool tc_supported(const Problem &pr);

// States of super-chunks m < nm (R chunks each) from a zero start, written to
// s_local[b][h][m] with a super-chunk extent of nsup.  dtT (nullable) is dt as float32
// in the [b][h][L] layout of G; with it, dt and G reach the kernel by bulk copies
// instead of per-thread loads.  `err` receives error bits.
// Whether launch_chunk_state_tc with these arguments zeroes s_local first (one
// cudaMemsetAsync): it does when a CTA's slice of stages cuts a super-chunk.
bool chunk_state_tc_memsets(const Problem &pr, int R, int nm);
cudaError_t launch_chunk_state_tc(const Problem &pr, const void *x, const void *dt, const float *dtT,
                                  const void *Bm, const float *G, float *s_local, int R, int nsup, int nm,
                                  int *err, cudaStream_t st);
// Output y for every super-chunk (R chunks, nsup of them): super-chunks m < hs_from
// start from h0 (NULL: zeros), the others from h_start[b][h][m]; the last super-chunk
// also writes h_final when it is not NULL.
cudaError_t launch_chunk_scan_tc(const Problem &pr, const void *x, const void *dt, const void *Bm,
                                 const void *Cm, const float *D, const float *G, const float *h0,
                                 const float *h_start, float *h_final, void *y, int R, int nsup, int hs_from,
                                 int *err, cudaStream_t st);

}  // namespace ssd
