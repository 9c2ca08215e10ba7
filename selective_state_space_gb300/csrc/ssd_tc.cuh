// ssd_tc.cuh -- tensor-core (tcgen05 / TMEM / TMA) kernels for the chunk_state
// and chunk_scan stages, for the shapes they are specialised for.
#pragma once

#include "ssd_common.cuh"

namespace ssd {

// True when the tensor-core kernels handle this problem shape.
bool tc_supported(const Problem &pr);

// The float32 path on the tensor cores (kind::tf32; ssd_tf32.cu): float32 inputs, H = 64,
// S = 64 or 128, L <= 1024.  One launch: one CTA per (batch, head) walks the sequence with
// the state in TMEM, its own in-chunk cumsum included; `err` (nullable) receives error bits.
bool tf32_supported(const Problem &pr);
cudaError_t launch_ssd_tf32(const Problem &pr, const void *x, const void *dt, const float *A, const void *Bm,
                            const void *Cm, const float *D, const float *h0, void *y, float *h_final, int *err,
                            cudaStream_t st);

// Heads per chunk_state CTA (the heads of one group that share its B tiles); a
// sequence run given to launch_chunk_state_tc must start and end on a multiple of it.
int state_heads_per_cta(const Problem &pr);

// States of super-chunks m < nm (R chunks each) from a zero start, for the sequences of
// `seqs`, written to s_local[(bh - seqs.lo) * nsup + m].  dtT (nullable) is dt as
// float32 in the [b][h][L] layout of G; with it, dt and G reach the kernel by bulk
// copies instead of per-thread loads.  `err` receives error bits.
// Whether launch_chunk_state_tc with these arguments zeroes s_local first (one
// cudaMemsetAsync): it does when a CTA's slice of stages cuts a super-chunk.
bool chunk_state_tc_memsets(const Problem &pr, SeqRange seqs, int R, int nm);
cudaError_t launch_chunk_state_tc(const Problem &pr, SeqRange seqs, const void *x, const void *dt,
                                  const float *dtT, const void *Bm, const float *G, float *s_local, int R,
                                  int nsup, int nm, int *err, cudaStream_t st);

// How the scan cuts the sequences ((batch, head) pairs in b * nh + h order) into
// super-chunks: sequences [0, split) into super-chunks of R0 chunks (nsup0 per
// sequence), the rest into super-chunks of R1 chunks (nsup1).  One CTA walks one
// super-chunk of one 64-column block of H.  Super-chunk m of sequence bh enters from
// h0 (zeros if NULL) when m < hs_from, else from the state at h_start index
// bh * nsup0 + m (first part) or base1 + (bh - split) * nsup1 + m (second part).
// When g_count is set, the CTAs that enter from h0 (m < hs_from) read nothing but G from the
// kernels before the scan: instead of waiting for all of them to finish, they wait until
// *g_count reaches g_target (the cumsum CTAs count themselves there, see launch_chunk_cumsum),
// so they do not wait for the chunk_state and state_passing launches the other CTAs need.
struct ScanSplit {
    int64_t split;
    int R0, nsup0, R1, nsup1;
    int hs_from;
    int64_t base1;
    const unsigned *g_count;
    unsigned g_target;
};

// Sequences per scan CTA: 2 (two heads of one B/C group) when S = 128, H = 64 and the
// heads per group are even, else 1.  With 2, both parts of a ScanSplit hold whole pairs.
int scan_seqs_per_cta(const Problem &pr);

// Output y for every super-chunk of `sp`; the last super-chunk of each sequence also
// writes h_final when it is not NULL.
cudaError_t launch_chunk_scan_tc(const Problem &pr, const void *x, const void *dt, const void *Bm,
                                 const void *Cm, const float *D, const float *G, const float *h0,
                                 const float *h_start, float *h_final, void *y, const ScanSplit &sp,
                                 int *err, cudaStream_t st);

}  // namespace ssd
