/*
 * ssd.h -- C ABI of libssd.so: the Mamba-2 selective-state-space (SSD) forward
 * pass in chunked form and its single-token recurrent decode, on one GPU.
 *
 * The method is the one described in the NVIDIA developer blog "Accelerating
 * Mamba-2 with High-Performance Forward Pass Kernels in NVIDIA CUDA Tile":
 *
 *   section "Mamba-2 architecture":
 *     h_t = exp(A dt_t) h_{t-1} + dt_t B_t x_t^T,      y_t = c_t^T h_t + D x_t
 *     G   = in-chunk cumsum of a_t = A dt_t
 *     h_{k+1} = exp(G_last) h_k + (exp(G_last - G) o b)^T X           (b = dt o B)
 *     Y_k     = exp(G) o (C h_k) + (exp(G - G^T) o (C B^T) o M) (dt o X) + D X
 *   sections "Kernel 1" .. "Kernel 3": the three stages chunk_cumsum,
 *   fwd_pass_state (split here into chunk_state + state_passing) and
 *   compute_out (here chunk_scan).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - All pointers are DEVICE pointers unless stated otherwise.  Every tensor is
 *    dense and row-major ("contiguous") in the layout given below.
 *  - The caller owns every buffer, the workspace included.  The library never
 *    allocates or frees device memory and keeps no state between calls.
 *  - Work is enqueued asynchronously on `stream` (a cudaStream_t; NULL means
 *    the legacy default stream).  A return of SSD_OK means the work was
 *    enqueued; errors in the kernels themselves surface on the stream.
 *  - Arguments are validated before anything is enqueued: every error other
 *    than SSD_ERR_CUDA means nothing was launched and no buffer was touched.
 *  - Symbols:  B batch, L seqlen, nh heads, H headdim, S dstate, G ngroups,
 *    T chunk, nc = ceil(L / T).  Head h reads B/C group h / (nh / G).
 *
 * Tensor layouts (dtype "in" = desc.in_dtype, "out" = desc.out_dtype):
 *    x   [B][L][nh][H]   in        y       [B][L][nh][H]  out
 *    dt  [B][L][nh]      in        A, D    [nh]           float32
 *    Bm  [B][L][G][S]    in        Cm      [B][L][G][S]   in
 *    h0, h_final [B][nh][H][S] float32  (state of head h: row p < H, column s < S)
 *  dt must already be the positive step (any softplus or bias applied by the
 *  caller); A must be negative for the usual decaying model (not enforced).
 */
#ifndef SSD_H_
#define SSD_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *ssd_stream_t;   /* identical to cudaStream_t */
typedef struct CUevent_st *ssd_event_t;     /* identical to cudaEvent_t  */

typedef enum { SSD_F32 = 0, SSD_BF16 = 1 } ssd_dtype;

/* ssd_desc.dt_dtype: dt in the dtype of x, Bm and Cm (the default), or dt in float32 beside
 * bfloat16 x, Bm, Cm.  The blog's first kernel ("Kernel 1: cumulative sum") takes dt up to
 * float32 before the cumulative sum of A dt, which sets every decay; with SSD_DT_FLOAT32 that
 * sum runs on the caller's float32 dt, and the later stages, where dt enters only products that
 * are rounded to bfloat16 as tensor-core operands, read a bfloat16 copy the cumsum writes into
 * the workspace.  Accepted by ssd_fwd, ssd_fwd_timed, ssd_fwd_noalloc, ssd_fwd_plan,
 * ssd_fwd_workspace_size, ssd_fwd_path and ssd_chunk_cumsum; the other entry points return
 * SSD_ERR_UNSUPPORTED for it. */
typedef enum { SSD_DT_AS_INPUTS = 0, SSD_DT_FLOAT32 = 1 } ssd_dt_dtype;

typedef enum {
    SSD_OK = 0,
    SSD_ERR_INVALID_ARG = 1,  /* null / misaligned pointer, negative size, bad dtype, G does not divide nh */
    SSD_ERR_UNSUPPORTED = 2,  /* well-formed problem outside what this library handles (see limits below;
                                 every entry point: arrays of 2^62 bytes or more, whose sizes could wrap;
                                 B * nh of 2^31 or more) */
    SSD_ERR_WORKSPACE = 3,    /* workspace NULL, smaller than ssd_fwd_workspace_size, or not 256-B aligned */
    SSD_ERR_CUDA = 4,         /* a CUDA runtime call or a kernel launch failed; call cudaGetLastError */
    SSD_ERR_TOO_LARGE = 5,    /* ssd_fwd_noalloc: the problem needs more scratch than SSD_NOALLOC_SCRATCH_BYTES */
    SSD_ERR_TIMEOUT = 6       /* ssd_fwd_check: a bounded wait inside a kernel expired; outputs are invalid */
} ssd_status;

/* Problem description.  Mirrors the blog's Mamba2ProblemSpec(batch_size,
 * num_tokens, num_groups, num_heads, state_size, head_size, chunk_size, dtype,
 * state_dtype) (section "Mamba-2 forward benchmark"); the state dtype is
 * always float32 here. */
typedef struct {
    int64_t batch;      /* B  >= 0 */
    int64_t seqlen;     /* L  >= 0 (0: y is empty, h_final = h0 or zeros) */
    int64_t nheads;     /* nh >= 0, a multiple of ngroups */
    int64_t headdim;    /* H  in [1, 1024] */
    int64_t dstate;     /* S  in [1, 256] */
    int64_t ngroups;    /* G  >= 1 */
    int64_t chunk;      /* T  in [1, 1024]; any L is accepted (the last chunk may be short) */
    int32_t in_dtype;   /* ssd_dtype of x, dt, Bm, Cm */
    int32_t out_dtype;  /* ssd_dtype of y */
    int32_t flags;      /* SSD_FLAG_* bits, 0 by default */
    int32_t dt_dtype;   /* ssd_dt_dtype of dt, SSD_DT_AS_INPUTS (0) by default */
} ssd_desc;

/* Use the CUDA-core kernels for every stage even where tensor-core kernels
 * exist for the shape (both are GPU code; this exists for cross-checking). */
#define SSD_FLAG_FORCE_SIMT 1

/* Test hook of the failure path: the tensor-core kernels run in a build of their own in
 * which every wait for another warp's work tests its barrier once and expires unless the
 * phase is already complete (the normal kernels wait up to 250 ms).  The call then winds
 * down without hanging -- each CTA still waits for the copies and MMAs it has issued
 * before it releases its tensor memory -- and ssd_fwd_check reports SSD_ERR_TIMEOUT; its
 * outputs are invalid.  The CUDA-core kernels have no such waits, and the float32 tensor-core
 * kernel waits only for its own MMAs; both ignore the flag.
 * Never set it in production code. */
#define SSD_FLAG_EXPIRE_WAITS 2

/* Human-readable name of a status code (static string, never NULL). */
const char *ssd_status_string(ssd_status s);

/* Bytes of device workspace ssd_fwd needs for `desc` (written to *bytes).
 * The workspace holds an error word, the in-chunk cumsum G, a float32 copy
 * of dt in G's [b][h][L] layout, the local (super-)chunk states and the
 * (super-)chunk-start states, all float32, and with SSD_DT_FLOAT32 a bfloat16
 * copy of dt in its own layout.
 * Errors: SSD_ERR_INVALID_ARG / SSD_ERR_UNSUPPORTED. */
ssd_status ssd_fwd_workspace_size(const ssd_desc *desc, size_t *bytes);

/* Whether ssd_fwd runs its chunk_state and chunk_scan stages on the tensor
 * cores (tcgen05) for `desc` (*uses_tensor_cores = 1) or on the CUDA cores
 * (0).  Both are GPU code; the choice depends only on the shape, the dtypes
 * and desc.flags. */
ssd_status ssd_fwd_path(const ssd_desc *desc, int32_t *uses_tensor_cores);

/* How ssd_fwd runs `desc` on the current device (written to *plan): which path,
 * how each sequence ((batch, head) pair, in b * nh + h order) is cut into
 * super-chunks (the tensor-core scan walks one super-chunk per CTA with the
 * state on chip; the CUDA-core path uses one chunk), and how many kernels and
 * cudaMemsetAsync calls one ssd_fwd call issues on its stream.  The first
 * split_sequences sequences are cut into super-chunks of super_tokens tokens,
 * the remaining ones into super-chunks of tail_super_tokens tokens (so that the
 * last wave of scan CTAs still covers the SMs).  Host-side query: it reads the
 * device's SM count and launches nothing.
 * Errors: SSD_ERR_INVALID_ARG / SSD_ERR_UNSUPPORTED, as for ssd_fwd. */
typedef struct {
    int32_t tensor_cores;          /* 1: tcgen05 kernels for chunk_state and chunk_scan   */
    int32_t super_tokens;          /* tokens per super-chunk, first split_sequences seqs  */
    int32_t n_super;               /* their super-chunks per sequence                     */
    int32_t split_sequences;       /* sequences cut with super_tokens (<= B * nh)         */
    int32_t tail_super_tokens;     /* tokens per super-chunk of the remaining sequences   */
    int32_t tail_n_super;          /* their super-chunks per sequence                     */
    int32_t kernel_launches;       /* kernels per ssd_fwd call (0 for an empty problem)   */
    int32_t memsets;               /* cudaMemsetAsync calls per ssd_fwd call              */
} ssd_plan;

ssd_status ssd_fwd_plan(const ssd_desc *desc, ssd_plan *plan);

/* Chunked SSD forward pass: y = SSD(x, dt, A, Bm, Cm, D; h0) and the state
 * after the last token (blog section "Mamba-2 architecture", the chunk jump
 * and chunk output; the stages of sections "Kernel 1".."Kernel 3").
 *   h0       nullable: NULL means a zero initial state.
 *   h_final  nullable: NULL means the final state is not written.
 *   workspace, ws_bytes: device scratch of at least ssd_fwd_workspace_size()
 *            bytes, 256-byte aligned, owned by the caller; its contents on
 *            entry are ignored and on exit are unspecified.
 * x, dt, Bm, Cm, y must be 16-byte aligned; A, D, h0, h_final 4-byte aligned.
 * y must not overlap any input.  Results are deterministic for a given input,
 * except when chunk_state splits a super-chunk between two CTAs (a plan with
 * two memsets): the two partial states are added with float atomics, in either
 * order, so results may differ between calls at the level of float rounding.
 * The work is ordered on `stream` like any other stream work; inside the call
 * the kernels after the first use programmatic dependent launch (each starts
 * while the previous one finishes and waits for its results).
 * dt is the positive step (the softplus output) and must be >= 0; it is not
 * scanned for sign.  A negative dt gives NaN outputs on the tensor-core path
 * (which evaluates the in-chunk decay times dt as one exp2 of G - log2 dt) and
 * is carried through the recurrence as written on the CUDA-core path. */
ssd_status ssd_fwd(const ssd_desc *desc, const void *x, const void *dt, const float *A,
                   const void *Bm, const void *Cm, const float *D, const float *h0, void *y,
                   float *h_final, void *workspace, size_t ws_bytes, ssd_stream_t stream);

/* Same as ssd_fwd, and records events around each stage on `stream`:
 * events[2*i] before and events[2*i+1] after stage i, for i = 0..3 in the order
 * chunk_cumsum, chunk_state, state_passing, chunk_scan.  `events` is a host
 * array of 8 created events (cudaEventCreate); used for per-stage timing. */
ssd_status ssd_fwd_timed(const ssd_desc *desc, const void *x, const void *dt, const float *A,
                         const void *Bm, const void *Cm, const float *D, const float *h0, void *y,
                         float *h_final, void *workspace, size_t ws_bytes, ssd_stream_t stream,
                         ssd_event_t const *events);

/* Synchronises `stream` and reports whether the last ssd_fwd that used
 * `workspace` hit a bounded device-side wait that expired (SSD_ERR_TIMEOUT:
 * the outputs of that call are invalid) or completed normally (SSD_OK).  The
 * tensor-core kernels bound every wait on a barrier (250 ms) and record expiry
 * in the workspace's error word instead of hanging. */
ssd_status ssd_fwd_check(const void *workspace, ssd_stream_t stream);

/* Forward pass on inputs and outputs in host memory (a convenience over ssd_fwd for callers
 * that hold them on the host; no counterpart on the pages).  x, dt, A, Bm, Cm, D, h0 (nullable)
 * are read from host memory and y, h_final (nullable) written to host memory, in the layouts
 * of ssd_fwd; page-locked host memory lets the copies run asynchronously.  The batch is cut
 * into up to 8 slices of whole batch rows: the library's two copy streams (one per direction,
 * one pair per device, created on first use) move slice k in and out while the forward pass
 * of the others runs on `stream`, so copies and computation overlap.  device_buffer: caller-
 * owned device memory of ssd_fwd_host_buffer_size() bytes, 256-byte aligned (inputs, outputs,
 * workspace; nothing is allocated).  The call only enqueues: `stream` reaches the point after
 * the outputs are in host memory once it is done, and the host buffers must stay valid until
 * then.  Calls on one device are enqueued under a lock; a call's copies start after all work
 * enqueued on `stream` before it.  Errors: those of ssd_fwd; SSD_ERR_WORKSPACE for a missing,
 * misaligned or short device_buffer. */
ssd_status ssd_fwd_host_buffer_size(const ssd_desc *desc, size_t *bytes);
ssd_status ssd_fwd_host(const ssd_desc *desc, const void *x, const void *dt, const float *A,
                        const void *Bm, const void *Cm, const float *D, const float *h0,
                        void *y, float *h_final, void *device_buffer, size_t buffer_bytes,
                        ssd_stream_t stream);
/* The ssd_fwd_check of ssd_fwd_host: synchronises `stream` and reports SSD_ERR_TIMEOUT if a
 * bounded device-side wait expired in any slice of the last call on device_buffer. */
ssd_status ssd_fwd_host_check(const void *device_buffer, ssd_stream_t stream);

/* One recurrent decode step for every (batch, head) (blog section "Mamba-2
 * architecture": the recurrent form suits sequential inference).
 * desc.seqlen and desc.chunk are ignored.  Layouts:
 *   x [B][nh][H] in, dt [B][nh] in, Bm, Cm [B][G][S] in, A, D [nh] float32,
 *   h [B][nh][H][S] float32 read and overwritten in place, y [B][nh][H] out.
 * All pointers 4-byte aligned (16 for h when S % 4 == 0 is used vectorised). */
ssd_status ssd_step(const ssd_desc *desc, const void *x, const void *dt, const float *A,
                    const void *Bm, const void *Cm, const float *D, float *h, void *y,
                    ssd_stream_t stream);

/* ---- The four stages of ssd_fwd, callable one by one --------------------
 * Intermediate layouts (all float32 unless stated):
 *   G        [B][nh][L]          log2(e) * inclusive in-chunk cumsum of A dt
 *   s_local  [B][nh][nc][H][S]   chunk state from a zero start
 *   h_start  [B][nh][nc][H][S]   state entering each chunk (the state dtype,
 *                                 float32; the chunk-output contraction casts it
 *                                 to its operand dtype)
 */

/* Stage 1 (blog section "Kernel 1: cumulative sum"): G from dt and A. */
ssd_status ssd_chunk_cumsum(const ssd_desc *desc, const void *dt, const float *A, float *G,
                            ssd_stream_t stream);

/* Stage 2 (blog section "Kernel 2: fwd_pass_state", the per-chunk contraction):
 * s_local[b][h][k] = sum_{t in chunk k} dt_t exp2(G_last - G_t) x_t B_t^T. */
ssd_status ssd_chunk_state(const ssd_desc *desc, const void *x, const void *dt, const void *Bm,
                           const float *G, float *s_local, ssd_stream_t stream);

/* Stage 3 (blog section "Kernel 2: fwd_pass_state", the sequential chunk loop):
 * h_start[k] = h_k with h_0 = h0 (NULL: zeros), h_{k+1} = exp2(G_last,k) h_k + s_local[k];
 * h_final (nullable) = h_nc.  s_local and h_start may not overlap. */
ssd_status ssd_state_passing(const ssd_desc *desc, const float *G, const float *s_local,
                             const float *h0, float *h_start, float *h_final, ssd_stream_t stream);

/* Stage 4 (blog section "Kernel 3: compute_out"): y from the chunk-start states:
 * Y_k = exp2(G) o (C h_k^T) + ((C B^T) o exp2(G_i - G_j) o [i >= j]) (dt o X) + D X. */
ssd_status ssd_chunk_scan(const ssd_desc *desc, const void *x, const void *dt, const void *Bm,
                          const void *Cm, const float *D, const float *G, const float *h_start,
                          void *y, ssd_stream_t stream);

/* ---- Gradients of the forward pass --------------------------------------
 * Reverse mode of the recurrence above, taken chunk by chunk ("Sasha Rush:
 * Mamba: The Hard Way", Part 3: the adjoint state runs the same scan
 * backwards; each coefficient's gradient pairs a forward and a backward
 * quantity).  For upstream gradients dy (of y) and dh_final (of h_final),
 * ssd_bwd writes the gradient of  sum(dy * y) + sum(dh_final * h_final)
 * with respect to every input of ssd_fwd:
 *   dx   [B][L][nh][H]  in      ddt [B][L][nh] in      dA, dD [nh] float32
 *   dB   [B][L][G][S]   in      dC  [B][L][G][S] in    dh0 [B][nh][H][S] float32
 * dy has the layout of y and the in dtype: the gradient pass requires
 * desc.in_dtype == desc.out_dtype.  dh_final, h0 and dh0 are nullable (zeros;
 * not written).  dB, dC sum over the heads of each group; dA, dD over batch
 * and tokens.
 * Limits: H <= 128, S <= 256, chunk <= 256, in_dtype == out_dtype; other
 * well-formed problems return SSD_ERR_UNSUPPORTED.  desc.flags is ignored.
 * All pointers aligned to their element size (2 bytes for bf16, 4 otherwise);
 * outputs must not overlap inputs or each other.  The forward states are
 * recomputed inside the call (nothing from an earlier ssd_fwd is reused).
 * Every sum is taken in a fixed order: results are deterministic.
 * workspace: at least ssd_bwd_workspace_size() bytes, 256-byte aligned. */
ssd_status ssd_bwd_workspace_size(const ssd_desc *desc, size_t *bytes);
ssd_status ssd_bwd(const ssd_desc *desc, const void *x, const void *dt, const float *A,
                   const void *Bm, const void *Cm, const float *D, const float *h0,
                   const void *dy, const float *dh_final, void *dx, void *ddt, float *dA,
                   void *dB, void *dC, float *dD, float *dh0, void *workspace, size_t ws_bytes,
                   ssd_stream_t stream);

/* ---- Mamba-1 selective scan (S6), forward --------------------------------
 * "Sasha Rush: Mamba: The Hard Way", Part 5: each channel d has a vector
 * state of N entries with its own A[d][n]; per token the step is discretised,
 *     abar = exp(delta_t A[d][n]),   bbar = delta_t B_t[n],
 * and the recurrence h[n] = abar h[n] + bbar x_t, y_t = sum_n C_t[n] h[n]
 * (+ D[d] x_t) runs over the tokens.  Channel d reads B/C group d / (dim / G).
 * Layouts (time innermost):
 *   x, delta, y  [B][dim][L]   (in, in, out dtype)      A   [dim][N] float32
 *   Bm, Cm       [B][G][N][L]  in dtype                 D   [dim] float32, nullable (no skip)
 *   h0, h_final  [B][dim][N]   float32, nullable (zeros / not written)
 * delta is the positive step (no softplus or bias applied inside).
 * Limits: 1 <= N <= 32, G divides dim, B <= 65535, B * dim * L * N * 16 < 2^62.  Pointers aligned to their
 * element size; y must not overlap an input.  Deterministic. */
typedef struct {
    int64_t batch;      /* B >= 0 */
    int64_t seqlen;     /* L >= 0 */
    int64_t dim;        /* channels >= 0, a multiple of ngroups */
    int64_t dstate;     /* N in [1, 32] */
    int64_t ngroups;    /* G >= 1 */
    int32_t in_dtype;   /* ssd_dtype of x, delta, Bm, Cm */
    int32_t out_dtype;  /* ssd_dtype of y */
    int32_t flags;      /* must be 0 */
    int32_t reserved;   /* must be 0 */
} ssd_s6_desc;

ssd_status ssd_s6_fwd(const ssd_s6_desc *desc, const void *x, const void *delta, const float *A, const void *Bm,
                  const void *Cm, const float *D, const float *h0, void *y, float *h_final,
                  ssd_stream_t stream);

/* ---- Forward pass for callers that cannot allocate device memory ---------
 * (The pages have no counterpart to this entry point: it is a deployment aid.)
 *
 * Some callers cannot call cudaMalloc at the point where they run the forward
 * pass: code running while a CUDA graph is being captured, allocator-less
 * embedded runtimes, or plug-ins whose host application owns every device
 * allocation.  ssd_fwd_noalloc computes exactly what ssd_fwd computes but takes
 * no workspace argument; it uses a scratch array that is part of libssd.so
 * itself (a file-scope __device__ array of SSD_NOALLOC_SCRATCH_BYTES bytes, which
 * every GPU that loads the library holds until the process exits).  The caller
 * still provides all inputs and outputs.  It calls no cudaMalloc, cudaFree or
 * other allocating routine.
 *
 *  - The first call in a CUDA context looks up the device address of the array
 *    (cudaGetSymbolAddress) in that context, with its device current; make that
 *    first call before any stream capture on that device.  The address is cached
 *    per context.
 *  - Problems whose workspace (ssd_fwd_workspace_size) exceeds
 *    SSD_NOALLOC_SCRATCH_BYTES are rejected with SSD_ERR_TOO_LARGE before
 *    anything is launched.
 *  - All calls in the process share the one array per device: calls whose
 *    executions overlap on the GPU (different streams, or different host
 *    threads without ordering) race on it and give wrong results.  Order them
 *    on one stream.  The array keeps the previous call's contents; each call
 *    clears what must start at zero (the error word, a counter, and the partial state
 *    sums when its plan adds them with atomics) and writes every other
 *    scratch byte before reading it.
 *  - A bounded wait that expired inside the call is reported by
 *    ssd_fwd_noalloc_check (the error word lives in the array too).
 * Arguments, layouts and the other errors are those of ssd_fwd.            */
#define SSD_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20)

ssd_status ssd_fwd_noalloc(const ssd_desc *desc, const void *x, const void *dt, const float *A,
                           const void *Bm, const void *Cm, const float *D, const float *h0,
                           void *y, float *h_final, ssd_stream_t stream);

/* The ssd_fwd_check of ssd_fwd_noalloc: synchronises `stream` and reports whether the last
 * ssd_fwd_noalloc call in the current context hit a bounded device-side wait that expired
 * (SSD_ERR_TIMEOUT: its outputs are invalid) or completed normally (SSD_OK).  Like
 * ssd_fwd_noalloc it allocates nothing; SSD_ERR_CUDA if the array's address cannot be
 * looked up or the copy of the error word fails. */
ssd_status ssd_fwd_noalloc_check(ssd_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* SSD_H_ */
