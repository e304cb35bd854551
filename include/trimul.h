/*
 * trimul.h -- C ABI of the GB300 (sm_103a) triangular multiplicative update (TriMul):
 * the forward pass and its backward pass (gradients).
 *
 * The operation is the pair-representation update built, in the fold-cp-ops
 * README ("Use" section), from the six sub-modules norm_in, p_in, g_in,
 * norm_out, p_out and g_out, run on one GPU (the README's cp = 1 case, which
 * it says is selected automatically for a single device).  With z' = LN_in(z)
 * and pair mask m:
 *
 *     a[b,i,j,c] = sigmoid(z' . W_ga[c]) * (z' . W_a[c]) * m[b,i,j]
 *     b[b,i,j,c] = sigmoid(z' . W_gb[c]) * (z' . W_b[c]) * m[b,i,j]
 *     outgoing:  x[b,i,j,c] = sum_k a[b,i,k,c] * b[b,j,k,c]
 *     incoming:  x[b,i,j,c] = sum_k a[b,k,i,c] * b[b,k,j,c]
 *     out[b,i,j,:] = sigmoid(z'[b,i,j,:] W_g^T) * (LN_out(x[b,i,j,:]) W_o^T)
 *
 * LN is torch.nn.LayerNorm (biased variance, eps under the square root).
 *
 * Conventions shared by every entry point
 *   - "bf16"/"fp16" buffers are arrays of uint16_t holding IEEE bfloat16 /
 *     binary16 bit patterns; "f32" buffers hold float.
 *   - Every tensor pointer is a DEVICE pointer on the handle's device unless
 *     the entry point says HOST.  All tensors are dense row-major (C order)
 *     with 16-byte aligned base addresses.  The caller owns every buffer it
 *     passes; the library keeps no reference after the call returns (device
 *     work may still be running on `stream`).
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *     Forward entry points only enqueue work: they never synchronise unless
 *     TRIMUL_FLAG_CHECK is given.
 *   - Sizes: B >= 1, N >= 1 with N % 8 == 0 (eight 16-bit elements = the 16-byte
 *     row granularity of the tensor-memory-access engine; the fold-cp-ops README
 *     states the same rule for its token axis), D and C multiples of 8 in [8, 256].
 *   - Every call returns a trimul_status; on a non-OK status a thread-local
 *     message is available from trimul_last_error().  Argument errors are
 *     detected before any device work is enqueued.
 *   - A handle is not re-entrant: its workspace serves one call at a time.
 *     Calls on one stream are ordered; calls on different streams with one
 *     handle must be ordered by the caller.
 */
#ifndef TRIMUL_H_
#define TRIMUL_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct trimul_handle_s* trimul_handle;

/* fold-cp-ops README, "Use": the layer's direction argument. */
typedef enum { TRIMUL_OUTGOING = 0, TRIMUL_INCOMING = 1 } trimul_direction;

typedef enum {
  TRIMUL_OK = 0,
  TRIMUL_ERR_INVALID_ARG = 1,       /* null pointer, bad enum, out-of-range value        */
  TRIMUL_ERR_SHAPE = 2,             /* size rule violated (N % 8, D, C limits, B, N)     */
  TRIMUL_ERR_UNSUPPORTED_ARCH = 3,  /* device is not compute capability 10.3 (sm_103)    */
  TRIMUL_ERR_OOM = 4,               /* device allocation failed                          */
  TRIMUL_ERR_CUDA = 5,              /* a CUDA runtime/driver call or a launch failed     */
  TRIMUL_ERR_TIMEOUT = 6            /* a kernel gave up on a bounded wait (see FLAG_CHECK) */
} trimul_status;

/* Flags for the forward entry points. */
enum {
  TRIMUL_FLAG_CHECK = 1u,           /* synchronise `stream`; report kernel wait timeouts and
                                       mask values outside [0, 1] */
  TRIMUL_FLAG_INJECT_STALL = 2u,    /* test hook: the first kernel's loads are never issued, so
                                       its consumers hit their bounded waits; with FLAG_CHECK the
                                       call returns TRIMUL_ERR_TIMEOUT and the context stays usable */
  TRIMUL_FLAG_DEFER_OUTPUT = 4u,    /* trimul_forward_host only: `stream` does not wait for the
                                       copy of out back to the host; call trimul_host_join before
                                       reading out_host (lets that copy overlap the next call's
                                       kernels) */
  TRIMUL_FLAG_FP8 = 8u              /* trimul_forward only, outgoing only: a and b are rounded to
                                       e4m3 (scaled by a power of two from the weights' bound on
                                       |a|, |b|) and the triangle contraction runs on the 8-bit
                                       tensor cores.  Less accurate than the default path: about
                                       4e-2 relative Frobenius error against the exact result
                                       instead of 2e-3.  Needs N % 16 == 0 (else TRIMUL_ERR_SHAPE);
                                       rejected with the incoming direction and by every other
                                       entry point (TRIMUL_ERR_INVALID_ARG). */
};

/*
 * Layer parameters (fold-cp-ops README, "Use": norm_in, p_in, g_in, norm_out,
 * p_out, g_out).  Weights use the nn.Linear (out_features, in_features) layout.
 * The README's p_in / g_in are Linear(D, 2D); their first C output rows are
 * W_a / W_ga and the next C rows are W_b / W_gb.  All pointers are DEVICE
 * pointers, read only during trimul_create (the handle keeps its own copies).
 */
typedef struct {
  int D;                     /* pair feature width (z, out) */
  int C;                     /* width of a, b, x (the README's layer has C = D) */
  const uint16_t* W_a;       /* bf16 [C][D] */
  const uint16_t* W_ga;      /* bf16 [C][D] */
  const uint16_t* W_b;       /* bf16 [C][D] */
  const uint16_t* W_gb;      /* bf16 [C][D] */
  const uint16_t* W_o;       /* bf16 [D][C]  (p_out) */
  const uint16_t* W_g;       /* bf16 [D][D]  (g_out) */
  const float* ln_in_gamma;  /* f32 [D] */
  const float* ln_in_beta;   /* f32 [D] */
  const float* ln_out_gamma; /* f32 [C] */
  const float* ln_out_beta;  /* f32 [C] */
  float eps;                 /* LayerNorm epsilon (nn.LayerNorm default 1e-5); must be > 0 */
} trimul_params;

/*
 * Create a handle on `device`: checks the architecture (10.3 required),
 * copies the weights into the kernels' layout (binary16, K-major, value/gate
 * rows interleaved) and allocates a small status word.  Weights must be
 * finite with |w| <= 65504 (binary16 range), and the input-projection bound
 * (sqrt(D) max|gamma_in| + ||beta_in||_2) * max_c ||W_{a,b}[c]||_2 must be
 * <= 65504 so that a and b fit binary16; otherwise TRIMUL_ERR_INVALID_ARG.
 * Synchronous.  On failure *out is set to NULL.
 * Logging: when the environment variable TRIMUL_LOG is set to a non-empty
 * value other than "0" at create, the handle prints one line to stderr at
 * create (its launch configuration: co-resident CTA pairs, ring depths) and
 * one per tiled kernel launch (tile range, grid, operand majors and types),
 * each starting with "trimul: ".  Nothing else changes.
 */
trimul_status trimul_create(trimul_handle* out, const trimul_params* p, int device);

/*
 * Optional: size the workspace (a, b: fp16 [B][C][N][N]; x: fp16 [B][C][N][N];
 * the LayerNorm statistics of z: float2 [B][N][N])
 * for calls up to B x N, so that the first forward does no allocation.  The
 * fold-cp-ops README's prepare(n_token, batch, masked) is likewise only a
 * scheduling choice.  `masked` is accepted for the same signature and unused.
 * Synchronous.  TRIMUL_ERR_OOM if the allocation fails (the old workspace is kept).
 */
trimul_status trimul_prepare(trimul_handle h, int B, int N, int masked);

/*
 * Full forward.  z: bf16 [B][N][N][D]; mask: bf16 [B][N][N] with values in
 * [0, 1], or NULL for all ones; out: bf16 [B][N][N][D], must not overlap z or
 * mask.  Grows the workspace if needed (that allocation synchronises the
 * device).  Enqueues a status reset and the kernels on `stream`.
 *
 * Mask values outside [0, 1] (or NaN) make the result undefined: the binary16
 * range of a and b rests on |m| <= 1.  The input projection flags them on the
 * device; with TRIMUL_FLAG_CHECK such a call returns TRIMUL_ERR_INVALID_ARG
 * (the check costs no extra pass over the mask).
 *
 * x is kept as binary16 x * 2^-s with s derived on the device from this
 * call's max |a|, |b| (the smallest s with N max^2 2^-s <= 32768), so x never
 * overflows and small x keep their precision whatever the layer's weights.
 *
 * CUDA graphs: once the workspace covers B x N (trimul_prepare or an earlier
 * call), a call without TRIMUL_FLAG_CHECK allocates nothing and does not wait
 * on the host, so it may be captured on `stream` and the graph replayed; the
 * graph keeps the pointers it was captured with.
 */
trimul_status trimul_forward(trimul_handle h, const uint16_t* z, const uint16_t* mask,
                             int B, int N, trimul_direction dir, uint16_t* out,
                             void* stream, unsigned flags);

/*
 * Same as trimul_forward with HOST buffers: z_host, mask_host (nullable) and
 * out_host are host pointers (page-locked memory gives asynchronous copies).
 * The handle stages them in device buffers it owns (two slots, used by
 * alternate calls).  The copies run on two streams of the handle and the
 * kernels on `stream`: above 256 MB of z the call works in 8 ranges of pair
 * tiles, so the input projection of a range follows its host-to-device copy
 * and the device-to-host copy of a range of out follows its output stage,
 * overlapping the other ranges' work; a call's input copies may also run
 * during the previous call's kernels.  The call returns after enqueueing;
 * `stream` completes only once out_host holds the result (synchronise it
 * before reading out_host).  z_host and mask_host must stay unchanged until
 * then.  Calls on one handle must not run concurrently from several threads.
 */
trimul_status trimul_forward_host(trimul_handle h, const uint16_t* z_host, const uint16_t* mask_host,
                                  int B, int N, trimul_direction dir, uint16_t* out_host,
                                  void* stream, unsigned flags);

/*
 * Stage 1 alone (LN_in + gated input projection + mask).  z, mask as above
 * (with TRIMUL_FLAG_CHECK, mask values outside [0, 1] give
 * TRIMUL_ERR_INVALID_ARG); a_out, b_out: fp16 [B][C][N][N] (channel-major planes).
 */
trimul_status trimul_inproj(trimul_handle h, const uint16_t* z, const uint16_t* mask,
                            int B, int N, uint16_t* a_out, uint16_t* b_out,
                            void* stream, unsigned flags);

/*
 * Stage 2 alone (the triangle contraction per channel plane).  a, b: fp16
 * [B][C][N][N]; x_out: fp16 [B][C][N][N] holding x * 2^-s with
 * s = trimul_x_scale_log2(h, N).  Outgoing computes X_c = A_c B_c^T, incoming
 * X_c = A_c^T B_c, with fp32 accumulation.  The power-of-two scale keeps x in
 * the binary16 range for every a, b the handle's input projection can produce
 * (|a|, |b| are bounded by the bound checked in trimul_create).
 */
trimul_status trimul_triangle(trimul_handle h, const uint16_t* a, const uint16_t* b,
                              int B, int N, trimul_direction dir, uint16_t* x_out,
                              void* stream, unsigned flags);

/*
 * Stage 3 alone (LN_out + output projection + output gate).  x: fp16
 * [B][C][N][N] holding x * 2^-s with s = trimul_x_scale_log2(h, N) (the format
 * trimul_triangle writes); z: bf16 [B][N][N][D]; out: bf16 [B][N][N][D].
 */
trimul_status trimul_outproj(trimul_handle h, const uint16_t* x, const uint16_t* z,
                             int B, int N, uint16_t* out, void* stream, unsigned flags);

/*
 * Optional per-stage timing.  With `events` non-NULL (four cudaEvent_t handles
 * passed as void*, created by the caller with timing enabled), every later
 * trimul_forward on this handle records events[0] before stage 1, events[1]
 * after stage 1, events[2] after stage 2 and events[3] after stage 3, on the
 * forward's stream.  The handle copies the four handles; NULL switches the
 * recording off.  The events must outlive their use.
 */
trimul_status trimul_set_stage_events(trimul_handle h, void* const* events);

/*
 * Forward without any device allocation.  (The pages have no counterpart of
 * this entry point; it serves callers of this library.)
 *
 * Some callers must not allocate device memory once they are running: a
 * framework whose caching allocator already owns the device memory (a
 * cudaMalloc from inside a library bypasses its accounting and can fail or
 * fragment the pool), or a serving loop that forbids allocation after
 * start-up so that a request can never stall on, or fail in, cudaMalloc.
 * trimul_forward grows a handle-owned workspace with cudaMalloc when a call
 * needs more than it holds; this entry point instead keeps its workspace
 * (a, b, x and the per-pair LayerNorm statistics) in a fixed scratch array that is part of the library's device image (64 MiB,
 * trimul_noalloc_scratch_bytes(), held by every GPU that loads the library
 * until the process exits).  It calls no cudaMalloc, cudaFree or allocating
 * routine; the handle itself must have been created beforehand.
 *
 * Arguments, layouts and results are those of trimul_forward.  A call whose
 * (6 * C + 8) * B * N * N bytes of scratch exceed the array returns
 * TRIMUL_ERR_SHAPE (use trimul_forward for those sizes).  The first call on a
 * device looks up the array's device address (cudaGetSymbolAddress); make
 * that first call before any stream capture.  Every call, from every handle,
 * shares the one array: calls that may overlap on the GPU (other streams,
 * other threads) race on it and must be ordered by the caller.  Nothing from
 * an earlier call is read: each call writes all the scratch it reads.
 */
trimul_status trimul_forward_noalloc(trimul_handle h, const uint16_t* z, const uint16_t* mask,
                                     int B, int N, trimul_direction dir, uint16_t* out,
                                     void* stream, unsigned flags);

/*
 * Gradients of the layer's parameters, written by trimul_backward.  All are
 * DEVICE pointers to f32 arrays in the parameters' own layouts; they are
 * overwritten (not accumulated into).
 */
typedef struct {
  float* dW_a;            /* f32 [C][D] */
  float* dW_ga;           /* f32 [C][D] */
  float* dW_b;            /* f32 [C][D] */
  float* dW_gb;           /* f32 [C][D] */
  float* dW_o;            /* f32 [D][C] */
  float* dW_g;            /* f32 [D][D] */
  float* d_ln_in_gamma;   /* f32 [D] */
  float* d_ln_in_beta;    /* f32 [D] */
  float* d_ln_out_gamma;  /* f32 [C] */
  float* d_ln_out_beta;   /* f32 [C] */
} trimul_grads;

/*
 * Backward pass: the gradients of a scalar loss L with respect to z and to
 * every parameter, given dout = dL/d out.  The pages ship the layer for
 * inference only; this is the plain reverse-mode derivative of the forward
 * defined above (LN_in, gated input projections, triangle, LN_out, gated
 * output projection, taken in reverse order).  The pair mask is data: it
 * gets no gradient.
 *
 * z, mask (nullable), dout: as trimul_forward's z, mask and out (bf16
 * [B][N][N][D], [B][N][N]); dz: bf16 [B][N][N][D], must not overlap z or
 * dout; grads: the ten gradient arrays (none NULL).  The forward is
 * recomputed inside the call (nothing is kept from an earlier forward).
 * The handle grows a backward workspace of
 * trimul_backward_workspace_bytes(h, B, N) bytes when needed (that
 * allocation synchronises the device).  Enqueues the kernels on `stream`;
 * flags as for trimul_forward (TRIMUL_FLAG_CHECK).
 *
 * Arithmetic: the gradient planes and the operands they meet in the tensor
 * cores are bf16 (a gradient's scale follows dout's, which the library cannot
 * bound, so it needs bf16's exponent range), accumulation is fp32, and the
 * sums over all pairs that make up the parameter gradients are fp32 and
 * reduced in a fixed order (the results are deterministic).
 */
trimul_status trimul_backward(trimul_handle h, const uint16_t* z, const uint16_t* mask, const uint16_t* dout,
                              int B, int N, trimul_direction dir, uint16_t* dz, const trimul_grads* grads,
                              void* stream, unsigned flags);

/* Bytes of the workspace trimul_backward uses for B x N (0 for a null handle or an empty shape). */
size_t trimul_backward_workspace_bytes(trimul_handle h, int B, int N);

/* Kernel launches one trimul_backward call enqueues for B x N (-1 for a null handle or an empty shape). */
int trimul_kernels_per_backward(trimul_handle h, int B, int N);

/*
 * The power of two s with which trimul_triangle stores x (as x * 2^-s in
 * fp16) for token count N, from the handle's bound on |a|, |b| (valid for any
 * a, b its input projection can produce); -1 for a null handle or N < 1.  The
 * forward entry points use a per-call s instead (see trimul_forward).
 */
int trimul_x_scale_log2(trimul_handle h, int N);

/* Size in bytes of the fixed scratch used by trimul_forward_noalloc. */
size_t trimul_noalloc_scratch_bytes(void);

/* Release the handle's device memory.  Synchronises the device.  NULL is accepted. */
trimul_status trimul_destroy(trimul_handle h);

/* Thread-local message describing the last non-OK status returned on this thread. */
const char* trimul_last_error(void);

/*
 * Kernel launches one trimul_forward (or trimul_forward_noalloc) call enqueues
 * for a B x N input, status reset excluded: the input projection, the
 * triangle GEMM (one launch per group of channel planes, sized so that the
 * CTA pairs of a launch stay within a few planes and share their operands in
 * L2), and the output projection.  -1 for a null handle or an empty shape.
 */
int trimul_kernels_per_forward(trimul_handle h, int B, int N);

/*
 * Make `stream` wait until every device-to-host copy of out that earlier
 * trimul_forward_host calls on this handle enqueued (with or without
 * TRIMUL_FLAG_DEFER_OUTPUT) has completed.  Enqueues a wait; returns at once.
 */
trimul_status trimul_host_join(trimul_handle h, void* stream);

/*
 * Kernels one trimul_forward_host call launches for a B x N input: as
 * trimul_forward, except that the input and output projections run once per
 * range of pair tiles when the call works in ranges (see
 * trimul_forward_host).  -1 for a null handle or an empty shape.
 */
int trimul_kernels_per_forward_host(trimul_handle h, int B, int N);

#ifdef __cplusplus
}
#endif

#endif /* TRIMUL_H_ */
