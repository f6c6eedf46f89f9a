/*
 * moe.h -- C ABI of the sparse Mixture-of-Experts feed-forward block on one
 * GB300 GPU (sm_103a).
 *
 * The block (from "Optimizing on-device inference for Apple Silicon",
 * Perplexity, 2026):
 *   section "Qwen creates three distinct workload shapes": a router scores E
 *   experts for each token and keeps the best k; one shared expert processes
 *   every token; experts therefore receive uneven numbers of tokens.
 *   section "Reduce intermediate traffic and dispatch traffic": each expert is
 *   two input projections with a gated activation followed by an output
 *   projection, scaled by the routing score and summed with the shared
 *   expert's result.
 * For token x (a row of d values):
 *   l_e   = Wr[e] . x + b_e                            (e < E)
 *   S     = indices of the k largest l_e (ties: lower index first)
 *   w_e   = exp(l_e) / sum_{e' in S} exp(l_e')         (= softmax over all E,
 *                                                        renormalised over S)
 *   E_e(x)= Wd[e] (silu(Wg[e] x) * (Wu[e] x)),  silu(z) = z / (1 + exp(-z))
 *   out   = sum_{e in S} w_e E_e(x) + Sd (silu(Sg x) * (Su x))
 *
 * Every pointer named "device" below must be a CUDA device pointer on the
 * device that was current when moe_create ran; "host" pointers are ordinary
 * host memory.  All matrices are row-major and contiguous.  Element type of x,
 * out and every weight is the handle's dtype (bfloat16 or float32); the
 * router bias is always float32.
 *
 * Errors: every function returns MOE_OK (0) or a negative MOE_ERR_* code and
 * leaves its outputs unspecified on error.  Device-side failures (a bounded
 * wait that ran out, an index out of range) cannot be returned by an
 * asynchronous call; they are recorded in a status word on the device and
 * returned by moe_status.  No call ever traps or asserts on the device.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MOE_OK 0
#define MOE_ERR_INVALID_ARG (-1)    /* null pointer, negative size, bad field */
#define MOE_ERR_ALIGNMENT (-2)      /* a pointer or row pitch is not 16-byte aligned */
#define MOE_ERR_UNSUPPORTED (-3)    /* dimensions outside what the kernels are built for */
#define MOE_ERR_CUDA (-4)           /* a CUDA runtime call failed */
#define MOE_ERR_DEVICE_TIMEOUT (-5) /* a bounded device wait ran out (from moe_status) */
#define MOE_ERR_DEVICE_BOUNDS (-6)  /* a device index check failed (from moe_status) */
#define MOE_ERR_OUT_OF_MEMORY (-7)  /* workspace allocation failed in moe_create */

typedef enum { MOE_BF16 = 0, MOE_F32 = 1 } moe_dtype;

typedef struct moe_handle moe_handle; /* opaque, owned by the library */

/*
 * Shapes and weights of one MoE layer.  Supported: d_model a multiple of 256
 * in [256, 16384]; d_ff a multiple of 128 in [128, 4096]; n_experts in
 * [1, 256]; top_k in [1, min(n_experts, 8)]; n_shared 0 or 1; max_tokens in
 * [1, 65536]; anything else returns MOE_ERR_UNSUPPORTED from moe_create.
 *
 * Weight layouts (all K-contiguous, i.e. the reduction index is innermost):
 *   w_router [E][d]          (the transpose of the mathematical x.Wr shape)
 *   w_gate   [E][F][d]       w_up [E][F][d]        w_down [E][d][F]
 *   s_gate   [F][d]          s_up [F][d]           s_down [d][F]
 *   router_bias [E] float32, or NULL for no bias
 * The caller owns the weights; the library keeps the pointers (it copies
 * nothing) so they must stay valid and unchanged until moe_destroy.
 */
typedef struct {
  int d_model;    /* d */
  int n_experts;  /* E */
  int top_k;      /* k */
  int d_ff;       /* F, intermediate width of every expert, shared one included */
  int n_shared;   /* 0 or 1 */
  int max_tokens; /* tokens per internal chunk; moe_forward splits longer inputs */
  moe_dtype dtype;
  const void *w_router;      /* device */
  const void *w_gate;        /* device */
  const void *w_up;          /* device */
  const void *w_down;        /* device */
  const void *s_gate;        /* device, NULL iff n_shared == 0 */
  const void *s_up;          /* device, NULL iff n_shared == 0 */
  const void *s_down;        /* device, NULL iff n_shared == 0 */
  const float *router_bias;  /* device, may be NULL */
} moe_config;

/*
 * Validate cfg, build the TMA descriptors for the weights and allocate the
 * device workspace sized for cfg->max_tokens tokens.  This is the only call
 * that allocates.  On success *out receives the handle.
 * Errors: INVALID_ARG, ALIGNMENT (weight pointers must be 16-byte aligned),
 * UNSUPPORTED, OUT_OF_MEMORY, CUDA.
 */
int moe_create(const moe_config *cfg, moe_handle **out);

/*
 * 4-bit group-affine expert weights ("Optimizing on-device inference for
 * Apple Silicon", section "Dequantise weights within matrix multiplication":
 * 4-bit codes with one scale and one bias per group of 64 weights; the block's
 * arithmetic is unchanged, only the weights are stored smaller).
 *
 * A matrix [rows][cols] (cols a multiple of 64, K-contiguous like the bf16
 * layouts above) is three device arrays:
 *   codes  [rows][cols / 2] uint8, two codes per byte along the row, the even
 *          column in the low nibble;
 *   scales [rows][cols / 64] bfloat16 bit patterns;
 *   biases [rows][cols / 64] bfloat16 bit patterns;
 * and element (r, c) is  w = scale[r][c / 64] * q + bias[r][c / 64]  with q the
 * 4-bit code (0..15).  All three pointers 16-byte aligned.
 */
typedef struct {
  const uint8_t *codes;
  const uint16_t *scales;
  const uint16_t *biases;
} moe_q4_matrix;

typedef struct {
  moe_q4_matrix gate;    /* [E * F][d] */
  moe_q4_matrix up;      /* [E * F][d] */
  moe_q4_matrix down;    /* [E * d][F] */
  moe_q4_matrix s_gate;  /* [F][d], all NULL iff n_shared == 0 */
  moe_q4_matrix s_up;    /* [F][d] */
  moe_q4_matrix s_down;  /* [d][F] */
} moe_q4_weights;

/*
 * moe_create for a layer whose expert weights (routed and shared) are 4-bit
 * group-affine; the router stays bfloat16.  cfg is as for moe_create with
 * dtype MOE_BF16 (tokens and outputs are bf16) and w_gate, w_up, w_down,
 * s_gate, s_up, s_down NULL; w holds the 4-bit matrices instead (kept by
 * pointer, like the bf16 weights).  Supported: as moe_create, with
 * (top_k + n_shared) * d_ff <= 10240.  The handle runs moe_route, moe_forward
 * with T == 1 (the batch-1 path, which reads 3.6x fewer weight bytes) and,
 * when d_model and d_ff are multiples of 512, moe_forward with T >= 2: the
 * grouped GEMMs dequantise each 64-column weight block into bf16 on the chip
 * (one rounding of s q + b) right before the tensor-core multiplication.  For
 * other shapes moe_forward with T >= 2 returns MOE_ERR_UNSUPPORTED.
 * Section "Dequantise weights within matrix multiplication".
 * Errors: INVALID_ARG, ALIGNMENT, UNSUPPORTED, OUT_OF_MEMORY, CUDA.
 */
int moe_create_q4(const moe_config *cfg, const moe_q4_weights *w, moe_handle **out);

/*
 * Quantise a device matrix w[rows][cols] (dtype MOE_BF16 or MOE_F32, cols a
 * multiple of 64) into the 4-bit group-affine format above: per group of 64
 * along a row, bias = min rounded to bfloat16, scale = (max - min) / 15 rounded
 * to bfloat16 (0 for a constant group), q = the nearest integer to
 * (w - bias) / scale clamped to 0..15 (0 when scale is 0).  Writes codes,
 * scales and biases (device, 16-byte aligned).  Asynchronous on cuda_stream.
 * Errors: INVALID_ARG, ALIGNMENT, CUDA.
 */
int moe_quantize_q4(const void *w, moe_dtype dtype, long long rows, int cols, uint8_t *codes,
                    uint16_t *scales, uint16_t *biases, void *cuda_stream);

/*
 * Routing only (the router and the routing half of the block): for T tokens
 * x[T][d] (device) writes, all device:
 *   topk_idx[T][k] int32   chosen experts of each token, by descending logit,
 *                          ties to the lower index;
 *   topk_w[T][k]   float32 their routing weights (sum to 1 per token);
 *   counts[E]      int32   number of tokens that chose each expert.
 * Sections "Qwen creates three distinct workload shapes" and "Keep expert
 * routing on the GPU" (histogram of assignments per expert).
 * Requires 1 <= T <= max_tokens (T == 0 is a no-op returning MOE_OK).
 * cuda_stream is a cudaStream_t (NULL = legacy default stream).  Asynchronous:
 * no host synchronisation, no allocation.
 */
int moe_route(moe_handle *h, const void *x, int T, int32_t *topk_idx, float *topk_w,
              int32_t *counts, void *cuda_stream);

/*
 * The whole block: out[T][d] = MoE(x[T][d]), both device, same dtype.  T == 1
 * takes the batch-1 decode kernels (section "Optimise the single-row weight
 * path"); T >= 2 takes the prefill kernels (section "Prefill: reuse weights and
 * keep routing on the GPU"), in chunks of at most max_tokens tokens (section
 * "Bound temporary memory with request chunking"; tokens are independent so
 * chunking does not change the result).  x and out must not overlap.
 * Asynchronous on cuda_stream: no host synchronisation, no allocation, no
 * device-to-host copy.  T == 0 is a no-op returning MOE_OK.
 */
int moe_forward(moe_handle *h, const void *x, int T, void *out, void *cuda_stream);

/*
 * moe_forward that also hands back the routing its own kernels computed and
 * used for this call (section "Keep expert routing on the GPU": the top-8,
 * the histogram of assignments per expert, all on the GPU).  Every path
 * writes what it actually used, not a second computation: the batch-1
 * kernels (T == 1), the small-batch router (the bf16 chunks that run the
 * grouped GEMVs, see MOE_OPT_GEMV_MAX_TOKENS) and the tensor-core or fp32
 * router of the others.
 *   topk_idx [T][k] int32  device, the chosen experts of each token, by
 *                          descending logit, ties to the lower index;
 *   topk_w   [T][k] float  device, their routing weights (sum 1 per token);
 *   counts   [E]    int32  device, tokens that chose each expert, summed over
 *                          all chunks of the call (zeroed on the stream first).
 * Each of the three may be NULL; with all three NULL this is moe_forward.
 * out and the other arguments as for moe_forward; asynchronous, no
 * allocation, no host synchronisation.  Errors: as moe_forward.
 */
int moe_forward_routed(moe_handle *h, const void *x, int T, void *out, int32_t *topk_idx,
                       float *topk_w, int32_t *counts, void *cuda_stream);

/*
 * The whole block on host buffers: out_host[T][d] = MoE(x_host[T][d]), the
 * same result as moe_forward on device copies of x, bit for bit.  Like
 * moe_forward it enqueues the work and returns (section "Keep expert routing
 * on the GPU": no host synchronisation inside the block).  The handle stages
 * batches through two device slots, used by alternate calls: the copy of
 * x_host into a slot runs on a copy-in stream of the handle's, the forward on
 * cuda_stream, the copy into out_host on a copy-out stream of the handle's.
 * A call's copy-in waits only for the forward two calls back (the slot's
 * previous user), so the copies of one batch overlap the forward of the
 * batches next to it.
 *   x_host, out_host: host, [T][d] in the handle's dtype, not overlapping.
 *     Page-locked memory (cudaHostAlloc, cudaHostRegister) gives asynchronous
 *     copies; pageable memory works, but the copies then hold up the host.
 *   The caller keeps x_host unchanged and out_host untouched until the work
 *   of a later moe_host_join on some stream has completed.
 * The first call, and any call with a larger T than all before it, allocates
 * the slots (2 x 2 x T x d elements of device memory) after draining the copy
 * streams and cuda_stream.  Calls on one handle must come from one host
 * thread and use one cuda_stream (the forward's workspace is the handle's).
 * Errors: INVALID_ARG, UNSUPPORTED (as moe_forward, checked before any copy),
 * OUT_OF_MEMORY (the slots), CUDA.  T == 0 is a no-op returning MOE_OK.
 */
int moe_forward_host(moe_handle *h, const void *x_host, int T, void *out_host,
                     void *cuda_stream);

/*
 * Make cuda_stream wait for every copy into a host buffer that
 * moe_forward_host has issued on this handle; once that stream's work has
 * completed (cudaStreamSynchronize, an event), all those results are in host
 * memory.  Asynchronous; a no-op before the first moe_forward_host.
 * Errors: INVALID_ARG, CUDA.
 */
int moe_host_join(moe_handle *h, void *cuda_stream);

/*
 * Synchronise cuda_stream, then return and clear the handle's device status
 * word: MOE_OK, MOE_ERR_DEVICE_TIMEOUT or MOE_ERR_DEVICE_BOUNDS.  If
 * detail != NULL it receives a library-defined code naming the kernel and the
 * wait or check that failed (0 when none).
 */
int moe_status(moe_handle *h, void *cuda_stream, int *detail);

/*
 * Tuning options of a handle; each keeps its default until set.
 * MOE_OPT_PAIR_MIN_TOKENS, MOE_OPT_MMA2_MIN_TOKENS,
 * MOE_OPT_MMA2_DOWN_MIN_TOKENS and MOE_OPT_ROUTER_PAIR_MIN_TOKENS change no
 * result bit (the same tiles are multiplied, and the same partial sums
 * added, in the same order either way);
 * MOE_OPT_GEMV_MAX_TOKENS picks
 * between two kernels that sum in different orders (both fp32, both within
 * the block's tolerance).
 *   MOE_OPT_PAIR_MIN_TOKENS: chunks of at least this many tokens through a
 *     bf16 handle run the grouped GEMMs on thread-block clusters of two CTAs
 *     that multiply consecutive 128-row tiles of one expert group with the
 *     same weight tile, each CTA loading half of the tile into both (section
 *     "Match tile size to expert load": large groups share weight traffic).
 *     Default 8192; 0 for every chunk, a value above max_tokens for none.
 *     Ignored where the device cannot run such clusters.
 *   MOE_OPT_MMA2_MIN_TOKENS: chunks of at least this many tokens through a
 *     bf16 handle run the gate/up GEMM on the two-CTA tensor-core MMA: a
 *     cluster of two CTAs computes a 256 x 256 tile of one expert group, each
 *     CTA staging its own 128 rows and half of the weight tile.  Takes
 *     precedence over MOE_OPT_PAIR_MIN_TOKENS.  Default 8192; 0 for every
 *     chunk, a value above max_tokens for none.  Ignored where the device
 *     cannot run such clusters.
 *   MOE_OPT_MMA2_DOWN_MIN_TOKENS: the same for the down GEMM (default
 *     16384: with groups of a few hundred rows the down GEMM's short K does
 *     not repay the half-empty tile pairs).
 *   MOE_OPT_ROUTER_PAIR_MIN_TOKENS: chunks of at least this many bf16 tokens
 *     that take the cluster router run it on clusters of two CTAs per 128
 *     tokens (each multiplying half of d) instead of four.  Default: the
 *     smallest chunk whose four-CTA clusters would not all be resident at
 *     once (128 * floor(SMs / 4) + 1 tokens).  0 for every such chunk, a
 *     value above max_tokens for none.
 *   MOE_OPT_GEMV_MAX_TOKENS: chunks of at most this many tokens (0..32)
 *     route on the small-batch router and run the experts as grouped GEMVs
 *     (warp-level MMAs over all SMs); larger chunks take the cluster router
 *     and the grouped GEMMs.  Default
 *     16 for bf16 weights and 32 for 4-bit ones (where the GEMMs dequantise
 *     every weight tile for few rows).  4-bit layers whose shapes the 4-bit
 *     GEMMs do not take use the GEMVs whatever the value.
 * Host-side only, takes effect at the next call; not to be changed while
 * a forward on the handle is being captured into a CUDA graph.
 * Errors: INVALID_ARG (null handle, unknown option, value out of range).
 */
#define MOE_OPT_PAIR_MIN_TOKENS 1
#define MOE_OPT_GEMV_MAX_TOKENS 3
#define MOE_OPT_MMA2_MIN_TOKENS 4
#define MOE_OPT_MMA2_DOWN_MIN_TOKENS 5
#define MOE_OPT_ROUTER_PAIR_MIN_TOKENS 6
int moe_set_option(moe_handle *h, int option, long long value);

/* Free the workspace and the handle.  NULL is accepted.  The caller must make
 * sure no work using the handle is still running. */
int moe_destroy(moe_handle *h);

/* Static string describing an error code. */
const char *moe_strerror(int code);

/*
 * Per-kernel timing with CUDA events recorded on the launching stream around
 * every kernel the handle launches.  moe_profile(h, 1) resets the totals and
 * starts recording, moe_profile(h, 0) stops.  moe_profile_read synchronises
 * the last recorded event and writes, for kernel kind i < n (see
 * MOE_KERNEL_*), the summed milliseconds to ms[i] and the number of launches
 * to launches[i] (either pointer may be NULL).  Kinds that have not run read 0.
 */
#define MOE_KERNEL_ROUTER 0
#define MOE_KERNEL_PERMUTE 1
#define MOE_KERNEL_GEMM_GATE_UP 2
#define MOE_KERNEL_GEMM_DOWN 3
#define MOE_KERNEL_COMBINE 4
#define MOE_KERNEL_DECODE_ROUTER 5
#define MOE_KERNEL_DECODE_GATE_UP 6
#define MOE_KERNEL_DECODE_DOWN 7
#define MOE_KERNEL_GEMV_GATE_UP 8 /* small batches: the grouped GEMVs */
#define MOE_KERNEL_GEMV_DOWN 9
#define MOE_KERNEL_KINDS 10
int moe_profile(moe_handle *h, int enable);
int moe_profile_read(moe_handle *h, float *ms, int64_t *launches, int n);

/*
 * Test hook for the device failure path: launch one small kernel on
 * cuda_stream that waits, with the same bounded wait the GEMM kernels use, on
 * a barrier nothing will ever signal, giving up after about wait_us
 * microseconds (1 <= wait_us <= 2000000).  The kernel then records
 * MOE_ERR_DEVICE_TIMEOUT in the handle's status word and returns; the context
 * stays usable.  Read the result with moe_status.  With h == NULL the kernel
 * records it in the status word of moe_decode_noalloc on the current device
 * instead (read it with moe_noalloc_status).
 */
int moe_debug_wait_timeout(moe_handle *h, int wait_us, void *cuda_stream);

/*
 * Batch-1 forward of one layer that allocates no device memory, for callers
 * that cannot call cudaMalloc (an application whose allocator owns the whole
 * device pool, a serving loop that must not allocate after start-up, a plugin
 * that is only handed device pointers) and so cannot use moe_create.  The
 * pages have no counterpart to this entry point.
 *
 * cfg describes the layer exactly as for moe_create (max_tokens is ignored);
 * x[d] and out[d] are device rows of cfg->dtype, 16-byte aligned, not
 * overlapping.  Result: out = MoE(x), computed by the same decode kernels as
 * moe_forward with T == 1 (bit for bit the same result).
 *
 * Scratch: one static device array of 66,576 bytes inside the library, which
 * every GPU that loads the library holds until the process exits.  It limits
 * (top_k + n_shared) * d_ff to 16384; larger layers return
 * MOE_ERR_UNSUPPORTED, as do the limits of moe_create.  The first call on a
 * device looks up the array's device address (once per device, with that
 * device current), so make that first call before any stream capture.  All
 * calls share the array: calls that overlap on the GPU, on different streams
 * or from different threads, race on it and must be serialised by the caller.
 * Within a call every scratch value is written before it is read, unless a
 * device-side failure cuts the call short: a bounded wait in the kernels
 * that runs out leaves out unspecified and records MOE_ERR_DEVICE_TIMEOUT in
 * a status word kept in the same array (the first failure wins until it is
 * read), which moe_noalloc_status returns.
 * Errors: INVALID_ARG, ALIGNMENT, UNSUPPORTED, CUDA.  Asynchronous on
 * cuda_stream; no host synchronisation.
 */
int moe_decode_noalloc(const moe_config *cfg, const void *x, void *out, void *cuda_stream);

/*
 * Synchronise cuda_stream, then return and clear the device status word of
 * moe_decode_noalloc on the current device: MOE_OK, MOE_ERR_DEVICE_TIMEOUT or
 * MOE_ERR_DEVICE_BOUNDS, the first device-side failure of any call since the
 * last read.  If detail != NULL it receives the library-defined code of the
 * kernel and wait that failed (0 when none).  Allocates nothing; like
 * moe_decode_noalloc, its first use on a device looks the array up.
 * Errors: CUDA.
 */
int moe_noalloc_status(void *cuda_stream, int *detail);

#ifdef __cplusplus
}
#endif
#endif /* MOE_GB300_H */
