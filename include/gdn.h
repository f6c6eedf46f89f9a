/* gdn.h -- C ABI of the Gated DeltaNet recurrent scan on GB300 (sm_103a).
 *
 * "Optimizing on-device inference for Apple Silicon", section "Qwen creates
 * three distinct workload shapes": a Gated DeltaNet layer keeps a recurrent
 * state of fixed size; a learned gate sets how much of the state survives
 * each token and a delta update writes the token in.  Section "Keep the
 * recurrent state on chip": the state is a matrix, kept (with its gate) in
 * 32-bit float, each column held in registers for the whole scan and written
 * back only at its end; the query and key (and value) activations are
 * bfloat16.  The update (the published gated delta rule), per value head h,
 * value coordinate j and token t, with S[h][j] the d_k-vector of column j:
 *
 *     r     = S[h][j] . k_t            (k_t, q_t of key head h / (H_v / H_k))
 *     u     = beta_t[h] * (v_t[h][j] - alpha_t[h] * r)
 *     S[h][j] = alpha_t[h] * S[h][j] + u * k_t
 *     o_t[h][j] = S[h][j] . q_t
 *
 * Columns are independent, so one call scans any number of heads; a long
 * sequence may be scanned in pieces, passing state_out of one piece as
 * state_in of the next.  Pieces cut at multiples of 8 tokens give results
 * bit-identical to one scan (the kernel takes tokens 8 at a time and passes
 * the state in the float32 it keeps it in); other cuts agree up to float
 * rounding.
 * The caller applies the model's preprocessing (normalising q and k, the
 * query scale, the gate and write-strength activations) before the call.
 */
#ifndef GDN_H
#define GDN_H

#include "moe.h" /* MOE_OK and the error codes */

#ifdef __cplusplus
extern "C" {
#endif

/* One scan over T tokens on `cuda_stream` (asynchronous; all pointers device
 * memory, owned by the caller, not retained after the call returns).
 *   q, k       bf16 [T][n_k_heads][d_k]
 *   v          bf16 [T][n_v_heads][d_v]
 *   alpha      float32 [T][n_v_heads], the gate (state kept), in [0, 1]
 *   beta       float32 [T][n_v_heads], the write strength
 *   state_in   float32 [n_v_heads][d_v][d_k] (column j of head h contiguous),
 *              or NULL for a zero state
 *   state_out  float32, same layout, written after the scan, or NULL; may be
 *              state_in (each column is read before it is written)
 *   o          bf16 [T][n_v_heads][d_v], round-to-nearest of the fp32 result
 * Supported: d_k == 128, d_v a multiple of 16, n_v_heads a multiple of
 * n_k_heads, T >= 0 (T == 0 copies state_in to state_out).
 * Returns MOE_OK; MOE_ERR_INVALID_ARG for NULL required pointers, negative
 * sizes or a head count that does not divide; MOE_ERR_UNSUPPORTED for other
 * dimensions; MOE_ERR_ALIGNMENT unless q, k, v are 16-byte aligned, the
 * state pointers 8-byte, alpha and beta 4-byte and o 2-byte aligned;
 * MOE_ERR_CUDA if a launch fails (nothing is written then).  All checks are
 * made on the host before anything is launched.
 * Device-side faults are not produced by this kernel (it waits on nothing
 * but block barriers). */
int gdn_scan(const void *q, const void *k, const void *v, const float *alpha, const float *beta,
             const float *state_in, float *state_out, void *o, int T, int n_k_heads,
             int n_v_heads, int d_k, int d_v, void *cuda_stream);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H */
