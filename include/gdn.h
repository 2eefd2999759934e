/*
 * C ABI of the Gated DeltaNet scan (same library as moe.h: libmoe_gb300.so).
 *
 * "Perplexity's Lily Beats MLX-LM by 1.35x Running Qwen3.6 on Apple Silicon":
 * section "What Lily actually does" (30 of the model's 40 layers are Gated
 * DeltaNet layers, linear attention with a fixed-size recurrent state) and
 * section "Prefill optimizations", third bullet (the scan keeps the state in
 * registers for the whole sequence). The page gives no formula; the scan is the
 * published gated delta rule (Yang, Kautz and Hatamizadeh, "Gated Delta
 * Networks", 2024). Per value head h, state S in R^{d_v x d_k}, token t:
 *
 *   S_t = alpha_t S_{t-1} + beta_t (v_t - alpha_t S_{t-1} k_t) k_t^T
 *   o_t = S_t q_t
 *
 * Value head h reads key/query head h / (n_v_heads / n_k_heads).
 *
 * Status codes, stream and ownership rules are those of moe.h.
 */
#ifndef MOE_GB300_GDN_H
#define MOE_GB300_GDN_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/*
 * moe_gdn_scan: the recurrence over T tokens for every value head, from the
 * state in `state` to the state after token T-1 (written back in place).
 *   q, k   bf16 [T][n_k_heads][d_k] device (used as given: any normalisation or
 *          scaling happens before the call); 16-byte aligned
 *   v      bf16 [T][n_v_heads][d_v] device; 16-byte aligned
 *   alpha  fp32 [T][n_v_heads] device, decay per token and value head
 *   beta   fp32 [T][n_v_heads] device, write strength per token and value head
 *   state  fp32 [n_v_heads][d_v][d_k] device, in/out; 16-byte aligned for d_k
 *          128, 8-byte for d_k 64
 *   out    fp32 [T][n_v_heads][d_v] device, o_t
 * d_k in {64, 128}; d_v a multiple of 8; n_v_heads a multiple of n_k_heads;
 * T >= 0 (T == 0 leaves the state unchanged and launches nothing). Others:
 * MOE_ERR_SHAPE. NULL pointers: MOE_ERR_NULL; misaligned ones: MOE_ERR_ALIGN.
 * One launch of one 8-warp block per 8 R state rows (R rows per warp: 4 when
 * d_v is a multiple of 32, else 2 or 1); every warp
 * carries its rows through all T tokens in registers (state traffic: one read
 * and one write of the state per call), the block staging 32 tokens of inputs
 * at a time in shared memory. fp32 arithmetic throughout. The launch is a
 * programmatic dependent of the previous one on the stream: it reads nothing
 * before that launch's memory is visible.
 */
int moe_gdn_scan(const uint16_t* q, const uint16_t* k, const uint16_t* v, const float* alpha,
                 const float* beta, int T, int n_k_heads, int n_v_heads, int d_k, int d_v,
                 float* state, float* out, void* stream);

/* flags of moe_gdn_scan_ex */
#define MOE_GDN_STATE_EARLY 1 /* the launch just before this one on the stream does not write
                                 `state`: the state is read before waiting for that launch */

/*
 * moe_gdn_scan_ex: moe_gdn_scan with flags (0 gives moe_gdn_scan). With
 * MOE_GDN_STATE_EARLY each block loads its state rows before it waits for the
 * previous launch on the stream (q, k, v, alpha, beta and out are still only
 * touched after the wait), so a chain of layers with distinct states overlaps
 * each layer's state read with the layer before it. The caller guarantees
 * that the previous launch does not write `state`; otherwise the result is
 * undefined. Unknown flag bits: MOE_ERR_SHAPE.
 */
int moe_gdn_scan_ex(const uint16_t* q, const uint16_t* k, const uint16_t* v, const float* alpha,
                    const float* beta, int T, int n_k_heads, int n_v_heads, int d_k, int d_v,
                    float* state, float* out, int flags, void* stream);

#ifdef __cplusplus
}
#endif

#endif
