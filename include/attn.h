/*
 * C ABI of batch-1 decode attention with grouped KV heads (same library as
 * moe.h: libmoe_gb300.so).
 *
 * "Perplexity's Lily Beats MLX-LM by 1.35x Running Qwen3.6 on Apple Silicon":
 * section "What Lily actually does" (10 of the model's 40 layers are full
 * attention) and section "Decode optimizations", the GQA paragraph (eight
 * query heads share one KV head; packing the query heads of a group into one
 * threadgroup lets them share the KV loads). The page gives no formula; this
 * is scaled dot-product attention of one new token over L cached positions:
 *
 *   o_h = sum_j softmax_j(scale * q_h . k_{g,j}) v_{g,j},  g = h / (n_q_heads / n_kv_heads)
 *
 * Status codes, stream and ownership rules are those of moe.h.
 */
#ifndef MOE_GB300_ATTN_H
#define MOE_GB300_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Workspace bytes moe_decode_attention needs for these sizes (an upper bound that
   does not depend on the GPU); 0 for unsupported sizes. */
size_t moe_decode_attention_workspace_bytes(int L, int n_q_heads, int n_kv_heads, int d);

/*
 * moe_decode_attention: out = attention of the new token's queries over the
 * cache.
 *   q      bf16 [n_q_heads][d] device, 16-byte aligned
 *   K, V   bf16 [L][n_kv_heads][d] device (position-major, as appended per
 *          token), 16-byte aligned
 *   scale  multiplies every score; <= 0 means 1 / sqrt(d)
 *   out    fp32 [n_q_heads][d] device
 *   ws     device, 4-byte aligned, >= moe_decode_attention_workspace_bytes
 * L >= 1; d in {64, 128, 256}; n_q_heads a multiple of n_kv_heads with at most
 * 8 query heads per KV head. Others: MOE_ERR_SHAPE. Two launches: a split
 * kernel (one block per KV head and slice of the cache, all of the head's
 * query heads together; online softmax per warp, at least 8 positions per
 * warp, the warps' states merged in a fixed order into one partial per block
 * and query head) and a combine kernel (one block per query head and 32
 * outputs, merging the partials with fixed-order block reductions). fp32
 * arithmetic.
 */
int moe_decode_attention(const uint16_t* q, const uint16_t* K, const uint16_t* V, int L,
                         int n_q_heads, int n_kv_heads, int d, float scale, float* out, void* ws,
                         size_t ws_bytes, void* stream);

#ifdef __cplusplus
}
#endif

#endif
