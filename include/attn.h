/* attn.h -- C ABI of the single-token (decode) attention in libmoe.so (sm_103a).
 *
 * Source: "Perplexity open-sources Lily" -- "three workload shapes" (10
 * full-attention layers, grouped-query attention with 16 query heads and 2 KV
 * heads; attention over a KV cache that grows with the context) and "Decode"
 * (the query heads of one KV group share each KV row read, "GQA packing",
 * +23.8 % at 32K; a fixed-block attention layout, +40.2 % at 128K).  Per query
 * head h, KV head g = h / (Hq / Hkv), over the L cached positions:
 *
 *   s_l = scale * (q_h . k_{l,g}),  o_h = sum_l softmax_l(s)_l * v_{l,g}
 *
 * Arithmetic: scores from bf16 products summed in fp32, softmax in fp32 (base-2
 * exponentials of the scores times scale * log2(e)), the weights rounded to
 * bf16 for the product with V (fp32 sums), blocks of positions (a multiple
 * of 64, sized so that the blocks fill the SMs once) combined in fp32, o
 * rounded once to bf16.
 *
 * Conventions as in moe.h: *_d pointers are device pointers, bf16 tensors are
 * raw 16-bit patterns, every device pointer 16-byte aligned, checks run on the
 * host before anything is enqueued, nothing is allocated or synchronised,
 * launch failures return MOE_ERR_CUDA.
 */
#ifndef ATTN_H
#define ATTN_H
#include "moe.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Bytes of workspace attn_decode needs for a cache of L positions and Hq
 * query heads of dimension D (the per-block partial results): 0 for bad
 * arguments. */
size_t attn_decode_workspace_bytes(int L, int Hq, int D);

/* One query token against a KV cache, on `stream` (a cudaStream_t, NULL for
 * the default stream).
 *   q_d     bf16 [Hq][D]          query (read)
 *   k_d     bf16 [L][Hkv][D]      key cache, position-major (read)
 *   v_d     bf16 [L][Hkv][D]      value cache, same layout (read)
 *   scale   fp32                  score scale; 0 means 1 / sqrt(D)
 *   ws_d    device workspace of ws_bytes >= attn_decode_workspace_bytes(L, Hq, D):
 *           scratch, except its first int32, a status word that the call only
 *           sets, to MOE_ERR_DEVICE_TIMEOUT, if a wait for cache rows gave up
 *           (after 1 s; the output is then invalid).  Zero it to use it.
 *   o_d     bf16 [Hq][D]          output (written)
 * Supported: D == 256, Hq == 8 * Hkv, 1 <= L <= 2^24.
 * Errors: MOE_ERR_INVALID_ARGUMENT (null pointer, L < 1, Hkv < 1, scale < 0 or
 * not finite), MOE_ERR_UNSUPPORTED (D, the head grouping, L too large),
 * MOE_ERR_MISALIGNED, MOE_ERR_WORKSPACE_TOO_SMALL, MOE_ERR_CUDA. */
moe_status attn_decode(const void *q_d, const void *k_d, const void *v_d, int L, int Hq, int Hkv, int D, float scale,
                       void *ws_d, size_t ws_bytes, void *o_d, void *stream);

#ifdef __cplusplus
}
#endif
#endif
