/* CPU oracle for the MoE expert layer -- TEST INFRASTRUCTURE ONLY.
 *
 * Only the test suite, the smoke check and the benchmark's CPU-baseline leg
 * may load or call this code.  The product library never links it, and it
 * shares no code, header or table with the product library.
 *
 * Every function here is a plain, slow, direct statement of the layer as the
 * source pages describe it ("Perplexity open-sources Lily, a Rust + Metal
 * inference engine for Qwen3.6-35B-A3B"; the news.ainew.jp translation is the
 * most complete copy):
 *   - section "three workload shapes": the router scores 256 experts, picks 8,
 *     and a shared expert processes every token;
 *   - section "Prefill": groupwise-affine 4-bit checkpoint, 64 weights share a
 *     bf16 scale and a bf16 bias; weights are rebuilt to bf16 tile by tile
 *     inside the grouped GEMM and accumulated in FP32; routing runs as
 *     histogram, prefix scan, scatter and block map.
 * Arithmetic the pages leave open (affine form, nibble order, rounding
 * points, softmax placement, ties, shared-expert gate) follows the readings
 * listed at each function.  All sums are taken in fp64 in natural order.
 */
#ifndef MOE_ORACLE_H
#define MOE_ORACLE_H
#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
  int H;        /* hidden size (K of gate/up, N of down)          */
  int E;        /* routed experts                                 */
  int k;        /* experts picked per token                       */
  int I;        /* expert intermediate size                       */
  int n_shared; /* 0 or 1 shared experts (stored at index E)      */
  int G;        /* quantisation group size along K (64)           */
} orc_dims;

typedef struct {
  const float *router;                    /* [E][H] fp32                       */
  const uint32_t *gate_q, *up_q;          /* [E+S][I][H/8], nibble k%8 at 4*(k%8) */
  const uint16_t *gate_s, *gate_b;        /* [E+S][I][H/G] bf16                */
  const uint16_t *up_s, *up_b;            /* [E+S][I][H/G] bf16                */
  const uint32_t *down_q;                 /* [E+S][H][I/8]                     */
  const uint16_t *down_s, *down_b;        /* [E+S][H][I/G] bf16                */
  const float *shared_gate;               /* [H] fp32 or NULL: the shared expert's
                                             output is scaled by sigmoid(x . gate) */
} orc_weights;

double orc_bf16_to_double(uint16_t h);
/* bf16 nearest-even rounding of the exact value hi + lo (|lo| <= ulp(hi)/2). */
uint16_t orc_round_bf16(double hi, double lo);
/* Packed bytes of one expert (gate + up + down, codes + scales + biases). */
size_t orc_expert_bytes(int H, int I, int G);

void orc_dequant(const uint32_t *q, const uint16_t *s, const uint16_t *b, int rows, int K, int G,
                 uint16_t *w);
void orc_logits(const uint16_t *x, int T, int H, const float *router, int E, const float *bias,
                float *keys);
void orc_select(const float *keys, int T, int E, int k, int32_t *ids, double *w);
void orc_route_maps(const int32_t *ids, int T, int E, int k, int n_shared, int BN,
                    int32_t *counts, int32_t *offsets, int32_t *perm, int32_t *inv,
                    int32_t *blockmap, int32_t *n_tiles);
void orc_rmsnorm(const uint16_t *r, int T, int H, double eps, uint16_t *x);
int orc_moe_layer(const orc_dims *d, const uint16_t *x, const uint16_t *res, int T,
                  const orc_weights *W, const float *bias, const float *keys_in,
                  uint16_t *out, double *out_exact, float *keys_out, int32_t *ids_out,
                  double *w_out, uint16_t *h_out, uint16_t *y_out);
int orc_num_threads(void);

#ifdef __cplusplus
}
#endif
#endif
