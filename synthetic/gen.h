/* Seeded, counter-based synthetic inputs for the MoE expert layer.
 *
 * This module draws random numbers and nothing else: it holds none of the
 * layer's arithmetic (no dequantisation, routing or GEMM).  Both the CPU
 * oracle's tests and the GPU path's tests and benchmarks take their inputs
 * from here, so the two sides see the same bytes.
 *
 * Generator: SplitMix64 (Steele, Lea & Flood, "Fast splittable pseudorandom
 * number generators", OOPSLA 2014).  A stream is named by (seed, tensor id,
 * layer, expert); draw i of a stream is mix64(key + (i + 1) * GAMMA), i.e. the
 * i-th output of a SplitMix64 whose state starts at `key`.  Any element can be
 * generated independently of the others.
 *
 * Value recipes (distributions of the pages' workload, model card shapes):
 *   uniform u  = (draw >> 11) * 2^-53                         in [0, 1)
 *   normal     = Box-Muller in double: sqrt(-2 ln(1-u1)) cos(2 pi u2) with
 *                u1 = uniform(draw 2i), u2 = uniform(draw 2i+1)
 *   bf16 value = the double rounded to fp32 (RNE), then to bf16 (RNE)
 *   4-bit code = 8 codes per 32-bit word, the word = low 32 bits of a draw
 */
#ifndef SYNTH_GEN_H
#define SYNTH_GEN_H
#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
  SYN_T_X = 1,       /* activations x [T][H] bf16 ~ N(0,1)           */
  SYN_T_ROUTER = 2,  /* router weight [E][H] fp32 ~ N(0, 0.02)       */
  SYN_T_GATE_Q = 3, SYN_T_GATE_S = 4, SYN_T_GATE_B = 5,
  SYN_T_UP_Q = 6, SYN_T_UP_S = 7, SYN_T_UP_B = 8,
  SYN_T_DOWN_Q = 9, SYN_T_DOWN_S = 10, SYN_T_DOWN_B = 11,
  SYN_T_ZIPF = 12,   /* permutation behind the Zipf expert ranking   */
  SYN_T_RESID = 13,  /* a separate residual stream [T][H] bf16        */
  SYN_T_SHGATE = 14, /* shared-expert gate vector [H] fp32 ~ N(0, 0.02) */
  /* Gated DeltaNet scan inputs */
  SYN_T_GDN_Q = 15, SYN_T_GDN_K = 16, SYN_T_GDN_V = 17, /* bf16                     */
  SYN_T_GDN_ALPHA = 18, SYN_T_GDN_BETA = 19,          /* fp32 ~ U(lo, hi)         */
  SYN_T_GDN_STATE = 20,                                /* fp32 initial state        */
  /* decode attention inputs: query, key cache, value cache, bf16 ~ N(0, 1) */
  SYN_T_ATT_Q = 21, SYN_T_ATT_K = 22, SYN_T_ATT_V = 23
};

uint64_t syn_key(uint64_t seed, uint32_t tensor, uint32_t layer, uint32_t expert);
uint64_t syn_draw(uint64_t key, uint64_t i);
double syn_uniform(uint64_t key, uint64_t i);
double syn_normal(uint64_t key, uint64_t i);
uint16_t syn_bf16_from_double(double v);

void syn_fill_normal_bf16(uint64_t key, double mean, double std, uint16_t *out, size_t n);
void syn_fill_normal_f32(uint64_t key, double mean, double std, float *out, size_t n);
void syn_fill_uniform_bf16(uint64_t key, double lo, double hi, uint16_t *out, size_t n);
void syn_fill_uniform_f32(uint64_t key, double lo, double hi, float *out, size_t n);
void syn_fill_words(uint64_t key, uint32_t *out, size_t n);

/* One expert's packed weights (gate, up: [I][H/8] words + [I][H/64] scale,
 * bias; down: [H][I/8] words + [H][I/64] scale, bias).  Scale ~ U(0.005,0.02),
 * bias ~ N(0, 0.01); with centred != 0 the bias is N(0,0.01) - 7.5*scale (the
 * scale taken as its bf16 value), which keeps the mean weight near zero. */
void syn_expert(uint64_t seed, uint32_t layer, uint32_t expert, int H, int I, int centred,
                uint32_t *gate_q, uint16_t *gate_s, uint16_t *gate_b,
                uint32_t *up_q, uint16_t *up_s, uint16_t *up_b,
                uint32_t *down_q, uint16_t *down_s, uint16_t *down_b);

/* All n_exp experts of one layer into [n_exp]-stacked arrays (OpenMP). */
void syn_layer_experts(uint64_t seed, uint32_t layer, int n_exp, int H, int I, int centred,
                       uint32_t *gate_q, uint16_t *gate_s, uint16_t *gate_b,
                       uint32_t *up_q, uint16_t *up_s, uint16_t *up_b,
                       uint32_t *down_q, uint16_t *down_s, uint16_t *down_b);

/* Zipf(s) logit bias: a seeded permutation gives each expert a rank in 1..E;
 * bias[e] = -s * ln(rank_e) (the log of the Zipf pmf up to a constant). */
void syn_zipf_bias(uint64_t seed, uint32_t layer, int E, double s, float *bias);

int syn_num_threads(void);

#ifdef __cplusplus
}
#endif
#endif
