/* Seeded, counter-based synthetic inputs (see gen.h for the recipes). */
#include "gen.h"

#include <math.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define SYN_GAMMA 0x9E3779B97F4A7C15ULL

static inline uint64_t mix64(uint64_t z) {
  /* SplitMix64 output function (Steele, Lea & Flood 2014). */
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

uint64_t syn_key(uint64_t seed, uint32_t tensor, uint32_t layer, uint32_t expert) {
  uint64_t k = mix64(seed + SYN_GAMMA);
  k = mix64(k ^ (((uint64_t)tensor << 40) | ((uint64_t)layer << 20) | (uint64_t)expert));
  return k;
}

uint64_t syn_draw(uint64_t key, uint64_t i) { return mix64(key + (i + 1) * SYN_GAMMA); }

double syn_uniform(uint64_t key, uint64_t i) {
  return (double)(syn_draw(key, i) >> 11) * (1.0 / 9007199254740992.0);
}

double syn_normal(uint64_t key, uint64_t i) {
  const double two_pi = 6.283185307179586476925286766559;
  double u1 = syn_uniform(key, 2 * i);
  double u2 = syn_uniform(key, 2 * i + 1);
  return sqrt(-2.0 * log(1.0 - u1)) * cos(two_pi * u2);
}

uint16_t syn_bf16_from_double(double v) {
  float f = (float)v; /* RNE to fp32 */
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return 0x7FC0;
  u += 0x7FFFu + ((u >> 16) & 1u); /* RNE to bf16 */
  return (uint16_t)(u >> 16);
}

void syn_fill_normal_bf16(uint64_t key, double mean, double std, uint16_t *out, size_t n) {
  for (size_t i = 0; i < n; ++i) out[i] = syn_bf16_from_double(mean + std * syn_normal(key, i));
}

void syn_fill_normal_f32(uint64_t key, double mean, double std, float *out, size_t n) {
  for (size_t i = 0; i < n; ++i) out[i] = (float)(mean + std * syn_normal(key, i));
}

void syn_fill_uniform_bf16(uint64_t key, double lo, double hi, uint16_t *out, size_t n) {
  for (size_t i = 0; i < n; ++i) out[i] = syn_bf16_from_double(lo + (hi - lo) * syn_uniform(key, i));
}

void syn_fill_uniform_f32(uint64_t key, double lo, double hi, float *out, size_t n) {
  for (size_t i = 0; i < n; ++i) out[i] = (float)(lo + (hi - lo) * syn_uniform(key, i));
}

void syn_fill_words(uint64_t key, uint32_t *out, size_t n) {
  for (size_t i = 0; i < n; ++i) out[i] = (uint32_t)syn_draw(key, i);
}

static double bf16_value(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

static void fill_matrix(uint64_t seed, uint32_t layer, uint32_t expert, uint32_t tq, uint32_t ts,
                        uint32_t tb, int rows, int K, int centred, uint32_t *q, uint16_t *s,
                        uint16_t *b) {
  size_t nw = (size_t)rows * (size_t)(K / 8);
  size_t ng = (size_t)rows * (size_t)(K / 64);
  syn_fill_words(syn_key(seed, tq, layer, expert), q, nw);
  syn_fill_uniform_bf16(syn_key(seed, ts, layer, expert), 0.005, 0.02, s, ng);
  uint64_t kb = syn_key(seed, tb, layer, expert);
  for (size_t i = 0; i < ng; ++i) {
    double v = 0.01 * syn_normal(kb, i);
    if (centred) v -= 7.5 * bf16_value(s[i]);
    b[i] = syn_bf16_from_double(v);
  }
}

void syn_expert(uint64_t seed, uint32_t layer, uint32_t expert, int H, int I, int centred,
                uint32_t *gate_q, uint16_t *gate_s, uint16_t *gate_b,
                uint32_t *up_q, uint16_t *up_s, uint16_t *up_b,
                uint32_t *down_q, uint16_t *down_s, uint16_t *down_b) {
  fill_matrix(seed, layer, expert, SYN_T_GATE_Q, SYN_T_GATE_S, SYN_T_GATE_B, I, H, centred,
              gate_q, gate_s, gate_b);
  fill_matrix(seed, layer, expert, SYN_T_UP_Q, SYN_T_UP_S, SYN_T_UP_B, I, H, centred,
              up_q, up_s, up_b);
  fill_matrix(seed, layer, expert, SYN_T_DOWN_Q, SYN_T_DOWN_S, SYN_T_DOWN_B, H, I, centred,
              down_q, down_s, down_b);
}

void syn_layer_experts(uint64_t seed, uint32_t layer, int n_exp, int H, int I, int centred,
                       uint32_t *gate_q, uint16_t *gate_s, uint16_t *gate_b,
                       uint32_t *up_q, uint16_t *up_s, uint16_t *up_b,
                       uint32_t *down_q, uint16_t *down_s, uint16_t *down_b) {
  const size_t gu_w = (size_t)I * (H / 8), gu_g = (size_t)I * (H / 64);
  const size_t dn_w = (size_t)H * (I / 8), dn_g = (size_t)H * (I / 64);
#pragma omp parallel for schedule(dynamic, 1)
  for (int e = 0; e < n_exp; ++e) {
    syn_expert(seed, layer, (uint32_t)e, H, I, centred,
               gate_q + e * gu_w, gate_s + e * gu_g, gate_b + e * gu_g,
               up_q + e * gu_w, up_s + e * gu_g, up_b + e * gu_g,
               down_q + e * dn_w, down_s + e * dn_g, down_b + e * dn_g);
  }
}

void syn_zipf_bias(uint64_t seed, uint32_t layer, int E, double s, float *bias) {
  /* Fisher-Yates shuffle of 0..E-1 with multiply-shift bounded draws. */
  int perm[4096];
  if (E > 4096) return;
  uint64_t key = syn_key(seed, SYN_T_ZIPF, layer, 0);
  for (int i = 0; i < E; ++i) perm[i] = i;
  for (int i = E - 1; i > 0; --i) {
    unsigned __int128 m = (unsigned __int128)syn_draw(key, (uint64_t)i) * (uint64_t)(i + 1);
    int j = (int)(m >> 64);
    int t = perm[i];
    perm[i] = perm[j];
    perm[j] = t;
  }
  /* perm[r] is the expert at rank r+1 */
  for (int r = 0; r < E; ++r) bias[perm[r]] = (float)(-s * log((double)(r + 1)));
}

int syn_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
