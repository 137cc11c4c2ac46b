/* CPU oracle for the MoE expert layer -- TEST INFRASTRUCTURE ONLY.
 * (Scope, sources and readings: see moe_oracle.h.)  Plain loops, fp64 sums in
 * natural order, one bf16 rounding at each point where the layer's definition
 * rounds.  OpenMP only spreads independent tokens or experts over cores.
 */
#include "moe_oracle.h"

#include <float.h>
#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

double orc_bf16_to_double(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

static uint16_t bits_of_float(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  return (uint16_t)(u >> 16);
}

uint16_t orc_round_bf16(double hi, double lo) {
  /* bf16: 8 significant bits, fp32's exponent range, smallest subnormal 2^-133.
   * The quantum of the binade of |hi| is 2^(e-8) for |hi| = m*2^e, m in [.5,1). */
  if (isnan(hi)) return 0x7FC0;
  if (isinf(hi)) return hi > 0 ? 0x7F80 : 0xFF80;
  if (hi == 0.0) return signbit(hi) ? 0x8000 : 0x0000;
  int e;
  (void)frexp(fabs(hi), &e);
  int qe = e - 8;
  if (qe < -133) qe = -133;
  double scaled = ldexp(hi, -qe); /* exact: a power-of-two scaling */
  double fl = floor(scaled);
  double frac = scaled - fl; /* exact */
  double r;
  if (frac > 0.5) {
    r = fl + 1.0;
  } else if (frac < 0.5) {
    r = fl;
  } else if (lo > 0) {
    r = fl + 1.0;
  } else if (lo < 0) {
    r = fl;
  } else {
    r = (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0; /* ties to even */
  }
  double v = ldexp(r, qe);
  if (fabs(v) > (double)FLT_MAX) return v > 0 ? 0x7F80 : 0xFF80;
  if (v == 0.0) return signbit(hi) ? 0x8000 : 0x0000;
  return bits_of_float((float)v); /* exact: v has at most 8 significant bits */
}

size_t orc_expert_bytes(int H, int I, int G) {
  size_t codes = 3 * (size_t)H * (size_t)I / 2;              /* 4 bits per weight  */
  size_t affine = 3 * 2 * 2 * ((size_t)H * (size_t)I / (size_t)G); /* bf16 scale+bias */
  return codes + affine;
}

/* Dequantisation ("Prefill" section: 64 weights share one bf16 scale and one
 * bf16 bias; weights are rebuilt to bf16).  Reading: w = scale*q + bias with
 * q the unsigned 4-bit code, the exact value rounded once to bf16 (RNE).
 * Packing reading: 8 codes per little-endian 32-bit word, code of column k at
 * bits 4*(k%8); rows are output features, groups run along K. */
void orc_dequant(const uint32_t *q, const uint16_t *s, const uint16_t *b, int rows, int K, int G,
                 uint16_t *w) {
  for (int n = 0; n < rows; ++n) {
    for (int k = 0; k < K; ++k) {
      uint32_t word = q[(size_t)n * (K / 8) + k / 8];
      int code = (int)((word >> (4 * (k % 8))) & 15u);
      double sc = orc_bf16_to_double(s[(size_t)n * (K / G) + k / G]);
      double bi = orc_bf16_to_double(b[(size_t)n * (K / G) + k / G]);
      double prod = sc * (double)code; /* exact: 8-bit times 4-bit significands */
      /* TwoSum: hi + lo == prod + bi exactly */
      double hi = prod + bi;
      double bb = hi - prod;
      double lo = (prod - (hi - bb)) + (bi - bb);
      w[(size_t)n * K + k] = orc_round_bf16(hi, lo);
    }
  }
}

/* Router scores ("three workload shapes": the router scores all experts).
 * Reading: fp32 logits = fp32 rounding of the fp64 dot product of the bf16
 * token with the fp32 router row; an optional per-expert bias is added in
 * fp32.  The result is the selection key. */
void orc_logits(const uint16_t *x, int T, int H, const float *router, int E, const float *bias,
                float *keys) {
#pragma omp parallel for schedule(static)
  for (int t = 0; t < T; ++t) {
    for (int e = 0; e < E; ++e) {
      double acc = 0.0;
      for (int h = 0; h < H; ++h)
        acc += orc_bf16_to_double(x[(size_t)t * H + h]) * (double)router[(size_t)e * H + h];
      float l = (float)acc;
      if (bias) l = l + bias[e];
      keys[(size_t)t * E + e] = l;
    }
  }
}

/* "a precedes b" in the selection order: larger key first, equal keys by the
 * lower expert index, NaN below every number; -0 and +0 compare equal. */
static int precedes(float ka, int ia, float kb, int ib) {
  int na = isnan(ka), nb = isnan(kb);
  if (na || nb) {
    if (na && nb) return ia < ib;
    return nb; /* a is a number, b is NaN */
  }
  if (ka > kb) return 1;
  if (ka < kb) return 0;
  return ia < ib;
}

/* Top-k selection and weights ("the router scores 256 experts and selects
 * 8").  Reading: select on the fp32 keys (softmax is monotone), k largest,
 * slot order = selection order; weights = softmax over the k selected keys,
 * which equals softmax over all experts renormalised over the k picked. */
void orc_select(const float *keys, int T, int E, int k, int32_t *ids, double *w) {
#pragma omp parallel for schedule(static)
  for (int t = 0; t < T; ++t) {
    const float *row = keys + (size_t)t * E;
    int *order = (int *)malloc(sizeof(int) * (size_t)E);
    for (int e = 0; e < E; ++e) order[e] = e;
    /* plain insertion sort of all E experts */
    for (int i = 1; i < E; ++i) {
      int cur = order[i], j = i - 1;
      while (j >= 0 && precedes(row[cur], cur, row[order[j]], order[j])) {
        order[j + 1] = order[j];
        --j;
      }
      order[j + 1] = cur;
    }
    double l0 = (double)row[order[0]];
    double den = 0.0;
    for (int j = 0; j < k; ++j) den += exp((double)row[order[j]] - l0);
    for (int j = 0; j < k; ++j) {
      ids[(size_t)t * k + j] = order[j];
      w[(size_t)t * k + j] = exp((double)row[order[j]] - l0) / den;
    }
    free(order);
  }
}

/* Histogram, prefix scan, scatter and block map ("Prefill" section: routing
 * histogram, prefix scan, scatter and block map).  Pairs are (token t, slot j)
 * with id t*k+j.  counts[e] = pairs routed to e; offsets = exclusive scan with
 * offsets[E] = k*T; perm lists, for each expert in index order, its pairs in
 * ascending token order; inv is perm's inverse.  The block map cuts every
 * expert's rows into tiles of at most BN rows -- entry (expert, first row,
 * rows, 0) -- and then the shared expert's T rows (rows k*T .. k*T+T-1). */
void orc_route_maps(const int32_t *ids, int T, int E, int k, int n_shared, int BN,
                    int32_t *counts, int32_t *offsets, int32_t *perm, int32_t *inv,
                    int32_t *blockmap, int32_t *n_tiles) {
  for (int e = 0; e < E; ++e) counts[e] = 0;
  for (int p = 0; p < T * k; ++p) counts[ids[p]] += 1;
  offsets[0] = 0;
  for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
  int *fill = (int *)calloc((size_t)E, sizeof(int));
  for (int t = 0; t < T; ++t) {
    for (int j = 0; j < k; ++j) {
      int p = t * k + j;
      int e = ids[p];
      int pos = offsets[e] + fill[e]++;
      perm[pos] = p;
      inv[p] = pos;
    }
  }
  free(fill);
  int nt = 0;
  if (blockmap && BN > 0) {
    for (int e = 0; e < E; ++e) {
      for (int r0 = 0; r0 < counts[e]; r0 += BN) {
        int32_t *ent = blockmap + 4 * (size_t)nt++;
        ent[0] = e;
        ent[1] = offsets[e] + r0;
        ent[2] = (counts[e] - r0 < BN) ? counts[e] - r0 : BN;
        ent[3] = 0;
      }
    }
    if (n_shared) {
      for (int t0 = 0; t0 < T; t0 += BN) {
        int32_t *ent = blockmap + 4 * (size_t)nt++;
        ent[0] = E;
        ent[1] = k * T + t0;
        ent[2] = (T - t0 < BN) ? T - t0 : BN;
        ent[3] = 0;
      }
    }
  }
  if (n_tiles) *n_tiles = nt;
}

/* Pre-norm between stacked layers (the pages' model has 40 layers; their norm
 * is not printed).  Reading: unit-gain RMSNorm, x = bf16(r / sqrt(mean(r^2) + eps)). */
void orc_rmsnorm(const uint16_t *r, int T, int H, double eps, uint16_t *x) {
#pragma omp parallel for schedule(static)
  for (int t = 0; t < T; ++t) {
    double ss = 0.0;
    for (int h = 0; h < H; ++h) {
      double v = orc_bf16_to_double(r[(size_t)t * H + h]);
      ss += v * v;
    }
    double scale = 1.0 / sqrt(ss / (double)H + eps);
    for (int h = 0; h < H; ++h)
      x[(size_t)t * H + h] = orc_round_bf16(orc_bf16_to_double(r[(size_t)t * H + h]) * scale, 0.0);
  }
}

static void dequant_to_double(const uint32_t *q, const uint16_t *s, const uint16_t *b, int rows,
                              int K, int G, double *wd, uint16_t *scratch) {
  orc_dequant(q, s, b, rows, K, G, scratch);
  for (size_t i = 0; i < (size_t)rows * K; ++i) wd[i] = orc_bf16_to_double(scratch[i]);
}

/* One expert's SwiGLU FFN on one token row (spec reading: SwiGLU,
 * h rounded to bf16, y rounded to bf16):
 *   g = x.Wg^T, u = x.Wu^T (fp64), h = bf16(silu(g)*u), silu(g) = g/(1+e^-g);
 *   y = bf16(h.Wd^T). */
static void expert_row(const double *xr, int H, int I, const double *wg, const double *wu,
                       const double *wd, uint16_t *h_row, uint16_t *y_row, double *hbuf) {
  for (int n = 0; n < I; ++n) {
    double g = 0.0, u = 0.0;
    for (int kk = 0; kk < H; ++kk) {
      g += xr[kk] * wg[(size_t)n * H + kk];
      u += xr[kk] * wu[(size_t)n * H + kk];
    }
    double silu = g / (1.0 + exp(-g));
    h_row[n] = orc_round_bf16(silu * u, 0.0);
    hbuf[n] = orc_bf16_to_double(h_row[n]);
  }
  for (int n = 0; n < H; ++n) {
    double acc = 0.0;
    for (int i = 0; i < I; ++i) acc += hbuf[i] * wd[(size_t)n * I + i];
    y_row[n] = orc_round_bf16(acc, 0.0);
  }
}

/* The whole layer.  Routing as orc_logits/orc_select/orc_route_maps (or from
 * the caller's keys when keys_in != NULL); every routed pair and every token's
 * shared-expert row runs expert_row; then the combine (spec reading:
 * bf16 weighted gather-combine with the shared expert and a residual add):
 *   out[t] = bf16(res[t] + y_shared[t] + sum_j w[t,j] * y[t,j]),
 * summed in that order in fp64; res = x when res == NULL.  The shared expert
 * enters with weight 1 and no gate (the pages print no gate).
 * Optional outputs: keys [T][E], ids/w [T][k], h [(k+S)T][I], y [(k+S)T][H],
 * rows in the block-map row order (routed pairs in perm order, then the
 * shared rows by token).  out_exact gets the fp64 sum before its rounding. */
int orc_moe_layer(const orc_dims *d, const uint16_t *x, const uint16_t *res, int T,
                  const orc_weights *W, const float *bias, const float *keys_in,
                  uint16_t *out, double *out_exact, float *keys_out, int32_t *ids_out,
                  double *w_out, uint16_t *h_out, uint16_t *y_out) {
  const int H = d->H, E = d->E, k = d->k, I = d->I, S = d->n_shared ? 1 : 0, G = d->G;
  if (T <= 0) return 0;
  if (H % G || I % G || G % 8 || k < 1 || k > E) return -1;
  const size_t P = (size_t)T * k, R = P + (size_t)S * T;

  float *keys = (float *)malloc(sizeof(float) * (size_t)T * E);
  int32_t *ids = (int32_t *)malloc(sizeof(int32_t) * P);
  double *w = (double *)malloc(sizeof(double) * P);
  int32_t *counts = (int32_t *)malloc(sizeof(int32_t) * (size_t)E);
  int32_t *offsets = (int32_t *)malloc(sizeof(int32_t) * (size_t)(E + 1));
  int32_t *perm = (int32_t *)malloc(sizeof(int32_t) * P);
  int32_t *inv = (int32_t *)malloc(sizeof(int32_t) * P);
  uint16_t *hrows = (uint16_t *)malloc(sizeof(uint16_t) * R * I);
  uint16_t *yrows = (uint16_t *)malloc(sizeof(uint16_t) * R * H);
  double *xd = (double *)malloc(sizeof(double) * (size_t)T * H);
  if (!keys || !ids || !w || !counts || !offsets || !perm || !inv || !hrows || !yrows || !xd) return -2;

  if (keys_in)
    memcpy(keys, keys_in, sizeof(float) * (size_t)T * E);
  else
    orc_logits(x, T, H, W->router, E, bias, keys);
  orc_select(keys, T, E, k, ids, w);
  orc_route_maps(ids, T, E, k, S, 0, counts, offsets, perm, inv, NULL, NULL);
  for (size_t i = 0; i < (size_t)T * H; ++i) xd[i] = orc_bf16_to_double(x[i]);

  const size_t gu_w = (size_t)I * (H / 8), gu_g = (size_t)I * (H / G);
  const size_t dn_w = (size_t)H * (I / 8), dn_g = (size_t)H * (I / G);
#pragma omp parallel
  {
    double *wg = (double *)malloc(sizeof(double) * (size_t)I * H);
    double *wu = (double *)malloc(sizeof(double) * (size_t)I * H);
    double *wd = (double *)malloc(sizeof(double) * (size_t)H * I);
    uint16_t *scratch = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)I * H);
    double *hbuf = (double *)malloc(sizeof(double) * (size_t)I);
#pragma omp for schedule(dynamic, 1)
    for (int e = 0; e < E + S; ++e) {
      int n_rows = (e < E) ? counts[e] : T;
      if (n_rows == 0) continue;
      dequant_to_double(W->gate_q + e * gu_w, W->gate_s + e * gu_g, W->gate_b + e * gu_g, I, H, G, wg, scratch);
      dequant_to_double(W->up_q + e * gu_w, W->up_s + e * gu_g, W->up_b + e * gu_g, I, H, G, wu, scratch);
      dequant_to_double(W->down_q + e * dn_w, W->down_s + e * dn_g, W->down_b + e * dn_g, H, I, G, wd, scratch);
      for (int r = 0; r < n_rows; ++r) {
        size_t row = (e < E) ? (size_t)(offsets[e] + r) : P + (size_t)r;
        int t = (e < E) ? perm[offsets[e] + r] / k : r;
        expert_row(xd + (size_t)t * H, H, I, wg, wu, wd, hrows + row * I, yrows + row * H, hbuf);
      }
    }
    free(wg);
    free(wu);
    free(wd);
    free(scratch);
    free(hbuf);
  }

#pragma omp parallel for schedule(static)
  for (int t = 0; t < T; ++t) {
    /* optional shared-expert gate: g = 1 / (1 + exp(-x . gate)), x the expert input */
    double g = 1.0;
    if (S && W->shared_gate) {
      double z = 0.0;
      for (int h = 0; h < H; ++h) z += xd[(size_t)t * H + h] * (double)W->shared_gate[h];
      g = 1.0 / (1.0 + exp(-z));
    }
    for (int n = 0; n < H; ++n) {
      double acc = orc_bf16_to_double((res ? res : x)[(size_t)t * H + n]);
      if (S) acc += g * orc_bf16_to_double(yrows[(P + (size_t)t) * H + n]);
      for (int j = 0; j < k; ++j) {
        size_t row = (size_t)inv[(size_t)t * k + j];
        acc += w[(size_t)t * k + j] * orc_bf16_to_double(yrows[row * H + n]);
      }
      out[(size_t)t * H + n] = orc_round_bf16(acc, 0.0);
      if (out_exact) out_exact[(size_t)t * H + n] = acc;
    }
  }

  if (keys_out) memcpy(keys_out, keys, sizeof(float) * (size_t)T * E);
  if (ids_out) memcpy(ids_out, ids, sizeof(int32_t) * P);
  if (w_out) memcpy(w_out, w, sizeof(double) * P);
  if (h_out) memcpy(h_out, hrows, sizeof(uint16_t) * R * I);
  if (y_out) memcpy(y_out, yrows, sizeof(uint16_t) * R * H);
  free(keys); free(ids); free(w); free(counts); free(offsets); free(perm); free(inv);
  free(hrows); free(yrows); free(xd);
  return 0;
}

int orc_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
