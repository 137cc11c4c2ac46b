// Per-token top-k selection shared by the grouped and the decode routing.
// Selection ("three workload shapes": the router scores every expert and
// picks k): the k best keys under this order -- larger key first, equal keys
// by the lower expert index, NaN below every number, -0 == +0 -- and the
// weights are a softmax over the k picked keys.
//
// A (key, expert) pair is encoded as one 64-bit integer whose unsigned order
// is exactly that order, so selection is plain integer max / compare:
//   high word: the fp32 key mapped to an order-preserving unsigned integer
//              (NaN -> 0, below every number; -0 mapped to +0)
//   low word : 0xFFFFFFFF - expert (lower index -> larger)
#pragma once
#include "common.cuh"

namespace moe {

__device__ __forceinline__ unsigned long long topk_code(float key, int e) {
  uint32_t u = __float_as_uint(key);
  if (u == 0x80000000u) u = 0u;  // -0 == +0
  uint32_t o = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  if (isnan(key)) o = 0u;
  return ((unsigned long long)o << 32) | (0xFFFFFFFFu - (uint32_t)e);
}

__device__ __forceinline__ int topk_code_expert(unsigned long long c) {
  return (int)(0xFFFFFFFFu - (uint32_t)(c & 0xFFFFFFFFull));
}

__device__ __forceinline__ unsigned long long shfl_xor_u64(unsigned long long v, int o) {
  const uint32_t lo = __shfl_xor_sync(0xffffffffu, (uint32_t)v, o);
  const uint32_t hi = __shfl_xor_sync(0xffffffffu, (uint32_t)(v >> 32), o);
  return ((unsigned long long)hi << 32) | lo;
}

// Weights of the picked keys: softmax over the k picked keys (max = slot 0),
// written with the ids; lane j < k owns slot j.  NaN/Inf keys set the status.
// counts (or null): the histogram over experts; ccounts (or null): the same
// per chunk of SCATTER_ENT consecutive (token, slot) pairs, [chunk][E], the
// token's first pair being number p0.
__device__ __forceinline__ void topk_finish(int lane, int k, int my_id, float my_key, int32_t *__restrict__ ids_out,
                                            float *__restrict__ w_out, int32_t *__restrict__ counts,
                                            int32_t *__restrict__ status, int32_t *__restrict__ ccounts = nullptr,
                                            int E = 0, size_t p0 = 0) {
  const float l0 = __shfl_sync(0xffffffffu, my_key, 0);
  const float ex = (lane < k) ? expf(my_key - l0) : 0.f;
  const float den = warp_sum(ex);
  const bool bad = (lane < k) && !isfinite(my_key);
  if (__any_sync(0xffffffffu, bad) && lane == 0) set_status(status, MOE_ERR_NONFINITE);
  if (lane < k) {
    ids_out[lane] = my_id;
    w_out[lane] = ex / den;
    if (counts) atomicAdd(&counts[my_id], 1);
    if (ccounts) atomicAdd(&ccounts[((p0 + lane) / SCATTER_ENT) * E + my_id], 1);
  }
}

// The keys of one token come either from row (KS == 0) or, with the router's
// K split into KS slices, as part[0][e] + part[1][e] + ... + part[KS-1][e]
// (+ bias[e]), added in slice order; those sums are stored to row.
// part points at the token's row of slice 0; slices are pstride floats apart.
struct KeySrc {
  const float *part;
  size_t pstride;
  int KS;
  const float *bias;
};

// One warp selects a token's top k (k <= 16) from E <= 32*KPL keys.  Lane l
// holds experts l, l+32, ...
// cand (KPL <= 8): a warp-private shared buffer of 256 + 16 codes; null: k
// rounds of a warp-wide maximum instead.
template <int KPL>
__device__ void topk_token(float *__restrict__ row, int E, int k, int lane, int32_t *__restrict__ ids_out,
                           float *__restrict__ w_out, int32_t *__restrict__ counts, int32_t *__restrict__ status,
                           KeySrc src = KeySrc{nullptr, 0, 0, nullptr}, unsigned long long *cand = nullptr,
                           int32_t *__restrict__ ccounts = nullptr, size_t p0 = 0) {
  unsigned long long c[KPL];
  float key[KPL];
  if (src.KS > 0) {
    // every slice's loads issued before the first sum (the sums stay in
    // slice order; the router splits K into at most 8 slices)
#pragma unroll
    for (int i = 0; i < KPL; ++i) key[i] = lane + 32 * i < E ? src.part[lane + 32 * i] : 0.f;
#pragma unroll
    for (int s = 1; s < 8; ++s) {
      if (s >= src.KS) break;
      float v[KPL];
#pragma unroll
      for (int i = 0; i < KPL; ++i) v[i] = lane + 32 * i < E ? src.part[(size_t)s * src.pstride + lane + 32 * i] : 0.f;
#pragma unroll
      for (int i = 0; i < KPL; ++i) key[i] += v[i];
    }
#pragma unroll
    for (int i = 0; i < KPL; ++i) {
      const int e = lane + 32 * i;
      if (e < E) {
        if (src.bias) key[i] += src.bias[e];
        row[e] = key[i];
      }
    }
    __syncwarp();  // the stored keys are read back below
  } else {
#pragma unroll
    for (int i = 0; i < KPL; ++i) key[i] = lane + 32 * i < E ? row[lane + 32 * i] : 0.f;
  }
#pragma unroll
  for (int i = 0; i < KPL; ++i) {
    const int e = lane + 32 * i;
    c[i] = (e < E) ? topk_code(key[i], e) : 0ull;  // 0: below every real code
  }
  int my_id = -1;
  float my_key = 0.f;
  if (KPL <= 8 && cand != nullptr) {
    // Threshold, then rank.  tau = the k-th largest of the 32 lane maxima's
    // key bits (k rounds of a warp maximum, each dropping the lanes that hold
    // it): k distinct keys reach it, so every selected key is at or above it.
    // The codes at or above it -- k of them, a few more when lanes hold
    // several large keys, all E when every key is equal -- are ranked against
    // one another; rank r < k is slot r.
    unsigned long long m = c[0];
#pragma unroll
    for (int i = 1; i < KPL; ++i) m = c[i] > m ? c[i] : m;
    uint32_t v = (uint32_t)(m >> 32), t = 0u;
    for (int r = 0; r < k; ++r) {
      t = __reduce_max_sync(0xffffffffu, v);
      if (v == t) v = 0u;
    }
    const unsigned long long tau = (unsigned long long)t << 32;
    int n = 0;
    const unsigned below = (1u << lane) - 1u;
#pragma unroll
    for (int i = 0; i < KPL; ++i) {
      const bool take = c[i] != 0ull && c[i] >= tau;
      const unsigned b = __ballot_sync(0xffffffffu, take);
      if (take) cand[n + __popc(b & below)] = c[i];
      n += __popc(b);
    }
    __syncwarp();
    for (int q = lane; q < n; q += 32) {
      const unsigned long long cq = cand[q];
      int rank = 0;
      for (int j = 0; j < n; ++j) rank += cand[j] > cq;
      if (rank < k) cand[256 + rank] = cq;  // slot order
    }
    __syncwarp();
    if (lane < k) my_id = topk_code_expert(cand[256 + lane]);
    __syncwarp();
  } else {
    for (int r = 0; r < k; ++r) {
      unsigned long long best = c[0];
#pragma unroll
      for (int i = 1; i < KPL; ++i) best = c[i] > best ? c[i] : best;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const unsigned long long other = shfl_xor_u64(best, o);
        best = other > best ? other : best;
      }
#pragma unroll
      for (int i = 0; i < KPL; ++i) c[i] = (c[i] == best) ? 0ull : c[i];  // the owner drops it
      if (r == lane) my_id = topk_code_expert(best);
    }
  }
  if (lane < k) my_key = row[my_id];
  topk_finish(lane, k, my_id, my_key, ids_out, w_out, counts, status, ccounts, E, p0);
}

}  // namespace moe
