// Per-token top-k selection shared by the grouped and the decode routing.
// Selection ("three workload shapes": the router scores every expert and
// picks k): the k best keys under `precedes` (larger first, ties to the lower
// index, NaN last), weights = softmax over the k picked keys.
#pragma once
#include "common.cuh"

namespace moe {

// One warp per token.  Lane l holds keys l, l+32, ...; k rounds of a warp
// arg-best under `precedes`; lane j keeps the j-th pick.
template <int KPL>
__device__ __forceinline__ void topk_row(const float *__restrict__ row, int E, int k, int lane,
                                         int &my_id, float &my_key) {
  float key[KPL];
  uint32_t taken = 0;
#pragma unroll
  for (int i = 0; i < KPL; ++i) {
    int e = lane + 32 * i;
    if (e < E)
      key[i] = row[e];
    else {
      key[i] = 0.f;
      taken |= 1u << i;
    }
  }
  my_id = -1;
  my_key = 0.f;
  for (int r = 0; r < k; ++r) {
    float bk = 0.f;
    int bi = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < KPL; ++i) {
      if (taken & (1u << i)) continue;
      int e = lane + 32 * i;
      if (bi == 0x7fffffff || precedes(key[i], e, bk, bi)) {
        bk = key[i];
        bi = e;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      float ok = __shfl_xor_sync(0xffffffffu, bk, o);
      int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (oi != 0x7fffffff && (bi == 0x7fffffff || precedes(ok, oi, bk, bi))) {
        bk = ok;
        bi = oi;
      }
    }
    if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
    if (r == lane) {
      my_id = bi;
      my_key = bk;
    }
  }
}

template <int KPL>
__device__ void topk_token(const float *__restrict__ row, int E, int k, int lane, int32_t *__restrict__ ids_out,
                           float *__restrict__ w_out, int32_t *__restrict__ counts, int32_t *__restrict__ status) {
  int my_id;
  float my_key;
  topk_row<KPL>(row, E, k, lane, my_id, my_key);
  const float l0 = __shfl_sync(0xffffffffu, my_key, 0);
  float ex = (lane < k) ? expf(my_key - l0) : 0.f;
  float den = warp_sum(ex);
  bool bad = (lane < k) && !isfinite(my_key);
  if (__any_sync(0xffffffffu, bad) && lane == 0) set_status(status, MOE_ERR_NONFINITE);
  if (lane < k) {
    ids_out[lane] = my_id;
    w_out[lane] = ex / den;
    if (counts) atomicAdd(&counts[my_id], 1);
  }
}

}  // namespace moe
