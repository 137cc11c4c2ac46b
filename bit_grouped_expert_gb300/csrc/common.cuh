// Shared device helpers and the plan's host layout for libmoe.so.
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "moe.h"

namespace moe {

// ----------------------------------------------------------------- plan

struct Layout {
  // status, counter (the decode epoch) and dtags (the decode kernel's tagged
  // exchange words) lie below keys: moe_workspace_init zeroes [0, keys)
  size_t status, counter, dtags, keys, topk_id, topk_w, counts, offsets, perm, inv, blockmap, n_tiles, blockmap2,
      n_tiles2, qctr, h, y, xg, rsplit, rpart, xn, trace, total;
};

}  // namespace moe

struct moe_plan {
  moe_config cfg;
  int32_t max_tokens;
  uint32_t flags;
  int32_t block_rows;  // rows per block-map tile
  int32_t max_tiles;
  int32_t block_rows2;  // rows per tile of the second block map (tensor-core down GEMM); 0: none
  int32_t max_tiles2;
  int32_t num_sms;
  bool use_tc;         // tensor-core grouped GEMMs (else the CUDA-core ones)
  bool use_router_tc;  // tensor-core router for T >= ROUTER_TC_MIN_T
  bool use_decode;     // one-launch decode layer for T == 1
  moe::Layout lay;
};

namespace moe {

// Sticky device status (values of moe_status); the first error wins.
__device__ __forceinline__ void set_status(int32_t *status, int32_t code) {
  atomicCAS(status, 0, code);
}

// ----------------------------------------------------------------- numbers

__device__ __forceinline__ float bf16_to_f32(uint16_t h) {
  return __uint_as_float(static_cast<uint32_t>(h) << 16);
}

__device__ __forceinline__ uint16_t f32_to_bf16(float f) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

// Selection order: larger key first, equal keys by lower index, NaN below
// every number; -0 == +0.
__device__ __forceinline__ bool precedes(float ka, int ia, float kb, int ib) {
  const bool na = isnan(ka), nb = isnan(kb);
  if (na || nb) return (na && nb) ? (ia < ib) : nb;
  if (ka > kb) return true;
  if (ka < kb) return false;
  return ia < ib;
}

// fast reciprocal division: within 2 ulp of fp32, far below the bf16 rounding of h
__device__ __forceinline__ float silu(float g) { return __fdividef(g, 1.0f + __expf(-g)); }

// Dequantise the 8 codes of one packed word into 4 bf16x2 pairs, each
// w = bf16_rne(s * q + b) with one rounding (fma.rn.bf16x2 rounds the exact
// s*q+b once).  s2/b2 hold the group's scale/bias in both halves.
__device__ __forceinline__ void dequant_word(uint32_t word, __nv_bfloat162 s2, __nv_bfloat162 b2,
                                             __nv_bfloat162 out[4]) {
  // q as bf16: 0x4300 | q is 128 + q exactly; subtracting 128 is exact.
  const uint32_t hi4 = word >> 4;
  const __nv_bfloat162 k128 = __floats2bfloat162_rn(128.0f, 128.0f);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    // result bytes [word.byte i, -, hi4.byte i, -]: the low nibble of byte 0 is
    // code 2i, the low nibble of byte 2 is code 2i+1 (element 2i in the low half)
    uint32_t t = __byte_perm(word, hi4, static_cast<uint32_t>(i | ((4 + i) << 8)));
    t = (t & 0x000F000Fu) | 0x43004300u;
    __nv_bfloat162 m = *reinterpret_cast<__nv_bfloat162 *>(&t);
    __nv_bfloat162 q = __hsub2(m, k128);
    out[i] = __hfma2(s2, q, b2);
  }
}

// The rebuild through subnormal codes.  The bf16 pattern 0x000q is the
// subnormal q * 2^-133 exactly, so with the scale taken times 2^133 (exact:
// a power of two) one fused multiply-add of the masked code pair gives
// bf16_rne(s*q + b) with a single rounding -- the same bits as the
// 0x4300 | q route, without its OR and subtraction.  s * 2^133 stays finite
// for |s| < 2^-5 (bf16 exponent field <= 121); larger scales take the other
// route.
__device__ __forceinline__ bool small_scale(__nv_bfloat162 s2) {
  return (*reinterpret_cast<const uint32_t *>(&s2) & 0x7F80u) < (122u << 7);
}
__device__ __forceinline__ __nv_bfloat162 scale_for_subnormal_codes(__nv_bfloat162 s2) {
  return __hmul2(__hmul2(s2, __floats2bfloat162_rn(0x1p127f, 0x1p127f)), __floats2bfloat162_rn(64.f, 64.f));
}
// Codes at bits 0..3 and 16..19 of t (other bits ignored) -> bf16x2 weights;
// s2x from scale_for_subnormal_codes.
__device__ __forceinline__ uint32_t dq_pair_subnormal(uint32_t t, __nv_bfloat162 s2x, __nv_bfloat162 b2) {
  t &= 0x000F000Fu;
  const __nv_bfloat162 r = __hfma2(s2x, *reinterpret_cast<const __nv_bfloat162 *>(&t), b2);
  return *reinterpret_cast<const uint32_t *>(&r);
}

__device__ __forceinline__ __nv_bfloat162 bf16x2_splat(uint16_t v) {
  uint32_t u = static_cast<uint32_t>(v) | (static_cast<uint32_t>(v) << 16);
  return *reinterpret_cast<__nv_bfloat162 *>(&u);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

}  // namespace moe

// Host-side helpers shared by the .cu files.
namespace moe {
inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
template <typename T>
inline T *ws_ptr(void *ws, size_t off) {
  return reinterpret_cast<T *>(static_cast<char *>(ws) + off);
}
}  // namespace moe
