// Shared device helpers and the plan's host layout for libmoe.so.
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "moe.h"

namespace moe {

// (token, slot) pairs per block of the scatter kernel; the top-k and the
// given-ids histogram count the pairs of every such chunk per expert.
constexpr int SCATTER_ENT = 2048;

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

// The rebuild of the code pairs (j, j+4), j = 0..3, of a packed word (code i
// at bits 4i): out[j] holds w = bf16_rne(s*q + b) of code j in its low half
// and of code j+4 in its high half.
//
// Usual route, for |s| < 2^-5: the bf16 bit patterns 0 .. 0x00FF are the
// values 0 .. 255 times 2^-133 exactly (subnormals up to 0x007F, then the
// first binade, whose step is the same), so a code masked in place -- at
// bits 0..3 of a half (q * 2^-133) or at bits 4..7 (q * 2^-129) -- is an exact
// bf16 operand, and with the scale taken times 2^133 or 2^129 (powers of two:
// exact while the product stays finite, i.e. |s| < 2^-5) one fused
// multiply-add rounds the exact s*q + b once.  A word costs one shift and four
// ANDs for its four pairs.
// Other scales: 0x4300 | q is the bf16 value 128 + q; subtracting 128 is
// exact and the fused multiply-add rounds once.
struct GroupScale {
  __nv_bfloat162 s133, s129;  // s * 2^133, s * 2^129 (usual route)
  __nv_bfloat162 s, b;
  bool small;                 // |s| < 2^-5 (bf16 exponent field <= 121)
};

__device__ __forceinline__ GroupScale group_scale(__nv_bfloat162 s2, __nv_bfloat162 b2) {
  GroupScale g;
  g.s = s2;
  g.b = b2;
  g.small = (*reinterpret_cast<const uint32_t *>(&s2) & 0x7F80u) < (122u << 7);
  g.s129 = __hmul2(__hmul2(s2, __floats2bfloat162_rn(0x1p127f, 0x1p127f)), __floats2bfloat162_rn(4.f, 4.f));
  g.s133 = __hmul2(g.s129, __floats2bfloat162_rn(16.f, 16.f));
  return g;
}

__device__ __forceinline__ uint32_t fma_pair(__nv_bfloat162 s2, uint32_t codes, __nv_bfloat162 b2) {
  const __nv_bfloat162 r = __hfma2(s2, *reinterpret_cast<const __nv_bfloat162 *>(&codes), b2);
  return *reinterpret_cast<const uint32_t *>(&r);
}

// Usual route (g.small).
__device__ __forceinline__ void dq_word_small(uint32_t w, const GroupScale &g, uint32_t out[4]) {
  const uint32_t w8 = w >> 8;
  out[0] = fma_pair(g.s133, w & 0x000F000Fu, g.b);   // codes 0, 4
  out[1] = fma_pair(g.s129, w & 0x00F000F0u, g.b);   // codes 1, 5
  out[2] = fma_pair(g.s133, w8 & 0x000F000Fu, g.b);  // codes 2, 6
  out[3] = fma_pair(g.s129, w8 & 0x00F000F0u, g.b);  // codes 3, 7
}

// Any scale.
__device__ __forceinline__ void dq_word_general(uint32_t w, const GroupScale &g, uint32_t out[4]) {
  const __nv_bfloat162 k128 = __floats2bfloat162_rn(128.0f, 128.0f);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    uint32_t t = ((w >> (4 * j)) & 0x000F000Fu) | 0x43004300u;
    const __nv_bfloat162 q = __hsub2(*reinterpret_cast<__nv_bfloat162 *>(&t), k128);
    const __nv_bfloat162 r = __hfma2(g.s, q, g.b);
    out[j] = *reinterpret_cast<const uint32_t *>(&r);
  }
}

// The 8 weights of a packed word in natural order (bf16, two per 32-bit
// word: out[i] holds codes 2i and 2i+1), through the pair rebuild above.
__device__ __forceinline__ void dequant_word(uint32_t w, const GroupScale &g, uint32_t out[4]) {
  uint32_t p[4];
  if (g.small)
    dq_word_small(w, g, p);
  else
    dq_word_general(w, g, p);
  out[0] = __byte_perm(p[0], p[1], 0x5410);
  out[1] = __byte_perm(p[2], p[3], 0x5410);
  out[2] = __byte_perm(p[0], p[1], 0x7632);
  out[3] = __byte_perm(p[2], p[3], 0x7632);
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
