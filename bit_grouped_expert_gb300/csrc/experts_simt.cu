// CUDA-core grouped expert GEMMs over the block map (the comparison path;
// the tensor-core kernels are in experts_tc.cu).
//
// "Prefill" section of the Lily pages: the 4-bit weights are rebuilt to bf16
// tile by tile inside the grouped GEMM, kept in on-chip memory and
// accumulated in FP32, so no unpacked weight array reaches memory.  Here a
// block rebuilds a 64-feature x 64-K tile of each matrix into shared memory
// per step and multiplies it with the tile's (up to 32) token rows.
#include "common.cuh"
#include "kernels.h"

namespace moe {

constexpr int SB_N = 64;  // output features per block
constexpr int SB_K = 64;  // K step (one quantisation group)

// Dequantise 4 consecutive words (32 codes) of one row into floats.
__device__ __forceinline__ void dequant4_to_float(uint4 words, uint16_t s, uint16_t b, float out[32]) {
  const GroupScale gs = group_scale(bf16x2_splat(s), bf16x2_splat(b));
  const uint32_t wv[4] = {words.x, words.y, words.z, words.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t p[4];
    dequant_word(wv[i], gs, p);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&p[j]));
      out[8 * i + 2 * j] = f.x;
      out[8 * i + 2 * j + 1] = f.y;
    }
  }
}

// GATEUP: rows are tokens of x (gathered through perm; shared rows are
// tokens directly), K = H, two matrices, epilogue h = bf16(silu(g) * u).
// !GATEUP: rows are h rows (contiguous), K = I, one matrix, y = bf16(acc).
template <bool GATEUP>
__global__ void __launch_bounds__(256) grouped_simt_kernel(const uint16_t *__restrict__ xin, int T, int H, int I,
                                                           int E, int k, const int32_t *__restrict__ perm,
                                                           const int32_t *__restrict__ blockmap,
                                                           const int32_t *__restrict__ n_tiles, ExpertPtrs w,
                                                           uint16_t *__restrict__ out) {
  const int tile = blockIdx.x;
  if (tile >= *n_tiles) return;
  const int4 ent = reinterpret_cast<const int4 *>(blockmap)[tile];
  const int e = ent.x, row0 = ent.y, nrows = min(ent.z, SIMT_ROWS);
  const int K = GATEUP ? H : I;   // reduction length
  const int NOUT = GATEUP ? I : H; // output features of this matrix
  const int n0 = blockIdx.y * SB_N;
  const int tid = threadIdx.x, tx = tid % 16, ty = tid / 16;

  __shared__ int s_src[SIMT_ROWS];
  __shared__ float xs[SB_K][SIMT_ROWS + 1];
  __shared__ float wa[SB_K][SB_N + 4];
  __shared__ float wb[GATEUP ? SB_K : 1][SB_N + 4];

  if (tid < SIMT_ROWS) {
    int src = -1;
    if (tid < nrows) {
      if (GATEUP)
        src = (e < E) ? perm[row0 + tid] / k : row0 + tid - k * T;  // token index
      else
        src = row0 + tid;  // h row
    }
    s_src[tid] = src;
  }
  __syncthreads();

  const uint32_t *qa;
  const uint16_t *sa, *ba;
  const uint32_t *qb = nullptr;
  const uint16_t *sb = nullptr, *bb = nullptr;
  const size_t wq = (size_t)NOUT * (K / 8), wg = (size_t)NOUT * (K / 64);
  if (GATEUP) {
    qa = w.gate_q + e * wq; sa = w.gate_s + e * wg; ba = w.gate_b + e * wg;
    qb = w.up_q + e * wq;   sb = w.up_s + e * wg;   bb = w.up_b + e * wg;
  } else {
    qa = w.down_q + e * wq; sa = w.down_s + e * wg; ba = w.down_b + e * wg;
  }

  float acc_a[2][4] = {}, acc_b[2][4] = {};
  for (int k0 = 0; k0 < K; k0 += SB_K) {
    {  // activations: 32 rows x 64 columns, one 16-byte chunk per thread
      const int r = tid / 8, c8 = tid % 8;
      const int src = s_src[r];
      uint4 v = make_uint4(0, 0, 0, 0);
      if (src >= 0) v = *reinterpret_cast<const uint4 *>(xin + (size_t)src * K + k0 + 8 * c8);
      const uint32_t vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        xs[8 * c8 + 2 * i][r] = __uint_as_float(vv[i] << 16);
        xs[8 * c8 + 2 * i + 1][r] = __uint_as_float(vv[i] & 0xFFFF0000u);
      }
    }
    // weights: (matrix, feature, half of the group) per thread, 32 codes each
    for (int job = tid; job < (GATEUP ? 2 : 1) * SB_N * 2; job += 256) {
      const int m = job / (SB_N * 2), f = (job % (SB_N * 2)) / 2, half = job % 2;
      const uint32_t *q = (m ? qb : qa) + (size_t)(n0 + f) * (K / 8) + k0 / 8 + 4 * half;
      const size_t gi = (size_t)(n0 + f) * (K / 64) + k0 / 64;
      const uint16_t s = (m ? sb : sa)[gi], b = (m ? bb : ba)[gi];
      float vals[32];
      dequant4_to_float(*reinterpret_cast<const uint4 *>(q), s, b, vals);
      float(*dst)[SB_N + 4] = m ? wb : wa;
#pragma unroll
      for (int i = 0; i < 32; ++i) dst[32 * half + i][f] = vals[i];
    }
    __syncthreads();
#pragma unroll 4
    for (int c = 0; c < SB_K; ++c) {
      const float x0 = xs[c][2 * ty], x1 = xs[c][2 * ty + 1];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float a = wa[c][4 * tx + j];
        acc_a[0][j] = fmaf(x0, a, acc_a[0][j]);
        acc_a[1][j] = fmaf(x1, a, acc_a[1][j]);
        if (GATEUP) {
          const float b = wb[c][4 * tx + j];
          acc_b[0][j] = fmaf(x0, b, acc_b[0][j]);
          acc_b[1][j] = fmaf(x1, b, acc_b[1][j]);
        }
      }
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int r = 2 * ty + i;
    if (r >= nrows) continue;
    uint16_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
      o[j] = GATEUP ? f32_to_bf16(silu(acc_a[i][j]) * acc_b[i][j]) : f32_to_bf16(acc_a[i][j]);
    uint2 pk = make_uint2(o[0] | ((uint32_t)o[1] << 16), o[2] | ((uint32_t)o[3] << 16));
    *reinterpret_cast<uint2 *>(out + (size_t)(row0 + r) * NOUT + n0 + 4 * tx) = pk;
  }
}

cudaError_t launch_gateup_simt(const uint16_t *x, int T, int H, int I, int E, int k, const int32_t *perm,
                               const int32_t *blockmap, const int32_t *n_tiles, int max_tiles, ExpertPtrs w,
                               uint16_t *h, cudaStream_t s) {
  dim3 grid(max_tiles, I / SB_N);
  prof_before(MOE_KERNEL_GATEUP, s);
  grouped_simt_kernel<true><<<grid, 256, 0, s>>>(x, T, H, I, E, k, perm, blockmap, n_tiles, w, h);
  prof_after(MOE_KERNEL_GATEUP, s);
  return cudaGetLastError();
}

cudaError_t launch_down_simt(const uint16_t *h, int T, int H, int I, int E, int k, const int32_t *blockmap,
                             const int32_t *n_tiles, int max_tiles, ExpertPtrs w, uint16_t *y, cudaStream_t s) {
  dim3 grid(max_tiles, H / SB_N);
  prof_before(MOE_KERNEL_DOWN, s);
  grouped_simt_kernel<false><<<grid, 256, 0, s>>>(h, T, H, I, E, k, nullptr, blockmap, n_tiles, w, y);
  prof_after(MOE_KERNEL_DOWN, s);
  return cudaGetLastError();
}

}  // namespace moe
