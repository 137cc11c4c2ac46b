// Weighted gather-combine, RMSNorm and the dequantisation test hook.
//
// combine:  out[t] = bf16(res[t] + g[t] * y_shared[t] + sum_j w[t,j] * y[inv[t*k+j]])
//           fp32, summed in that order (the layer's bf16 weighted gather-combine
//           with the shared expert's output and a residual add); g[t] = 1, or
//           with a shared-expert gate vector, sigmoid(x[t] . gate) in fp32.
// rmsnorm:  x = bf16(r / sqrt(mean(r^2) + eps)), fp32 (between stacked layers);
//           the combine can also write it for its own output rows (the next
//           layer's input in a stack), with the same arithmetic in the same
//           order as the separate kernel, so the two agree bit for bit.
// dequant:  w = bf16_rne(scale * q + bias) ("Prefill": 64 weights share one bf16
//           scale and bias; weights are rebuilt to bf16).
#include "common.cuh"
#include "kernels.h"

namespace moe {

__device__ __forceinline__ void unpack8(uint4 v, float f[8]) {
  const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(u[i] << 16);
    f[2 * i + 1] = __uint_as_float(u[i] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ uint4 pack8(const float f[8]) {
  uint32_t u[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) u[i] = f32_to_bf16(f[2 * i]) | ((uint32_t)f32_to_bf16(f[2 * i + 1]) << 16);
  return make_uint4(u[0], u[1], u[2], u[3]);
}

// RMSNorm of row r (bf16, H values) into xo, by the whole block (256
// threads, thread t owning columns 8t, 8t + 2048, ...): the sum of squares
// per thread in column order, warp sums, the warps' partials in warp order.
// Every thread of the block calls it; s_part holds 8 floats.
__device__ __forceinline__ void rmsnorm_row(const uint16_t *r, int H, float eps, uint16_t *xo, float *s_part) {
  float ss = 0.f;
  for (int c = threadIdx.x * 8; c < H; c += blockDim.x * 8) {
    float v[8];
    unpack8(*reinterpret_cast<const uint4 *>(r + c), v);
#pragma unroll
    for (int i = 0; i < 8; ++i) ss = fmaf(v[i], v[i], ss);
  }
  ss = warp_sum(ss);
  if ((threadIdx.x & 31) == 0) s_part[threadIdx.x >> 5] = ss;
  __syncthreads();
  float tot = 0.f;
  for (int w = 0; w < (int)(blockDim.x >> 5); ++w) tot += s_part[w];
  const float scale = rsqrtf(tot / (float)H + eps);
  for (int c = threadIdx.x * 8; c < H; c += blockDim.x * 8) {
    float v[8];
    unpack8(*reinterpret_cast<const uint4 *>(r + c), v);
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] *= scale;
    *reinterpret_cast<uint4 *>(xo + c) = pack8(v);
  }
}

// One block per token; each thread owns 8 consecutive columns.  KMAX >= k:
// the rows' loads are all in flight before the sums.  xnorm (or null): also
// the RMSNorm of the output row, for the next layer of a stack (x may alias
// it: this block reads row t of x before it writes row t of xnorm).
template <int KMAX>
__global__ void __launch_bounds__(256) combine_kernel(const uint16_t *res, const uint16_t *__restrict__ y,
                                                      const int32_t *__restrict__ inv,
                                                      const float *__restrict__ topk_w, const uint16_t *x,
                                                      const float *__restrict__ sh_gate, int T, int H, int k, int S,
                                                      uint16_t *out, uint16_t *xnorm, float eps) {
  const int t = blockIdx.x;
  __shared__ int s_row[16];
  __shared__ float s_w[16];
  __shared__ float s_part[8];
  // launched as a programmatic dependent of the down GEMM: its y first
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (threadIdx.x < k) {
    s_row[threadIdx.x] = inv[(size_t)t * k + threadIdx.x];
    s_w[threadIdx.x] = topk_w[(size_t)t * k + threadIdx.x];
  }
  float gsh = 1.f;  // the shared expert's gate
  if (S && sh_gate) {
    float z = 0.f;
    for (int c = threadIdx.x * 8; c < H; c += blockDim.x * 8) {
      float v[8];
      unpack8(*reinterpret_cast<const uint4 *>(x + (size_t)t * H + c), v);
      const float4 g0 = *reinterpret_cast<const float4 *>(sh_gate + c);
      const float4 g1 = *reinterpret_cast<const float4 *>(sh_gate + c + 4);
      z = fmaf(v[0], g0.x, z);
      z = fmaf(v[1], g0.y, z);
      z = fmaf(v[2], g0.z, z);
      z = fmaf(v[3], g0.w, z);
      z = fmaf(v[4], g1.x, z);
      z = fmaf(v[5], g1.y, z);
      z = fmaf(v[6], g1.z, z);
      z = fmaf(v[7], g1.w, z);
    }
    z = warp_sum(z);
    if ((threadIdx.x & 31) == 0) s_part[threadIdx.x >> 5] = z;
    __syncthreads();
    z = 0.f;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) z += s_part[w];
    gsh = 1.f / (1.f + expf(-z));
  }
  __syncthreads();
  for (int c = threadIdx.x * 8; c < H; c += blockDim.x * 8) {
    // every row's 16 bytes are requested before the first sum; the sums then
    // run in the fixed order
    uint4 yv[KMAX];
    const uint4 rv = *reinterpret_cast<const uint4 *>(res + (size_t)t * H + c);
    const uint4 sv = S ? *reinterpret_cast<const uint4 *>(y + ((size_t)k * T + t) * H + c) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int j = 0; j < KMAX; ++j)
      if (j < k) yv[j] = *reinterpret_cast<const uint4 *>(y + (size_t)s_row[j] * H + c);
    float acc[8], v[8];
    unpack8(rv, acc);
    if (S) {
      unpack8(sv, v);
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = fmaf(gsh, v[i], acc[i]);
    }
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
      if (j >= k) break;
      unpack8(yv[j], v);
      const float wj = s_w[j];
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = fmaf(wj, v[i], acc[i]);
    }
    *reinterpret_cast<uint4 *>(out + (size_t)t * H + c) = pack8(acc);
  }
  if (xnorm) {  // the block's writes of the row are visible to it after the barrier
    __syncthreads();
    rmsnorm_row(out + (size_t)t * H, H, eps, xnorm + (size_t)t * H, s_part);
  }
}

__global__ void __launch_bounds__(256) rmsnorm_kernel(const uint16_t *__restrict__ r, int H, float eps,
                                                      uint16_t *__restrict__ x) {
  __shared__ float s_part[8];
  const int t = blockIdx.x;
  rmsnorm_row(r + (size_t)t * H, H, eps, x + (size_t)t * H, s_part);
}

// One thread per packed word (8 weights).
__global__ void dequant_kernel(const uint32_t *__restrict__ q, const uint16_t *__restrict__ sc,
                               const uint16_t *__restrict__ b, int rows, int K, int G, uint16_t *__restrict__ w) {
  const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  const size_t words = (size_t)rows * (K / 8);
  if (i >= words) return;
  const size_t n = i / (K / 8), kw = i % (K / 8);
  const size_t g = n * (K / G) + (kw * 8) / G;
  uint32_t p[4];
  dequant_word(q[i], group_scale(bf16x2_splat(sc[g]), bf16x2_splat(b[g])), p);
  *reinterpret_cast<uint4 *>(w + n * K + kw * 8) = make_uint4(p[0], p[1], p[2], p[3]);
}

cudaError_t launch_combine(const uint16_t *res, const uint16_t *y, const int32_t *inv, const float *topk_w,
                           const uint16_t *x, const float *shared_gate, int T, int H, int k, int S, uint16_t *out,
                           uint16_t *xnorm, float eps, cudaStream_t s) {
  const bool pdl = prof_chain(MOE_KERNEL_COMBINE);  // a dependent of the down GEMM
  prof_before(MOE_KERNEL_COMBINE, s);
  const cudaError_t e =
      k <= 8 ? launch_dep(pdl, combine_kernel<8>, dim3(T), dim3(256), 0, s, res, y, inv, topk_w, x, shared_gate, T, H,
                          k, S, out, xnorm, eps)
             : launch_dep(pdl, combine_kernel<16>, dim3(T), dim3(256), 0, s, res, y, inv, topk_w, x, shared_gate, T,
                          H, k, S, out, xnorm, eps);
  prof_after(MOE_KERNEL_COMBINE, s);
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_rmsnorm(const uint16_t *r, int T, int H, float eps, uint16_t *x, cudaStream_t s) {
  prof_before(MOE_KERNEL_RMSNORM, s);
  rmsnorm_kernel<<<T, 256, 0, s>>>(r, H, eps, x);
  prof_after(MOE_KERNEL_RMSNORM, s);
  return cudaGetLastError();
}

cudaError_t launch_dequant(const uint32_t *q, const uint16_t *sc, const uint16_t *b, int rows, int K, int G,
                           uint16_t *w, cudaStream_t s) {
  const size_t words = (size_t)rows * (K / 8);
  const unsigned blocks = (unsigned)((words + 255) / 256);
  dequant_kernel<<<blocks, 256, 0, s>>>(q, sc, b, rows, K, G, w);
  return cudaGetLastError();
}

}  // namespace moe
