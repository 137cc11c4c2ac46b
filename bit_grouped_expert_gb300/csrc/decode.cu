// T == 1 decode path ("Decode" section of the Lily pages: at batch 1 there is
// almost no weight reuse, so bandwidth sets the ceiling; only the bytes of the
// selected experts are streamed).  Three launches:
//   decode_router_kernel   keys = x . router^T (+bias); the last block to
//                          finish picks the top k (no host sync, no spin)
//   decode_gateup_kernel   one warp per (slot, row): g, u over the packed
//                          gate/up rows of the k picked experts and the
//                          shared one; h = bf16(silu(g) * u)
//   decode_down_kernel     one warp per output feature: y_j = bf16(h_j . Wd_j)
//                          for every slot, then out = bf16(res + y_shared +
//                          sum_j w_j * y_j) -- the combine and residual add
//                          fused into the down projection
// All weight reads are 16-byte (gate/up) or 8-byte (down) coalesced loads
// of the packed codes; nothing unpacked is written to memory.
#include "common.cuh"
#include "kernels.h"
#include "topk.cuh"

namespace moe {

// ---------------------------------------------------------------- router
// Block b: experts 2b and 2b+1, four warps per expert row, each warp a
// quarter of H.  Partial sums are added in a fixed order.
__global__ void __launch_bounds__(256) decode_router_kernel(const uint16_t *__restrict__ x, int H,
                                                            const float *__restrict__ router, int E,
                                                            const float *__restrict__ bias, float *__restrict__ keys,
                                                            int k, int32_t *__restrict__ topk_id,
                                                            float *__restrict__ topk_w, int32_t *__restrict__ counter,
                                                            int32_t *__restrict__ status) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int e = blockIdx.x * 2 + (warp >> 2), q = warp & 3;
  const int seg = H / 4;
  float acc = 0.f;
  if (e < E) {
    const float *wrow = router + (size_t)e * H + (size_t)q * seg;
    const uint16_t *xr = x + (size_t)q * seg;
    for (int c = lane * 4; c < seg; c += 128) {
      const float4 wv = *reinterpret_cast<const float4 *>(wrow + c);
      const uint2 xv = *reinterpret_cast<const uint2 *>(xr + c);
      acc = fmaf(__uint_as_float(xv.x << 16), wv.x, acc);
      acc = fmaf(__uint_as_float(xv.x & 0xFFFF0000u), wv.y, acc);
      acc = fmaf(__uint_as_float(xv.y << 16), wv.z, acc);
      acc = fmaf(__uint_as_float(xv.y & 0xFFFF0000u), wv.w, acc);
    }
  }
  acc = warp_sum(acc);
  __shared__ float s_part[8];
  __shared__ int s_last;
  if (lane == 0) s_part[warp] = acc;
  __syncthreads();
  if (tid < 2) {
    const int ee = blockIdx.x * 2 + tid;
    if (ee < E) {
      float l = ((s_part[4 * tid] + s_part[4 * tid + 1]) + s_part[4 * tid + 2]) + s_part[4 * tid + 3];
      if (bias) l += bias[ee];
      keys[ee] = l;
    }
    __threadfence();
  }
  __syncthreads();
  if (tid == 0) s_last = (atomicAdd(counter, 1) == (int)gridDim.x - 1);
  __syncthreads();
  if (!s_last) return;
  // Last block: every other block's keys are visible (fence + counter).
  __threadfence();
  __shared__ float s_keys[1024];
  for (int i = tid; i < E; i += blockDim.x) s_keys[i] = __ldcg(keys + i);
  __syncthreads();
  if (warp == 0) {
    if (E <= 256)
      topk_token<8>(s_keys, E, k, lane, topk_id, topk_w, nullptr, status);
    else
      topk_token<32>(s_keys, E, k, lane, topk_id, topk_w, nullptr, status);
  }
  if (tid == 0) *counter = 0;  // ready for the next call on this workspace
}

// ---------------------------------------------------------------- gate/up
// x is staged in shared memory lane-major: element 32u + j (u = 16-byte
// chunk of packed codes, j = code within it) sits at (u/32)*1024 + j*32 +
// u%32, so lane u%32 reads bank u%32 for every j.
__global__ void __launch_bounds__(256) decode_gateup_kernel(const uint16_t *__restrict__ x, int H, int E, int k,
                                                            int I, int S, ExpertPtrs w,
                                                            const int32_t *__restrict__ topk_id,
                                                            uint16_t *__restrict__ hbuf) {
  extern __shared__ float s_x[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  for (int kk = tid; kk < H; kk += blockDim.x) {
    const int u = kk >> 5, j = kk & 31;
    s_x[(u >> 5) * 1024 + j * 32 + (u & 31)] = bf16_to_f32(x[kk]);
  }
  __syncthreads();
  const int gw = blockIdx.x * 8 + warp;
  const int slot = gw / I, n = gw % I;
  if (slot >= k + S) return;
  const int e = (slot < k) ? topk_id[slot] : E;
  const size_t rq = ((size_t)e * I + n) * (H / 8), rg = ((size_t)e * I + n) * (H / 64);
  const uint4 *gq = reinterpret_cast<const uint4 *>(w.gate_q + rq);
  const uint4 *uq = reinterpret_cast<const uint4 *>(w.up_q + rq);
  float ag = 0.f, au = 0.f;
  // every load of the row is issued before any arithmetic (up to 4 x 16 B per
  // matrix per lane in flight), then the rows are dequantised and reduced
  constexpr int MAXIT = 4;
  const int nu = H / 32;
  for (int u0 = 0; u0 < nu; u0 += 32 * MAXIT) {
    uint4 wg4[MAXIT], wu4[MAXIT];
    uint16_t sgv[MAXIT], bgv[MAXIT], suv[MAXIT], buv[MAXIT];
#pragma unroll
    for (int it = 0; it < MAXIT; ++it) {
      const int u = u0 + lane + 32 * it;
      if (u < nu) {
        wg4[it] = __ldg(gq + u);
        wu4[it] = __ldg(uq + u);
        sgv[it] = __ldg(w.gate_s + rg + (u >> 1));
        bgv[it] = __ldg(w.gate_b + rg + (u >> 1));
        suv[it] = __ldg(w.up_s + rg + (u >> 1));
        buv[it] = __ldg(w.up_b + rg + (u >> 1));
      }
    }
#pragma unroll
    for (int it = 0; it < MAXIT; ++it) {
      const int u = u0 + lane + 32 * it;
      if (u >= nu) break;
      const __nv_bfloat162 sg = bf16x2_splat(sgv[it]), bg = bf16x2_splat(bgv[it]);
      const __nv_bfloat162 su = bf16x2_splat(suv[it]), bu = bf16x2_splat(buv[it]);
      const float *xs = s_x + (u >> 5) * 1024 + (u & 31);
      const uint32_t wgv[4] = {wg4[it].x, wg4[it].y, wg4[it].z, wg4[it].w};
      const uint32_t wuv[4] = {wu4[it].x, wu4[it].y, wu4[it].z, wu4[it].w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        __nv_bfloat162 pg[4], pu[4];
        dequant_word(wgv[i], sg, bg, pg);
        dequant_word(wuv[i], su, bu, pu);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float x0 = xs[(8 * i + 2 * j) * 32], x1 = xs[(8 * i + 2 * j + 1) * 32];
          const float2 fg = __bfloat1622float2(pg[j]), fu = __bfloat1622float2(pu[j]);
          ag = fmaf(x0, fg.x, ag);
          ag = fmaf(x1, fg.y, ag);
          au = fmaf(x0, fu.x, au);
          au = fmaf(x1, fu.y, au);
        }
      }
    }
  }
  ag = warp_sum(ag);
  au = warp_sum(au);
  if (lane == 0) hbuf[(size_t)slot * I + n] = f32_to_bf16(silu(ag) * au);
}

// ---------------------------------------------------------------- down + combine
// h of every slot staged lane-major like x above (8-byte chunks of 16 codes).
__global__ void __launch_bounds__(256) decode_down_kernel(const uint16_t *__restrict__ hbuf,
                                                          const uint16_t *__restrict__ res, int H, int E, int k, int I,
                                                          int S, ExpertPtrs w, const int32_t *__restrict__ topk_id,
                                                          const float *__restrict__ topk_w,
                                                          uint16_t *__restrict__ out) {
  extern __shared__ float s_h[];  // [slots][ceil(I/512)*512]
  __shared__ int s_e[17];
  __shared__ float s_w[17];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nslot = k + S;
  const int hs = ((I + 511) / 512) * 512;
  for (int i = tid; i < nslot * I; i += blockDim.x) {
    const int sl = i / I, kk = i % I;
    const int u = kk >> 4, j = kk & 15;
    s_h[sl * hs + (u >> 5) * 512 + j * 32 + (u & 31)] = bf16_to_f32(hbuf[i]);
  }
  if (tid < nslot) {
    s_e[tid] = (tid < k) ? topk_id[tid] : E;
    s_w[tid] = (tid < k) ? topk_w[tid] : 1.f;
  }
  __syncthreads();
  const int n = blockIdx.x * 8 + warp;
  if (n >= H) return;
  // all slots' code and scale loads are issued first (one 8-byte chunk of 16
  // codes per lane per slot and pass), then dequantised and reduced
  float acc[17];
#pragma unroll
  for (int sl = 0; sl < 17; ++sl) acc[sl] = 0.f;
  const int nu = I / 16;
  for (int u0 = 0; u0 < nu; u0 += 32) {
    const int u = u0 + lane;
    uint2 wv[17];
    uint16_t sv[17], bv[17];
#pragma unroll
    for (int sl = 0; sl < 17; ++sl) {
      if (sl < nslot && u < nu) {
        const size_t r = (size_t)s_e[sl] * H + n;
        wv[sl] = __ldg(reinterpret_cast<const uint2 *>(w.down_q + r * (I / 8)) + u);
        sv[sl] = __ldg(w.down_s + r * (I / 64) + (u >> 2));
        bv[sl] = __ldg(w.down_b + r * (I / 64) + (u >> 2));
      }
    }
#pragma unroll
    for (int sl = 0; sl < 17; ++sl) {
      if (sl < nslot && u < nu) {
        const __nv_bfloat162 s2 = bf16x2_splat(sv[sl]), b2 = bf16x2_splat(bv[sl]);
        const float *hs_ = s_h + sl * hs + (u >> 5) * 512 + (u & 31);
        const uint32_t wvv[2] = {wv[sl].x, wv[sl].y};
        float a = 0.f;
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          __nv_bfloat162 p[4];
          dequant_word(wvv[i], s2, b2, p);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float2 f = __bfloat1622float2(p[j]);
            a = fmaf(hs_[(8 * i + 2 * j) * 32], f.x, a);
            a = fmaf(hs_[(8 * i + 2 * j + 1) * 32], f.y, a);
          }
        }
        acc[sl] += a;
      }
    }
  }
#pragma unroll
  for (int sl = 0; sl < 17; ++sl)
    if (sl < nslot) acc[sl] = warp_sum(acc[sl]);
  if (lane == 0) {
    float o = bf16_to_f32(res[n]);
#pragma unroll
    for (int sl = 0; sl < 17; ++sl)
      if (S && sl == k) o += bf16_to_f32(f32_to_bf16(acc[sl]));
#pragma unroll
    for (int sl = 0; sl < 16; ++sl)
      if (sl < k) o = fmaf(s_w[sl], bf16_to_f32(f32_to_bf16(acc[sl])), o);
    out[n] = f32_to_bf16(o);
  }
}

cudaError_t launch_decode(const uint16_t *x, const uint16_t *res, int H, int E, int k, int I, int S,
                          const float *router, const float *bias, ExpertPtrs w, float *keys, int32_t *topk_id,
                          float *topk_w, int32_t *counter, uint16_t *hbuf, uint16_t *out, int32_t *status,
                          int *launches, cudaStream_t s) {
  prof_before(MOE_KERNEL_DECODE_ROUTER, s);
  decode_router_kernel<<<(E + 1) / 2, 256, 0, s>>>(x, H, router, E, bias, keys, k, topk_id, topk_w, counter, status);
  prof_after(MOE_KERNEL_DECODE_ROUTER, s);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  const size_t xs_bytes = (size_t)((H + 1023) / 1024) * 1024 * sizeof(float);
  const int gu_blocks = ((k + S) * I + 7) / 8;
  prof_before(MOE_KERNEL_DECODE_GATEUP, s);
  decode_gateup_kernel<<<gu_blocks, 256, xs_bytes, s>>>(x, H, E, k, I, S, w, topk_id, hbuf);
  prof_after(MOE_KERNEL_DECODE_GATEUP, s);
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  const size_t hs_bytes = (size_t)(k + S) * ((I + 511) / 512) * 512 * sizeof(float);
  prof_before(MOE_KERNEL_DECODE_DOWN, s);
  decode_down_kernel<<<(H + 7) / 8, 256, hs_bytes, s>>>(hbuf, res, H, E, k, I, S, w, topk_id, topk_w, out);
  prof_after(MOE_KERNEL_DECODE_DOWN, s);
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  *launches += 3;
  return cudaSuccess;
}

}  // namespace moe
