// T == 1 decode path ("Decode" section of the Lily pages: at batch 1 there is
// almost no weight reuse, so bandwidth sets the ceiling; only the bytes of the
// selected experts are streamed, and the step's kernels overlap instead of
// running as hundreds of sequential launches).
//
// One cooperative launch per layer: every CTA (one per SM) runs
//   P0  x = bf16(r / sqrt(mean(r^2) + eps)) (pre-norm plans) or x = input,
//       computed redundantly into shared memory
//   P1  router keys (fp32, one warp per expert row) and the shared expert's
//       gate/up rows (h = bf16(silu(g) * u))
//   --- grid barrier ---
//   P2  top-k over the keys (every CTA, same order, same result); the routed
//       experts' gate/up rows
//   --- grid barrier ---
//   P3  the down rows of every slot for this CTA's output features, y_j =
//       bf16(h_j . Wd_j), out = bf16(res + y_shared + sum_j w_j * y_j)
// Weight rows reach shared memory by 16-byte cp.async issued by all threads
// as soon as their addresses are known: P1 and the shared expert's down rows
// at launch, the routed experts' gate/up and down rows right after the top-k,
// so the down rows arrive while P2 computes.  The GEMVs run on mma.sync
// m16n8k16: A = the activation vector broadcast to 16 rows, B = 8 weight rows
// dequantised in registers (w = bf16_rne(scale*q + bias)), fp32 accumulate.
// The grid barrier is a monotonic 64-bit arrival counter in the workspace;
// every wait is bounded (MOE_ERR_DEVICE_TIMEOUT).
#include "common.cuh"
#include "kernels.h"
#include "tc_ptx.cuh"
#include "topk.cuh"

namespace moe {
namespace {

constexpr int DTHREADS = 512;
constexpr int DWARPS = DTHREADS / 32;
constexpr unsigned long long DTIMEOUT_NS = 1000000000ull;

struct DecArgs {
  const uint16_t *xin;  // x, or the residual stream r for pre-norm plans
  const uint16_t *res;  // residual added by the combine
  uint16_t *out;
  const float *router, *bias;
  ExpertPtrs w;
  float *keys;
  int32_t *topk_id;
  float *topk_w;
  uint16_t *hbuf;  // [k+S][I]
  unsigned long long *bar;  // monotonic arrival counter of the grid barrier
  int32_t *status;
  uint64_t *trace;  // [3][16] phase timestamps or null
  int H, E, k, I, S, prenorm;
  float eps;
  // schedule
  int n_su, rp_cta0, rp_ctas, n_ru, n_ou;
  // shared-memory layout (bytes)
  int off_x, off_h, off_red, off_keys, off_p1, off_p2, off_p3;
  int ug, ud;  // bytes of one gate/up unit (8 rows, 2 matrices) and one down slot block (8 rows)
};

__device__ __forceinline__ unsigned long long ld_acquire64(const unsigned long long *p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ unsigned long long atom_add_release64(unsigned long long *p, unsigned long long v) {
  unsigned long long old;
  asm volatile("atom.add.release.gpu.global.u64 %0, [%1], %2;" : "=l"(old) : "l"(p), "l"(v) : "memory");
  return old;
}

// Grid barrier on a monotonic arrival counter: a CTA's arrival number `old`
// belongs to the round ending at the next multiple of the grid size, so no
// reset is needed between barriers or launches (bounded wait).
__device__ bool grid_sync(unsigned long long *bar, int32_t *status) {
  __shared__ int s_ok;
  __syncthreads();
  if (threadIdx.x == 0) {
    int ok = 1;
    const unsigned long long G = gridDim.x;
    const unsigned long long old = atom_add_release64(bar, 1ull);
    const unsigned long long target = (old / G + 1ull) * G;
    if (ld_acquire64(bar) < target) {
      const uint64_t t0 = ptx::globaltimer();
      while (ld_acquire64(bar) < target) {
        if (ptx::globaltimer() - t0 > DTIMEOUT_NS) {
          set_status(status, MOE_ERR_DEVICE_TIMEOUT);
          ok = 0;
          break;
        }
      }
    }
    s_ok = ok;
  }
  __syncthreads();
  return s_ok != 0;
}

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%4,%5,%5}, {%6,%7}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(b0), "r"(b1));
}

// Codes 2q and 2q+1 of a word (its byte q) as w = bf16_rne(s*q + b), packed.
__device__ __forceinline__ uint32_t dq_pair(uint32_t word, int q, __nv_bfloat162 s2, __nv_bfloat162 b2) {
  uint32_t t = __byte_perm(word, word >> 4, (uint32_t)(q | ((4 + q) << 8)));
  t = (t & 0x000F000Fu) | 0x43004300u;
  const __nv_bfloat162 m = *reinterpret_cast<__nv_bfloat162 *>(&t);
  const __nv_bfloat162 r = __hfma2(s2, __hsub2(m, __floats2bfloat162_rn(128.f, 128.f)), b2);
  return *reinterpret_cast<const uint32_t *>(&r);
}

// One 32-K step of an 8-row GEMV: lane (g = lane/4, q = lane%4) dequantises
// row g's codes 2q,2q+1 and 2q+8,2q+9 of both 16-K halves.
__device__ __forceinline__ void gemv_step(float (&d)[4], const uint8_t *crow, const uint16_t *srow,
                                          const uint16_t *brow, const uint16_t *xs, int kk, int q) {
  const uint4 w = *reinterpret_cast<const uint4 *>(crow + kk / 2);
  const __nv_bfloat162 s2 = bf16x2_splat(srow[kk >> 6]), b2 = bf16x2_splat(brow[kk >> 6]);
  const uint32_t xa0 = *reinterpret_cast<const uint32_t *>(xs + kk + 2 * q);
  const uint32_t xb0 = *reinterpret_cast<const uint32_t *>(xs + kk + 8 + 2 * q);
  const uint32_t xa1 = *reinterpret_cast<const uint32_t *>(xs + kk + 16 + 2 * q);
  const uint32_t xb1 = *reinterpret_cast<const uint32_t *>(xs + kk + 24 + 2 * q);
  mma16816(d, xa0, xb0, dq_pair(w.x, q, s2, b2), dq_pair(w.y, q, s2, b2));
  mma16816(d, xa1, xb1, dq_pair(w.z, q, s2, b2), dq_pair(w.w, q, s2, b2));
}

// d += x[k0:k1] . W[8 rows][k0:k1] (k0, k1 multiples of 64).  Two
// accumulators alternate over the 32-K steps so consecutive MMAs are
// independent; after the call lane q holds rows 2q (d[0]) and 2q+1 (d[1]).
__device__ __forceinline__ void gemv8(const uint8_t *codes, int rs, const uint16_t *sc, const uint16_t *bi, int gs,
                                      const uint16_t *xs, int k0, int k1, int lane, float (&d)[4]) {
  const int g = lane >> 2, q = lane & 3;
  const uint8_t *crow = codes + g * rs;
  const uint16_t *srow = sc + g * gs, *brow = bi + g * gs;
  float e[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 2
  for (int kk = k0; kk < k1; kk += 64) {
    gemv_step(d, crow, srow, brow, xs, kk, q);
    gemv_step(e, crow, srow, brow, xs, kk + 32, q);
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) d[i] += e[i];
}

// Gate and up rows of one unit over the same K range, interleaved so the four
// accumulator chains overlap.
__device__ __forceinline__ void gemv8x2(const uint8_t *cg, const uint8_t *cu, int rs, const uint16_t *sg,
                                        const uint16_t *bg, const uint16_t *su, const uint16_t *bu, int gs,
                                        const uint16_t *xs, int k0, int k1, int lane, float (&dg)[4],
                                        float (&du)[4]) {
  const int g = lane >> 2, q = lane & 3;
  float eg[4] = {0.f, 0.f, 0.f, 0.f}, eu[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
  for (int kk = k0; kk < k1; kk += 64) {
    gemv_step(dg, cg + g * rs, sg + g * gs, bg + g * gs, xs, kk, q);
    gemv_step(du, cu + g * rs, su + g * gs, bu + g * gs, xs, kk, q);
    gemv_step(eg, cg + g * rs, sg + g * gs, bg + g * gs, xs, kk + 32, q);
    gemv_step(eu, cu + g * rs, su + g * gs, bu + g * gs, xs, kk + 32, q);
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    dg[i] += eg[i];
    du[i] += eu[i];
  }
}

// Shared-memory image of one gate/up unit: for each matrix, 8 code rows
// (stride H/2 + 16 to spread banks), then 8 scale rows and 8 bias rows.
__device__ __forceinline__ int gu_rs(int H) { return H / 2 + 16; }
__device__ __forceinline__ int gu_mat_bytes(int H) { return 8 * gu_rs(H) + 2 * (H / 4); }
__device__ __forceinline__ int dn_rs(int I) { return I / 2 + 16; }

__device__ __forceinline__ int ilog2(int v) { return 31 - __clz(v); }

// Stage one gate/up unit (expert e, rows r0..r0+7, both matrices) with
// 16-byte cp.async copies spread over all threads of the CTA (H is a power
// of two, so chunk indices split with shifts).
__device__ void stage_gu(const DecArgs &a, uint8_t *dst, int e, int r0) {
  const int H = a.H, rs = gu_rs(H), mb = gu_mat_bytes(H);
  const int lc = ilog2(H / 32);  // log2 of the 16-byte chunks per code row
  const size_t row = (size_t)e * a.I + r0;
  const uint8_t *q0 = reinterpret_cast<const uint8_t *>(a.w.gate_q) + row * (H / 2);
  const uint8_t *q1 = reinterpret_cast<const uint8_t *>(a.w.up_q) + row * (H / 2);
  for (int c = threadIdx.x; c < (16 << lc); c += DTHREADS) {
    const int mat = c >> (lc + 3), r = (c >> lc) & 7, j = c & ((1 << lc) - 1);
    ptx::cp_async_16(dst + mat * mb + r * rs + j * 16, (mat ? q1 : q0) + r * (H / 2) + j * 16, 16);
  }
  const int ls = ilog2(H / 64);  // chunks per 8-row scale (or bias) block: 8 * H/64 * 2 / 16
  for (int c = threadIdx.x; c < (4 << ls); c += DTHREADS) {
    const int which = c >> ls, j = c & ((1 << ls) - 1);  // 0 gate s, 1 gate b, 2 up s, 3 up b
    const uint16_t *src = which == 0 ? a.w.gate_s : which == 1 ? a.w.gate_b : which == 2 ? a.w.up_s : a.w.up_b;
    ptx::cp_async_16(dst + (which >> 1) * mb + 8 * rs + (which & 1) * (H / 4) + j * 16,
                     reinterpret_cast<const uint8_t *>(src + row * (H / 64)) + j * 16, 16);
  }
}

// Stage one down block: expert e, output rows n0..n0+7.
__device__ void stage_dn(const DecArgs &a, uint8_t *dst, int e, int n0) {
  const int I = a.I, rs = dn_rs(I);
  const int lc = ilog2(I / 32), ls = ilog2(I / 64);
  const size_t row = (size_t)e * a.H + n0;
  const uint8_t *q = reinterpret_cast<const uint8_t *>(a.w.down_q) + row * (I / 2);
  for (int c = threadIdx.x; c < (8 << lc); c += DTHREADS) {
    const int r = c >> lc, j = c & ((1 << lc) - 1);
    ptx::cp_async_16(dst + r * rs + j * 16, q + r * (I / 2) + j * 16, 16);
  }
  for (int c = threadIdx.x; c < (2 << ls); c += DTHREADS) {
    const int which = c >> ls, j = c & ((1 << ls) - 1);
    const uint16_t *src = which ? a.w.down_b : a.w.down_s;
    ptx::cp_async_16(dst + 8 * rs + which * (I / 4) + j * 16,
                     reinterpret_cast<const uint8_t *>(src + row * (I / 64)) + j * 16, 16);
  }
}

// Stage router rows e0, e0+stride, ... (n rows, fp32, H values each).
__device__ void stage_router(const DecArgs &a, float *dst, int e0, int stride, int n) {
  const int lc = ilog2(a.H / 4);
  for (int c = threadIdx.x; c < (n << lc); c += DTHREADS) {
    const int r = c >> lc, j = c & ((1 << lc) - 1);
    ptx::cp_async_16(dst + r * a.H + j * 4, a.router + (size_t)(e0 + r * stride) * a.H + j * 4, 16);
  }
}

// Top-k of one token by all threads of the CTA: each key's rank is the number
// of keys whose order code is larger (codes are distinct), so the picked
// experts land in slot order directly; warp 0 then computes the weights.
__device__ void topk_block(const float *keys, int E, int k, unsigned long long *codes, int32_t *ids, float *w,
                           int32_t *status) {
  const int tid = threadIdx.x;
  for (int e = tid; e < E; e += DTHREADS) codes[e] = topk_code(keys[e], e);
  __syncthreads();
  for (int e = tid; e < E; e += DTHREADS) {
    const unsigned long long c = codes[e];
    int rank = 0;
#pragma unroll 8
    for (int j = 0; j < E; ++j) rank += codes[j] > c;
    if (rank < k) ids[rank] = e;
  }
  __syncthreads();
  if (tid < 32) {
    const int lane = tid;
    const int my_id = lane < k ? ids[lane] : -1;
    const float my_key = lane < k ? keys[my_id] : 0.f;
    topk_finish(lane, k, my_id, my_key, ids, w, nullptr, status);
  }
}

// One gate/up unit slice: a warp reduces K range [c*len, (c+1)*len) of the
// unit at `base` and leaves 8 gate and 8 up partial sums in red[0..15].
__device__ __forceinline__ void gu_slice(const uint8_t *base, int H, int mb, const uint16_t *xs, int c, int len,
                                         int lane, float *red) {
  float dg[4] = {0.f, 0.f, 0.f, 0.f}, du[4] = {0.f, 0.f, 0.f, 0.f};
  const uint16_t *sg = reinterpret_cast<const uint16_t *>(base + 8 * gu_rs(H));
  const uint16_t *su = reinterpret_cast<const uint16_t *>(base + mb + 8 * gu_rs(H));
  gemv8x2(base, base + mb, gu_rs(H), sg, sg + 8 * (H / 64), su, su + 8 * (H / 64), H / 64, xs, c * len,
          (c + 1) * len, lane, dg, du);
  if (lane < 4) {
    red[2 * lane] = dg[0];
    red[2 * lane + 1] = dg[1];
    red[8 + 2 * lane] = du[0];
    red[8 + 2 * lane + 1] = du[1];
  }
}

__device__ __forceinline__ int k_chunks(int units, int H) {
  int kc = units > 0 ? DWARPS / units : 1;
  if (kc < 1) kc = 1;
  while (kc > 1 && (H / 64) % kc) kc >>= 1;
  return kc;
}

// Phase timestamp for the trace of CTAs 0, G/2 and G-1 (thread 0).
__device__ __forceinline__ void trace_at(const DecArgs &a, int slot) {
  if (!a.trace || threadIdx.x != 0) return;
  const int c = blockIdx.x, G = gridDim.x;
  const int row = c == 0 ? 0 : (c == G / 2 ? 1 : (c == G - 1 ? 2 : -1));
  if (row >= 0) a.trace[row * 16 + slot] = ptx::globaltimer();
}

__global__ void __launch_bounds__(DTHREADS, 1) decode_layer_kernel(const DecArgs a) {
  extern __shared__ __align__(1024) uint8_t sm[];
  __shared__ int s_ids[17];
  __shared__ float s_w[17];
  __shared__ float s_part[DWARPS];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int cta = blockIdx.x, G = gridDim.x;
  const int H = a.H, I = a.I, E = a.E, k = a.k, S = a.S, NS = k + S;
  uint16_t *xs = reinterpret_cast<uint16_t *>(sm + a.off_x);
  uint16_t *hs = reinterpret_cast<uint16_t *>(sm + a.off_h);
  float *red = reinterpret_cast<float *>(sm + a.off_red);
  float *keys = reinterpret_cast<float *>(sm + a.off_keys);
  uint8_t *p1 = sm + a.off_p1, *p2 = sm + a.off_p2, *p3 = sm + a.off_p3;
  const int mb = gu_mat_bytes(H);
  const int nsu = (cta < a.n_su) ? (a.n_su - 1 - cta) / G + 1 : 0;  // shared gate/up units of this CTA
  const int rc = cta - a.rp_cta0;                                    // index among the router CTAs
  const int nre = (rc >= 0 && rc < a.rp_ctas && rc < E) ? (E - 1 - rc) / a.rp_ctas + 1 : 0;  // router rows
  const int nou = (cta < a.n_ou) ? (a.n_ou - 1 - cta) / G + 1 : 0;  // output units of this CTA
  float *rrows = reinterpret_cast<float *>(p1 + nsu * a.ug);
  trace_at(a, 0);

  // ---------------------------------------------------------------- copies known at launch (group 0)
  for (int i = 0; i < nsu; ++i) stage_gu(a, p1 + i * a.ug, E, (cta + i * G) * 8);
  if (nre) stage_router(a, rrows, rc, a.rp_ctas, nre);
  if (S)
    for (int i = 0; i < nou; ++i) stage_dn(a, p3 + (i * NS + k) * a.ud, E, (cta + i * G) * 8);
  ptx::cp_async_commit();
  trace_at(a, 1);

  // ---------------------------------------------------------------- P0: x
  if (a.prenorm) {
    float ss = 0.f;
    for (int i = tid; i < H; i += DTHREADS) {
      const float v = bf16_to_f32(a.xin[i]);
      ss = fmaf(v, v, ss);
    }
    ss = warp_sum(ss);
    if (lane == 0) s_part[warp] = ss;
    __syncthreads();
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < DWARPS; ++w) tot += s_part[w];
    const float scale = rsqrtf(tot / (float)H + a.eps);
    for (int i = tid; i < H; i += DTHREADS) xs[i] = f32_to_bf16(bf16_to_f32(a.xin[i]) * scale);
  } else {
    for (int i = tid; i < H; i += DTHREADS) xs[i] = a.xin[i];
  }
  trace_at(a, 2);
  ptx::cp_async_wait_all();
  __syncthreads();
  trace_at(a, 3);

  // ---------------------------------------------------------------- P1: shared gate/up, router rows
  if (nsu > 0) {
    const int kc = k_chunks(nsu, H), len = H / kc;
    if (warp < nsu * kc) gu_slice(p1 + (warp / kc) * a.ug, H, mb, xs, warp % kc, len, lane, red + warp * 16);
    __syncthreads();
    if (tid < nsu * 8) {
      const int u = tid / 8, r = tid % 8;
      float g = 0.f, uu = 0.f;
      for (int c = 0; c < kc; ++c) {
        g += red[(u * kc + c) * 16 + r];
        uu += red[(u * kc + c) * 16 + 8 + r];
      }
      a.hbuf[(size_t)k * I + (cta + u * G) * 8 + r] = f32_to_bf16(silu(g) * uu);
    }
  }
  for (int i = warp; i < nre; i += DWARPS) {  // one warp per router row, fp32 FMA
    const float *row = rrows + i * H;
    float acc = 0.f;
    for (int kk = 4 * lane; kk < H; kk += 128) {
      const float4 wv = *reinterpret_cast<const float4 *>(row + kk);
      const uint2 xv = *reinterpret_cast<const uint2 *>(xs + kk);
      acc = fmaf(__uint_as_float(xv.x << 16), wv.x, acc);
      acc = fmaf(__uint_as_float(xv.x & 0xFFFF0000u), wv.y, acc);
      acc = fmaf(__uint_as_float(xv.y << 16), wv.z, acc);
      acc = fmaf(__uint_as_float(xv.y & 0xFFFF0000u), wv.w, acc);
    }
    acc = warp_sum(acc);
    const int e = rc + i * a.rp_ctas;
    if (lane == 0) a.keys[e] = a.bias ? acc + a.bias[e] : acc;
  }
  trace_at(a, 4);
  bool ok = grid_sync(a.bar, a.status);
  trace_at(a, 5);

  // ---------------------------------------------------------------- P2: routing, routed gate/up
  const int upr = I / 8;
  const int nru = (cta < a.n_ru) ? (a.n_ru - 1 - cta) / G + 1 : 0;
  if (ok) {
    for (int e = tid; e < E; e += DTHREADS) keys[e] = __ldcg(a.keys + e);
    __syncthreads();
    trace_at(a, 6);
    topk_block(keys, E, k, reinterpret_cast<unsigned long long *>(p2), s_ids, s_w, a.status);
    __syncthreads();
    trace_at(a, 14);
    if (cta == 0 && tid < k) {
      a.topk_id[tid] = s_ids[tid];
      a.topk_w[tid] = s_w[tid];
    }
    // group 1: routed gate/up units u = slot * (I/8) + rowblock with u % G == cta
    for (int i = 0; i < nru; ++i) {
      const int u = cta + i * G;
      stage_gu(a, p2 + i * a.ug, s_ids[u / upr], (u % upr) * 8);
    }
    ptx::cp_async_commit();
    // group 2: the routed experts' down rows of this CTA's output units
    for (int i = 0; i < nou; ++i)
      for (int j = 0; j < k; ++j) stage_dn(a, p3 + (i * NS + j) * a.ud, s_ids[j], (cta + i * G) * 8);
    ptx::cp_async_commit();
    trace_at(a, 7);
    ptx::cp_async_wait_1();
    __syncthreads();
    trace_at(a, 8);
    if (nru > 0) {
      const int kc = k_chunks(nru, H), len = H / kc;
      if (warp < nru * kc) gu_slice(p2 + (warp / kc) * a.ug, H, mb, xs, warp % kc, len, lane, red + warp * 16);
      __syncthreads();
      if (tid < nru * 8) {
        const int ul = tid / 8, r = tid % 8, u = cta + ul * G;
        float g = 0.f, uu = 0.f;
        for (int c = 0; c < kc; ++c) {
          g += red[(ul * kc + c) * 16 + r];
          uu += red[(ul * kc + c) * 16 + 8 + r];
        }
        a.hbuf[(size_t)(u / upr) * I + (u % upr) * 8 + r] = f32_to_bf16(silu(g) * uu);
      }
    }
  }
  trace_at(a, 9);
  ok = grid_sync(a.bar, a.status) && ok;
  trace_at(a, 10);

  // ---------------------------------------------------------------- P3: down + combine
  ptx::cp_async_wait_all();  // also drains every copy of a CTA that gave up
  if (ok) {
    // h of every slot, 16 bytes per load, all loads in flight together
    const int nvec = NS * I / 8;
    for (int i = tid; i < nvec; i += DTHREADS)
      reinterpret_cast<uint4 *>(hs)[i] = __ldcg(reinterpret_cast<const uint4 *>(a.hbuf) + i);
    __syncthreads();
    trace_at(a, 11);
    // tasks (output unit, slot, K half): partial sums, then bf16(y) per slot
    float *yp = red;  // [nou][NS][2][8] partials
    const int ntask = nou * NS * 2;
    for (int t = warp; t < ntask; t += DWARPS) {
      const int half = t & 1, ol = (t >> 1) / NS, j = (t >> 1) % NS;
      const uint8_t *base = p3 + (ol * NS + j) * a.ud;
      const uint16_t *sd = reinterpret_cast<const uint16_t *>(base + 8 * dn_rs(I));
      float d[4] = {0.f, 0.f, 0.f, 0.f};
      gemv8(base, dn_rs(I), sd, sd + 8 * (I / 64), I / 64, hs + j * I, half * (I / 2), (half + 1) * (I / 2), lane, d);
      if (lane < 4) {
        yp[t * 8 + 2 * lane] = d[0];
        yp[t * 8 + 2 * lane + 1] = d[1];
      }
    }
    __syncthreads();
    trace_at(a, 12);
    if (tid < nou * 8) {
      const int ol = tid / 8, r = tid % 8;
      const int n = (cta + ol * G) * 8 + r;
      auto y = [&](int j) {
        const int t = (ol * NS + j) * 2;
        return bf16_to_f32(f32_to_bf16(yp[t * 8 + r] + yp[(t + 1) * 8 + r]));
      };
      float o = bf16_to_f32(a.res[n]);
      if (S) o += y(k);
      for (int j = 0; j < k; ++j) o = fmaf(s_w[j], y(j), o);
      a.out[n] = f32_to_bf16(o);
    }
  }
  trace_at(a, 13);
}

struct DecPlan {
  DecArgs a;
  int grid, smem;
};

DecPlan make_plan(int H, int E, int k, int I, int S, int num_sms) {
  DecPlan p{};
  DecArgs &a = p.a;
  a.H = H;
  a.E = E;
  a.k = k;
  a.I = I;
  a.S = S;
  const int G = num_sms;
  a.n_su = S ? I / 8 : 0;
  a.rp_cta0 = a.n_su < G ? a.n_su : 0;
  a.rp_ctas = a.n_su < G ? G - a.n_su : G;
  a.n_ru = k * (I / 8);
  a.n_ou = H / 8;
  a.ug = 2 * (8 * (H / 2 + 16) + 2 * (H / 4));
  a.ud = 8 * (I / 2 + 16) + 2 * (I / 4);
  const int max_su = (a.n_su + G - 1) / G;
  const int max_re = (E + a.rp_ctas - 1) / a.rp_ctas;
  const int max_ru = (a.n_ru + G - 1) / G;
  const int max_ou = (a.n_ou + G - 1) / G;
  auto al = [](int v) { return (v + 127) & ~127; };
  int o = 0;
  a.off_x = o;
  o = al(o + H * 2);
  a.off_h = o;
  o = al(o + (k + S) * I * 2);
  a.off_red = o;
  o = al(o + 4096);
  a.off_keys = o;
  o = al(o + E * 4);
  a.off_p1 = o;
  o = al(o + max_su * a.ug + max_re * H * 4);
  a.off_p2 = o;
  o = al(o + max_ru * a.ug);
  a.off_p3 = o;
  o = al(o + max_ou * (k + S) * a.ud);
  p.smem = o;
  p.grid = G;
  // reduction scratch: 16 floats per warp task, 16 per (output unit, slot)
  if (max_ou * (k + S) * 16 * 4 > 4096) p.smem = -1;
  return p;
}

}  // namespace

// Dynamic shared memory the decode kernel may use on the current device: the
// per-block opt-in maximum less the kernel's static shared memory.
static int decode_smem_limit() {
  int dev = 0, optin = 0;
  cudaFuncAttributes fa;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess ||
      cudaFuncGetAttributes(&fa, decode_layer_kernel) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return optin - (int)fa.sharedSizeBytes;
}

bool decode_supported(int H, int E, int k, int I, int S, int num_sms) {
  auto pow2 = [](int v) { return v > 0 && (v & (v - 1)) == 0; };
  if (!pow2(H) || !pow2(I) || H < 128 || I < 128 || num_sms <= 0 || k > 16) return false;
  if ((size_t)E * 8 > (size_t)((k * (I / 8) + num_sms - 1) / num_sms) * (2 * (8 * (H / 2 + 16) + 2 * (H / 4))))
    return false;  // the top-k codes borrow the P2 staging area
  DecPlan p = make_plan(H, E, k, I, S, num_sms);
  return p.smem > 0 && p.smem <= decode_smem_limit();
}

cudaError_t decode_prepare(int H, int E, int k, int I, int S, int num_sms) {
  // The opt-in is per kernel and device, shared by every plan: set it to the
  // device maximum so that plans of different shapes cannot shrink it under
  // one another (decode_supported has checked this shape's need against it).
  (void)H, (void)E, (void)k, (void)I, (void)S, (void)num_sms;
  const int lim = decode_smem_limit();
  if (lim <= 0) return cudaErrorInvalidValue;
  return cudaFuncSetAttribute(decode_layer_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, lim);
}

cudaError_t launch_decode(const uint16_t *x, const uint16_t *res, int H, int E, int k, int I, int S, int prenorm,
                          float eps, const float *router, const float *bias, ExpertPtrs w, float *keys,
                          int32_t *topk_id, float *topk_w, unsigned long long *bar, uint16_t *hbuf, uint16_t *out,
                          int32_t *status, uint64_t *trace, int num_sms, int *launches, cudaStream_t s) {
  DecPlan p = make_plan(H, E, k, I, S, num_sms);
  DecArgs &a = p.a;
  a.xin = x;
  a.res = res;
  a.out = out;
  a.router = router;
  a.bias = bias;
  a.w = w;
  a.keys = keys;
  a.topk_id = topk_id;
  a.topk_w = topk_w;
  a.hbuf = hbuf;
  a.bar = bar;
  a.status = status;
  a.trace = trace;
  a.prenorm = prenorm;
  a.eps = eps;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.grid);
  cfg.blockDim = dim3(DTHREADS);
  cfg.dynamicSmemBytes = p.smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  prof_before(MOE_KERNEL_DECODE_LAYER, s);
  // the grid barrier needs every CTA resident at once: launch cooperatively or not at all
  cudaError_t e = cudaLaunchKernelEx(&cfg, decode_layer_kernel, a);
  prof_after(MOE_KERNEL_DECODE_LAYER, s);
  if (e != cudaSuccess) return e;
  *launches += 1;
  return cudaSuccess;
}

}  // namespace moe
