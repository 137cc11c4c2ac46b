// Gated DeltaNet scan with the recurrent state held in registers.
//
// Recurrence (gated delta rule, per value head h and token t, state S[dk][dv]):
//   S_t = alpha_t (I - beta_t k_t k_t^T) S_{t-1} + beta_t k_t v_t^T,  o_t = S_t^T q_t
// taken per token as: u = S^T k (what the state holds for k), delta =
// beta (v - alpha u), S = alpha S + k delta^T, o = S^T q.
//
// Work split: one CTA per (value head, 32 value columns), 512 threads.  Thread
// (column c, row part r of 16) keeps S[8 r .. 8 r + 7][c] in 8 registers for
// the whole sequence; the sixteen parts of a column are neighbouring lanes, so
// the column sums u and o take four xor-shuffles.  (Four warps per scheduler
// give it independent work while each token's chain waits; with eight row
// parts the scan took 7 % longer.)  Per token the CTA needs
// k_t and q_t of its key head, its 32 values of v_t, alpha_t and beta_t (600
// bytes).  Tokens move in blocks of GDN_BLK: cp.async brings block j+2 into a
// ring of three raw blocks in shared memory while the threads that copied
// block j+1 convert it to fp32 in a double buffer and every thread runs the
// tokens of block j from the other buffer.  One block barrier per block, not
// per token, so a thread goes from token to token with only its own warp's
// shuffles in between.  State traffic is one read and one write per sequence.
#include <cuda_bf16.h>

#include "common.cuh"
#include "gdn.h"
#include "kernels.h"

namespace moe {
namespace {

constexpr int GDN_DK = 128;
constexpr int GDN_COLS = 32;                // value columns per CTA
constexpr int GDN_RQ = 16;                  // row parts per column
constexpr int GDN_ROWS = GDN_DK / GDN_RQ;   // state rows per thread
constexpr int GDN_THREADS = GDN_COLS * GDN_RQ;
constexpr int GDN_BLK = 8;                  // tokens per block
constexpr int GDN_RAWB = 3;                 // raw blocks in the ring
constexpr int GDN_KPAD = GDN_ROWS + 4;      // fp32 row-part stride: the parts' 16-byte reads on distinct banks
// one token's raw bytes in the ring: k (256 B), q (256 B), v (64 B), alpha, beta
constexpr int RAW_K = 0, RAW_Q = 256, RAW_V = 512, RAW_A = 576, RAW_B = 580, RAW_BYTES = 592;

struct GdnArgs {
  const uint16_t *q, *k, *v;
  const float *alpha, *beta;
  float *state;
  uint16_t *o;
  int T, Hk, Hv, dv;
};

__device__ __forceinline__ void cp_async16(void *dst, const void *src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
               "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async4(void *dst, const void *src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
               "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__global__ void __launch_bounds__(GDN_THREADS) gdn_scan_kernel(const __grid_constant__ GdnArgs a) {
  __shared__ __align__(16) uint8_t raw[GDN_RAWB * GDN_BLK][RAW_BYTES];
  __shared__ __align__(16) float kf[2][GDN_BLK][GDN_RQ * GDN_KPAD], qf[2][GDN_BLK][GDN_RQ * GDN_KPAD];
  __shared__ float vf[2][GDN_BLK][GDN_COLS], ab[2][GDN_BLK][2];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int h = blockIdx.x, cb = blockIdx.y, kh = h / (a.Hv / a.Hk);
  constexpr int CPW = 32 / GDN_RQ;  // columns per warp
  const int r = lane % GDN_RQ, cl = warp * CPW + lane / GDN_RQ, c = cb * GDN_COLS + cl;
  const int T = a.T, nblk = (T + GDN_BLK - 1) / GDN_BLK;
  // copy jobs: (token tt of a block, piece p), 16-byte pieces 0-15 k, 16-31
  // q, 32-35 v; 36 alpha, 37 beta.  A thread converts the pieces it copied.
  constexpr int PIECES = 38, JOBS = PIECES * GDN_BLK;
  auto issue = [&](int j) {  // block j into raw block j % GDN_RAWB
    for (int job = tid; job < JOBS; job += GDN_THREADS) {
      const int tt = job / PIECES, p = job % PIECES, t = j * GDN_BLK + tt;
      if (j >= nblk || t >= T) break;
      uint8_t *slot = raw[(j % GDN_RAWB) * GDN_BLK + tt];
      if (p < 16)
        cp_async16(slot + RAW_K + p * 16, a.k + ((size_t)t * a.Hk + kh) * GDN_DK + p * 8);
      else if (p < 32)
        cp_async16(slot + RAW_Q + (p - 16) * 16, a.q + ((size_t)t * a.Hk + kh) * GDN_DK + (p - 16) * 8);
      else if (p < 36)
        cp_async16(slot + RAW_V + (p - 32) * 16, a.v + ((size_t)t * a.Hv + h) * a.dv + cb * GDN_COLS + (p - 32) * 8);
      else if (p == 36)
        cp_async4(slot + RAW_A, a.alpha + (size_t)t * a.Hv + h);
      else
        cp_async4(slot + RAW_B, a.beta + (size_t)t * a.Hv + h);
    }
    cp_async_commit();  // one group per block, empty past the end
  };
  auto convert = [&](int j) {  // this thread's pieces of block j, to fp32 buffer j & 1
    const int b = j & 1;
    for (int job = tid; job < JOBS; job += GDN_THREADS) {
      const int tt = job / PIECES, p = job % PIECES, t = j * GDN_BLK + tt;
      if (j >= nblk || t >= T) break;
      const uint8_t *slot = raw[(j % GDN_RAWB) * GDN_BLK + tt];
      if (p < 36) {
        const uint4 w = *reinterpret_cast<const uint4 *>(slot + (p < 16 ? RAW_K + p * 16
                                                                 : p < 32 ? RAW_Q + (p - 16) * 16
                                                                          : RAW_V + (p - 32) * 16));
        const uint32_t pw[4] = {w.x, w.y, w.z, w.w};
        float f[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          f[2 * i] = __uint_as_float(pw[i] << 16);
          f[2 * i + 1] = __uint_as_float(pw[i] & 0xFFFF0000u);
        }
        float *dst;
        if (p < 32) {
          const int e = (p & 15) * 8;  // element of k or q; 8 consecutive stay in one row part
          dst = (p < 16 ? kf[b][tt] : qf[b][tt]) + (e / GDN_ROWS) * GDN_KPAD + e % GDN_ROWS;
        } else {
          dst = vf[b][tt] + (p - 32) * 8;
        }
        *reinterpret_cast<float4 *>(dst) = make_float4(f[0], f[1], f[2], f[3]);
        *reinterpret_cast<float4 *>(dst + 4) = make_float4(f[4], f[5], f[6], f[7]);
      } else {
        ab[b][tt][p - 36] = *reinterpret_cast<const float *>(slot + (p == 36 ? RAW_A : RAW_B));
      }
    }
  };

  float S[GDN_ROWS];
  float *st = a.state + ((size_t)h * GDN_DK + r * GDN_ROWS) * a.dv + c;
#pragma unroll
  for (int i = 0; i < GDN_ROWS; ++i) S[i] = st[(size_t)i * a.dv];

  issue(0);
  issue(1);
  cp_async_wait<1>();  // block 0
  convert(0);
  issue(2);
  __syncthreads();

  for (int j = 0; j < nblk; ++j) {
    cp_async_wait<1>();  // block j+1 has landed (block j+2 may still be in flight)
    convert(j + 1);
    const int b = j & 1, n = min(GDN_BLK, T - j * GDN_BLK);
    // each token's output partial; the column sums wait for the block's end,
    // off the chain from one token's state to the next
    float op[GDN_BLK] = {};
#pragma unroll
    for (int tt2 = 0; tt2 < GDN_BLK; ++tt2) {
      if (tt2 >= n) break;
      const float *kb = kf[b][tt2] + r * GDN_KPAD, *qb = qf[b][tt2] + r * GDN_KPAD;
      const float al = ab[b][tt2][0], be = ab[b][tt2][1];
      float u4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int i = 0; i < GDN_ROWS; i += 4) {
        const float4 kv = *reinterpret_cast<const float4 *>(kb + i);
        u4[0] = fmaf(S[i], kv.x, u4[0]);
        u4[1] = fmaf(S[i + 1], kv.y, u4[1]);
        u4[2] = fmaf(S[i + 2], kv.z, u4[2]);
        u4[3] = fmaf(S[i + 3], kv.w, u4[3]);
      }
      float u = (u4[0] + u4[1]) + (u4[2] + u4[3]);
#pragma unroll
      for (int m = 1; m < GDN_RQ; m <<= 1) u += __shfl_xor_sync(0xffffffffu, u, m);
      const float d = be * (vf[b][tt2][cl] - al * u);
      float o4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int i = 0; i < GDN_ROWS; i += 4) {
        const float4 kv = *reinterpret_cast<const float4 *>(kb + i);
        const float4 qv = *reinterpret_cast<const float4 *>(qb + i);
        S[i] = fmaf(al, S[i], kv.x * d);
        S[i + 1] = fmaf(al, S[i + 1], kv.y * d);
        S[i + 2] = fmaf(al, S[i + 2], kv.z * d);
        S[i + 3] = fmaf(al, S[i + 3], kv.w * d);
        o4[0] = fmaf(S[i], qv.x, o4[0]);
        o4[1] = fmaf(S[i + 1], qv.y, o4[1]);
        o4[2] = fmaf(S[i + 2], qv.z, o4[2]);
        o4[3] = fmaf(S[i + 3], qv.w, o4[3]);
      }
      op[tt2] = (o4[0] + o4[1]) + (o4[2] + o4[3]);
    }
#pragma unroll
    for (int m = 1; m < GDN_RQ; m <<= 1)
#pragma unroll
      for (int tt2 = 0; tt2 < GDN_BLK; ++tt2) op[tt2] += __shfl_xor_sync(0xffffffffu, op[tt2], m);
    if (r == 0)
#pragma unroll
      for (int tt2 = 0; tt2 < GDN_BLK; ++tt2)
        if (tt2 < n) a.o[((size_t)(j * GDN_BLK + tt2) * a.Hv + h) * a.dv + c] = f32_to_bf16(op[tt2]);
    __syncthreads();  // buffer j & 1 and raw block j are free; buffer (j + 1) & 1 is published
    issue(j + 3);     // into raw block j's slots
  }
  cp_async_wait<0>();
#pragma unroll
  for (int i = 0; i < GDN_ROWS; ++i) st[(size_t)i * a.dv] = S[i];
}

bool overlaps(const void *p, size_t np, const void *q, size_t nq) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(p), b = reinterpret_cast<uintptr_t>(q);
  return np && nq && a < b + nq && b < a + np;
}

}  // namespace
}  // namespace moe

extern "C" moe_status gdn_scan(const void *q_d, const void *k_d, const void *v_d, const float *alpha_d,
                               const float *beta_d, float *state_d, void *o_d, int T, int Hk, int Hv, int dk, int dv,
                               void *stream) {
  using moe::aligned16;
  if (T < 0 || Hk < 1 || Hv < 1 || Hv % Hk) return MOE_ERR_INVALID_ARGUMENT;
  if (dk != moe::GDN_DK || dv <= 0 || dv % moe::GDN_COLS) return MOE_ERR_UNSUPPORTED;
  if (T == 0) return MOE_OK;
  if (!q_d || !k_d || !v_d || !alpha_d || !beta_d || !state_d || !o_d) return MOE_ERR_INVALID_ARGUMENT;
  if (!aligned16(q_d) || !aligned16(k_d) || !aligned16(v_d) || !aligned16(alpha_d) || !aligned16(beta_d) ||
      !aligned16(state_d) || !aligned16(o_d))
    return MOE_ERR_MISALIGNED;
  const size_t nqk = (size_t)T * Hk * dk * 2, nv = (size_t)T * Hv * dv * 2, nab = (size_t)T * Hv * 4,
               ns = (size_t)Hv * dk * dv * 4, no = nv;
  if (moe::overlaps(o_d, no, q_d, nqk) || moe::overlaps(o_d, no, k_d, nqk) || moe::overlaps(o_d, no, v_d, nv) ||
      moe::overlaps(o_d, no, alpha_d, nab) || moe::overlaps(o_d, no, beta_d, nab) ||
      moe::overlaps(o_d, no, state_d, ns))
    return MOE_ERR_INVALID_ARGUMENT;
  moe::GdnArgs a;
  a.q = static_cast<const uint16_t *>(q_d);
  a.k = static_cast<const uint16_t *>(k_d);
  a.v = static_cast<const uint16_t *>(v_d);
  a.alpha = alpha_d;
  a.beta = beta_d;
  a.state = state_d;
  a.o = static_cast<uint16_t *>(o_d);
  a.T = T;
  a.Hk = Hk;
  a.Hv = Hv;
  a.dv = dv;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  moe::prof_before(MOE_KERNEL_GDN_SCAN, s);
  moe::gdn_scan_kernel<<<dim3(Hv, dv / moe::GDN_COLS), moe::GDN_THREADS, 0, s>>>(a);
  moe::prof_after(MOE_KERNEL_GDN_SCAN, s);
  return moe::note_cuda_error(cudaGetLastError());
}
