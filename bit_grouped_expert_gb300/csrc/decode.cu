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
//
// Weights reach shared memory through the tensor-memory accelerator as soon
// as their addresses are known -- P1 and the shared expert's down rows at
// launch, the routed experts' rows right after the top-k -- and each routed
// gate/up unit has its own mbarrier, so its GEMV starts when its bytes land
// while later units are still in flight.  Packed codes arrive in the 128-byte
// swizzled layout: for 8 rows and one K-chunk of 256 codes, [row][128 B] with
// the 16-byte pieces of row r permuted by XOR r, which makes the GEMV's
// 16-byte reads of eight rows conflict-free.
//
// The GEMVs run on mma.sync m16n8k16 with the activation vector broadcast
// over the 16 A rows and 8 weight rows as B, dequantised in registers
// (w = bf16_rne(scale * q + bias), fp32 accumulate).  The k index of the MMA
// may map onto any 16 positions of K as long as A and B agree, so lane
// (g, q) owns one whole quantisation group of row g -- 64 codes, one scale,
// one bias -- and keeps that group's 64 x values in registers across all the
// rows it visits.
//
// The grid barrier is a monotonic 64-bit arrival counter; every wait is
// bounded (MOE_ERR_DEVICE_TIMEOUT).
#include <cudaTypedefs.h>

#include "common.cuh"
#include "kernels.h"
#include "tc.h"
#include "tc_ptx.cuh"
#include "topk.cuh"

namespace moe {
namespace {

constexpr int DTHREADS = 512;
constexpr int DWARPS = DTHREADS / 32;
constexpr int KCH = 256;   // codes per K-chunk: 4 groups, 128 bytes of a code row
constexpr int XPAD = 72;   // bf16 slots per 64-value group of x / h in shared memory
constexpr int MAX_RU = 8;  // routed gate/up units (mbarriers) per CTA
constexpr unsigned long long DTIMEOUT_NS = 1000000000ull;

struct DecMaps {
  CUtensorMap gate, up, down;  // packed codes, [rows][K/2] bytes, 128B-swizzled 8-row boxes
};

struct DecArgs {
  const uint16_t *xin;  // x, or the residual stream r for pre-norm plans
  const uint16_t *res;  // residual added by the combine
  uint16_t *out;
  const float *router, *bias;
  ExpertPtrs w;
  float *keys;
  int32_t *topk_id;
  float *topk_w;
  uint16_t *hbuf;           // [k+S][I]
  unsigned long long *bar;  // monotonic arrival counter of the grid barrier
  int32_t *status;
  uint64_t *trace;  // [3][16] phase timestamps or null
  int H, E, k, I, S, prenorm;
  float eps;
  int map3d;  // 1: one TMA op per matrix (3-D map over the K-chunks), 0: one per K-chunk
  // schedule
  int n_su, rp_cta0, rp_ctas, n_ru, n_ou;
  // shared-memory layout (bytes from the 1024-aligned base)
  int off_dc, off_ru, off_su, off_rr, off_x, off_h, off_ds, off_rus, off_sus, off_red, off_keys, off_cand,
      off_gmax, off_bar, off_ys;
};

__device__ __forceinline__ unsigned long long ld_acquire64(const unsigned long long *p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

// Grid barrier on a monotonic arrival counter.  Every launch adds exactly
// two arrivals per CTA, so at launch the counter is a multiple of the grid
// size G; a CTA rounds the value it first reads down to that multiple (no CTA
// can have completed the first round before it arrives) and barrier b of the
// launch ends when the counter reaches base + b * G.  Arrival is a release
// reduction that needs no reply; the wait is bounded.
__device__ __forceinline__ void red_add_release64(unsigned long long *p, unsigned long long v) {
  asm volatile("red.release.gpu.global.add.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ bool grid_sync(unsigned long long *bar, unsigned long long target, int32_t *status) {
  __shared__ int s_ok;
  __syncthreads();
  if (threadIdx.x == 0) {
    int ok = 1;
    red_add_release64(bar, 1ull);
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

// Bounded wait for phase 0 of a one-shot mbarrier.
__device__ bool wait_bar(uint64_t *bar, int32_t *status) {
  if (ptx::mbar_try_wait(bar, 0)) return true;
  const uint64_t t0 = ptx::globaltimer();
  while (!ptx::mbar_try_wait_sleep(bar, 0, 20000)) {
    if (ptx::globaltimer() - t0 > DTIMEOUT_NS) {
      set_status(status, MOE_ERR_DEVICE_TIMEOUT);
      return false;
    }
  }
  return true;
}

__device__ __forceinline__ void expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(ptx::smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%4,%5,%5}, {%6,%7}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(b0), "r"(b1));
}

// Codes 2b and 2b+1 of a word (its byte b) as bf16_rne(s*q + bias), packed;
// w4 = w >> 4.  0x4300 | q is the bf16 value 128 + q, so one subtraction and
// one fused multiply-add (a single rounding) rebuild the weight.
__device__ __forceinline__ uint32_t dq(uint32_t w, uint32_t w4, int b, __nv_bfloat162 s2, __nv_bfloat162 b2) {
  uint32_t t = __byte_perm(w, w4, (uint32_t)(b | ((4 + b) << 8)));
  t = (t & 0x000F000Fu) | 0x43004300u;
  const __nv_bfloat162 m = *reinterpret_cast<__nv_bfloat162 *>(&t);
  const __nv_bfloat162 r = __hfma2(s2, __hsub2(m, __floats2bfloat162_rn(128.f, 128.f)), b2);
  return *reinterpret_cast<const uint32_t *>(&r);
}

// The 64 values of quantisation group `grp` (bf16 pairs) of a padded shared
// vector (XPAD slots per group).
__device__ __forceinline__ void load_group(const uint16_t *v, int grp, uint32_t (&xr)[32]) {
  const uint4 *p = reinterpret_cast<const uint4 *>(v + grp * XPAD);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint4 t = p[i];
    xr[4 * i] = t.x;
    xr[4 * i + 1] = t.y;
    xr[4 * i + 2] = t.z;
    xr[4 * i + 3] = t.w;
  }
}

// d += x . W over one K-chunk of 8 rows.  chunk: the swizzled [8][128 B] code
// image of the chunk; s, b: the rows' scales and biases ([8][gpr] bf16);
// lane (g, q) handles group grp = 4 * chunk + q of row g.  After the call
// lane q holds rows 2q (d[0]) and 2q+1 (d[1]).
__device__ __forceinline__ void gemv_chunk(const uint8_t *chunk, const uint16_t *s, const uint16_t *b, int gpr,
                                           int grp, const uint32_t (&xr)[32], int g, int q, float (&d)[4]) {
  const uint8_t *row = chunk + g * 128;
  const uint4 c0 = *reinterpret_cast<const uint4 *>(row + (((2 * q) ^ g) << 4));
  const uint4 c1 = *reinterpret_cast<const uint4 *>(row + (((2 * q + 1) ^ g) << 4));
  const __nv_bfloat162 s2 = bf16x2_splat(s[g * gpr + grp]), b2 = bf16x2_splat(b[g * gpr + grp]);
  const uint32_t wv[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
  // four accumulators: chains of four dependent MMAs instead of sixteen
  float e[4][4] = {};
#pragma unroll
  for (int i = 0; i < 8; ++i) {  // word i holds codes 8i..8i+7: MMAs 2i and 2i+1
    const uint32_t w = wv[i], w4 = w >> 4;
    mma16816(e[(2 * i) & 3], xr[4 * i], xr[4 * i + 1], dq(w, w4, 0, s2, b2), dq(w, w4, 1, s2, b2));
    mma16816(e[(2 * i + 1) & 3], xr[4 * i + 2], xr[4 * i + 3], dq(w, w4, 2, s2, b2), dq(w, w4, 3, s2, b2));
  }
#pragma unroll
  for (int r = 0; r < 4; ++r) d[r] += (e[0][r] + e[1][r]) + (e[2][r] + e[3][r]);
}

__device__ __forceinline__ int gu_ops(const DecArgs &a) { return 2 * (a.map3d ? 1 : a.H / KCH) + 4; }
__device__ __forceinline__ int dn_ops(const DecArgs &a) { return (a.map3d ? 1 : a.I / KCH) + 2; }

// Gate/up image of one unit: codes [2 matrices][H/256 chunks][8 rows][128 B]
// (8H bytes) and scales [gate_s, gate_b, up_s, up_b][8 rows][H/64] (H bytes).
// Issues copy o of the unit (code boxes of both matrices, then 4 scale rows).
__device__ void gu_op(const DecArgs &a, const DecMaps &mp, int o, uint8_t *cdst, uint8_t *sdst, int e, int r0,
                      uint64_t *bar) {
  const int H = a.H, nco = a.map3d ? 1 : H / KCH;
  const int row = e * a.I + r0;
  if (o < 2 * nco) {
    const int mat = o / nco, c = o % nco;
    uint8_t *dst = cdst + mat * 4 * H + c * 1024;
    const CUtensorMap *map = mat ? &mp.up : &mp.gate;
    if (a.map3d)
      ptx::tma_load_3d(dst, map, bar, 0, row, 0);
    else
      ptx::tma_load_2d(dst, map, bar, c * 128, row);
  } else {
    const int which = o - 2 * nco;  // 0 gate_s, 1 gate_b, 2 up_s, 3 up_b
    const uint16_t *src = which == 0 ? a.w.gate_s : which == 1 ? a.w.gate_b : which == 2 ? a.w.up_s : a.w.up_b;
    ptx::bulk_g2s(sdst + which * (H / 4), src + (size_t)row * (H / 64), H / 4, bar);
  }
}

// Down image of one (output unit, slot): codes [I/256 chunks][8 rows][128 B]
// (4I bytes) and scales [down_s, down_b][8 rows][I/64] (I/2 bytes).
__device__ void dn_op(const DecArgs &a, const DecMaps &mp, int o, uint8_t *cdst, uint8_t *sdst, int e, int n0,
                      uint64_t *bar) {
  const int I = a.I, nco = a.map3d ? 1 : I / KCH;
  const int row = e * a.H + n0;
  if (o < nco) {
    if (a.map3d)
      ptx::tma_load_3d(cdst, &mp.down, bar, 0, row, 0);
    else
      ptx::tma_load_2d(cdst + o * 1024, &mp.down, bar, o * 128, row);
  } else {
    const int which = o - nco;  // 0 down_s, 1 down_b
    ptx::bulk_g2s(sdst + which * (I / 4), (which ? a.w.down_b : a.w.down_s) + (size_t)row * (I / 64), I / 4, bar);
  }
}

// Partial gate/up dot products of `nu` unit images against x (padded, in
// shared memory) into red[(u * nkc + kc) * 16 + r] (r < 8 gate rows, 8 + r up
// rows).  Warps split the K-chunks first, then the row sets (unit, matrix);
// with `bars`, unit u is read once bars[u] completes.  Returns false on a
// timeout.
__device__ bool gu_compute(const DecArgs &a, const uint8_t *codes, const uint8_t *scales, int nu, uint64_t *bars,
                           const uint16_t *xs, float *red) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, q = lane & 3;
  const int H = a.H, nkc = H / KCH, WK = nkc < DWARPS ? nkc : DWARPS, WR = DWARPS / WK;
  const int kg = warp % WK, rg = warp / WK, gpr = H / 64;
  if (rg >= 2 * nu) return true;
  for (int kc = kg; kc < nkc; kc += WK) {
    uint32_t xr[32];
    load_group(xs, 4 * kc + q, xr);
    for (int rs = rg; rs < 2 * nu; rs += WR) {
      const int u = rs >> 1, mat = rs & 1;  // gate (0) or up (1) rows of unit u
      if (bars && !wait_bar(&bars[u], a.status)) return false;
      const uint16_t *su = reinterpret_cast<const uint16_t *>(scales + (size_t)u * H) + mat * 16 * gpr;
      float d[4] = {0.f, 0.f, 0.f, 0.f};
      gemv_chunk(codes + (size_t)u * 8 * H + mat * 4 * H + kc * 1024, su, su + 8 * gpr, gpr, 4 * kc + q, xr, g, q,
                 d);
      if (g == 0) {
        float *r = red + (u * nkc + kc) * 16 + mat * 8;
        r[2 * q] = d[0];
        r[2 * q + 1] = d[1];
      }
    }
  }
  return true;
}

// h = bf16(silu(gate) * up) of `nu` units from the partials; unit u's 8 rows
// go to hbuf from element row_of(u).
template <typename RowOf>
__device__ void gu_finish(const DecArgs &a, int nu, const float *red, RowOf row_of) {
  const int nkc = a.H / KCH;
  for (int t = threadIdx.x; t < nu * 8; t += DTHREADS) {
    const int u = t >> 3, r = t & 7;
    float gs = 0.f, us = 0.f;
    for (int kc = 0; kc < nkc; ++kc) {
      gs += red[(u * nkc + kc) * 16 + r];
      us += red[(u * nkc + kc) * 16 + 8 + r];
    }
    a.hbuf[row_of(u) + r] = f32_to_bf16(silu(gs) * us);
  }
}

// Top-k of one token by all threads of the CTA.  Codes (topk_code) order the
// keys exactly as the selection does and are distinct.  The k-th largest of
// the maxima of 16-key groups is a lower bound for the k-th largest key (k
// distinct keys reach it), so only keys at or above it can be selected; their
// rank among themselves is their slot.
__device__ void topk_block(const float *keys, int E, int k, unsigned long long *cand, unsigned long long *gmax,
                           int32_t *ids, float *w, int32_t *status) {
  __shared__ int s_n;
  const int tid = threadIdx.x, lane = tid & 31;
  const int NG = (E + 15) / 16;
  for (int base = 0; base < E; base += DTHREADS) {
    const int e = base + tid;
    unsigned long long c = e < E ? topk_code(keys[e], e) : 0ull;
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) {  // maximum over the 16 lanes of the half-warp
      const unsigned long long other = shfl_xor_u64(c, o);
      c = other > c ? other : c;
    }
    if ((tid & 15) == 0 && e < E) gmax[e >> 4] = c;
  }
  if (tid == 0) s_n = 0;
  __syncthreads();
  // every warp finds the threshold itself (NG <= 64): no block barrier
  unsigned long long tau = 0ull;
  if (NG >= k) {
    const unsigned long long m0 = lane < NG ? gmax[lane] : 0ull, m1 = lane + 32 < NG ? gmax[lane + 32] : 0ull;
    int r0 = 0, r1 = 0;
#pragma unroll 4
    for (int j = 0; j < NG; ++j) {
      const unsigned long long gj = gmax[j];
      r0 += gj > m0;
      r1 += gj > m1;
    }
    unsigned long long t = (lane < NG && r0 == k - 1) ? m0 : ((lane + 32 < NG && r1 == k - 1) ? m1 : 0ull);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const unsigned long long other = shfl_xor_u64(t, o);
      t = other > t ? other : t;
    }
    tau = t;
  }
  for (int base = 0; base < E; base += DTHREADS) {
    const int e = base + tid;
    const unsigned long long c = e < E ? topk_code(keys[e], e) : 0ull;
    const bool take = e < E && c >= tau;
    const unsigned m = __ballot_sync(0xffffffffu, take);
    int pos = 0;
    if (lane == 0 && m) pos = atomicAdd(&s_n, __popc(m));
    pos = __shfl_sync(0xffffffffu, pos, 0);
    if (take) cand[pos + __popc(m & ((1u << lane) - 1u))] = c;
  }
  __syncthreads();
  const int n = s_n;
  for (int t = tid; t < n; t += DTHREADS) {
    const unsigned long long c = cand[t];
    int rank = 0;
    for (int j = 0; j < n; ++j) rank += cand[j] > c;
    if (rank < k) ids[rank] = topk_code_expert(c);
  }
  __syncthreads();
  if (tid < 32) {
    const int my_id = lane < k ? ids[lane] : -1;
    const float my_key = lane < k ? keys[my_id] : 0.f;
    topk_finish(lane, k, my_id, my_key, ids, w, nullptr, status);
  }
}

// Phase timestamp for the trace of CTAs 0, G/2 and G-1 (thread 0).
__device__ __forceinline__ void trace_at(const DecArgs &a, int slot) {
  if (!a.trace || threadIdx.x != 0) return;
  const int c = blockIdx.x, G = gridDim.x;
  const int row = c == 0 ? 0 : (c == G / 2 ? 1 : (c == G - 1 ? 2 : -1));
  if (row >= 0) a.trace[row * 16 + slot] = ptx::globaltimer();
}

__global__ void __launch_bounds__(DTHREADS, 1) decode_layer_kernel(const __grid_constant__ DecMaps mp,
                                                                   const DecArgs a) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ int s_ids[16];
  __shared__ float s_w[16];
  __shared__ float s_part[DWARPS];
  // 1024-byte aligned base for the swizzled code images (keeps the shared space)
  uint8_t *sm = smem_raw + ((1024u - (ptx::smem_u32(smem_raw) & 1023u)) & 1023u);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int cta = blockIdx.x, G = gridDim.x;
  const int H = a.H, I = a.I, E = a.E, k = a.k, S = a.S, NS = k + S;
  uint8_t *dc = sm + a.off_dc, *ru = sm + a.off_ru, *su = sm + a.off_su, *ds = sm + a.off_ds,
          *rus = sm + a.off_rus, *sus = sm + a.off_sus;
  float *rr = reinterpret_cast<float *>(sm + a.off_rr);
  uint16_t *xs = reinterpret_cast<uint16_t *>(sm + a.off_x);
  uint16_t *hs = reinterpret_cast<uint16_t *>(sm + a.off_h);
  float *red = reinterpret_cast<float *>(sm + a.off_red);
  float *keys = reinterpret_cast<float *>(sm + a.off_keys);
  uint64_t *bars = reinterpret_cast<uint64_t *>(sm + a.off_bar);
  uint64_t *bar_p1 = bars, *bar_dsh = bars + 1, *bar_drt = bars + 2, *bar_ru = bars + 3;
  const int nsu = (cta < a.n_su) ? (a.n_su - 1 - cta) / G + 1 : 0;  // shared gate/up units of this CTA
  const int rc = cta - a.rp_cta0;                                    // index among the router CTAs
  const int nre = (rc >= 0 && rc < a.rp_ctas && rc < E) ? (E - 1 - rc) / a.rp_ctas + 1 : 0;  // router rows
  const int nru = (cta < a.n_ru) ? (a.n_ru - 1 - cta) / G + 1 : 0;  // routed gate/up units
  const int nou = (cta < a.n_ou) ? (a.n_ou - 1 - cta) / G + 1 : 0;  // output units
  const int upr = I / 8;
  trace_at(a, 0);

  if (tid == 0) {
    for (int i = 0; i < 3 + MAX_RU; ++i) ptx::mbar_init(&bars[i], 1);
    ptx::fence_mbar_init();
    if (a.map3d) {
      ptx::prefetch_tmap(&mp.gate);
      ptx::prefetch_tmap(&mp.up);
      ptx::prefetch_tmap(&mp.down);
    }
    expect_tx(bar_p1, (uint32_t)(nsu * 9 * H + nre * 4 * H));
    expect_tx(bar_dsh, S ? (uint32_t)(nou * (4 * I + I / 2)) : 0u);
  }
  __syncthreads();

  // ---------------------------------------------------------------- copies known at launch
  // (issued by the first two lanes of every warp: one warp alone issues slowly)
  const int issuer = lane < 2 ? warp * 2 + lane : -1;
  if (issuer >= 0) {
    const int ngu = gu_ops(a), ndn = dn_ops(a);
    const int n1 = nsu * ngu, n2 = n1 + nre, n3 = n2 + (S ? nou * ndn : 0);
    for (int o = issuer; o < n3; o += 2 * DWARPS) {
      if (o < n1) {
        const int i = o / ngu;
        gu_op(a, mp, o % ngu, su + i * 8 * H, sus + i * H, E, (cta + i * G) * 8, bar_p1);
      } else if (o < n2) {
        const int i = o - n1;
        ptx::bulk_g2s(rr + i * H, a.router + (size_t)(rc + i * a.rp_ctas) * H, 4 * H, bar_p1);
      } else {
        const int ol = (o - n2) / ndn;
        dn_op(a, mp, (o - n2) % ndn, dc + (ol * NS + k) * 4 * I, ds + (ol * NS + k) * (I / 2), E,
              (cta + ol * G) * 8, bar_dsh);
      }
    }
  }
  trace_at(a, 1);

  // ---------------------------------------------------------------- P0: x (padded groups)
  // The input (and the workspace) may still be written by the previous layer's
  // launch when this one starts early: wait for it here, after the weight
  // copies are on their way.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  __shared__ unsigned long long s_base;
  if (tid == 0) {  // a relaxed read: only the value matters, not ordering
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(a.bar) : "memory");
    s_base = v / (unsigned long long)G * (unsigned long long)G;
  }
  // the residual of this CTA's output rows, read now rather than at the end
  float res_v = 0.f;
  if (tid < nou * 8) res_v = bf16_to_f32(a.res[(cta + (tid >> 3) * G) * 8 + (tid & 7)]);
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
    for (int i = tid; i < H; i += DTHREADS)
      xs[(i >> 6) * XPAD + (i & 63)] = f32_to_bf16(bf16_to_f32(a.xin[i]) * scale);
  } else {
    for (int i = tid; i < H / 8; i += DTHREADS)
      *reinterpret_cast<uint4 *>(xs + (i >> 3) * XPAD + (i & 7) * 8) = reinterpret_cast<const uint4 *>(a.xin)[i];
  }
  __syncthreads();
  trace_at(a, 2);

  // ---------------------------------------------------------------- P1: shared gate/up, router rows
  bool ok = wait_bar(bar_p1, a.status);
  trace_at(a, 3);
  if (ok && nsu > 0) ok = gu_compute(a, su, sus, nsu, nullptr, xs, red);
  if (ok)
    for (int i = warp; i < nre; i += DWARPS) {  // one warp per router row, fp32 FMA
      const float *row = rr + i * H;
      float acc = 0.f;
      for (int kk = 4 * lane; kk < H; kk += 128) {
        const float4 wv = *reinterpret_cast<const float4 *>(row + kk);
        const uint2 xv = *reinterpret_cast<const uint2 *>(xs + (kk >> 6) * XPAD + (kk & 63));
        acc = fmaf(__uint_as_float(xv.x << 16), wv.x, acc);
        acc = fmaf(__uint_as_float(xv.x & 0xFFFF0000u), wv.y, acc);
        acc = fmaf(__uint_as_float(xv.y << 16), wv.z, acc);
        acc = fmaf(__uint_as_float(xv.y & 0xFFFF0000u), wv.w, acc);
      }
      acc = warp_sum(acc);
      const int e = rc + i * a.rp_ctas;
      if (lane == 0) a.keys[e] = a.bias ? acc + a.bias[e] : acc;
    }
  ok = __syncthreads_and(ok) != 0;  // every flag below stays uniform across the CTA
  if (ok && nsu > 0) gu_finish(a, nsu, red, [&](int u) { return (size_t)k * I + (size_t)(cta + u * G) * 8; });
  trace_at(a, 4);
  ok = grid_sync(a.bar, s_base + (unsigned long long)G, a.status) && ok;
  trace_at(a, 5);

  // ---------------------------------------------------------------- P2: routing, routed gate/up
  bool issued2 = false;
  if (ok) {
    for (int e = tid; e < E; e += DTHREADS) keys[e] = __ldcg(a.keys + e);
    __syncthreads();
    trace_at(a, 6);
    topk_block(keys, E, k, reinterpret_cast<unsigned long long *>(sm + a.off_cand),
               reinterpret_cast<unsigned long long *>(sm + a.off_gmax), s_ids, s_w, a.status);
    __syncthreads();
    trace_at(a, 14);
    if (cta == 0 && tid < k) {
      a.topk_id[tid] = s_ids[tid];
      a.topk_w[tid] = s_w[tid];
    }
    if (tid == 0) {
      for (int i = 0; i < nru; ++i) expect_tx(&bar_ru[i], (uint32_t)(9 * H));
      expect_tx(bar_drt, (uint32_t)(nou * k * (4 * I + I / 2)));
    }
    __syncthreads();
    if (issuer >= 0) {
      const int ngu = gu_ops(a), ndn = dn_ops(a);
      const int n1 = nru * ngu, n2 = n1 + nou * k * ndn;
      for (int o = issuer; o < n2; o += 2 * DWARPS) {
        if (o < n1) {
          const int i = o / ngu, u = cta + i * G;
          gu_op(a, mp, o % ngu, ru + i * 8 * H, rus + i * H, s_ids[u / upr], (u % upr) * 8, &bar_ru[i]);
        } else {
          const int b = (o - n1) / ndn, ol = b / k, j = b % k;
          dn_op(a, mp, (o - n1) % ndn, dc + (ol * NS + j) * 4 * I, ds + (ol * NS + j) * (I / 2), s_ids[j],
                (cta + ol * G) * 8, bar_drt);
        }
      }
    }
    issued2 = true;
    trace_at(a, 7);
    const bool ok2 = __syncthreads_and(gu_compute(a, ru, rus, nru, bar_ru, xs, red)) != 0;
    trace_at(a, 8);
    if (ok2 && nru > 0)
      gu_finish(a, nru, red, [&](int u) {
        const int uu = cta + u * G;
        return (size_t)(uu / upr) * I + (size_t)(uu % upr) * 8;
      });
    ok = ok && ok2;
  }
  trace_at(a, 9);
  ok = grid_sync(a.bar, s_base + 2ull * (unsigned long long)G, a.status) && ok;
  trace_at(a, 10);

  // ---------------------------------------------------------------- P3: down + combine
  // let the next launch in the stream start its prologue and weight copies
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (ok) ok = __syncthreads_and(wait_bar(bar_dsh, a.status) && wait_bar(bar_drt, a.status)) != 0;
  if (ok) {
    const int nv = NS * I / 8;  // h of every slot, 16 bytes per load, into padded groups
    for (int i = tid; i < nv; i += DTHREADS) {
      const int j = i / (I / 8), c8 = i % (I / 8);
      *reinterpret_cast<uint4 *>(hs + (j * (I / 64) + (c8 >> 3)) * XPAD + (c8 & 7) * 8) =
          __ldcg(reinterpret_cast<const uint4 *>(a.hbuf) + i);
    }
    __syncthreads();
    trace_at(a, 11);
    const int nkcd = I / KCH, gpr = I / 64, g = lane >> 2, q = lane & 3;
    const int nitem = nou * NS * nkcd;
    for (int t = warp; t < nitem; t += DWARPS) {
      const int kc = t % nkcd, j = (t / nkcd) % NS, ol = t / (nkcd * NS);
      uint32_t xr[32];
      load_group(hs + j * (I / 64) * XPAD, 4 * kc + q, xr);
      const uint16_t *sc = reinterpret_cast<const uint16_t *>(ds + (ol * NS + j) * (I / 2));
      float d[4] = {0.f, 0.f, 0.f, 0.f};
      gemv_chunk(dc + (ol * NS + j) * 4 * I + kc * 1024, sc, sc + 8 * gpr, gpr, 4 * kc + q, xr, g, q, d);
      if (g == 0) {
        red[t * 8 + 2 * q] = d[0];
        red[t * 8 + 2 * q + 1] = d[1];
      }
    }
    __syncthreads();
    trace_at(a, 12);
    // y_j = bf16(h_j . Wd_j) of every (row, slot) in parallel, then the combine
    float *ys = reinterpret_cast<float *>(sm + a.off_ys);  // [nou * 8][NS]
    for (int t = tid; t < nou * 8 * NS; t += DTHREADS) {
      const int ol = t / (8 * NS), r = (t / NS) & 7, j = t % NS;
      float v = 0.f;
      for (int kc = 0; kc < nkcd; ++kc) v += red[((ol * NS + j) * nkcd + kc) * 8 + r];
      ys[t] = bf16_to_f32(f32_to_bf16(v));
    }
    __syncthreads();
    if (tid < nou * 8) {
      const float *yr = ys + tid * NS;
      float o = res_v;
      if (S) o += yr[k];
      for (int j = 0; j < k; ++j) o = fmaf(s_w[j], yr[j], o);
      a.out[(cta + (tid >> 3) * G) * 8 + (tid & 7)] = f32_to_bf16(o);
    }
  }
  // never leave with copies in flight into this CTA's shared memory
  if (tid == 0 && !ok) {
    wait_bar(bar_p1, a.status);
    wait_bar(bar_dsh, a.status);
    if (issued2) {
      wait_bar(bar_drt, a.status);
      for (int i = 0; i < nru; ++i) wait_bar(&bar_ru[i], a.status);
    }
  }
  trace_at(a, 13);
}

struct DecPlan {
  DecArgs a;
  int grid, smem, max_ru;
};

DecPlan make_plan(int H, int E, int k, int I, int S, int num_sms) {
  DecPlan p{};
  DecArgs &a = p.a;
  a.H = H;
  a.E = E;
  a.k = k;
  a.I = I;
  a.S = S;
  const int G = num_sms, NS = k + S;
  a.n_su = S ? I / 8 : 0;
  a.rp_cta0 = a.n_su < G ? a.n_su : 0;
  a.rp_ctas = a.n_su < G ? G - a.n_su : G;
  a.n_ru = k * (I / 8);
  a.n_ou = H / 8;
  const int max_su = (a.n_su + G - 1) / G;
  const int max_re = (E + a.rp_ctas - 1) / a.rp_ctas;
  const int max_ru = (a.n_ru + G - 1) / G;
  const int max_ou = (a.n_ou + G - 1) / G;
  const int nkc = H / KCH, nkcd = I / KCH;
  auto al = [](int v, int m) { return (v + m - 1) / m * m; };
  int o = 0;
  a.off_dc = o;
  o = al(o + max_ou * NS * 4 * I, 1024);
  a.off_ru = o;
  o = al(o + max_ru * 8 * H, 1024);
  a.off_su = o;
  o = al(o + max_su * 8 * H, 1024);
  a.off_rr = o;
  o = al(o + max_re * 4 * H, 128);
  a.off_x = o;
  o = al(o + (H / 64) * XPAD * 2, 128);
  a.off_h = o;
  o = al(o + NS * (I / 64) * XPAD * 2, 128);
  a.off_ds = o;
  o = al(o + max_ou * NS * (I / 2), 128);
  a.off_rus = o;
  o = al(o + max_ru * H, 128);
  a.off_sus = o;
  o = al(o + max_su * H, 128);
  a.off_red = o;
  const int red_gu = (max_ru > max_su ? max_ru : max_su) * nkc * 16 * 4;
  const int red_dn = max_ou * NS * nkcd * 8 * 4;
  o = al(o + (red_gu > red_dn ? red_gu : red_dn), 128);
  a.off_keys = o;
  o = al(o + E * 4, 128);
  a.off_cand = o;
  o = al(o + E * 8, 128);
  a.off_gmax = o;
  o = al(o + ((E + 15) / 16) * 8, 128);
  a.off_bar = o;
  o = al(o + (3 + MAX_RU) * 8, 128);
  a.off_ys = o;
  o = al(o + max_ou * 8 * NS * 4, 128);
  p.smem = o + 1024;  // slack for aligning the base
  p.grid = G;
  p.max_ru = max_ru;
  return p;
}

// Dynamic shared memory the decode kernel may use on the current device: the
// per-block opt-in maximum less the kernel's static shared memory.
int decode_smem_limit() {
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

// Codes as bytes [rows][K/2]: either one 3-D box per 8 rows (dims 128 B x
// rows x K/256 chunks, the chunk stride 128 B) or 2-D boxes of 8 rows x 128 B
// taken one K-chunk at a time.  Both land as [chunk][row][128 B], swizzled.
cudaError_t codes_map(CUtensorMap *m, const uint32_t *codes, int rows, int K, bool three_d) {
  auto enc = tensor_map_encoder();
  if (!enc) return cudaErrorInitializationError;
  CUresult r;
  if (three_d) {
    cuuint64_t dims[3] = {128, (cuuint64_t)rows, (cuuint64_t)(K / KCH)};
    cuuint64_t strides[2] = {(cuuint64_t)(K / 2), 128};
    cuuint32_t box[3] = {128, 8, (cuuint32_t)(K / KCH)};
    cuuint32_t estr[3] = {1, 1, 1};
    r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint32_t *>(codes), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  } else {
    cuuint64_t dims[2] = {(cuuint64_t)(K / 2), (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)(K / 2)};
    cuuint32_t box[2] = {128, 8};
    cuuint32_t estr[2] = {1, 1};
    r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint32_t *>(codes), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  }
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t make_maps(DecMaps *m, const ExpertPtrs &w, int H, int E, int I, int S, bool three_d) {
  const int E_tot = E + S;
  cudaError_t e = codes_map(&m->gate, w.gate_q, E_tot * I, H, three_d);
  if (e == cudaSuccess) e = codes_map(&m->up, w.up_q, E_tot * I, H, three_d);
  if (e == cudaSuccess) e = codes_map(&m->down, w.down_q, E_tot * H, I, three_d);
  return e;
}

}  // namespace

bool decode_supported(int H, int E, int k, int I, int S, int num_sms) {
  auto pow2 = [](int v) { return v > 0 && (v & (v - 1)) == 0; };
  if (!pow2(H) || !pow2(I) || H < KCH || I < KCH || num_sms <= 0 || k > 16 || E > 1024) return false;
  DecPlan p = make_plan(H, E, k, I, S, num_sms);
  return p.max_ru <= MAX_RU && p.smem <= decode_smem_limit();
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
  DecMaps maps;
  a.map3d = 1;
  cudaError_t e = make_maps(&maps, w, H, E, I, S, true);
  if (e != cudaSuccess) {  // the driver refused the 3-D view: one 2-D box per K-chunk
    a.map3d = 0;
    if ((e = make_maps(&maps, w, H, E, I, S, false)) != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.grid);
  cfg.blockDim = dim3(DTHREADS);
  cfg.dynamicSmemBytes = p.smem;
  cfg.stream = s;
  // The grid barrier needs every CTA resident at once: launch cooperatively
  // or not at all.  Programmatic serialisation lets the launch begin while
  // the previous kernel in the stream drains (the kernel waits for it before
  // it reads its input); drivers that refuse the pair get a plain cooperative
  // launch.
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  prof_before(MOE_KERNEL_DECODE_LAYER, s);
  e = cudaLaunchKernelEx(&cfg, decode_layer_kernel, maps, a);
  if (e != cudaSuccess) {
    cudaGetLastError();
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, decode_layer_kernel, maps, a);
  }
  prof_after(MOE_KERNEL_DECODE_LAYER, s);
  if (e != cudaSuccess) return e;
  *launches += 1;
  return cudaSuccess;
}

}  // namespace moe
