// T == 1 decode path ("Decode" section of the Lily pages: a single token uses
// each weight it reads once, so HBM bandwidth bounds the step; only the
// selected experts' bytes are read, and the work of a step is overlapped
// rather than issued as a long chain of small launches).
//
// One cooperative launch runs up to MAXL layers; for each layer every CTA
// (one per SM) runs
//   P0  x = bf16(r / sqrt(mean(r^2) + eps)) (pre-norm plans) or x = input,
//       computed redundantly into shared memory
//   P1  router keys (fp32, one warp per expert row) or, on the CTAs without
//       router rows, the shared expert's gate/up rows (h = bf16(silu(g) * u))
//   P2  top-k over the keys (every CTA, same order, same result); the routed
//       experts' gate/up rows
//   P3  the down rows of every slot for this CTA's output rows, y_j =
//       bf16(h_j . Wd_j), out = bf16(res + y_shared + sum_j w_j * y_j)
// The keys, h and the next layer's residual cross CTAs as epoch-tagged words
// (see ld_relaxed64): a CTA waits for exactly the values it reads, with no
// grid barrier.
//
// Weights reach shared memory through the tensor-memory accelerator as soon
// as their addresses are known -- the next layer's router rows, shared rows
// and shared down rows during this layer, the routed experts' rows right
// after the top-k -- and each routed gate/up unit has its own mbarrier, so
// its GEMV starts when its bytes land while later units are still in flight.
// Packed codes arrive in the 128-byte swizzled layout: for 8 rows and one
// K-chunk of 256 codes, [row][128 B] with the 16-byte pieces of row r
// permuted by XOR r, which makes the GEMV's 16-byte reads of eight rows
// conflict-free.
//
// The GEMVs run on mma.sync m16n8k16 with the weights as the A operand,
// dequantised in registers (w = bf16_rne(scale * q + bias), fp32
// accumulate) and the activation vector in B's first two columns.  The k
// index of the MMA may map onto any 16 positions of K as long as A and B
// agree, so lane (g, q) owns one whole quantisation group of row g -- 64
// codes, one scale, one bias -- and the vector is kept in shared memory in
// the order in which the codes unpack (see perm8).
//
// Every wait is bounded (MOE_ERR_DEVICE_TIMEOUT).
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
constexpr int MAXL = 7;    // layers per launch (the parameters stay under 4 KB)
constexpr int DN_ITEMS = 4;  // down items (output unit, slot, K-chunk) per warp at most
constexpr int XREG = 4;    // uint2 of r a thread holds in the RMSNorm: H <= 4 * XREG * DTHREADS

struct DecMaps {
  CUtensorMap gate, up, down;  // packed codes, [rows][K/2] bytes, 128B-swizzled 8-row boxes
};

// One layer's weights: router fp32 [E][H], logit bias [E] or null, experts.
struct LayerW {
  const float *router, *bias;
  ExpertPtrs w;
};

struct DecArgs {
  DecMaps maps[MAXL];   // per layer (the tensor maps must live in the parameters)
  LayerW lw[MAXL];
  int nl;               // layers of this launch
  const uint16_t *xin;  // x, or the residual stream r for pre-norm plans (layers > 0: r)
  const uint16_t *res;  // residual added by the first layer's combine (later layers: r)
  uint16_t *out;        // output (stacks: r, updated in place layer by layer)
  float *keys;
  int32_t *topk_id;
  float *topk_w;
  // tagged exchange buffers (see ld_relaxed64) and the epoch counter
  unsigned long long *tkeys;  // [2][key_words(E)] fp32 router keys, then the shared-expert gate's x . gate
  unsigned long long *th;     // [2][(k+S)*I/2]   h, bf16 pairs
  unsigned long long *tr;     // [2][H/2]         residual stream between layers, bf16 pairs
  unsigned long long *epoch;  // epochs used so far (low 32 bits)
  int32_t *status;
  uint64_t *trace;  // [MOE_TRACE_CTAS][MOE_TRACE_SLOTS] phase timestamps or null
  unsigned long long timeout_ns;  // limit of every bounded wait
  int withhold;                   // test aid: expert 0's router key is never published
  int H, E, k, I, S, prenorm;
  float eps;
  int map3d;  // 1: one TMA op per matrix (3-D map over the K-chunks), 0: one per K-chunk
  // schedule
  int n_su, rp_cta0, rp_ctas, n_ru, n_ou;
  int max_su, max_ru, max_ou;  // per-CTA maxima (strides of the scale images)
  // shared-memory layout (bytes from the 1024-aligned base)
  int off_dc, off_ru, off_su, off_rr, off_x, off_xn, off_h, off_rus, off_sus, off_red, off_keys, off_cand,
      off_gmax, off_bar, off_ys;
};
static_assert(sizeof(DecArgs) <= 4000, "kernel parameters stay under 4 KB");


// CTAs hand values to one another without grid barriers: every value that
// crosses CTAs (router keys, h, the residual stream between layers) travels
// in a 64-bit word whose high half is its layer's epoch and whose low half is
// the payload (an fp32 key or two bf16).  An aligned 64-bit store is seen
// whole, so a reader that finds the current epoch in a word has its payload.
// Each layer of each launch has its own epoch -- a counter read at launch and
// advanced by the launch's layer count -- and the buffers alternate with the
// epoch's parity.  Every layer rewrites all words of its parity, so a buffer
// never holds a tag more than two epochs old and the 32-bit epoch may wrap.
// A buffer is rewritten two layers later only by a CTA that has waited for
// values every CTA produced after it had read that buffer.
__device__ __forceinline__ unsigned long long ld_relaxed64(const unsigned long long *p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_relaxed64(unsigned long long *p, unsigned long long v) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// Tagged words per parity for the router keys and the shared-expert gate's
// dot product (E + 1), rounded up to 16 so that the h and residual words
// after them start on a 128-byte line: the down items poll h 32 bytes per lane.
__host__ __device__ constexpr int key_words(int E) { return (E + 1 + 15) / 16 * 16; }

__device__ __forceinline__ unsigned long long tagged(uint32_t ep, uint32_t payload) {
  return ((unsigned long long)ep << 32) | payload;
}

__device__ __forceinline__ bool has_tag(unsigned long long w, uint32_t ep) { return (uint32_t)(w >> 32) == ep; }

// w[i] = src[idx[i]] once that word carries epoch ep (idx[i] < 0: no word);
// false, with the status set, when the wait times out.
template <int N>
__device__ bool poll_tagged(const unsigned long long *src, const int (&idx)[N], unsigned long long (&w)[N],
                            uint32_t ep, int32_t *status, unsigned long long timeout_ns) {
  bool done = true;
#pragma unroll
  for (int i = 0; i < N; ++i) w[i] = idx[i] >= 0 ? ld_relaxed64(src + idx[i]) : tagged(ep, 0u);
#pragma unroll
  for (int i = 0; i < N; ++i) done = done && has_tag(w[i], ep);
  if (done) return true;
  const uint64_t t0 = ptx::globaltimer();
  while (true) {
    done = true;
#pragma unroll
    for (int i = 0; i < N; ++i)
      if (!has_tag(w[i], ep)) {
        w[i] = ld_relaxed64(src + idx[i]);
        done = done && has_tag(w[i], ep);
      }
    if (done) return true;
    if (ptx::globaltimer() - t0 > timeout_ns) {
      set_status(status, MOE_ERR_DEVICE_TIMEOUT);
      return false;
    }
  }
}

// Bounded wait for the phase of an mbarrier with the given parity.
__device__ bool wait_bar(uint64_t *bar, uint32_t parity, int32_t *status, unsigned long long timeout_ns) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer();
  while (!ptx::mbar_try_wait_sleep(bar, parity, 20000)) {
    if (ptx::globaltimer() - t0 > timeout_ns) {
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

// D += A.B on bf16 fragments, fp32 accumulators (m16n8k16).
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Vectors the GEMV reads (x, h) sit in shared memory in groups of 64 values,
// XPAD slots apart, each 8-value run (one code word) stored in the order
// p0 p4 p1 p5 | p2 p6 p3 p7: the code pairs (0,4) (2,6) (1,5) (3,7) of the
// word's rebuild (common.cuh), as the GEMV feeds them to the MMA.  perm8 takes a run in
// natural order (v0 = p0 p1, v1 = p2 p3, v2 = p4 p5, v3 = p6 p7) to that order.
__device__ __forceinline__ uint4 perm8(uint32_t v0, uint32_t v1, uint32_t v2, uint32_t v3) {
  return make_uint4(__byte_perm(v0, v2, 0x5410), __byte_perm(v0, v2, 0x7632), __byte_perm(v1, v3, 0x5410),
                    __byte_perm(v1, v3, 0x7632));
}

// x . W over one K-chunk of 8 rows.  chunk: the swizzled [8][128 B] code
// image of the chunk; sv, bv: the scale and bias of this lane's group (row g,
// group q of the chunk); xg: the chunk's first group of the permuted vector.  Lane (g, q) takes
// group q of the chunk in row g; the weights are the A operand: rows g and
// g+8 of A are codes {j, j+4 : j = 0, 1} and {j, j+4 : j = 2, 3} of a word of
// row g, and B columns 0 and 1 (lanes g = 0 and 1) carry the matching x
// values, so D[g][0] + D[g+8][1] sums row g over the 32 values of the word
// and its three quad partners.  Returns row g's sum in the lanes with q == 0.
__device__ __forceinline__ float gemv_chunk(const uint8_t *chunk, uint16_t sv, uint16_t bv, const uint16_t *xg, int g,
                                            int q) {
  const uint8_t *row = chunk + g * 128;
  const uint4 c0 = *reinterpret_cast<const uint4 *>(row + (((2 * q) ^ g) << 4));
  const uint4 c1 = *reinterpret_cast<const uint4 *>(row + (((2 * q + 1) ^ g) << 4));
  const __nv_bfloat162 s2 = bf16x2_splat(sv), b2 = bf16x2_splat(bv);
  const uint32_t wv[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
  const uint2 *xp = reinterpret_cast<const uint2 *>(xg + q * XPAD) + (g & 1);
  // four accumulators: chains of two dependent MMAs
  float e[4][4] = {};
  const GroupScale gs = group_scale(s2, b2);
  if (gs.small) {  // the usual route (common.cuh)
#pragma unroll
    for (int i = 0; i < 8; ++i) {  // word i: codes 8i..8i+7 of the group
      uint32_t p[4];  // pairs (0,4) (1,5) (2,6) (3,7)
      dq_word_small(wv[i], gs, p);
      const uint2 xv = xp[2 * i];
      mma16816(e[i & 3], p[0], p[2], p[1], p[3], xv.x, xv.y);
    }
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      uint32_t p[4];
      dq_word_general(wv[i], gs, p);
      const uint2 xv = xp[2 * i];
      mma16816(e[i & 3], p[0], p[2], p[1], p[3], xv.x, xv.y);
    }
  }
  return ((e[0][0] + e[1][0]) + (e[2][0] + e[3][0])) + ((e[0][3] + e[1][3]) + (e[2][3] + e[3][3]));
}

// Copies.  Code images: one 3-D TMA box per 8 rows and matrix (or one 2-D box
// per K-chunk where the driver refused the 3-D view), landing as
// [chunk][8 rows][128 B], swizzled.  Scales and biases: one bulk copy per
// array for a run of consecutive 8-row units of one expert.
__device__ __forceinline__ int code_ops(const DecArgs &a, int K) { return a.map3d ? 1 : K / KCH; }

// Gate/up codes of one unit (rows r0 .. r0+7 of expert e): copy o of
// 2 * code_ops, gate then up; cdst = [2 matrices][K/256 chunks][8][128 B] (8H bytes).
__device__ void gu_codes(const DecArgs &a, const DecMaps &mp, int o, uint8_t *cdst, int e, int r0, uint64_t *bar) {
  const int H = a.H, nco = code_ops(a, H), row = e * a.I + r0;
  const int mat = o / nco, c = o % nco;
  uint8_t *dst = cdst + mat * 4 * H + c * 1024;
  const CUtensorMap *map = mat ? &mp.up : &mp.gate;
  if (a.map3d)
    ptx::tma_load_3d(dst, map, bar, 0, row, 0);
  else
    ptx::tma_load_2d(dst, map, bar, c * 128, row);
}

// Array `which` (0 gate_s, 1 gate_b, 2 up_s, 3 up_b) of n units from rows r0
// of expert e: n * H/4 bytes, [n][8 rows][H/64] bf16.
__device__ void gu_scales(const DecArgs &a, const LayerW &L, int which, uint8_t *sdst, int e, int r0, int n,
                          uint64_t *bar) {
  const int H = a.H;
  const uint16_t *src = which == 0 ? L.w.gate_s : which == 1 ? L.w.gate_b : which == 2 ? L.w.up_s : L.w.up_b;
  ptx::bulk_g2s(sdst, src + ((size_t)e * a.I + r0) * (H / 64), n * (H / 4), bar);
}

// Down codes of one (output unit, slot): rows n0 .. n0+7 of expert e, copy o
// of code_ops; cdst = [I/256 chunks][8][128 B] (4I bytes).
__device__ void dn_codes(const DecArgs &a, const DecMaps &mp, int o, uint8_t *cdst, int e, int n0, uint64_t *bar) {
  const int row = e * a.H + n0;
  if (a.map3d)
    ptx::tma_load_3d(cdst, &mp.down, bar, 0, row, 0);
  else
    ptx::tma_load_2d(cdst + o * 1024, &mp.down, bar, o * 128, row);
}

// Partial gate/up dot products of `nu` unit images against x (padded, in
// shared memory) into red[(u * nkc + kc) * 16 + r] (r < 8 gate rows, 8 + r up
// rows).  scales: [4 arrays][ustride units][8 rows][H/64] bf16.  Warps split
// the K-chunks first, then the row sets (unit, matrix); with `bars`, unit u is
// read once bars[u] (its codes) and bars[0] (every unit's scales) complete.
// Returns false on a timeout.
__device__ bool gu_compute(const DecArgs &a, const uint8_t *codes, const uint8_t *scales, int ustride, int nu,
                           uint64_t *bars, uint32_t parity, const uint16_t *xs, float *red) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, q = lane & 3;
  const int H = a.H, nkc = H / KCH, WK = nkc < DWARPS ? nkc : DWARPS, WR = DWARPS / WK;
  const int kg = warp % WK, rg = warp / WK, gpr = H / 64;
  if (rg >= 2 * nu) return true;
  for (int kc = kg; kc < nkc; kc += WK) {
    for (int rs = rg; rs < 2 * nu; rs += WR) {
      const int u = rs >> 1, mat = rs & 1;  // gate (0) or up (1) rows of unit u
      if (bars && !(wait_bar(&bars[0], parity, a.status, a.timeout_ns) &&
                    wait_bar(&bars[u], parity, a.status, a.timeout_ns)))
        return false;
      const uint16_t *sc = reinterpret_cast<const uint16_t *>(scales + (size_t)(2 * mat * ustride + u) * (H / 4));
      const uint16_t *bi = reinterpret_cast<const uint16_t *>(scales + (size_t)((2 * mat + 1) * ustride + u) * (H / 4));
      const float d = gemv_chunk(codes + (size_t)u * 8 * H + mat * 4 * H + kc * 1024, sc[g * gpr + 4 * kc + q],
                                 bi[g * gpr + 4 * kc + q], xs + 4 * kc * XPAD, g, q);
      if (q == 0) red[(u * nkc + kc) * 16 + mat * 8 + g] = d;
    }
  }
  return true;
}

// h = bf16(silu(gate) * up) of `nu` units from the partials; unit u's 8 rows
// are elements row_of(u) .. +7 of the h vectors [k+S][I], written as tagged
// bf16 pairs into th (this epoch's half).
template <typename RowOf>
__device__ void gu_finish(const DecArgs &a, int nu, const float *red, unsigned long long *th, uint32_t ep,
                          RowOf row_of) {
  const int nkc = a.H / KCH;
  for (int t = threadIdx.x; t < nu * 4; t += DTHREADS) {
    const int u = t >> 2, r = (t & 3) * 2;
    uint32_t hv[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      float gs = 0.f, us = 0.f;
      for (int kc = 0; kc < nkc; ++kc) {
        gs += red[(u * nkc + kc) * 16 + r + i];
        us += red[(u * nkc + kc) * 16 + 8 + r + i];
      }
      hv[i] = f32_to_bf16(silu(gs) * us);
    }
    st_relaxed64(th + (row_of(u) + r) / 2, tagged(ep, hv[0] | (hv[1] << 16)));
  }
}

// Top-k of one token by one warp, for E <= 256 keys in shared memory:
// lane l holds the codes of experts l, l+32, ...  A bound taken from the 32
// lane maxima bounds the k-th largest key from below, so only the keys at or
// above it -- at most 8k unless lane maxima tie, all E at worst (cand holds
// E codes) -- are ranked, each against the others.  Same order and tie rule
// as topk_block.  Leaves the
// ids and their keys by rank in ids and w; topk_weights turns the keys into
// weights.
__device__ void topk_warp(const float *keys, int E, int k, unsigned long long *cand, int32_t *ids, float *w,
                          int32_t *status, uint64_t *tr) {
  const int lane = threadIdx.x & 31;
  auto mark = [&](int slot) {
    if (tr && lane == 0) tr[slot] = ptx::globaltimer();
  };
  float kv[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) kv[i] = lane + 32 * i < E ? keys[lane + 32 * i] : 0.f;
  unsigned long long c[8], m = 0ull;
  mark(18);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    c[i] = lane + 32 * i < E ? topk_code(kv[i], lane + 32 * i) : 0ull;
    m = c[i] > m ? c[i] : m;
  }
  // A lower bound on the k-th largest key: the k-th largest of the key bits
  // (upper word) of the 32 lane maxima -- k lanes hold distinct keys that
  // reach it.  Each lane counts the maxima at or above its own (all 32 read
  // from shared memory at once, no dependent chain), and the largest value
  // that at least k maxima reach is the k-th largest.
  __shared__ uint32_t s_lmax[32];
  const uint32_t v = (uint32_t)(m >> 32);
  s_lmax[lane] = v;
  __syncwarp();
  int ge = 0;
#pragma unroll
  for (int j = 0; j < 32; ++j) ge += s_lmax[j] >= v;
  const uint32_t tau_hi = __reduce_max_sync(0xffffffffu, ge >= k ? v : 0u);
  const unsigned long long tau = (unsigned long long)tau_hi << 32;  // 0: every key is a candidate
  mark(19);
  int n = 0;
  const unsigned below = (1u << lane) - 1u;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const bool take = c[i] != 0ull && c[i] >= tau;
    const unsigned b = __ballot_sync(0xffffffffu, take);
    if (take) cand[n + __popc(b & below)] = c[i];
    n += __popc(b);
  }
  __syncwarp();
  for (int t = lane; t < n; t += 32) {
    const unsigned long long ct = cand[t];
    int rank = 0;
    int j = 0;
    for (; j + 4 <= n; j += 4)  // four independent loads a step
      rank += (cand[j] > ct) + (cand[j + 1] > ct) + (cand[j + 2] > ct) + (cand[j + 3] > ct);
    for (; j < n; ++j) rank += cand[j] > ct;
    if (rank < k) {
      ids[rank] = topk_code_expert(ct);
      // the key back from its code (a NaN stays a NaN, -0 becomes +0: same weights)
      const uint32_t o = (uint32_t)(ct >> 32);
      w[rank] = __uint_as_float((o & 0x80000000u) ? (o & 0x7FFFFFFFu) : ~o);
    }
  }
  __syncwarp();
  mark(20);
}

// The softmax weights of the picked keys (in w, by rank) replace the keys:
// run by one warp after topk_warp, once the copies the ids decide are on
// their way.
__device__ void topk_weights(int k, int32_t *ids, float *w, int32_t *status) {
  const int lane = threadIdx.x & 31;
  const int my_id = lane < k ? ids[lane] : -1;
  const float my_key = lane < k ? w[lane] : 0.f;
  __syncwarp();
  topk_finish(lane, k, my_id, my_key, ids, w, nullptr, status);
  __syncwarp();
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
  if (!a.trace || threadIdx.x != 0 || blockIdx.x >= MOE_TRACE_CTAS) return;
  a.trace[blockIdx.x * MOE_TRACE_SLOTS + slot] = ptx::globaltimer();
}

// GATE: some layer of the launch has a shared-expert gate vector (the
// variant without one carries none of its code).
template <bool GATE>
__global__ void __launch_bounds__(DTHREADS, 1) decode_layer_kernel(const __grid_constant__ DecArgs a) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ int s_ids[16];
  __shared__ float s_w[16];
  __shared__ float s_gz;  // x . gate of the shared expert's sigmoid gate
  __shared__ float s_part[DWARPS];
  __shared__ uint32_t s_ep0;
  // 1024-byte aligned base for the swizzled code images (keeps the shared space)
  uint8_t *sm = smem_raw + ((1024u - (ptx::smem_u32(smem_raw) & 1023u)) & 1023u);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int cta = blockIdx.x, G = gridDim.x;
  const int H = a.H, I = a.I, E = a.E, k = a.k, S = a.S, NS = k + S;
  uint8_t *dc = sm + a.off_dc, *ru = sm + a.off_ru, *su = sm + a.off_su,
          *rus = sm + a.off_rus, *sus = sm + a.off_sus;
  float *rr = reinterpret_cast<float *>(sm + a.off_rr);
  uint16_t *xs = reinterpret_cast<uint16_t *>(sm + a.off_x);   // x, permuted groups (GEMV operand)
  uint16_t *xn = reinterpret_cast<uint16_t *>(sm + a.off_xn);  // x in natural order (router)
  uint16_t *hs = reinterpret_cast<uint16_t *>(sm + a.off_h);
  float *red = reinterpret_cast<float *>(sm + a.off_red);
  float *keys = reinterpret_cast<float *>(sm + a.off_keys);
  uint64_t *bars = reinterpret_cast<uint64_t *>(sm + a.off_bar);
  uint64_t *bar_p1 = bars, *bar_dsh = bars + 1, *bar_drt = bars + 2, *bar_ru = bars + 3;
  const int nsu = (cta < a.n_su) ? (a.n_su - 1 - cta) / G + 1 : 0;  // shared gate/up units of this CTA
  const int rc = cta - a.rp_cta0;                                    // index among the router CTAs
  // router rows of this CTA: experts rc, rc + rp_ctas, ... < E, and row E,
  // the shared-expert gate vector, in layers that have one
  auto rows_below = [&](int n) { return (rc >= 0 && rc < a.rp_ctas && rc < n) ? (n - 1 - rc) / a.rp_ctas + 1 : 0; };
  const int nre0 = rows_below(E), nre1 = rows_below(E + 1);
  auto nre_of = [&](int l) { return (GATE && S && a.lw[l].w.shared_gate) ? nre1 : nre0; };
  // Routed gate/up units: a run of consecutive units per CTA (so that one
  // copy per array brings a run's scales), the CTAs counted from the first one
  // without a shared unit, so that those take the extra units.
  const int rcta = (cta + G - a.n_su % G) % G;
  const int nru = a.n_ru / G + (rcta < a.n_ru % G), u0 = rcta * (a.n_ru / G) + min(rcta, a.n_ru % G);
  // output units: a run of consecutive 8-row units, rows o0 ..
  const int nou = a.n_ou / G + (cta < a.n_ou % G);
  const int o0 = 8 * (cta * (a.n_ou / G) + min(cta, a.n_ou % G));
  const int upr = I / 8;
  // copies are issued by the first two lanes of every warp: one warp alone issues slowly
  const int issuer = lane < 2 ? warp * 2 + lane : -1;
  const bool trace0 = a.trace != nullptr;
  // phases of the launch's last layer (its first one has the prologue's copies)
  auto trace = [&](int slot, int l) {
    if (trace0 && l == a.nl - 1) trace_at(a, slot);
  };
  trace_at(a, 0);

  // Layer l's router rows and shared gate/up unit (bar_p1) and its shared
  // expert's down rows (bar_dsh); each mbarrier completes once per layer, so
  // layer l waits on parity l & 1.
  auto issue_p1 = [&](int l) {
    const LayerW &L = a.lw[l];
    if (issuer >= 0) {
      const int ngu = 2 * code_ops(a, H) + 4, n1 = nsu * ngu, n2 = n1 + nre_of(l);
      for (int o = issuer; o < n2; o += 2 * DWARPS) {
        if (o < n1) {
          const int i = o / ngu, c = o % ngu;
          if (c < ngu - 4)
            gu_codes(a, a.maps[l], c, su + i * 8 * H, E, (cta + i * G) * 8, bar_p1);
          else
            gu_scales(a, L, c - (ngu - 4), sus + ((c - (ngu - 4)) * a.max_su + i) * (H / 4), E, (cta + i * G) * 8, 1,
                      bar_p1);
        } else {
          const int i = o - n1, e = rc + i * a.rp_ctas;
          ptx::bulk_g2s(rr + i * H, e < E ? L.router + (size_t)e * H : L.w.shared_gate, 4 * H, bar_p1);
        }
      }
    }
  };
  // the shared expert's down rows (its scales and biases are loaded into
  // registers by the down items themselves)
  auto issue_dsh = [&](int l) {
    if (issuer >= 0 && S) {
      const int ndn = code_ops(a, I);
      for (int o = issuer; o < nou * ndn; o += 2 * DWARPS) {
        const int ol = o / ndn;
        dn_codes(a, a.maps[l], o % ndn, dc + (ol * NS + k) * 4 * I, E, o0 + ol * 8, bar_dsh);
      }
    }
  };
  auto p1_bytes = [&](int l) { return (uint32_t)(nsu * 9 * H + nre_of(l) * 4 * H); };
  const uint32_t dsh_bytes = S ? (uint32_t)(nou * 4 * I) : 0u;

  if (tid == 0) {
    for (int i = 0; i < 3 + MAX_RU; ++i) ptx::mbar_init(&bars[i], 1);
    ptx::fence_mbar_init();
    if (a.map3d)
      for (int l = 0; l < a.nl; ++l) {
        ptx::prefetch_tmap(&a.maps[l].gate);
        ptx::prefetch_tmap(&a.maps[l].up);
        ptx::prefetch_tmap(&a.maps[l].down);
      }
    expect_tx(bar_p1, p1_bytes(0));
    expect_tx(bar_dsh, dsh_bytes);
  }
  __syncthreads();
  // ---------------------------------------------------------------- copies known at launch
  issue_p1(0);
  issue_dsh(0);
  trace_at(a, 1);
  // The input (and the workspace) may still be written by the previous
  // launch in the stream when this one starts early: wait for it here, after
  // the weight copies are on their way.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // This launch's layers take epochs ep0 + 1 .. ep0 + nl (CTA 0 advances the
  // counter when it is done, by which time every CTA has read it).
  if (tid == 0) s_ep0 = (uint32_t)ld_relaxed64(a.epoch);
  // the residual of this CTA's output rows: read once; later layers keep
  // their own output, which is the next layer's residual
  float res_v = 0.f;
  if (tid < nou * 8) res_v = bf16_to_f32(a.res[o0 + tid]);
  __syncthreads();
  const uint32_t ep0 = s_ep0;
  bool ok = true;
  uint32_t n_p1 = 1, n_dsh = 1, n_drt = 0;  // phases armed so far, for the drain on failure
  const int hw = NS * I / 2;                // words of one h buffer
  int l = 0;
  for (; l < a.nl && ok; ++l) {
    const LayerW &L = a.lw[l];
    const uint32_t ph = (uint32_t)l & 1u, ep = ep0 + (uint32_t)l + 1u, pb = ep & 1u;
    unsigned long long *tk = a.tkeys + pb * key_words(E), *thb = a.th + (size_t)pb * hw;
    trace(2, l);
    // this layer's tensor maps, for the copies issued after the routing
    if (tid == 0 && a.map3d && l > 0) {
      ptx::prefetch_tmap(&a.maps[l].gate);
      ptx::prefetch_tmap(&a.maps[l].up);
      ptx::prefetch_tmap(&a.maps[l].down);
    }
    // -------------------------------------------------------------- P0: x (padded groups)
    if (a.prenorm) {
      // r into registers (4 values a thread a round): layer 0 from the
      // input, later layers from the previous layer's tagged words; RMS, scale
      uint2 rv[XREG];
      bool got = true;
      if (l == 0) {
#pragma unroll
        for (int j = 0; j < XREG; ++j) {
          const int i = tid + j * DTHREADS;
          rv[j] = i < H / 4 ? __ldcg(reinterpret_cast<const uint2 *>(a.xin) + i) : make_uint2(0u, 0u);
        }
      } else {
        int idx[2 * XREG];
        unsigned long long w[2 * XREG];
#pragma unroll
        for (int j = 0; j < XREG; ++j) {
          const int i = tid + j * DTHREADS;
          idx[2 * j] = i < H / 4 ? 2 * i : -1;
          idx[2 * j + 1] = i < H / 4 ? 2 * i + 1 : -1;
        }
        got = poll_tagged(a.tr + (size_t)pb * (H / 2), idx, w, ep, a.status, a.timeout_ns);
#pragma unroll
        for (int j = 0; j < XREG; ++j) rv[j] = make_uint2((uint32_t)w[2 * j], (uint32_t)w[2 * j + 1]);
      }
      float ss = 0.f;
#pragma unroll
      for (int j = 0; j < XREG; ++j) {
        const float v0 = __uint_as_float(rv[j].x << 16), v1 = __uint_as_float(rv[j].x & 0xFFFF0000u);
        const float v2 = __uint_as_float(rv[j].y << 16), v3 = __uint_as_float(rv[j].y & 0xFFFF0000u);
        ss = fmaf(v0, v0, ss);
        ss = fmaf(v1, v1, ss);
        ss = fmaf(v2, v2, ss);
        ss = fmaf(v3, v3, ss);
      }
      ss = warp_sum(ss);
      if (lane == 0) s_part[warp] = ss;
      ok = __syncthreads_and(got) != 0;
      if (!ok) break;
      float tot = 0.f;
#pragma unroll
      for (int w = 0; w < DWARPS; ++w) tot += s_part[w];
      const float scale = rsqrtf(tot / (float)H + a.eps);
#pragma unroll
      for (int j = 0; j < XREG; ++j) {
        const int i = tid + j * DTHREADS;  // H / 4 is a multiple of 32: whole warps take this branch
        if (i < H / 4) {
          const uint32_t y0 = f32_to_bf16(__uint_as_float(rv[j].x << 16) * scale);
          const uint32_t y1 = f32_to_bf16(__uint_as_float(rv[j].x & 0xFFFF0000u) * scale);
          const uint32_t y2 = f32_to_bf16(__uint_as_float(rv[j].y << 16) * scale);
          const uint32_t y3 = f32_to_bf16(__uint_as_float(rv[j].y & 0xFFFF0000u) * scale);
          const uint32_t lo = y0 | (y1 << 16), hi = y2 | (y3 << 16);
          reinterpret_cast<uint2 *>(xn)[i] = make_uint2(lo, hi);
          // lanes 2c and 2c+1 hold the halves of word c: swap one register
          const bool odd = (lane & 1) != 0;
          const uint32_t got2 = __shfl_xor_sync(0xffffffffu, odd ? lo : hi, 1);
          const uint4 pw = odd ? perm8(got2, got2, lo, hi) : perm8(lo, hi, got2, got2);
          *reinterpret_cast<uint2 *>(xs + (i >> 4) * XPAD + (i & 15) * 4) =
              odd ? make_uint2(pw.z, pw.w) : make_uint2(pw.x, pw.y);
        }
      }
    } else {  // one layer (launches of several layers are pre-norm)
      for (int i = tid; i < H / 8; i += DTHREADS) {
        const uint4 v = __ldcg(reinterpret_cast<const uint4 *>(a.xin) + i);
        reinterpret_cast<uint4 *>(xn)[i] = v;
        *reinterpret_cast<uint4 *>(xs + (i >> 3) * XPAD + (i & 7) * 8) = perm8(v.x, v.y, v.z, v.w);
      }
    }
    __syncthreads();
    trace(3, l);

    // -------------------------------------------------------------- P1: router rows, shared gate/up
    ok = wait_bar(bar_p1, ph, a.status, a.timeout_ns);
    trace(4, l);
    if (ok)
      for (int i = warp; i < nre_of(l); i += DWARPS) {  // one warp per router row, fp32 FMA
        const float *row = rr + i * H;
        float acc = 0.f;
        for (int kk = 4 * lane; kk < H; kk += 128) {
          const float4 wv = *reinterpret_cast<const float4 *>(row + kk);
          const uint2 xv = *reinterpret_cast<const uint2 *>(xn + kk);
          acc = fmaf(__uint_as_float(xv.x << 16), wv.x, acc);
          acc = fmaf(__uint_as_float(xv.x & 0xFFFF0000u), wv.y, acc);
          acc = fmaf(__uint_as_float(xv.y << 16), wv.z, acc);
          acc = fmaf(__uint_as_float(xv.y & 0xFFFF0000u), wv.w, acc);
        }
        acc = warp_sum(acc);
        const int e = rc + i * a.rp_ctas;
        if (lane == 0) {
          const float key = (L.bias && e < E) ? acc + L.bias[e] : acc;
          if (e < E) a.keys[e] = key;
          if (!(a.withhold && e == 0)) st_relaxed64(tk + e, tagged(ep, __float_as_uint(key)));
        }
      }
    trace(5, l);
    // the shared expert's units (CTAs without router rows)
    if (ok && nsu > 0) ok = gu_compute(a, su, sus, a.max_su, nsu, nullptr, 0u, xs, red);
    ok = __syncthreads_and(ok) != 0;  // every flag below stays uniform across the CTA
    if (!ok) break;
    if (nsu > 0)
      gu_finish(a, nsu, red, thb, ep, [&](int u) { return (size_t)k * I + (size_t)(cta + u * G) * 8; });
    trace(6, l);
    // the next layer's router rows and shared unit, into the buffers P1 has
    // finished with (read by this CTA's generic loads, written by TMA next)
    if (l + 1 < a.nl) {
      ptx::fence_proxy_async_smem();
      if (tid == 0) expect_tx(bar_p1, p1_bytes(l + 1));
      __syncthreads();
      issue_p1(l + 1);
      n_p1 = l + 2;
    }
    trace(7, l);

    // -------------------------------------------------------------- P2: routing, routed gate/up
    // the keys: every thread polls a word or two (many pollers with few words
    // each see the last store sooner than a few pollers with many)
    bool got;
    {
      const int idx[2] = {tid < E ? tid : -1, tid + DTHREADS < E ? tid + DTHREADS : -1};
      unsigned long long w[2];
      got = poll_tagged(tk, idx, w, ep, a.status, a.timeout_ns);
      if (tid < E) keys[tid] = __uint_as_float((uint32_t)w[0]);
      if (tid + DTHREADS < E) keys[tid + DTHREADS] = __uint_as_float((uint32_t)w[1]);
    }
    ok = __syncthreads_and(got) != 0;
    if (!ok) break;
    if (E <= 256) {
      if (warp == 0)
        topk_warp(keys, E, k, reinterpret_cast<unsigned long long *>(sm + a.off_cand), s_ids, s_w, a.status,
                  trace0 && l == a.nl - 1 && cta < MOE_TRACE_CTAS ? a.trace + cta * MOE_TRACE_SLOTS : nullptr);
    } else {
      topk_block(keys, E, k, reinterpret_cast<unsigned long long *>(sm + a.off_cand),
                 reinterpret_cast<unsigned long long *>(sm + a.off_gmax), s_ids, s_w, a.status);
    }
    ptx::fence_proxy_async_smem();  // the routed buffers were last read by generic loads
    if (tid == 0) {
      // unit 0's barrier also takes every unit's scales
      for (int i = 0; i < nru; ++i) expect_tx(&bar_ru[i], (uint32_t)(8 * H + (i ? 0 : nru * H)));
      expect_tx(bar_drt, (uint32_t)(nou * k * 4 * I));
    }
    __syncthreads();
    trace(8, l);
    n_drt = l + 1;
    // the gate/up rows first (a block barrier keeps the down rows behind them
    // in the copy engine's queue): the scales of the unit run (one or two runs
    // of one slot each), then the code images unit by unit
    if (issuer >= 0 && nru > 0) {
      const int ua = u0, ub = min(u0 + nru, (u0 / upr + 1) * upr), uc = u0 + nru;  // runs [ua,ub) [ub,uc)
      const int nseg = ub < uc ? 2 : 1, ngc = 2 * code_ops(a, H);
      for (int o = issuer; o < 4 * nseg + nru * ngc; o += 2 * DWARPS) {
        if (o < 4 * nseg) {
          const int sg = o >> 2, which = o & 3, f = sg ? ub : ua, n = sg ? uc - ub : ub - ua;
          gu_scales(a, L, which, rus + (which * a.max_ru + (f - u0)) * (H / 4), s_ids[f / upr], (f % upr) * 8, n,
                    &bar_ru[0]);
        } else {
          const int i = (o - 4 * nseg) / ngc, u = u0 + i;
          gu_codes(a, a.maps[l], (o - 4 * nseg) % ngc, ru + i * 8 * H, s_ids[u / upr], (u % upr) * 8, &bar_ru[i]);
        }
      }
    }
    trace(21, l);
    __syncthreads();
    if (issuer >= 0) {  // routed down rows: code images per (unit, slot)
      const int ndn = code_ops(a, I), nc = nou * k * ndn;
      for (int o = issuer; o < nc; o += 2 * DWARPS) {
        const int b = o / ndn, ol = b / k, j = b % k;
        dn_codes(a, a.maps[l], o % ndn, dc + (ol * NS + j) * 4 * I, s_ids[j], o0 + ol * 8, bar_drt);
      }
    }
    trace(22, l);
    // the weights (only the combine needs them) while the copies are in flight
    if (warp == 0) {
      if (E <= 256) topk_weights(k, s_ids, s_w, a.status);
      if (cta == 0 && tid < k) {
        a.topk_id[tid] = s_ids[tid];
        a.topk_w[tid] = s_w[tid];
      }
    }
    trace(9, l);
    ok = __syncthreads_and(gu_compute(a, ru, rus, a.max_ru, nru, bar_ru, ph, xs, red)) != 0;
    trace(10, l);
    if (!ok) break;
    if (nru > 0)
      gu_finish(a, nru, red, thb, ep, [&](int u) {
        const int uu = u0 + u;
        return (size_t)(uu / upr) * I + (size_t)(uu % upr) * 8;
      });
    trace(11, l);

    // -------------------------------------------------------------- P3: down + combine
    // let the next launch in the stream start its prologue and weight copies
    if (l + 1 == a.nl) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    {
      // h of every slot comes into shared memory first (padded 64-value
      // groups in the MMA operand order), all threads polling at once and
      // before the down rows are waited for; the down items (output unit ol,
      // slot j, K-chunk kc), warp by warp, then read it there.  (Items that
      // polled their own h paid one L2 round trip each, in sequence.)
      const int nkcd = I / KCH, gpr = I / 64, g = lane >> 2, q = lane & 3;
      const int nitem = nou * NS * nkcd;
      // this lane's scale and bias for each of the warp's items (row g, group
      // q of the chunk), loaded while h is on its way
      uint16_t dsv[DN_ITEMS], dbv[DN_ITEMS];
#pragma unroll
      for (int i = 0; i < DN_ITEMS; ++i) {
        const int t = warp + i * DWARPS;
        dsv[i] = dbv[i] = 0;
        if (t < nitem) {
          const int kc = t % nkcd, j = (t / nkcd) % NS, ol = t / (nkcd * NS);
          const size_t at = ((size_t)(j < k ? s_ids[j] : E) * H + o0 + ol * 8 + g) * gpr + 4 * kc + q;
          dsv[i] = __ldg(L.w.down_s + at);
          dbv[i] = __ldg(L.w.down_b + at);
        }
      }
      bool gotw = true;
      {
        const int n8 = NS * I / 8;  // runs of 8 values (4 tagged words), two per thread and round
        for (int u = tid; u < n8; u += 2 * DTHREADS) {
          const int v = u + DTHREADS < n8 ? 4 * (u + DTHREADS) : -4;
          const int idx[8] = {4 * u, 4 * u + 1, 4 * u + 2, 4 * u + 3, v, v + 1, v + 2, v + 3};
          unsigned long long w[8];
          gotw = poll_tagged(thb, idx, w, ep, a.status, a.timeout_ns);
          if (!gotw) break;
          *reinterpret_cast<uint4 *>(hs + (u >> 3) * XPAD + (u & 7) * 8) =
              perm8((uint32_t)w[0], (uint32_t)w[1], (uint32_t)w[2], (uint32_t)w[3]);
          if (v >= 0) {
            const int u2 = u + DTHREADS;
            *reinterpret_cast<uint4 *>(hs + (u2 >> 3) * XPAD + (u2 & 7) * 8) =
                perm8((uint32_t)w[4], (uint32_t)w[5], (uint32_t)w[6], (uint32_t)w[7]);
          }
        }
      }
      trace(13, l);
      if (GATE && S && L.w.shared_gate && tid == 0) {  // x . gate, published with the keys
        const int gi[1] = {E};
        unsigned long long gw[1];
        gotw = gotw && poll_tagged(tk, gi, gw, ep, a.status, a.timeout_ns);
        s_gz = __uint_as_float((uint32_t)gw[0]);
      }
      gotw = gotw && wait_bar(bar_drt, ph, a.status, a.timeout_ns) && wait_bar(bar_dsh, ph, a.status, a.timeout_ns);
      gotw = __syncthreads_and(gotw) != 0;  // h is in shared memory
      trace(12, l);
#pragma unroll
      for (int i = 0; i < DN_ITEMS; ++i) {
        const int t = warp + i * DWARPS;
        if (t >= nitem || !gotw) break;  // gotw is uniform across the CTA here
        const int kc = t % nkcd, j = (t / nkcd) % NS, ol = t / (nkcd * NS);
        const float d = gemv_chunk(dc + (ol * NS + j) * 4 * I + kc * 1024, dsv[i], dbv[i],
                                   hs + ((j * I + kc * KCH) / 64) * XPAD, g, q);
        if (q == 0) red[t * 8 + g] = d;
      }
      trace(14, l);
      ok = __syncthreads_and(gotw) != 0;
      if (!ok) break;
      trace(15, l);
      // y_j = bf16(h_j . Wd_j) of every (row, slot) in parallel, then the combine
      float *ys = reinterpret_cast<float *>(sm + a.off_ys);  // [nou * 8][NS]
      for (int t = tid; t < nou * 8 * NS; t += DTHREADS) {
        const int ol = t / (8 * NS), r = (t / NS) & 7, j = t % NS;
        float v = 0.f;
        for (int kc = 0; kc < nkcd; ++kc) v += red[((ol * NS + j) * nkcd + kc) * 8 + r];
        ys[t] = bf16_to_f32(f32_to_bf16(v));
      }
      __syncthreads();
      // rows of this CTA (nou * 8 <= 16 of them, all in warp 0): out, and the
      // next epoch's tagged words (row pairs)
      if (warp == 0) {
        uint32_t ob = 0u;
        const int n = o0 + tid;
        if (tid < nou * 8) {
          const float *yr = ys + tid * NS;
          float o = res_v;
          if (GATE && S && L.w.shared_gate) o = fmaf(1.f / (1.f + expf(-s_gz)), yr[k], o);
          else if (S) o += yr[k];
          for (int j = 0; j < k; ++j) o = fmaf(s_w[j], yr[j], o);
          ob = f32_to_bf16(o);
          if (l + 1 == a.nl) a.out[n] = (uint16_t)ob;
          res_v = bf16_to_f32((uint16_t)ob);  // the next layer's residual for this row
        }
        const uint32_t other = __shfl_xor_sync(0xffffffffu, ob, 1);
        if (tid < nou * 8 && !(tid & 1))
          st_relaxed64(a.tr + (size_t)((ep + 1u) & 1u) * (H / 2) + n / 2, tagged(ep + 1u, ob | (other << 16)));
      }
      // the next layer's shared down rows, into the slots the down items have
      // finished with (after the residual words, which every CTA waits for)
      if (l + 1 < a.nl) {
        ptx::fence_proxy_async_smem();
        if (tid == 0) expect_tx(bar_dsh, dsh_bytes);
        __syncthreads();
        issue_dsh(l + 1);
        n_dsh = l + 2;
      }
      trace(16, l);
    }
    trace(17, l);
  }
  if (cta == 0 && tid == 0) st_relaxed64(a.epoch, (unsigned long long)(uint32_t)(ep0 + (uint32_t)a.nl));
  // never leave with copies in flight into this CTA's shared memory
  // (a phase that has completed passes at once)
  // (the copies complete by themselves: these waits take the full second
  // whatever limit the layer's waits had)
  if (tid == 0 && !ok) {
    constexpr unsigned long long DRAIN_NS = 1000000000ull;
    wait_bar(bar_p1, (n_p1 - 1) & 1u, a.status, DRAIN_NS);
    wait_bar(bar_dsh, (n_dsh - 1) & 1u, a.status, DRAIN_NS);
    if (n_drt > 0) {
      wait_bar(bar_drt, (n_drt - 1) & 1u, a.status, DRAIN_NS);
      for (int i = 0; i < nru; ++i) wait_bar(&bar_ru[i], (n_drt - 1) & 1u, a.status, DRAIN_NS);
    }
  }
  trace_at(a, MOE_TRACE_SLOTS - 1);
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
  const int max_re = (E + 1 + a.rp_ctas - 1) / a.rp_ctas;  // experts and the shared-expert gate row
  const int max_ru = (a.n_ru + G - 1) / G;
  const int max_ou = (a.n_ou + G - 1) / G;
  a.max_su = max_su > 0 ? max_su : 1;
  a.max_ru = max_ru;
  a.max_ou = max_ou;
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
  a.off_xn = o;
  o = al(o + H * 2, 128);
  a.off_h = o;  // h of every slot, padded 64-value groups
  o = al(o + (NS * I / 64) * XPAD * 2, 128);
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
  cudaFuncAttributes fa, fg;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess ||
      cudaFuncGetAttributes(&fa, decode_layer_kernel<false>) != cudaSuccess ||
      cudaFuncGetAttributes(&fg, decode_layer_kernel<true>) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return optin - (int)(fa.sharedSizeBytes > fg.sharedSizeBytes ? fa.sharedSizeBytes : fg.sharedSizeBytes);
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
  if (!pow2(H) || !pow2(I) || H < KCH || I < KCH || H > 4 * XREG * DTHREADS || num_sms <= 0 || k > 16 ||
      E > 1024)
    return false;
  DecPlan p = make_plan(H, E, k, I, S, num_sms);
  const int dn_items = p.a.max_ou * (k + S) * (I / KCH);  // down items of the busiest CTA
  return p.max_ru <= MAX_RU && dn_items <= DN_ITEMS * DWARPS && p.smem <= decode_smem_limit();
}

cudaError_t decode_prepare(int H, int E, int k, int I, int S, int num_sms) {
  // The opt-in is per kernel and device, shared by every plan: set it to the
  // device maximum so that plans of different shapes cannot shrink it under
  // one another (decode_supported has checked this shape's need against it).
  (void)H, (void)E, (void)k, (void)I, (void)S, (void)num_sms;
  const int lim = decode_smem_limit();
  if (lim <= 0) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(decode_layer_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, lim);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(decode_layer_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, lim);
}

namespace {

// One cooperative launch of layers [0, nl) of lw (nl <= MAXL).
cudaError_t launch_layers(const uint16_t *x, const uint16_t *res, uint16_t *out, int H, int E, int k, int I, int S,
                          int prenorm, float eps, const LayerW *lw, int nl, const DecodeScratch &sc, bool trace,
                          int num_sms, cudaStream_t s) {
  if (nl < 1 || nl > MAXL || (nl > 1 && !prenorm)) return cudaErrorInvalidValue;
  DecPlan p = make_plan(H, E, k, I, S, num_sms);
  DecArgs &a = p.a;
  a.nl = nl;
  a.xin = x;
  a.res = res;
  a.out = out;
  a.keys = sc.keys;
  a.topk_id = sc.topk_id;
  a.topk_w = sc.topk_w;
  a.tkeys = sc.tags;
  a.th = sc.tags + 2 * (size_t)key_words(E);
  a.tr = a.th + (size_t)(k + S) * I;
  a.epoch = sc.epoch;
  a.status = sc.status;
  a.trace = trace ? sc.trace : nullptr;
  a.timeout_ns = sc.timeout_ns;
  a.withhold = sc.withhold;
  a.prenorm = prenorm;
  a.eps = eps;
  a.map3d = 1;
  for (int l = 0; l < nl; ++l) {
    a.lw[l] = lw[l];
    cudaError_t e = make_maps(&a.maps[l], lw[l].w, H, E, I, S, a.map3d != 0);
    if (e != cudaSuccess && l == 0) {  // the driver refused the 3-D view: one 2-D box per K-chunk
      a.map3d = 0;
      e = make_maps(&a.maps[l], lw[l].w, H, E, I, S, false);
    }
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.grid);
  cfg.blockDim = dim3(DTHREADS);
  cfg.dynamicSmemBytes = p.smem;
  cfg.stream = s;
  // CTAs wait for values other CTAs produce, so every CTA must be resident at
  // once: launch cooperatively or not at all.  Programmatic serialisation lets the launch begin while
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
  bool gate = false;
  for (int l = 0; l < nl; ++l) gate = gate || (S && lw[l].w.shared_gate);
  void (*kern)(DecArgs) = gate ? decode_layer_kernel<true> : decode_layer_kernel<false>;
  prof_before(MOE_KERNEL_DECODE_LAYER, s);
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, a);
  if (e != cudaSuccess) {
    cudaGetLastError();
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kern, a);
  }
  prof_after(MOE_KERNEL_DECODE_LAYER, s);
  return e;
}

}  // namespace

size_t decode_tag_words(int H, int E, int k, int I, int S) {
  // keys and the shared-expert gate [2][key_words(E)], h [2][(k+S) I / 2], residual [2][H / 2]
  return 2 * (size_t)key_words(E) + (size_t)(k + S) * I + (size_t)H;
}

cudaError_t launch_decode(const uint16_t *x, const uint16_t *res, int H, int E, int k, int I, int S, int prenorm,
                          float eps, const float *router, const float *bias, ExpertPtrs w, uint16_t *out,
                          const DecodeScratch &sc, int num_sms, int *launches, cudaStream_t s) {
  const LayerW lw{router, bias, w};
  const cudaError_t e = launch_layers(x, res, out, H, E, k, I, S, prenorm, eps, &lw, 1, sc, true, num_sms, s);
  if (e != cudaSuccess) return e;
  *launches += 1;
  return cudaSuccess;
}

cudaError_t launch_decode_stack(uint16_t *r, int n_layers, int H, int E, int k, int I, int S, float eps,
                                const float *const *router, const float *const *bias, const ExpertPtrs *w,
                                const DecodeScratch &sc, int num_sms, int *launches, cudaStream_t s) {
  for (int l0 = 0; l0 < n_layers; l0 += MAXL) {
    const int nl = n_layers - l0 < MAXL ? n_layers - l0 : MAXL;
    LayerW lw[MAXL];
    for (int l = 0; l < nl; ++l) lw[l] = LayerW{router[l0 + l], bias ? bias[l0 + l] : nullptr, w[l0 + l]};
    const cudaError_t e = launch_layers(r, r, r, H, E, k, I, S, 1, eps, lw, nl, sc, l0 == 0, num_sms, s);
    if (e != cudaSuccess) return e;
    *launches += 1;
  }
  return cudaSuccess;
}

}  // namespace moe
