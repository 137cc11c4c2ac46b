// Single-token attention over a KV cache with grouped query heads.
//
// o_h = sum_l softmax_l(scale * q_h . k_{l,g}) v_{l,g}, g = h / 8, D = 256.
//
// Fixed blocks of positions: one CTA per (block, KV head), so each K and V row
// is read once for all eight query heads that share it (their eight rows fill
// the useful half of the tensor-core tiles below).  The block length is a
// multiple of 64 chosen per call so that the CTAs fill the SMs once (one CTA
// per SM: the staging buffers take 198 KB), which spreads the cache evenly and
// pays each CTA's prologue and merge once per SM.  The CTA's four warps take a
// quarter of the block each and run a flash-decoding pass over it in sub-tiles
// of 16 positions:
//   scores  S[8 heads x 16] = Q . K^T   mma.sync m16n8k16 (bf16 in, fp32 sums),
//           Q in registers for the whole pass, K fragments from shared memory;
//   softmax running maximum and sum per head (base-2 exponentials);
//   output  O[8 heads x 256] += P . V   P rounded to bf16 and taken straight
//           from the score fragments, V fragments by ldmatrix.trans.
// K and V sub-tiles arrive by bulk copies (TMA, one 512-byte row each, on a
// per-stage mbarrier), three sub-tiles ahead, into each warp's own buffers
// (rows padded to 528 bytes: the fragment reads hit 32 distinct banks).  The
// waits are bounded: a wait that gives up sets MOE_ERR_DEVICE_TIMEOUT in the
// workspace's status word.  The warps' (max, sum, O) merge in shared memory
// into the block's partial result; a second kernel, launched as its
// programmatic dependent so that it is resident when the pass ends, combines
// the blocks.
#include <cuda_bf16.h>
#include <math.h>

#include <algorithm>

#include "attn.h"
#include "common.cuh"
#include "kernels.h"
#include "tc_ptx.cuh"

namespace moe {
namespace {

constexpr int AT_D = 256, AT_G = 8;         // head dimension, query heads per KV head
constexpr int AT_QUANT = 64;                // block lengths are multiples of this
constexpr int AT_MAXBLK = 512;              // blocks per KV head at most
constexpr int AT_WARPS = 4, AT_THREADS = AT_WARPS * 32;
constexpr int AT_SUB = 16;                  // positions per sub-tile
constexpr int AT_ROW = AT_D * 2 + 16;       // padded smem row (528 bytes)
constexpr int AT_TILE = AT_SUB * AT_ROW;    // one K or V sub-tile
constexpr int AT_STAGE = 2 * AT_TILE;       // K and V
constexpr int AT_NSTAGE = 3;               // sub-tiles in flight per warp
constexpr int AT_WARP_SMEM = AT_NSTAGE * AT_STAGE;
constexpr int AT_SMEM = AT_WARPS * AT_WARP_SMEM;  // 202,752 bytes

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a2, uint32_t b0, uint32_t b1) {
  // rows 8-15 of A are zero: only the eight query heads of rows 0-7 are real
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(0u), "r"(a2), "r"(0u), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}


__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  return (uint32_t)f32_to_bf16(lo) | ((uint32_t)f32_to_bf16(hi) << 16);
}

constexpr unsigned long long AT_TIMEOUT_NS = 1000000000ull;  // a copy wait gives up after 1 s

// Bounded wait on an mbarrier phase; false once AT_TIMEOUT_NS has passed.
__device__ bool at_wait(uint64_t *bar, uint32_t parity) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer();
  while (!ptx::mbar_try_wait_sleep(bar, parity, 20000u))
    if (ptx::globaltimer() - t0 > AT_TIMEOUT_NS) return false;
  return true;
}

struct AttnArgs {
  const uint16_t *q, *k, *v;
  int32_t *status;                  // sticky MOE_ERR_DEVICE_TIMEOUT
  float *part_o, *part_m, *part_l;  // [nblk][Hq][D], [nblk][Hq], [nblk][Hq]
  int L, Hq, Hkv;
  int blk_len, nsub;                // positions per block, sub-tiles per warp (blk_len / 64)
  float scale_log2;                 // scale * log2(e)
};

__global__ void __launch_bounds__(AT_THREADS) attn_block_kernel(const __grid_constant__ AttnArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];
  __shared__ uint64_t bars[AT_WARPS][AT_NSTAGE];
  // the combine kernel may be scheduled now; it waits for this grid to finish
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int blk = blockIdx.x, g = blockIdx.y;
  const int r = lane >> 2, c = lane & 3;  // fragment row (head / position) and column pair
  const int L = a.L, Hkv = a.Hkv;
  const int nsub = a.nsub, p_warp = blk * a.blk_len + warp * (a.blk_len / AT_WARPS);
  uint8_t *ws = smem + warp * AT_WARP_SMEM;

  // this warp's sub-tile st into stage st % AT_NSTAGE: 16 rows of K and of V
  // (512 bytes each, one bulk copy per row: lane i copies row i % 16 of K for
  // i < 16, of V otherwise).  Rows past L are not copied.
  uint64_t *wbar = bars[warp];
  if (lane == 0) {
    for (int s = 0; s < AT_NSTAGE; ++s) ptx::mbar_init(&wbar[s], 1);
    ptx::fence_mbar_init();
  }
  __syncwarp();
  auto issue = [&](int st) {
    if (st >= nsub) return;
    const int stg = st % AT_NSTAGE, p0 = p_warp + st * AT_SUB;
    const int nvalid = min(AT_SUB, L - p0);
    if (nvalid <= 0) return;
    ptx::fence_proxy_async_smem();  // this stage's earlier reads come before the copies
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive_expect_tx(&wbar[stg], (uint32_t)(2 * nvalid * AT_D * 2));
    __syncwarp();
    const int row = lane & (AT_SUB - 1), kv = lane >> 4;
    if (row < nvalid)
      ptx::bulk_g2s(ws + stg * AT_STAGE + kv * AT_TILE + row * AT_ROW,
                    (kv ? a.v : a.k) + ((size_t)(p0 + row) * Hkv + g) * AT_D, AT_D * 2, &wbar[stg]);
  };

  // the query rows of the group, as the A fragments of the 16 k-steps
  uint32_t qa[16], qb[16];
  {
    const uint32_t *qrow = reinterpret_cast<const uint32_t *>(a.q + (size_t)(g * AT_G + r) * AT_D);
#pragma unroll
    for (int s = 0; s < 16; ++s) {
      qa[s] = __ldg(qrow + 8 * s + c);
      qb[s] = __ldg(qrow + 8 * s + 4 + c);
    }
  }
  float o[32][4];
#pragma unroll
  for (int t = 0; t < 32; ++t) o[t][0] = o[t][1] = o[t][2] = o[t][3] = 0.f;
  float m = -INFINITY, l = 0.f;  // running maximum (base-2 units) and this lane's part of the sum

  for (int st = 0; st < AT_NSTAGE - 1; ++st) issue(st);
  bool ok = true;
  int st_fail = 0;
  for (int st = 0; st < nsub; ++st) {
    const int p0 = p_warp + st * AT_SUB;
    issue(st + AT_NSTAGE - 1);  // into the stage sub-tile st-1 used (every lane has finished it)
    if (p0 < L && ok) {  // warp-uniform
      ok = __all_sync(0xffffffffu, at_wait(&wbar[st % AT_NSTAGE], (uint32_t)(st / AT_NSTAGE) & 1u));
      if (!ok) {
        if (lane == 0) atomicExch(a.status, (int32_t)MOE_ERR_DEVICE_TIMEOUT);
        st_fail = st;
        break;
      }
      uint8_t *ks = ws + (st % AT_NSTAGE) * AT_STAGE, *vs = ks + AT_TILE;
      if (p0 + AT_SUB > L) {  // the cache's last sub-tile: V rows past L read as zeros
        for (int row = L - p0; row < AT_SUB; ++row)
          *reinterpret_cast<uint4 *>(vs + row * AT_ROW + lane * 16) = make_uint4(0u, 0u, 0u, 0u);
        __syncwarp();
      }
      // scores of n-tiles 0 and 1 (positions p0 .. p0+7, p0+8 .. p0+15), each
      // summed in four independent chains of four k-steps, then added
      float sc[2][4];
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const uint32_t *krow = reinterpret_cast<const uint32_t *>(ks + (8 * j + r) * AT_ROW);
        float part[4][4] = {};
#pragma unroll
        for (int s = 0; s < 16; ++s) mma16816(part[s & 3], qa[s], qb[s], krow[8 * s + c], krow[8 * s + 4 + c]);
#pragma unroll
        for (int e = 0; e < 2; ++e) sc[j][e] = (part[0][e] + part[1][e]) + (part[2][e] + part[3][e]);
      }
      // row r = head; this lane's positions p0 + 8j + 2c + {0, 1}
      float x[4];
      float tmax = -INFINITY;
#pragma unroll
      for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int pos = p0 + 8 * j + 2 * c + e;
          const float v = pos < L ? sc[j][e] * a.scale_log2 : -INFINITY;
          x[2 * j + e] = v;
          tmax = fmaxf(tmax, v);
        }
      tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 1));
      tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 2));
      const float mn = fmaxf(m, tmax);  // finite: position p0 is valid
      const float alpha = exp2f(m - mn);
      m = mn;
      float pr[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) pr[e] = exp2f(x[e] - mn);
      l = l * alpha + ((pr[0] + pr[1]) + (pr[2] + pr[3]));
      if (__any_sync(0xffffffffu, alpha != 1.f)) {  // a head's maximum moved: rescale its sums
#pragma unroll
        for (int t = 0; t < 32; ++t) {
          o[t][0] *= alpha;
          o[t][1] *= alpha;
        }
      }
      const uint32_t pa0 = pack_bf16x2(pr[0], pr[1]), pa2 = pack_bf16x2(pr[2], pr[3]);
      // O += P . V, 16 output dimensions per ldmatrix
      const uint32_t vs_u32 = static_cast<uint32_t>(__cvta_generic_to_shared(vs));
      const int mat = lane >> 3, row = (mat & 1) * 8 + (lane & 7);
#pragma unroll
      for (int d16 = 0; d16 < AT_D / 16; ++d16) {
        uint32_t b[4];
        ldsm_x4_trans(b, vs_u32 + row * AT_ROW + (d16 * 16 + (mat >> 1) * 8) * 2);
        mma16816(o[2 * d16], pa0, pa2, b[0], b[1]);
        mma16816(o[2 * d16 + 1], pa0, pa2, b[2], b[3]);
      }
    }
    __syncwarp();  // every lane is done with this stage before it is refilled
  }
  if (!ok) {  // let the copies still in flight land (bounded) before the buffers are reused
    for (int st = st_fail; st < min(nsub, st_fail + AT_NSTAGE); ++st)
      if (p_warp + st * AT_SUB < L) at_wait(&wbar[st % AT_NSTAGE], (uint32_t)(st / AT_NSTAGE) & 1u);
  }
  __syncthreads();  // the staging buffers become the merge area

  // merge the four warps: per warp m[8], l[8], O[8][256]
  l += __shfl_xor_sync(0xffffffffu, l, 1);
  l += __shfl_xor_sync(0xffffffffu, l, 2);
  float *om = reinterpret_cast<float *>(smem);             // [warp][8][256]
  float *mm = om + AT_WARPS * AT_G * AT_D;                 // [warp][8]
  float *lm = mm + AT_WARPS * AT_G;                        // [warp][8]
  if (c == 0) {
    mm[warp * AT_G + r] = m;
    lm[warp * AT_G + r] = l;
  }
#pragma unroll
  for (int t = 0; t < 32; ++t)
    *reinterpret_cast<float2 *>(om + (warp * AT_G + r) * AT_D + 8 * t + 2 * c) = make_float2(o[t][0], o[t][1]);
  __syncthreads();
  const int hq0 = g * AT_G;
  for (int i = tid; i < AT_G * AT_D; i += AT_THREADS) {
    const int h = i / AT_D, d = i % AT_D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < AT_WARPS; ++w) M = fmaxf(M, mm[w * AT_G + h]);
    float acc = 0.f, den = 0.f;
#pragma unroll
    for (int w = 0; w < AT_WARPS; ++w) {
      const float mw = mm[w * AT_G + h];
      const float f = mw == -INFINITY ? 0.f : exp2f(mw - M);  // a warp with no valid position adds nothing
      acc = fmaf(f, om[(w * AT_G + h) * AT_D + d], acc);
      den = fmaf(f, lm[w * AT_G + h], den);
    }
    const size_t row = (size_t)blk * a.Hq + hq0 + h;
    a.part_o[row * AT_D + d] = acc;
    if (d == 0) {
      a.part_m[row] = M;
      a.part_l[row] = den;
    }
  }
}

// o[h][d] = bf16(sum_b 2^(m_b - M) O_b[h][d] / sum_b 2^(m_b - M) l_b[h]).  One
// CTA per (head, 32 dimensions); its eight warps take every eighth block with
// a running maximum, then merge in shared memory.
__global__ void __launch_bounds__(256) attn_combine_kernel(const float *__restrict__ part_o,
                                                           const float *__restrict__ part_m,
                                                           const float *__restrict__ part_l, int nblk, int Hq,
                                                           uint16_t *__restrict__ out) {
  __shared__ float sm_m[8][32], sm_n[8][32], sm_d[8][32];
  // launched as a programmatic dependent of the block pass: resident early,
  // it reads the partials only once that grid has completed
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int h = blockIdx.x, wg = threadIdx.x >> 5, lane = threadIdx.x & 31, d = blockIdx.y * 32 + lane;
  // blocks wg, wg + 8, ... in groups of eight, each group's loads issued
  // together, merged into a running maximum
  float M = -INFINITY, num = 0.f, den = 0.f;
  for (int b0 = wg; b0 < nblk; b0 += 64) {
    float mb[8], ob[8], lb[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int b = b0 + 8 * i;
      const size_t row = (size_t)(b < nblk ? b : b0) * Hq + h;
      mb[i] = b < nblk ? part_m[row] : -INFINITY;
      ob[i] = part_o[row * AT_D + d];
      lb[i] = part_l[row];
    }
    float mx = M;
#pragma unroll
    for (int i = 0; i < 8; ++i) mx = fmaxf(mx, mb[i]);
    const float fo = exp2f(M - mx);  // 0 while M is still -inf
    num *= fo;
    den *= fo;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float f = exp2f(mb[i] - mx);  // 0 for the slots past nblk
      num = fmaf(f, ob[i], num);
      den = fmaf(f, lb[i], den);
    }
    M = mx;
  }
  sm_m[wg][lane] = M;
  sm_n[wg][lane] = num;
  sm_d[wg][lane] = den;
  __syncthreads();
  if (wg == 0) {
    float Mx = -INFINITY;
#pragma unroll
    for (int w = 0; w < 8; ++w) Mx = fmaxf(Mx, sm_m[w][lane]);
    float n = 0.f, dd = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) {
      const float f = sm_m[w][lane] == -INFINITY ? 0.f : exp2f(sm_m[w][lane] - Mx);  // warps with no block
      n = fmaf(f, sm_n[w][lane], n);
      dd = fmaf(f, sm_d[w][lane], dd);
    }
    out[(size_t)h * AT_D + d] = f32_to_bf16(n / dd);
  }
}

// Blocks per KV head and their length (a multiple of AT_QUANT) for L
// positions: enough CTAs to give every SM one, at most AT_MAXBLK.
void block_split(int L, int Hkv, int num_sms, int *nblk, int *blk_len) {
  int want = (num_sms + Hkv - 1) / Hkv;
  want = want < 1 ? 1 : want > AT_MAXBLK ? AT_MAXBLK : want;
  int len = (L + want - 1) / want;
  len = (len + AT_QUANT - 1) / AT_QUANT * AT_QUANT;
  *blk_len = len;
  *nblk = (L + len - 1) / len;
}

// Workspace: the status word (256 bytes reserved), partial outputs, maxima, sums.
size_t ws_layout(int nblk, int Hq, size_t *off_m, size_t *off_l) {
  const size_t o = 256 + (size_t)nblk * Hq * AT_D * 4;
  *off_m = o;
  *off_l = o + (((size_t)nblk * Hq * 4 + 255) / 256) * 256;
  return *off_l + (size_t)nblk * Hq * 4;
}

}  // namespace
}  // namespace moe

extern "C" size_t attn_decode_workspace_bytes(int L, int Hq, int D) {
  if (L < 1 || Hq < 1 || D != moe::AT_D || L > (1 << 24)) return 0;
  // the most blocks any device could use: one per AT_QUANT positions, at most AT_MAXBLK
  const int nb = std::min((L + moe::AT_QUANT - 1) / moe::AT_QUANT, moe::AT_MAXBLK);
  size_t om, ol;
  return moe::ws_layout(nb, Hq, &om, &ol);
}

extern "C" moe_status attn_decode(const void *q_d, const void *k_d, const void *v_d, int L, int Hq, int Hkv, int D,
                                  float scale, void *ws_d, size_t ws_bytes, void *o_d, void *stream) {
  using moe::aligned16;
  if (!q_d || !k_d || !v_d || !ws_d || !o_d || L < 1 || Hkv < 1 || Hq < 1 || !(scale >= 0.f) || isinf(scale))
    return MOE_ERR_INVALID_ARGUMENT;
  if (D != moe::AT_D || Hq != moe::AT_G * Hkv || L > (1 << 24)) return MOE_ERR_UNSUPPORTED;
  if (!aligned16(q_d) || !aligned16(k_d) || !aligned16(v_d) || !aligned16(ws_d) || !aligned16(o_d))
    return MOE_ERR_MISALIGNED;
  if (ws_bytes < attn_decode_workspace_bytes(L, Hq, D)) return MOE_ERR_WORKSPACE_TOO_SMALL;
  int dev = 0, num_sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return moe::note_cuda_error(e);
  int nblk = 0, blk_len = 0;
  moe::block_split(L, Hkv, num_sms, &nblk, &blk_len);
  size_t off_m, off_l;
  moe::ws_layout(nblk, Hq, &off_m, &off_l);
  // per device and cheap: set on every call rather than remembered
  const cudaError_t attr =
      cudaFuncSetAttribute(moe::attn_block_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, moe::AT_SMEM);
  if (attr != cudaSuccess) return moe::note_cuda_error(attr);
  if (scale == 0.f) scale = 1.f / sqrtf((float)D);
  uint8_t *ws = static_cast<uint8_t *>(ws_d);
  moe::AttnArgs a;
  a.q = static_cast<const uint16_t *>(q_d);
  a.k = static_cast<const uint16_t *>(k_d);
  a.v = static_cast<const uint16_t *>(v_d);
  a.status = reinterpret_cast<int32_t *>(ws);
  a.part_o = reinterpret_cast<float *>(ws + 256);
  a.part_m = reinterpret_cast<float *>(ws + off_m);
  a.part_l = reinterpret_cast<float *>(ws + off_l);
  a.L = L;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.blk_len = blk_len;
  a.nsub = blk_len / (moe::AT_WARPS * moe::AT_SUB);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  moe::prof_before(MOE_KERNEL_ATTN_DECODE, s);
  moe::attn_block_kernel<<<dim3(nblk, Hkv), moe::AT_THREADS, moe::AT_SMEM, s>>>(a);
  moe::prof_after(MOE_KERNEL_ATTN_DECODE, s);
  e = cudaGetLastError();
  if (e != cudaSuccess) return moe::note_cuda_error(e);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(Hq, moe::AT_D / 32);
  cfg.blockDim = dim3(256);
  cfg.stream = s;
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = pdl;
  cfg.numAttrs = 1;
  uint16_t *out = static_cast<uint16_t *>(o_d);
  e = cudaLaunchKernelEx(&cfg, moe::attn_combine_kernel, (const float *)a.part_o, (const float *)a.part_m,
                         (const float *)a.part_l, nblk, Hq, out);
  if (e != cudaSuccess) {  // a driver that refuses the attribute: a plain launch after the block pass
    cudaGetLastError();
    cfg.numAttrs = 0;
    e = cudaLaunchKernelEx(&cfg, moe::attn_combine_kernel, (const float *)a.part_o, (const float *)a.part_m,
                           (const float *)a.part_l, nblk, Hq, out);
  }
  return moe::note_cuda_error(e);
}
