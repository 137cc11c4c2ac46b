// Routing on the device ("Prefill" section of the Lily pages: histogram,
// prefix scan, scatter and block map stay in one GPU submission with no CPU
// sync inside the layer; "three workload shapes": the router scores every
// expert and picks k).
//
//   router_logits_kernel   keys[t][e] = fp32(x[t] . router[e]) (+ bias[e])
//   topk_kernel            per token: k best keys, softmax weights, histogram
//   scatter_kernel         per expert: offset (scan of the histogram), stable
//                          scatter of its pairs (perm / inv) and its block-map
//                          tiles; the last expert's block also appends the
//                          shared expert's tiles.
#include "common.cuh"
#include "kernels.h"
#include "topk.cuh"

namespace moe {

// ---------------------------------------------------------------- router
// fp32 CUDA-core GEMM: a block computes 32 tokens x 64 experts, K in steps
// of 32; each thread owns 2 tokens x 4 experts.
constexpr int RT_M = 32, RT_N = 64, RT_K = 32;

__global__ void __launch_bounds__(256) router_logits_kernel(const uint16_t *__restrict__ x, int T, int H,
                                                            const float *__restrict__ router, int E,
                                                            const float *__restrict__ bias,
                                                            float *__restrict__ keys) {
  __shared__ float xs[RT_K][RT_M + 1];
  __shared__ float ws[RT_K][RT_N + 1];
  const int tid = threadIdx.x;
  const int t0 = blockIdx.x * RT_M, e0 = blockIdx.y * RT_N;
  const int tx = tid % 16, ty = tid / 16;
  float acc[2][4] = {};
  for (int k0 = 0; k0 < H; k0 += RT_K) {
    // x tile: 32 tokens x 32 k  (1024 values, 4 per thread)
    for (int i = tid; i < RT_M * RT_K; i += 256) {
      int r = i / RT_K, c = i % RT_K;
      int t = t0 + r;
      xs[c][r] = (t < T) ? bf16_to_f32(x[(size_t)t * H + k0 + c]) : 0.f;
    }
    for (int i = tid; i < RT_N * RT_K; i += 256) {
      int r = i / RT_K, c = i % RT_K;
      int e = e0 + r;
      ws[c][r] = (e < E) ? router[(size_t)e * H + k0 + c] : 0.f;
    }
    __syncthreads();
#pragma unroll 8
    for (int c = 0; c < RT_K; ++c) {
      float a0 = xs[c][2 * ty], a1 = xs[c][2 * ty + 1];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        float b = ws[c][4 * tx + j];
        acc[0][j] = fmaf(a0, b, acc[0][j]);
        acc[1][j] = fmaf(a1, b, acc[1][j]);
      }
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    int t = t0 + 2 * ty + i;
    if (t >= T) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      int e = e0 + 4 * tx + j;
      if (e < E) keys[(size_t)t * E + e] = bias ? acc[i][j] + bias[e] : acc[i][j];
    }
  }
}

// ---------------------------------------------------------------- top-k
// (per-token selection: topk.cuh)
// With part != null the keys are first summed from the router's KS K-slice
// partial sums ([KS][T][E], in slice order, + bias) and stored to keys.
template <int KPL>
__global__ void __launch_bounds__(256) topk_kernel(float *__restrict__ keys, int T, int E, int k,
                                                   int32_t *__restrict__ topk_id, float *__restrict__ topk_w,
                                                   int32_t *__restrict__ counts, int32_t *__restrict__ status,
                                                   const float *__restrict__ part, int KS,
                                                   const float *__restrict__ bias) {
  // per warp: the candidates (up to 256 codes) and the k picked ones
  __shared__ unsigned long long s_cand[KPL <= 8 ? 8 : 1][KPL <= 8 ? 256 + 16 : 1];
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) / 32, lane = threadIdx.x % 32;
  if (warp >= T) return;
  const KeySrc src{part ? part + (size_t)warp * E : nullptr, (size_t)T * E, part ? KS : 0, bias};
  topk_token<KPL>(keys + (size_t)warp * E, E, k, lane, topk_id + (size_t)warp * k, topk_w + (size_t)warp * k,
                  counts, status, src, KPL <= 8 ? s_cand[threadIdx.x / 32] : nullptr);
}

// Histogram of given expert ids ([T][k]); ids outside [0, E) are not counted
// and set MOE_ERR_DEVICE_BOUNDS; with debug, so does an expert named twice
// by one token.
__global__ void __launch_bounds__(256) ids_histogram_kernel(const int32_t *__restrict__ ids, int T, int E, int k,
                                                            int32_t *__restrict__ counts, int32_t *__restrict__ status,
                                                            int debug) {
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= T) return;
  const int32_t *row = ids + (size_t)t * k;
  for (int j = 0; j < k; ++j) {
    const int e = row[j];
    if (e < 0 || e >= E) {
      set_status(status, MOE_ERR_DEVICE_BOUNDS);
      continue;
    }
    atomicAdd(&counts[e], 1);
    if (debug)
      for (int i = 0; i < j; ++i)
        if (row[i] == e) set_status(status, MOE_ERR_DEVICE_BOUNDS);
  }
}

// ---------------------------------------------------------------- scatter
// One block per expert e.  offsets[e] and the first tile index of e are
// sums over counts[0..e-1] (each block recomputes them: E values).  The
// scatter walks tokens in ascending order, so perm is stable.
constexpr int SCATTER_THREADS = 1024;  // 4 tokens a thread: one round covers 4096 tokens

__global__ void __launch_bounds__(SCATTER_THREADS) scatter_kernel(const int32_t *__restrict__ topk_id, int T, int E, int k,
                                                      int BN, int S, const int32_t *__restrict__ counts,
                                                      int32_t *__restrict__ offsets, int32_t *__restrict__ perm,
                                                      int32_t *__restrict__ inv, int32_t *__restrict__ blockmap,
                                                      int32_t *__restrict__ n_tiles, int max_tiles, int BN2,
                                                      int32_t *__restrict__ blockmap2, int32_t *__restrict__ n_tiles2,
                                                      int max_tiles2, int32_t *__restrict__ status, int debug,
                                                      int32_t *__restrict__ qctr) {
  __shared__ int s_a[32], s_b[32], s_c[32];
  __shared__ int s_warp[SCATTER_THREADS / 32];
  __shared__ int s_off, s_tb, s_tb2;
  const int e = blockIdx.x, tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  if (qctr && e == 0 && tid == 0) {  // the grouped GEMMs' work-queue counters start the layer at zero
    qctr[0] = 0;
    qctr[1] = 0;
  }
  int off = 0, tb = 0, tb2 = 0;
  for (int i = tid; i < e; i += blockDim.x) {
    int c = counts[i];
    off += c;
    tb += (c + BN - 1) / BN;
    tb2 += (c + BN2 - 1) / BN2;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    off += __shfl_xor_sync(0xffffffffu, off, o);
    tb += __shfl_xor_sync(0xffffffffu, tb, o);
    tb2 += __shfl_xor_sync(0xffffffffu, tb2, o);
  }
  if (lane == 0) {
    s_a[wid] = off;
    s_b[wid] = tb;
    s_c[wid] = tb2;
  }
  __syncthreads();
  if (tid == 0) {
    int a = 0, b = 0, c = 0;
    for (int w = 0; w < (int)(blockDim.x / 32); ++w) {
      a += s_a[w];
      b += s_b[w];
      c += s_c[w];
    }
    s_off = a;
    s_tb = b;
    s_tb2 = c;
  }
  __syncthreads();
  off = s_off;
  tb = s_tb;
  tb2 = s_tb2;
  const int ce = counts[e];
  // one block map per tile height: rows of BN (and, when blockmap2 is given, of BN2)
  auto write_map = [&](int32_t *map, int32_t *nt, int mt, int bn, int tbase) {
    const int ntile_e = (ce + bn - 1) / bn;
    if (e == E - 1) {
      const int routed_tiles = tbase + ntile_e;
      const int shared_tiles = S ? (T + bn - 1) / bn : 0;
      if (tid == 0) {
        *nt = routed_tiles + shared_tiles;
        if (debug && (off + ce != k * T || routed_tiles + shared_tiles > mt)) set_status(status, MOE_ERR_DEVICE_BOUNDS);
      }
      for (int s = tid; s < shared_tiles; s += blockDim.x) {
        int idx = routed_tiles + s;
        if (idx < mt) {
          int4 ent = make_int4(E, k * T + s * bn, min(bn, T - s * bn), 0);
          reinterpret_cast<int4 *>(map)[idx] = ent;
        }
      }
    }
    for (int r = tid; r < ntile_e; r += blockDim.x) {
      int idx = tbase + r;
      if (idx < mt) {
        int4 ent = make_int4(e, off + r * bn, min(bn, ce - r * bn), 0);
        reinterpret_cast<int4 *>(map)[idx] = ent;
      }
    }
  };
  if (tid == 0) offsets[e] = off;
  if (e == E - 1 && tid == 0) offsets[E] = off + ce;
  write_map(blockmap, n_tiles, max_tiles, BN, tb);
  if (blockmap2) write_map(blockmap2, n_tiles2, max_tiles2, BN2, tb2);
  if (ce == 0) return;
  // Tokens in rounds of blockDim.x * TPT: thread tid takes TPT consecutive
  // tokens, so (thread, token) order is token order and a block-wide scan of
  // the per-thread match counts gives every match its rank.
  constexpr int TPT = 4;
  const bool vec = (k % 4) == 0;  // a token's k ids as int4 loads (rows are 16-byte aligned)
  int running = 0;
  for (int t0 = 0; t0 < T; t0 += blockDim.x * TPT) {
    int jf[TPT];
    int c = 0;
#pragma unroll
    for (int i = 0; i < TPT; ++i) {
      const int t = t0 + tid * TPT + i;
      jf[i] = -1;
      if (t < T) {
        const int32_t *row = topk_id + (size_t)t * k;
        if (vec) {
          for (int j4 = 0; j4 < k; j4 += 4) {
            const int4 v = *reinterpret_cast<const int4 *>(row + j4);
            if (v.x == e) jf[i] = j4;
            if (v.y == e) jf[i] = j4 + 1;
            if (v.z == e) jf[i] = j4 + 2;
            if (v.w == e) jf[i] = j4 + 3;
          }
        } else {
          for (int j = 0; j < k; ++j)
            if (row[j] == e) jf[i] = j;
        }
      }
      c += jf[i] >= 0;
    }
    int incl = c;  // inclusive scan of the counts over the warp
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += n;
    }
    if (lane == 31) s_warp[wid] = incl;
    __syncthreads();
    int before = 0, total = 0;
#pragma unroll 8
    for (int w = 0; w < SCATTER_THREADS / 32; ++w) {
      const int cw = s_warp[w];
      before += (w < wid) ? cw : 0;
      total += cw;
    }
    int pos = off + running + before + incl - c;
#pragma unroll
    for (int i = 0; i < TPT; ++i) {
      if (jf[i] < 0) continue;
      const int p = (t0 + tid * TPT + i) * k + jf[i];
      if (pos < off + ce) {  // always checked: a stale histogram must not write out of bounds
        perm[pos] = p;
        inv[p] = pos;
      } else {
        set_status(status, MOE_ERR_DEVICE_BOUNDS);
      }
      ++pos;
    }
    running += total;
    __syncthreads();
  }
  if (debug && tid == 0 && running != ce) set_status(status, MOE_ERR_DEVICE_BOUNDS);
}

// ---------------------------------------------------------------- launchers

cudaError_t launch_router_logits(const uint16_t *x, int T, int H, const float *router, int E, const float *bias,
                                 float *keys, cudaStream_t s) {
  dim3 grid((T + RT_M - 1) / RT_M, (E + RT_N - 1) / RT_N);
  prof_before(MOE_KERNEL_ROUTER, s);
  router_logits_kernel<<<grid, 256, 0, s>>>(x, T, H, router, E, bias, keys);
  prof_after(MOE_KERNEL_ROUTER, s);
  return cudaGetLastError();
}

cudaError_t launch_topk(float *keys, int T, int E, int k, int32_t *topk_id, float *topk_w, int32_t *counts,
                        int32_t *status, const float *part, int KS, const float *bias, cudaStream_t s) {
  // a warp per token: eight tokens per block, or two when T is small (so
  // that small T still spreads over many SMs)
  const int tpb = T >= 1024 ? 8 : 2;
  const int blocks = (T + tpb - 1) / tpb;
  const int kpl = (E + 31) / 32;
  prof_before(MOE_KERNEL_TOPK, s);
#define MOE_TOPK(K) topk_kernel<K><<<blocks, 32 * tpb, 0, s>>>(keys, T, E, k, topk_id, topk_w, counts, status, part, KS, bias)
  if (kpl <= 1)
    MOE_TOPK(1);
  else if (kpl <= 2)
    MOE_TOPK(2);
  else if (kpl <= 4)
    MOE_TOPK(4);
  else if (kpl <= 8)
    MOE_TOPK(8);
  else if (kpl <= 16)
    MOE_TOPK(16);
  else
    MOE_TOPK(32);
#undef MOE_TOPK
  prof_after(MOE_KERNEL_TOPK, s);
  return cudaGetLastError();
}

cudaError_t launch_ids_histogram(const int32_t *ids, int T, int E, int k, int32_t *counts, int32_t *status, int debug,
                                 cudaStream_t s) {
  ids_histogram_kernel<<<(T + 255) / 256, 256, 0, s>>>(ids, T, E, k, counts, status, debug);
  return cudaGetLastError();
}

cudaError_t launch_scatter(const int32_t *topk_id, int T, int E, int k, int BN, int S, const int32_t *counts,
                           int32_t *offsets, int32_t *perm, int32_t *inv, int32_t *blockmap, int32_t *n_tiles,
                           int max_tiles, int BN2, int32_t *blockmap2, int32_t *n_tiles2, int max_tiles2,
                           int32_t *status, int debug, int32_t *qctr, cudaStream_t s) {
  if (!blockmap2) BN2 = BN;
  prof_before(MOE_KERNEL_SCATTER, s);
  scatter_kernel<<<E, SCATTER_THREADS, 0, s>>>(topk_id, T, E, k, BN, S, counts, offsets, perm, inv, blockmap, n_tiles, max_tiles,
                                   BN2, blockmap2, n_tiles2, max_tiles2, status, debug, qctr);
  prof_after(MOE_KERNEL_SCATTER, s);
  return cudaGetLastError();
}

}  // namespace moe
