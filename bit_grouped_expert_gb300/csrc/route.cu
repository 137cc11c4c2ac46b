// Routing on the device ("Prefill" section of the Lily pages: histogram,
// prefix scan, scatter and block map stay in one GPU submission with no CPU
// sync inside the layer; "three workload shapes": the router scores every
// expert and picks k).
//
//   router_logits_kernel   keys[t][e] = fp32(x[t] . router[e]) (+ bias[e])
//   topk_kernel            per token: k best keys, softmax weights, histogram
//                          (over all pairs and per chunk of SCATTER_ENT pairs)
//   scatter_kernel         per chunk of pairs: the experts' offsets (scan of the
//                          histogram), stable ranks of the chunk's pairs and
//                          their scatter (perm / inv); the blocks share the
//                          block-map tiles out by expert, the shared expert's
//                          tiles last.
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
  // counts[0 .. E) is the histogram, then one histogram per chunk of pairs
  // per warp: the candidates (up to 256 codes) and the k picked ones
  __shared__ unsigned long long s_cand[KPL <= 8 ? 8 : 1][KPL <= 8 ? 256 + 16 : 1];
  // launched as a programmatic dependent of the router: its keys first
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) / 32, lane = threadIdx.x % 32;
  if (warp >= T) return;
  const KeySrc src{part ? part + (size_t)warp * E : nullptr, (size_t)T * E, part ? KS : 0, bias};
  topk_token<KPL>(keys + (size_t)warp * E, E, k, lane, topk_id + (size_t)warp * k, topk_w + (size_t)warp * k,
                  counts, status, src, KPL <= 8 ? s_cand[threadIdx.x / 32] : nullptr, counts + E,
                  (size_t)warp * k);
}

// Histogram of given expert ids ([T][k]), over all pairs and per chunk of
// SCATTER_ENT pairs (as the top-k kernel); ids outside [0, E) are not counted
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
    atomicAdd(&counts[(size_t)E + (((size_t)t * k + j) / SCATTER_ENT) * E + e], 1);  // the pair's chunk
    if (debug)
      for (int i = 0; i < j; ++i)
        if (row[i] == e) set_status(status, MOE_ERR_DEVICE_BOUNDS);
  }
}

// ---------------------------------------------------------------- scatter
// One block per chunk of SCATTER_ENT consecutive (token, slot) pairs.  Every
// block scans the histogram (E values) for the experts' offsets and first
// tiles; the pairs of expert e in earlier chunks (the per-chunk histograms)
// put the chunk's first pair of e at base[e].  Within the chunk each warp
// takes SCATTER_ENT / 8 consecutive pairs in rounds of 32: a match over the
// warp counts each expert's pairs (per warp), a scan over the warps turns the
// counts into starts, and a second pass hands out the ranks in pair order.
// The scatter is therefore stable: perm lists each expert's pairs in
// ascending pair index.  The blocks share the block-map entries out by
// expert (e = block, block + gridDim.x, ...); the last block also writes the
// shared expert's tiles, n_tiles and offsets[E].
constexpr int SCATTER_THREADS = 256;
constexpr int SCATTER_WARPS = SCATTER_THREADS / 32;

// Exclusive scan over the block of one value per expert (E <= 4 * 256 = 1024:
// thread i holds experts 4i .. 4i+3); returns the total.
__device__ __forceinline__ int block_exscan4(int v[4], int *s_warp) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int tsum = v[0] + v[1] + v[2] + v[3];
  int incl = tsum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += n;
  }
  if (lane == 31) s_warp[wid] = incl;
  __syncthreads();
  int before = 0, total = 0;
#pragma unroll
  for (int w = 0; w < SCATTER_WARPS; ++w) {
    const int cw = s_warp[w];
    before += (w < wid) ? cw : 0;
    total += cw;
  }
  __syncthreads();  // s_warp is reused by the next scan
  int run = before + incl - tsum;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int x = v[i];
    v[i] = run;
    run += x;
  }
  return total;
}

__global__ void __launch_bounds__(SCATTER_THREADS) scatter_kernel(
    const int32_t *__restrict__ topk_id, int T, int E, int k, int BN, int S, const int32_t *__restrict__ counts,
    int32_t *__restrict__ offsets, int32_t *__restrict__ perm, int32_t *__restrict__ inv,
    int32_t *__restrict__ blockmap, int32_t *__restrict__ n_tiles, int max_tiles, int BN2,
    int32_t *__restrict__ blockmap2, int32_t *__restrict__ n_tiles2, int max_tiles2, int32_t *__restrict__ status,
    int debug, int32_t *__restrict__ qctr) {
  // shared: start of each expert in the chunk, per warp ([warp][E]); the
  // experts' offsets and first tiles ([3][E])
  extern __shared__ int s_dyn[];
  int *s_hist = s_dyn;
  int *s_off = s_dyn + SCATTER_WARPS * E, *s_tb = s_off + E, *s_tb2 = s_tb + E;
  __shared__ int s_warp[SCATTER_WARPS];
  // launched as a programmatic dependent of the top-k: its ids and counts first
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5, b = blockIdx.x;
  const int n_pairs = T * k;
  // this warp's pairs of the chunk: ids loaded first, so that their latency
  // overlaps the scans below
  constexpr int PER_WARP = SCATTER_ENT / SCATTER_WARPS, ROUNDS = PER_WARP / 32;
  const int p0 = b * SCATTER_ENT + wid * PER_WARP;
  int ev[ROUNDS];
#pragma unroll
  for (int r = 0; r < ROUNDS; ++r) {
    const int p = p0 + r * 32 + lane;
    const int e = p < n_pairs ? __ldg(topk_id + p) : -1;
    ev[r] = (e >= 0 && e < E) ? e : -1;  // out-of-range ids were flagged when they were counted
  }
  if (qctr && b == 0 && tid == 0) {  // the grouped GEMMs' work-queue counters start the layer at zero
    qctr[0] = 0;
    qctr[1] = 0;
  }
  // the experts' offsets and first tiles: scans of the histogram
  int vo[4], vt[4], vt2[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int e = 4 * tid + i;
    const int c = e < E ? counts[e] : 0;
    vo[i] = c;
    vt[i] = (c + BN - 1) / BN;
    vt2[i] = (c + BN2 - 1) / BN2;
  }
  const int total = block_exscan4(vo, s_warp);
  const int routed_tiles = block_exscan4(vt, s_warp);
  const int routed_tiles2 = block_exscan4(vt2, s_warp);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int e = 4 * tid + i;
    if (e < E) {
      s_off[e] = vo[i];
      s_tb[e] = vt[i];
      s_tb2[e] = vt2[i];
    }
  }
  for (int i = tid; i < SCATTER_WARPS * E; i += SCATTER_THREADS) s_hist[i] = 0;
  __syncthreads();
  auto end_of = [&](int e) { return e + 1 < E ? s_off[e + 1] : total; };

  // block-map entries: expert e = b + i * gridDim.x goes to thread i
  auto write_map = [&](int32_t *map, int mt, int bn, const int *tbase) {
    for (int e = b + tid * gridDim.x; e < E; e += SCATTER_THREADS * gridDim.x) {
      const int o = s_off[e], ce = end_of(e) - o;
      for (int r = 0; r * bn < ce; ++r) {
        const int idx = tbase[e] + r;
        if (idx < mt) reinterpret_cast<int4 *>(map)[idx] = make_int4(e, o + r * bn, min(bn, ce - r * bn), 0);
      }
    }
  };
  auto write_shared = [&](int32_t *map, int32_t *nt, int mt, int bn, int rtiles) {
    const int shared_tiles = S ? (T + bn - 1) / bn : 0;
    if (tid == 0) {
      *nt = rtiles + shared_tiles;
      if (debug && (total != k * T || rtiles + shared_tiles > mt)) set_status(status, MOE_ERR_DEVICE_BOUNDS);
    }
    for (int s = tid; s < shared_tiles; s += SCATTER_THREADS) {
      const int idx = rtiles + s;
      if (idx < mt) reinterpret_cast<int4 *>(map)[idx] = make_int4(E, k * T + s * bn, min(bn, T - s * bn), 0);
    }
  };
  write_map(blockmap, max_tiles, BN, s_tb);
  if (blockmap2) write_map(blockmap2, max_tiles2, BN2, s_tb2);
  if (b == gridDim.x - 1) {
    write_shared(blockmap, n_tiles, max_tiles, BN, routed_tiles);
    if (blockmap2) write_shared(blockmap2, n_tiles2, max_tiles2, BN2, routed_tiles2);
  }
  if (b == 0)
    for (int e = tid; e <= E; e += SCATTER_THREADS) offsets[e] = e < E ? s_off[e] : total;

  int *hw = s_hist + wid * E;
  unsigned peers[ROUNDS];
#pragma unroll
  for (int r = 0; r < ROUNDS; ++r) {  // pass 1: pairs per expert and warp
    peers[r] = __match_any_sync(0xffffffffu, ev[r]);
    if (ev[r] >= 0 && lane == __ffs(peers[r]) - 1) hw[ev[r]] += __popc(peers[r]);
    __syncwarp();
  }
  __syncthreads();
  for (int e = tid; e < E; e += SCATTER_THREADS) {  // starts: the experts' pairs in earlier chunks and warps
    int run = s_off[e];
    for (int c0 = 0; c0 < b; c0 += 16) {  // earlier chunks' counts, sixteen loads in flight at a time
      int v[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) v[i] = c0 + i < b ? counts[(size_t)E + (size_t)(c0 + i) * E + e] : 0;
#pragma unroll
      for (int i = 0; i < 16; ++i) run += v[i];
    }
#pragma unroll
    for (int w = 0; w < SCATTER_WARPS; ++w) {
      const int x = s_hist[w * E + e];
      s_hist[w * E + e] = run;
      run += x;
    }
  }
  __syncthreads();
  const unsigned lt = (1u << lane) - 1u;
#pragma unroll
  for (int r = 0; r < ROUNDS; ++r) {  // pass 2: ranks in pair order
    const int e = ev[r];
    const int pos = e >= 0 ? hw[e] + __popc(peers[r] & lt) : 0;
    __syncwarp();
    if (e >= 0) {
      if (lane == __ffs(peers[r]) - 1) hw[e] += __popc(peers[r]);
      const int p = p0 + r * 32 + lane;
      if (pos < end_of(e)) {  // always checked: a stale histogram must not write out of bounds
        perm[pos] = p;
        inv[p] = pos;
      } else {
        set_status(status, MOE_ERR_DEVICE_BOUNDS);
      }
    }
    __syncwarp();
  }
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
                        int32_t *status, const float *part, int KS, const float *bias, bool after_kernel,
                        cudaStream_t s) {
  // a warp per token: eight tokens per block, or two when T is small (so
  // that small T still spreads over many SMs)
  const int tpb = T >= 1024 ? 8 : 2;
  const int blocks = (T + tpb - 1) / tpb;
  const int kpl = (E + 31) / 32;
  // a programmatic dependent of the router kernel (not of a memset)
  const bool pdl = after_kernel && prof_chain(MOE_KERNEL_TOPK);
  prof_before(MOE_KERNEL_TOPK, s);
  cudaError_t e = cudaSuccess;
#define MOE_TOPK(K)                                                                                               \
  e = launch_dep(pdl, topk_kernel<K>, dim3(blocks), dim3(32 * tpb), 0, s, keys, T, E, k, topk_id, topk_w, counts, \
                 status, part, KS, bias)
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
  return e != cudaSuccess ? e : cudaGetLastError();
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
  if (E > 4 * SCATTER_THREADS) return cudaErrorInvalidValue;
  const int blocks = (T * k + SCATTER_ENT - 1) / SCATTER_ENT;
  const size_t smem = (size_t)(SCATTER_WARPS + 3) * E * sizeof(int);
  const bool pdl = prof_chain(MOE_KERNEL_SCATTER);  // a dependent of the top-k or the ids histogram
  prof_before(MOE_KERNEL_SCATTER, s);
  const cudaError_t e = launch_dep(pdl, scatter_kernel, dim3(blocks), dim3(SCATTER_THREADS), smem, s, topk_id, T, E,
                                   k, BN, S, counts, offsets, perm, inv, blockmap, n_tiles, max_tiles, BN2, blockmap2,
                                   n_tiles2, max_tiles2, status, debug, qctr);
  prof_after(MOE_KERNEL_SCATTER, s);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace moe
