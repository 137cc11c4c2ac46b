// The C ABI (include/moe.h): plan, workspace layout, argument checks and the
// enqueue order of the layer's kernels.  Host code only; nothing here
// allocates device memory or synchronises (moe_device_status excepted).
#include <stdlib.h>
#include <string.h>

#include <new>
#include <algorithm>
#include <vector>

#include "common.cuh"
#include "kernels.h"
#include "tc.h"

namespace {

thread_local int32_t g_last_launches = 0;
thread_local cudaError_t g_last_cuda = cudaSuccess;

// Profiling hook state, per kernel id (moe_profile_events), per thread.
constexpr int kProfKernels = 16;
struct ProfState {
  int n = 0;
  int stride = 1;                   // bracket every stride-th launch
  unsigned long long seen = 0;      // launches of the kernel since the hook was set
  unsigned long long next = 0;
  cudaEvent_t start[4096];
  cudaEvent_t stop[4096];
  bool open = false;
};
thread_local ProfState *g_prof[kProfKernels] = {};

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

int tiles_bound(int T, int k, int E, int S, int BN) {
  // sum_e ceil(c_e / BN) <= k*T/BN + E, plus the shared expert's tiles
  return (k * T + BN - 1) / BN + E + (S ? (T + BN - 1) / BN : 0);
}

// The down GEMM's mode for T tokens (tensor-core plans), from the average
// rows per expert k T / E:
//   < 12: two output tiles per item, two items in flight, over the second
//         block map cut into short tiles (TC_SHORT_ROWS; T = 256: 66 -> 61
//         us; at T = 512 with skewed routing, 16 rows on average, the busiest
//         experts' many short tiles made it slower: 37 -> 39 us);
//   < 96: two output tiles per item over the first map, whose items share
//         their token rows (measured: T = 256 86 -> 66 us, T = 2048 94 -> 82
//         us against one tile per item);
//   else: one output tile per item over the second map's taller tiles, whose
//         two accumulators hide the epilogue (T = 4096: 105 us against 125).
int down_mode(const moe_plan_t *p, int T) {
  const int64_t kt = (int64_t)p->cfg.top_k * T, e = p->cfg.n_experts;
  if (!p->block_rows2) return moe::TC_DOWN_PAIR;
  if (kt < 12 * e) return moe::TC_DOWN_PAIR_SHORT;
  if (kt < 96 * e) return moe::TC_DOWN_PAIR;
  return moe::TC_DOWN_ONE;
}

// Tile height of the second block map for T tokens (0: no second map).
int block_rows2_at(const moe_plan_t *p, int T) {
  if (!p->block_rows2) return 0;
  return down_mode(p, T) == moe::TC_DOWN_PAIR_SHORT ? moe::TC_SHORT_ROWS : p->block_rows2;
}

// Tiles of the second block map a plan's workspace holds: enough for either height.
int max_tiles2_of(const moe_plan_t *p, int Tmax) {
  if (!p->block_rows2) return 0;
  const moe_config &c = p->cfg;
  int m = tiles_bound(Tmax, c.top_k, c.n_experts, c.n_shared, p->block_rows2);
  const int t_short = (int)std::min<int64_t>(Tmax, (12 * (int64_t)c.n_experts + c.top_k - 1) / c.top_k);
  return std::max(m, tiles_bound(t_short, c.top_k, c.n_experts, c.n_shared, moe::TC_SHORT_ROWS));
}

moe::Layout make_layout(const moe_config &c, int Tmax, int max_tiles, int max_tiles2, bool tc,
                        size_t rpart_floats = 0) {
  moe::Layout L;
  size_t o = 0;
  auto take = [&](size_t bytes) {
    size_t at = o;
    o = align_up(o + bytes, 256);
    return at;
  };
  const size_t E = c.n_experts, k = c.top_k, S = c.n_shared, H = c.hidden, I = c.inter, T = Tmax;
  L.status = take(64);
  L.counter = take(64);
  L.dtags = take(moe::decode_tag_words(c.hidden, c.n_experts, c.top_k, c.inter, c.n_shared) * 8);
  L.keys = take(T * E * 4);
  L.topk_id = take(T * k * 4);
  L.topk_w = take(T * k * 4);
  // the histogram, then one per chunk of SCATTER_ENT (token, slot) pairs (the scatter kernel's blocks)
  L.counts = take((1 + (k * T + moe::SCATTER_ENT - 1) / moe::SCATTER_ENT) * E * 4);
  L.offsets = take((E + 1) * 4);
  L.perm = take(k * T * 4);
  L.inv = take(k * T * 4);
  L.blockmap = take((size_t)max_tiles * 16);
  L.n_tiles = take(16);
  L.blockmap2 = take((size_t)max_tiles2 * 16);
  L.n_tiles2 = take(16);
  L.qctr = take(16);  // the grouped GEMMs' work-queue counters
  L.h = take((k + S) * T * I * 2);
  L.y = take((k + S) * T * H * 2);
  L.xg = take(tc ? (k + S) * T * H * 2 : 0);  // x rows gathered in block-map row order (tensor-core gate/up)
  L.rsplit = take(3 * E * H * 2);
  L.rpart = take(rpart_floats * 4);  // the tensor-core router's K-slice partial sums
  L.xn = take(T * H * 2);  // normalised x of pre-norm plans
  L.trace = take(MOE_TRACE_CTAS * MOE_TRACE_SLOTS * 8);
  L.total = o;
  return L;
}

moe::DecodeScratch decode_scratch(const moe_plan_t *plan, void *ws_d) {
  const moe::Layout &L = plan->lay;
  moe::DecodeScratch sc;
  sc.keys = moe::ws_ptr<float>(ws_d, L.keys);
  sc.topk_id = moe::ws_ptr<int32_t>(ws_d, L.topk_id);
  sc.topk_w = moe::ws_ptr<float>(ws_d, L.topk_w);
  sc.epoch = moe::ws_ptr<unsigned long long>(ws_d, L.counter);
  sc.tags = moe::ws_ptr<unsigned long long>(ws_d, L.dtags);
  sc.status = moe::ws_ptr<int32_t>(ws_d, L.status);
  sc.trace = (plan->flags & MOE_FLAG_TRACE) ? moe::ws_ptr<uint64_t>(ws_d, L.trace) : nullptr;
  if (plan->flags & MOE_FLAG_TEST_WITHHOLD) {  // one key is never published; waits give up after 1 ms
    sc.timeout_ns = 1000000ull;
    sc.withhold = 1;
  }
  return sc;
}

bool weights_aligned(const moe_weights *w) {
  using moe::aligned16;
  return aligned16(w->router_d) && aligned16(w->gate_q_d) && aligned16(w->up_q_d) && aligned16(w->gate_s_d) &&
         aligned16(w->gate_b_d) && aligned16(w->up_s_d) && aligned16(w->up_b_d) && aligned16(w->down_q_d) &&
         aligned16(w->down_s_d) && aligned16(w->down_b_d) && aligned16(w->shared_gate_d) &&
         aligned16(w->router_split_d);
}

bool weights_present(const moe_weights *w) {
  return w->router_d && w->gate_q_d && w->up_q_d && w->gate_s_d && w->gate_b_d && w->up_s_d && w->up_b_d &&
         w->down_q_d && w->down_s_d && w->down_b_d;
}

moe_status check_call(const moe_plan_t *p, int32_t T, const void *ws, size_t ws_bytes) {
  if (!p) return MOE_ERR_INVALID_ARGUMENT;
  if (T < 1) return MOE_ERR_INVALID_ARGUMENT;
  if (T > p->max_tokens) return MOE_ERR_TOO_MANY_TOKENS;
  if (!ws) return MOE_ERR_INVALID_ARGUMENT;
  if (!moe::aligned16(ws)) return MOE_ERR_MISALIGNED;
  if (ws_bytes < p->lay.total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  return MOE_OK;
}

// Checked after every argument check: no device means nothing can be enqueued.
moe_status device_ready(const moe_plan_t *p) { return p->num_sms > 0 ? MOE_OK : MOE_ERR_CUDA; }

moe_status cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return MOE_OK;
  g_last_cuda = e;
  return MOE_ERR_CUDA;
}

// How enqueue_route gets its selection: router keys from x, given keys
// already in the workspace, or given ids and weights already in the
// workspace's top-k buffers.
enum class RouteFrom { kX, kKeys, kIds };

// Routing kernels for T tokens.  split: the router's bf16 parts or null.
moe_status enqueue_route(const moe_plan_t *p, const uint16_t *x, int T, const float *router, const uint16_t *split,
                         const float *bias, void *ws, RouteFrom from, cudaStream_t s, int *launches) {
  const moe_config &c = p->cfg;
  const moe::Layout &L = p->lay;
  float *keys = moe::ws_ptr<float>(ws, L.keys);
  int32_t *status = moe::ws_ptr<int32_t>(ws, L.status);
  int32_t *counts = moe::ws_ptr<int32_t>(ws, L.counts);
  const size_t chunks = ((size_t)T * c.top_k + moe::SCATTER_ENT - 1) / moe::SCATTER_ENT;
  const int n_counts = (int)(c.n_experts * (1 + chunks));
  // the tensor-core router zeroes the histograms itself (no memset between
  // the kernels); every other path clears them here
  const bool tc_router = from == RouteFrom::kX && p->use_router_tc && T >= moe::ROUTER_TC_MIN_T;
  cudaError_t err = cudaSuccess;
  if (!tc_router && (err = cudaMemsetAsync(counts, 0, sizeof(int32_t) * n_counts, s)) != cudaSuccess)
    return cuda_status(err);
  const float *part = nullptr;  // the tensor-core router's K-slice partial sums, when it splits K
  int ks = 0;
  if (from == RouteFrom::kX) {
    if (tc_router) {
      err = moe::launch_router_tc(x, T, c.hidden, router, c.n_experts, bias, split,
                                  moe::ws_ptr<uint16_t>(ws, L.rsplit), moe::ws_ptr<float>(ws, L.rpart), keys, status,
                                  counts, n_counts, p->num_sms, &ks, launches, s);
      if (err != cudaSuccess) return cuda_status(err);
      if (ks > 1) part = moe::ws_ptr<float>(ws, L.rpart);
    } else {
      if ((err = moe::launch_router_logits(x, T, c.hidden, router, c.n_experts, bias, keys, s)) != cudaSuccess)
        return cuda_status(err);
      ++*launches;
    }
  }
  if (from == RouteFrom::kIds) {
    err = moe::launch_ids_histogram(moe::ws_ptr<int32_t>(ws, L.topk_id), T, c.n_experts, c.top_k, counts, status,
                                    (p->flags & MOE_FLAG_DEBUG_CHECKS) ? 1 : 0, s);
  } else {
    err = moe::launch_topk(keys, T, c.n_experts, c.top_k, moe::ws_ptr<int32_t>(ws, L.topk_id),
                           moe::ws_ptr<float>(ws, L.topk_w), counts, status, part, ks, part ? bias : nullptr,
                           from == RouteFrom::kX, s);
  }
  if (err != cudaSuccess) return cuda_status(err);
  ++*launches;
  const int max_tiles = tiles_bound(T, c.top_k, c.n_experts, c.n_shared, p->block_rows);
  const int bn2 = block_rows2_at(p, T);
  const int max_tiles2 = bn2 ? tiles_bound(T, c.top_k, c.n_experts, c.n_shared, bn2) : 0;
  if ((err = moe::launch_scatter(moe::ws_ptr<int32_t>(ws, L.topk_id), T, c.n_experts, c.top_k, p->block_rows,
                                 c.n_shared, counts, moe::ws_ptr<int32_t>(ws, L.offsets),
                                 moe::ws_ptr<int32_t>(ws, L.perm), moe::ws_ptr<int32_t>(ws, L.inv),
                                 moe::ws_ptr<int32_t>(ws, L.blockmap), moe::ws_ptr<int32_t>(ws, L.n_tiles), max_tiles,
                                 bn2, bn2 ? moe::ws_ptr<int32_t>(ws, L.blockmap2) : nullptr,
                                 moe::ws_ptr<int32_t>(ws, L.n_tiles2), max_tiles2, status,
                                 (p->flags & MOE_FLAG_DEBUG_CHECKS) ? 1 : 0, moe::ws_ptr<int32_t>(ws, L.qctr),
                                 s)) != cudaSuccess)
    return cuda_status(err);
  ++*launches;
  return MOE_OK;
}

moe::ExpertPtrs expert_ptrs(const moe_weights *w) {
  moe::ExpertPtrs e;
  e.gate_q = w->gate_q_d;
  e.up_q = w->up_q_d;
  e.down_q = w->down_q_d;
  e.gate_s = w->gate_s_d;
  e.gate_b = w->gate_b_d;
  e.up_s = w->up_s_d;
  e.up_b = w->up_b_d;
  e.down_s = w->down_s_d;
  e.down_b = w->down_b_d;
  e.shared_gate = w->shared_gate_d;
  return e;
}

}  // namespace

namespace moe {
moe_status note_cuda_error(cudaError_t e) { return cuda_status(e); }

// Inside a stream capture the records become external event-record nodes,
// which time like ordinary records when the graph runs.
static void prof_record(cudaEvent_t ev, cudaStream_t s) {
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  cudaStreamIsCapturing(s, &cap);
  if (cap == cudaStreamCaptureStatusActive)
    cudaEventRecordWithFlags(ev, s, cudaEventRecordExternal);
  else
    cudaEventRecord(ev, s);
}
void prof_before(int kernel, cudaStream_t s) {
  ProfState *p = (kernel > 0 && kernel < kProfKernels) ? g_prof[kernel] : nullptr;
  if (!p || p->n == 0) return;
  if (p->seen++ % (unsigned long long)p->stride) return;
  prof_record(p->start[p->next % p->n], s);
  p->open = true;
}
bool prof_quiet(int kernel) {
  const ProfState *p = (kernel > 0 && kernel < kProfKernels) ? g_prof[kernel] : nullptr;
  return !p || p->n == 0 || (p->seen % (unsigned long long)p->stride) != 0;
}
thread_local bool g_after_recorded = false;  // the last prof_after recorded an event
bool prof_chain(int kernel) { return !g_after_recorded && prof_quiet(kernel); }
void prof_after(int kernel, cudaStream_t s) {
  ProfState *p = (kernel > 0 && kernel < kProfKernels) ? g_prof[kernel] : nullptr;
  g_after_recorded = false;
  if (!p || p->n == 0 || !p->open) return;
  prof_record(p->stop[p->next % p->n], s);
  g_after_recorded = true;
  p->open = false;
  ++p->next;
}
}  // namespace moe

extern "C" {

moe_status moe_profile_events(int32_t kernel, void *const *start_events, void *const *stop_events, int32_t n) {
  if (kernel < MOE_KERNEL_ROUTER || kernel > MOE_KERNEL_ATTN_DECODE || n < 0 || n > 4096) return MOE_ERR_INVALID_ARGUMENT;
  if (n > 0 && (!start_events || !stop_events)) return MOE_ERR_INVALID_ARGUMENT;
  for (int i = 0; i < n; ++i)
    if (!start_events[i] || !stop_events[i]) return MOE_ERR_INVALID_ARGUMENT;
  ProfState *&p = g_prof[kernel];
  if (n == 0) {
    delete p;
    p = nullptr;
    return MOE_OK;
  }
  if (!p) p = new (std::nothrow) ProfState;
  if (!p) return MOE_ERR_INVALID_ARGUMENT;
  p->n = n;
  p->stride = 1;
  p->seen = 0;
  p->next = 0;
  p->open = false;
  for (int i = 0; i < n; ++i) {
    p->start[i] = static_cast<cudaEvent_t>(start_events[i]);
    p->stop[i] = static_cast<cudaEvent_t>(stop_events[i]);
  }
  return MOE_OK;
}

moe_status moe_profile_stride(int32_t kernel, int32_t stride) {
  if (kernel < MOE_KERNEL_ROUTER || kernel > MOE_KERNEL_ATTN_DECODE || stride < 1) return MOE_ERR_INVALID_ARGUMENT;
  ProfState *p = g_prof[kernel];
  if (!p) return MOE_ERR_INVALID_ARGUMENT;
  p->stride = stride;
  p->seen = 0;
  return MOE_OK;
}

const char *moe_status_str(moe_status s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARGUMENT: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported dimensions";
    case MOE_ERR_MISALIGNED: return "device pointer not 16-byte aligned";
    case MOE_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case MOE_ERR_TOO_MANY_TOKENS: return "T exceeds the plan's max_tokens";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_DEVICE_TIMEOUT: return "device wait timed out";
    case MOE_ERR_NONFINITE: return "non-finite router key";
    case MOE_ERR_DEVICE_BOUNDS: return "device bounds check failed";
  }
  return "unknown status";
}

moe_status moe_plan(const moe_config *cfg, int32_t max_tokens, uint32_t flags, moe_plan_t **out) {
  if (!cfg || !out) return MOE_ERR_INVALID_ARGUMENT;
  *out = nullptr;
  const uint32_t known = MOE_FLAG_DEBUG_CHECKS | MOE_FLAG_FORCE_GROUPED | MOE_FLAG_SIMT_EXPERTS |
                         MOE_FLAG_TILE_ROWS_64 | MOE_FLAG_PRENORM | MOE_FLAG_TRACE | MOE_FLAG_TEST_WITHHOLD;
  if (flags & ~known) return MOE_ERR_INVALID_ARGUMENT;
  if (max_tokens < 1 || max_tokens > 65536) return MOE_ERR_INVALID_ARGUMENT;
  const moe_config &c = *cfg;
  if (c.hidden <= 0 || c.n_experts <= 0 || c.top_k <= 0 || c.inter <= 0) return MOE_ERR_INVALID_ARGUMENT;
  if (c.hidden % 128 || c.inter % 64 || c.group_size != 64 || c.n_experts > 1024 || c.top_k > 16 ||
      c.top_k > c.n_experts || (c.n_shared != 0 && c.n_shared != 1) || c.hidden > 12288 || c.inter > 8192)
    return MOE_ERR_UNSUPPORTED;
  moe_plan_t *p = new (std::nothrow) moe_plan_t;
  if (!p) return MOE_ERR_INVALID_ARGUMENT;
  p->cfg = c;
  p->max_tokens = max_tokens;
  p->flags = flags;
  const bool simt = (flags & MOE_FLAG_SIMT_EXPERTS) != 0 || !moe::tc_supported(c);
  p->use_tc = !simt;
  p->block_rows = simt ? moe::SIMT_ROWS : ((flags & MOE_FLAG_TILE_ROWS_64) ? 64 : moe::TC_ROWS);
  p->max_tiles = tiles_bound(max_tokens, c.top_k, c.n_experts, c.n_shared, p->block_rows);
  // the tensor-core down GEMM takes tiles of up to TC_DOWN_ROWS rows
  p->block_rows2 = simt ? 0 : ((flags & MOE_FLAG_TILE_ROWS_64) ? 64 : moe::TC_DOWN_ROWS);
  p->max_tiles2 = max_tiles2_of(p, max_tokens);
  p->lay = make_layout(c, max_tokens, p->max_tiles, p->max_tiles2, !simt);
  p->num_sms = 0;
  p->use_router_tc = false;
  p->use_decode = false;
  int dev = 0, count = 0;
  if (cudaGetDeviceCount(&count) == cudaSuccess && count > 0 && cudaGetDevice(&dev) == cudaSuccess) {
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, dev) == cudaSuccess) p->num_sms = prop.multiProcessorCount;
    if (p->use_tc && p->num_sms > 0 && moe::tc_prepare() != cudaSuccess) {
      cudaGetLastError();
      p->use_tc = false;  // no tensor-core kernels on this device: CUDA-core path
      p->block_rows = moe::SIMT_ROWS;
      p->max_tiles = tiles_bound(max_tokens, c.top_k, c.n_experts, c.n_shared, p->block_rows);
      p->block_rows2 = 0;
      p->max_tiles2 = 0;
      p->lay = make_layout(c, max_tokens, p->max_tiles, p->max_tiles2, false);
    }
    if (p->num_sms > 0 &&
        moe::decode_supported(c.hidden, c.n_experts, c.top_k, c.inter, c.n_shared, p->num_sms)) {
      p->use_decode =
          moe::decode_prepare(c.hidden, c.n_experts, c.top_k, c.inter, c.n_shared, p->num_sms) == cudaSuccess;
      if (!p->use_decode) cudaGetLastError();
    }
    if (p->num_sms > 0 && moe::router_tc_supported(c.n_experts, c.hidden)) {
      p->use_router_tc = moe::router_tc_prepare() == cudaSuccess;
      if (!p->use_router_tc) cudaGetLastError();
      if (p->use_router_tc)  // room for its K-slice partial sums
        p->lay = make_layout(c, max_tokens, p->max_tiles, p->max_tiles2, p->use_tc,
                             moe::router_tc_partial_floats(max_tokens, c.n_experts, c.hidden, p->num_sms));
    }
  } else {
    cudaGetLastError();  // no device: host-side checks still work, launches report MOE_ERR_CUDA
  }
  *out = p;
  return MOE_OK;
}

void moe_plan_destroy(moe_plan_t *plan) { delete plan; }

size_t moe_workspace_bytes(const moe_plan_t *plan) { return plan ? plan->lay.total : 0; }

moe_status moe_workspace_init(const moe_plan_t *plan, void *ws_d, size_t ws_bytes, void *stream) {
  if (!plan || !ws_d) return MOE_ERR_INVALID_ARGUMENT;
  if (!moe::aligned16(ws_d)) return MOE_ERR_MISALIGNED;
  if (ws_bytes < plan->lay.total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  if (device_ready(plan) != MOE_OK) return MOE_ERR_CUDA;
  // status, the decode epoch counter and its tagged words
  return cuda_status(cudaMemsetAsync(ws_d, 0, plan->lay.keys, static_cast<cudaStream_t>(stream)));
}

moe_status moe_route(const moe_plan_t *plan, const void *x_d, int32_t T, const float *router_d,
                     const float *logit_bias_d, void *ws_d, size_t ws_bytes, void *stream) {
  g_last_launches = 0;
  moe_status st = check_call(plan, T, ws_d, ws_bytes);
  if (st != MOE_OK) return st;
  if (!x_d || !router_d) return MOE_ERR_INVALID_ARGUMENT;
  if (!moe::aligned16(x_d) || !moe::aligned16(router_d) || !moe::aligned16(logit_bias_d))
    return MOE_ERR_MISALIGNED;
  if ((st = device_ready(plan)) != MOE_OK) return st;
  int launches = 0;
  st = enqueue_route(plan, static_cast<const uint16_t *>(x_d), T, router_d, nullptr, logit_bias_d, ws_d,
                     RouteFrom::kX, static_cast<cudaStream_t>(stream), &launches);
  g_last_launches = launches;
  return st;
}

moe_status moe_route_from_logits(const moe_plan_t *plan, const float *keys_d, int32_t T, void *ws_d,
                                 size_t ws_bytes, void *stream) {
  g_last_launches = 0;
  moe_status st = check_call(plan, T, ws_d, ws_bytes);
  if (st != MOE_OK) return st;
  if (!keys_d) return MOE_ERR_INVALID_ARGUMENT;
  if (!moe::aligned16(keys_d)) return MOE_ERR_MISALIGNED;
  if ((st = device_ready(plan)) != MOE_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  float *keys = moe::ws_ptr<float>(ws_d, plan->lay.keys);
  if (keys != keys_d) {
    cudaError_t err =
        cudaMemcpyAsync(keys, keys_d, sizeof(float) * (size_t)T * plan->cfg.n_experts, cudaMemcpyDeviceToDevice, s);
    if (err != cudaSuccess) return cuda_status(err);
  }
  int launches = 0;
  st = enqueue_route(plan, nullptr, T, nullptr, nullptr, nullptr, ws_d, RouteFrom::kKeys, s, &launches);
  g_last_launches = launches;
  return st;
}

moe_status moe_route_from_ids(const moe_plan_t *plan, const int32_t *ids_d, const float *w_d, int32_t T, void *ws_d,
                              size_t ws_bytes, void *stream) {
  g_last_launches = 0;
  moe_status st = check_call(plan, T, ws_d, ws_bytes);
  if (st != MOE_OK) return st;
  if (!ids_d || !w_d) return MOE_ERR_INVALID_ARGUMENT;
  if (!moe::aligned16(ids_d) || !moe::aligned16(w_d)) return MOE_ERR_MISALIGNED;
  if ((st = device_ready(plan)) != MOE_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t n = (size_t)T * plan->cfg.top_k;
  int32_t *ids = moe::ws_ptr<int32_t>(ws_d, plan->lay.topk_id);
  float *w = moe::ws_ptr<float>(ws_d, plan->lay.topk_w);
  cudaError_t err = cudaSuccess;
  if (ids != ids_d) err = cudaMemcpyAsync(ids, ids_d, n * sizeof(int32_t), cudaMemcpyDeviceToDevice, s);
  if (err == cudaSuccess && w != w_d) err = cudaMemcpyAsync(w, w_d, n * sizeof(float), cudaMemcpyDeviceToDevice, s);
  if (err != cudaSuccess) return cuda_status(err);
  int launches = 0;
  st = enqueue_route(plan, nullptr, T, nullptr, nullptr, nullptr, ws_d, RouteFrom::kIds, s, &launches);
  g_last_launches = launches;
  return st;
}

// One layer.  For the chunk loop of pre-norm stacks (grouped path only):
// norm_in -- the workspace's normalised x already holds RMSNorm(x_d) (the
// previous layer's combine wrote it), so the norm kernel is skipped;
// norm_out -- the combine also writes RMSNorm(out) there for the next layer.
static moe_status forward_impl(const moe_plan_t *plan, const void *x_d, const void *residual_d, int32_t T,
                               const moe_weights *w, const float *logit_bias_d, void *out_d, void *ws_d,
                               size_t ws_bytes, void *stream, bool norm_in, bool norm_out) {
  g_last_launches = 0;
  moe_status st = check_call(plan, T, ws_d, ws_bytes);
  if (st != MOE_OK) return st;
  const bool prenorm = (plan->flags & MOE_FLAG_PRENORM) != 0;
  if (!x_d || !w || !out_d || !weights_present(w)) return MOE_ERR_INVALID_ARGUMENT;
  if (out_d == x_d && !prenorm) return MOE_ERR_INVALID_ARGUMENT;
  if (prenorm && residual_d) return MOE_ERR_INVALID_ARGUMENT;
  if (!moe::aligned16(x_d) || !moe::aligned16(residual_d) || !moe::aligned16(out_d) ||
      !moe::aligned16(logit_bias_d) || !weights_aligned(w))
    return MOE_ERR_MISALIGNED;
  if ((st = device_ready(plan)) != MOE_OK) return st;
  const moe_config &c = plan->cfg;
  const moe::Layout &L = plan->lay;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const uint16_t *x = static_cast<const uint16_t *>(x_d);
  const uint16_t *res = residual_d ? static_cast<const uint16_t *>(residual_d) : x;
  uint16_t *out = static_cast<uint16_t *>(out_d);
  const moe::ExpertPtrs ep = expert_ptrs(w);
  int32_t *status = moe::ws_ptr<int32_t>(ws_d, L.status);
  int launches = 0;

  if (T == 1 && plan->use_decode && !(plan->flags & MOE_FLAG_FORCE_GROUPED)) {
    cudaError_t err = moe::launch_decode(x, res, c.hidden, c.n_experts, c.top_k, c.inter, c.n_shared,
                                         prenorm ? 1 : 0, 1e-6f, w->router_d, logit_bias_d, ep, out,
                                         decode_scratch(plan, ws_d), plan->num_sms, &launches, s);
    g_last_launches = launches;
    return cuda_status(err);
  }

  uint16_t *xnorm_next = nullptr;
  if (prenorm) {  // x = RMSNorm(r) into the workspace; the residual is r
    uint16_t *xn = moe::ws_ptr<uint16_t>(ws_d, L.xn);
    if (!norm_in) {
      cudaError_t err = moe::launch_rmsnorm(x, T, c.hidden, 1e-6f, xn, s);
      if (err != cudaSuccess) return cuda_status(err);
      ++launches;
    }
    x = xn;
    if (norm_out) xnorm_next = xn;
  }
  st = enqueue_route(plan, x, T, w->router_d, w->router_split_d, logit_bias_d, ws_d, RouteFrom::kX, s, &launches);
  if (st != MOE_OK) return st;
  const int max_tiles = tiles_bound(T, c.top_k, c.n_experts, c.n_shared, plan->block_rows);
  const int32_t *perm = moe::ws_ptr<int32_t>(ws_d, L.perm);
  const int32_t *bm = moe::ws_ptr<int32_t>(ws_d, L.blockmap);
  const int32_t *nt = moe::ws_ptr<int32_t>(ws_d, L.n_tiles);
  uint16_t *h = moe::ws_ptr<uint16_t>(ws_d, L.h);
  uint16_t *y = moe::ws_ptr<uint16_t>(ws_d, L.y);
  cudaError_t err;
  if (!plan->use_tc) {
    err = moe::launch_gateup_simt(x, T, c.hidden, c.inter, c.n_experts, c.top_k, perm, bm, nt, max_tiles, ep, h, s);
    if (err != cudaSuccess) return cuda_status(err);
    err = moe::launch_down_simt(h, T, c.hidden, c.inter, c.n_experts, c.top_k, bm, nt, max_tiles, ep, y, s);
    if (err != cudaSuccess) return cuda_status(err);
    launches += 2;
  } else {
    const int bn2 = block_rows2_at(plan, T);
    const int max_tiles2 = bn2 ? tiles_bound(T, c.top_k, c.n_experts, c.n_shared, bn2) : 0;
    err = moe::launch_experts_tc(plan, x, T, perm, bm, nt, max_tiles, down_mode(plan, T),
                                 moe::ws_ptr<int32_t>(ws_d, L.blockmap2), moe::ws_ptr<int32_t>(ws_d, L.n_tiles2),
                                 max_tiles2, ep, h, y,
                                 moe::ws_ptr<uint16_t>(ws_d, L.xg), moe::ws_ptr<int32_t>(ws_d, L.qctr),
                                 status,
                                 (plan->flags & MOE_FLAG_TRACE) ? moe::ws_ptr<uint64_t>(ws_d, L.trace) : nullptr,
                                 &launches, s);
    if (err != cudaSuccess) return cuda_status(err);
  }
  err = moe::launch_combine(res, y, moe::ws_ptr<int32_t>(ws_d, L.inv), moe::ws_ptr<float>(ws_d, L.topk_w), x,
                            ep.shared_gate, T, c.hidden, c.top_k, c.n_shared, out, xnorm_next, 1e-6f, s);
  if (err != cudaSuccess) return cuda_status(err);
  ++launches;
  g_last_launches = launches;
  return MOE_OK;
}

moe_status moe_forward(const moe_plan_t *plan, const void *x_d, const void *residual_d, int32_t T,
                       const moe_weights *w, const float *logit_bias_d, void *out_d, void *ws_d, size_t ws_bytes,
                       void *stream) {
  return forward_impl(plan, x_d, residual_d, T, w, logit_bias_d, out_d, ws_d, ws_bytes, stream, false, false);
}

moe_status moe_decode_stack(const moe_plan_t *plan, void *r_d, int32_t n_layers, const moe_weights *w,
                            const float *const *logit_bias_d, void *ws_d, size_t ws_bytes, void *stream) {
  g_last_launches = 0;
  moe_status st = check_call(plan, 1, ws_d, ws_bytes);
  if (st != MOE_OK) return st;
  if (!r_d || !w || n_layers < 1) return MOE_ERR_INVALID_ARGUMENT;
  if (!moe::aligned16(r_d)) return MOE_ERR_MISALIGNED;
  for (int l = 0; l < n_layers; ++l) {
    if (!weights_present(&w[l])) return MOE_ERR_INVALID_ARGUMENT;
    if (!weights_aligned(&w[l]) || (logit_bias_d && !moe::aligned16(logit_bias_d[l]))) return MOE_ERR_MISALIGNED;
  }
  if ((st = device_ready(plan)) != MOE_OK) return st;
  if (!plan->use_decode) return MOE_ERR_UNSUPPORTED;
  const moe_config &c = plan->cfg;
  const moe::Layout &L = plan->lay;
  std::vector<const float *> router(n_layers);
  std::vector<moe::ExpertPtrs> ep(n_layers);
  for (int l = 0; l < n_layers; ++l) {
    router[l] = w[l].router_d;
    ep[l] = expert_ptrs(&w[l]);
  }
  int launches = 0;
  const cudaError_t err = moe::launch_decode_stack(
      static_cast<uint16_t *>(r_d), n_layers, c.hidden, c.n_experts, c.top_k, c.inter, c.n_shared, 1e-6f,
      router.data(), logit_bias_d, ep.data(), decode_scratch(plan, ws_d), plan->num_sms, &launches,
      static_cast<cudaStream_t>(stream));
  g_last_launches = launches;
  return cuda_status(err);
}

moe_status moe_prefill_stack(const moe_plan_t *plan, void *r_d, int32_t T, int32_t n_layers, const moe_weights *w,
                             const float *const *logit_bias_d, void *ws_d, size_t ws_bytes, void *stream) {
  g_last_launches = 0;
  if (!plan || !r_d || !w || n_layers < 1 || T < 1) return MOE_ERR_INVALID_ARGUMENT;
  if (!(plan->flags & MOE_FLAG_PRENORM)) return MOE_ERR_INVALID_ARGUMENT;
  moe_status st = check_call(plan, 1, ws_d, ws_bytes);
  if (st != MOE_OK) return st;
  if (!moe::aligned16(r_d)) return MOE_ERR_MISALIGNED;
  for (int l = 0; l < n_layers; ++l) {
    if (!weights_present(&w[l])) return MOE_ERR_INVALID_ARGUMENT;
    if (!weights_aligned(&w[l]) || (logit_bias_d && !moe::aligned16(logit_bias_d[l]))) return MOE_ERR_MISALIGNED;
  }
  if ((st = device_ready(plan)) != MOE_OK) return st;
  const size_t H = plan->cfg.hidden;
  const int m = plan->max_tokens;
  uint16_t *r = static_cast<uint16_t *>(r_d);
  int launches = 0;
  for (int c0 = 0; c0 < T; c0 += m) {  // chunk-major: each chunk through every layer
    const int n = T - c0 < m ? T - c0 : m;
    uint16_t *rc = r + (size_t)c0 * H;
    // on the grouped path each layer's combine also normalises its output
    // for the next layer (bit for bit the norm kernel's result)
    const bool grouped = !(n == 1 && plan->use_decode && !(plan->flags & MOE_FLAG_FORCE_GROUPED));
    for (int l = 0; l < n_layers; ++l) {
      st = forward_impl(plan, rc, nullptr, n, &w[l], logit_bias_d ? logit_bias_d[l] : nullptr, rc, ws_d, ws_bytes,
                        stream, grouped && l > 0, grouped && l + 1 < n_layers);
      launches += g_last_launches;
      if (st != MOE_OK) {
        g_last_launches = launches;
        return st;
      }
    }
  }
  g_last_launches = launches;
  return MOE_OK;
}

size_t moe_router_split_bytes(int32_t E, int32_t H) {
  return (E > 0 && H > 0) ? (size_t)3 * (size_t)E * (size_t)H * 2 : 0;
}

moe_status moe_router_split(const float *router_d, int32_t E, int32_t H, void *split_d, size_t split_bytes,
                            void *stream) {
  g_last_launches = 0;
  if (!router_d || !split_d || E < 1 || H < 1 || ((size_t)E * H) % 4) return MOE_ERR_INVALID_ARGUMENT;
  if (!moe::aligned16(router_d) || !moe::aligned16(split_d)) return MOE_ERR_MISALIGNED;
  if (split_bytes < moe_router_split_bytes(E, H)) return MOE_ERR_WORKSPACE_TOO_SMALL;
  cudaError_t err = moe::launch_router_split(router_d, E, H, static_cast<uint16_t *>(split_d),
                                             static_cast<cudaStream_t>(stream));
  g_last_launches = 1;
  return cuda_status(err);
}

moe_status moe_route_view(const moe_plan_t *plan, void *ws_d, int32_t T, moe_route_ptrs *out) {
  if (!plan || !ws_d || !out) return MOE_ERR_INVALID_ARGUMENT;
  if (T < 1) return MOE_ERR_INVALID_ARGUMENT;
  if (T > plan->max_tokens) return MOE_ERR_TOO_MANY_TOKENS;
  const moe::Layout &L = plan->lay;
  out->keys_d = moe::ws_ptr<float>(ws_d, L.keys);
  out->topk_id_d = moe::ws_ptr<int32_t>(ws_d, L.topk_id);
  out->topk_w_d = moe::ws_ptr<float>(ws_d, L.topk_w);
  out->counts_d = moe::ws_ptr<int32_t>(ws_d, L.counts);
  out->offsets_d = moe::ws_ptr<int32_t>(ws_d, L.offsets);
  out->perm_d = moe::ws_ptr<int32_t>(ws_d, L.perm);
  out->inv_d = moe::ws_ptr<int32_t>(ws_d, L.inv);
  out->blockmap_d = moe::ws_ptr<int32_t>(ws_d, L.blockmap);
  out->n_tiles_d = moe::ws_ptr<int32_t>(ws_d, L.n_tiles);
  out->h_d = moe::ws_ptr<uint16_t>(ws_d, L.h);
  out->y_d = moe::ws_ptr<uint16_t>(ws_d, L.y);
  out->status_d = moe::ws_ptr<int32_t>(ws_d, L.status);
  out->trace_d = moe::ws_ptr<uint64_t>(ws_d, L.trace);
  out->max_tiles = tiles_bound(T, plan->cfg.top_k, plan->cfg.n_experts, plan->cfg.n_shared, plan->block_rows);
  out->block_rows = plan->block_rows;
  out->blockmap2_d = moe::ws_ptr<int32_t>(ws_d, L.blockmap2);
  out->n_tiles2_d = moe::ws_ptr<int32_t>(ws_d, L.n_tiles2);
  const int bn2 = block_rows2_at(plan, T);
  out->max_tiles2 = bn2 ? tiles_bound(T, plan->cfg.top_k, plan->cfg.n_experts, plan->cfg.n_shared, bn2) : 0;
  out->block_rows2 = bn2;
  return MOE_OK;
}

moe_status moe_rmsnorm(const void *r_d, int32_t T, int32_t H, float eps, void *x_d, void *stream) {
  g_last_launches = 0;
  if (!r_d || !x_d || T < 1 || H < 8 || H % 8 || !(eps >= 0.f)) return MOE_ERR_INVALID_ARGUMENT;
  if (r_d == x_d) return MOE_ERR_INVALID_ARGUMENT;
  if (!moe::aligned16(r_d) || !moe::aligned16(x_d)) return MOE_ERR_MISALIGNED;
  cudaError_t err = moe::launch_rmsnorm(static_cast<const uint16_t *>(r_d), T, H, eps, static_cast<uint16_t *>(x_d),
                                        static_cast<cudaStream_t>(stream));
  g_last_launches = 1;
  return cuda_status(err);
}

moe_status moe_dequant(const uint32_t *q_d, const uint16_t *s_d, const uint16_t *b_d, int32_t rows, int32_t K,
                       int32_t G, void *w_d, void *stream) {
  g_last_launches = 0;
  if (!q_d || !s_d || !b_d || !w_d || rows < 1 || K < 8) return MOE_ERR_INVALID_ARGUMENT;
  if (G != 64 || K % G) return MOE_ERR_UNSUPPORTED;
  if (!moe::aligned16(q_d) || !moe::aligned16(w_d)) return MOE_ERR_MISALIGNED;
  cudaError_t err = moe::launch_dequant(q_d, s_d, b_d, rows, K, G, static_cast<uint16_t *>(w_d),
                                        static_cast<cudaStream_t>(stream));
  g_last_launches = 1;
  return cuda_status(err);
}

moe_status moe_device_status(const moe_plan_t *plan, void *ws_d, void *stream, int32_t *host_status,
                             int32_t reset) {
  if (!plan || !ws_d || !host_status) return MOE_ERR_INVALID_ARGUMENT;
  if (!moe::aligned16(ws_d)) return MOE_ERR_MISALIGNED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t *status = moe::ws_ptr<int32_t>(ws_d, plan->lay.status);
  cudaError_t err = cudaMemcpyAsync(host_status, status, sizeof(int32_t), cudaMemcpyDeviceToHost, s);
  if (err == cudaSuccess && reset) err = cudaMemsetAsync(status, 0, sizeof(int32_t), s);
  if (err == cudaSuccess) err = cudaStreamSynchronize(s);
  return cuda_status(err);
}

int32_t moe_last_launch_count(void) { return g_last_launches; }

const char *moe_last_cuda_error(void) { return cudaGetErrorString(g_last_cuda); }

}  // extern "C"
