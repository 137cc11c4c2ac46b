// moe_decode_static: the single-token layer of moe_forward's decode path for
// callers that cannot allocate device memory.  Its scratch -- the status
// word, the decode epoch counter, the tagged exchange words, the router keys
// and the top-k ids and weights -- lives in one file-scope __device__ array
// instead of a caller-allocated workspace.
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace {

constexpr int kMaxDevices = 64;

// Every device that loads the library holds this array until the process
// exits.  In host code the symbol is only a stand-in: its device address comes
// from cudaGetSymbolAddress, taken once per device with that device current.
__device__ __align__(256) uint8_t g_decode_scratch[MOE_DECODE_STATIC_SCRATCH_BYTES];

// Byte offsets inside the array (256-byte aligned).
constexpr size_t kStatus = 0, kCounter = 64, kTags = 256;
constexpr size_t al256(size_t v) { return (v + 255) / 256 * 256; }

struct Scratch {
  size_t tag_bytes, keys, topk_id, topk_w, total;
};

Scratch scratch_layout(const moe_config &c) {
  Scratch s;
  s.tag_bytes = moe::decode_tag_words(c.hidden, c.n_experts, c.top_k, c.inter, c.n_shared) * 8;
  s.keys = al256(kTags + s.tag_bytes);
  s.topk_id = al256(s.keys + (size_t)c.n_experts * 4);
  s.topk_w = al256(s.topk_id + (size_t)c.top_k * 4);
  s.total = s.topk_w + (size_t)c.top_k * 4;
  return s;
}

struct DeviceState {
  bool ready = false;
  uint8_t *scratch = nullptr;  // device address of g_decode_scratch on this device
  int num_sms = 0;
  moe_config last{};  // dimensions of the previous call: its tagged words lie in another layout
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];

// First call on a device: resolve the array's address, read the SM count and
// raise the decode kernel's shared-memory opt-in.  Later calls only read.
moe_status device_setup(DeviceState **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return moe::note_cuda_error(e);
  if (dev < 0 || dev >= kMaxDevices) return MOE_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState &d = g_dev[dev];
  if (!d.ready) {
    void *ptr = nullptr;
    if ((e = cudaGetSymbolAddress(&ptr, g_decode_scratch)) != cudaSuccess) return moe::note_cuda_error(e);
    int sms = 0;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return moe::note_cuda_error(e);
    // the opt-in is set to the device maximum, whatever the layer's shape
    if ((e = moe::decode_prepare(0, 0, 0, 0, 0, sms)) != cudaSuccess) return moe::note_cuda_error(e);
    d.scratch = static_cast<uint8_t *>(ptr);
    d.num_sms = sms;
    d.ready = true;
  }
  *out = &d;
  return MOE_OK;
}

bool present(const moe_weights *w) {
  return w->router_d && w->gate_q_d && w->up_q_d && w->gate_s_d && w->gate_b_d && w->up_s_d && w->up_b_d &&
         w->down_q_d && w->down_s_d && w->down_b_d;
}

bool aligned(const moe_weights *w) {
  using moe::aligned16;
  return aligned16(w->router_d) && aligned16(w->gate_q_d) && aligned16(w->up_q_d) && aligned16(w->gate_s_d) &&
         aligned16(w->gate_b_d) && aligned16(w->up_s_d) && aligned16(w->up_b_d) && aligned16(w->down_q_d) &&
         aligned16(w->down_s_d) && aligned16(w->down_b_d) && aligned16(w->shared_gate_d);
}

}  // namespace

extern "C" moe_status moe_decode_static(const moe_config *cfg, const void *x_d, const void *residual_d,
                                        const moe_weights *w, const float *logit_bias_d, void *out_d,
                                        int32_t *status_d, uint32_t flags, void *stream) {
  if (!cfg || !x_d || !w || !out_d || !present(w)) return MOE_ERR_INVALID_ARGUMENT;
  if (flags & ~MOE_FLAG_PRENORM) return MOE_ERR_INVALID_ARGUMENT;
  const bool prenorm = (flags & MOE_FLAG_PRENORM) != 0;
  if (out_d == x_d && !prenorm) return MOE_ERR_INVALID_ARGUMENT;
  if (prenorm && residual_d) return MOE_ERR_INVALID_ARGUMENT;
  const moe_config &c = *cfg;
  if (c.hidden <= 0 || c.n_experts <= 0 || c.top_k <= 0 || c.inter <= 0) return MOE_ERR_INVALID_ARGUMENT;
  if (c.hidden % 128 || c.inter % 64 || c.group_size != 64 || c.n_experts > 1024 || c.top_k > 16 ||
      c.top_k > c.n_experts || (c.n_shared != 0 && c.n_shared != 1) || c.hidden > 12288 || c.inter > 8192)
    return MOE_ERR_UNSUPPORTED;
  const Scratch L = scratch_layout(c);
  if (L.total > MOE_DECODE_STATIC_SCRATCH_BYTES) return MOE_ERR_WORKSPACE_TOO_SMALL;
  if (!moe::aligned16(x_d) || !moe::aligned16(residual_d) || !moe::aligned16(out_d) ||
      !moe::aligned16(logit_bias_d) || !aligned(w) || (reinterpret_cast<uintptr_t>(status_d) & 3))
    return MOE_ERR_MISALIGNED;

  DeviceState *d = nullptr;
  moe_status st = device_setup(&d);
  if (st != MOE_OK) return st;
  if (!moe::decode_supported(c.hidden, c.n_experts, c.top_k, c.inter, c.n_shared, d->num_sms))
    return MOE_ERR_UNSUPPORTED;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // The array keeps the previous call's contents (zero before the first).
  // The status word starts at zero; the epoch counter and the tagged words
  // carry over from call to call, except that the words are cleared when the
  // dimensions change (a word of the old layout must not pass for the new);
  // keys and top-k are rewritten in full.
  bool same;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    same = std::memcmp(&d->last, &c, sizeof c) == 0;
    d->last = c;
  }
  cudaError_t e = cudaMemsetAsync(d->scratch + kStatus, 0, 64, s);
  if (e == cudaSuccess && !same) e = cudaMemsetAsync(d->scratch + kTags, 0, L.tag_bytes, s);
  if (e == cudaSuccess && status_d) e = cudaMemsetAsync(status_d, 0, sizeof(int32_t), s);
  if (e != cudaSuccess) return moe::note_cuda_error(e);

  moe::ExpertPtrs ep;
  ep.gate_q = w->gate_q_d;
  ep.up_q = w->up_q_d;
  ep.down_q = w->down_q_d;
  ep.gate_s = w->gate_s_d;
  ep.gate_b = w->gate_b_d;
  ep.up_s = w->up_s_d;
  ep.up_b = w->up_b_d;
  ep.down_s = w->down_s_d;
  ep.down_b = w->down_b_d;
  ep.shared_gate = w->shared_gate_d;
  const uint16_t *x = static_cast<const uint16_t *>(x_d);
  const uint16_t *res = residual_d ? static_cast<const uint16_t *>(residual_d) : x;
  uint8_t *sc = d->scratch;
  int32_t *status = status_d ? status_d : reinterpret_cast<int32_t *>(sc + kStatus);
  moe::DecodeScratch ds;
  ds.keys = reinterpret_cast<float *>(sc + L.keys);
  ds.topk_id = reinterpret_cast<int32_t *>(sc + L.topk_id);
  ds.topk_w = reinterpret_cast<float *>(sc + L.topk_w);
  ds.epoch = reinterpret_cast<unsigned long long *>(sc + kCounter);
  ds.tags = reinterpret_cast<unsigned long long *>(sc + kTags);
  ds.status = status;
  ds.trace = nullptr;
  int launches = 0;
  e = moe::launch_decode(x, res, c.hidden, c.n_experts, c.top_k, c.inter, c.n_shared, prenorm ? 1 : 0, 1e-6f,
                         w->router_d, logit_bias_d, ep, static_cast<uint16_t *>(out_d), ds, d->num_sms, &launches,
                         s);
  return e == cudaSuccess ? MOE_OK : moe::note_cuda_error(e);
}
