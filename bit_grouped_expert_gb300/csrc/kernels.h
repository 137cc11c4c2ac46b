// Launchers of libmoe.so's kernels (host declarations, one place).
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include "moe.h"

namespace moe {

// Records e as the calling thread's last CUDA error (moe_last_cuda_error)
// and returns MOE_ERR_CUDA, or MOE_OK for cudaSuccess.
moe_status note_cuda_error(cudaError_t e);

// Profiling hook (moe_profile_events): record events around a kernel launch.
void prof_before(int kernel, cudaStream_t s);
void prof_after(int kernel, cudaStream_t s);
// true when the kernel's next launch records no timing event (a launch that
// follows another kernel directly may then start as its programmatic dependent)
bool prof_quiet(int kernel);
// true when no timing event was recorded after the last kernel and none will
// be recorded before this one: the launch may start as a programmatic
// dependent of the kernel before it
bool prof_chain(int kernel);

// Launch of kernel(args...); with pdl, as a programmatic dependent of the
// previous kernel in the stream (the kernel waits for it with
// griddepcontrol.wait before touching its outputs); a plain launch where the
// attribute is refused.
template <typename... P, typename... A>
cudaError_t launch_dep(bool pdl, void (*kernel)(P...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       A... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = pdl ? 1 : 0;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, args...);
  if (e != cudaSuccess && pdl) {
    cudaGetLastError();
    cfg.numAttrs = 0;
    e = cudaLaunchKernelEx(&cfg, kernel, args...);
  }
  return e;
}

// Every member starts null: a pointer a caller leaves unset reads as absent.
struct ExpertPtrs {
  const uint32_t *gate_q = nullptr, *up_q = nullptr, *down_q = nullptr;
  const uint16_t *gate_s = nullptr, *gate_b = nullptr, *up_s = nullptr, *up_b = nullptr, *down_s = nullptr,
                 *down_b = nullptr;
  const float *shared_gate = nullptr;  // [H] fp32 or null: the shared expert's output is scaled by sigmoid(x . gate)
};

// route.cu
cudaError_t launch_router_logits(const uint16_t *x, int T, int H, const float *router, int E, const float *bias,
                                 float *keys, cudaStream_t s);
// part: null (keys given) or the router's KS K-slice partial sums [KS][T][E],
// summed in slice order (+ bias) into keys before the selection.
// after_kernel: the launch directly follows the router kernel in the stream
// (it may then start as that kernel's programmatic dependent).
cudaError_t launch_topk(float *keys, int T, int E, int k, int32_t *topk_id, float *topk_w, int32_t *counts,
                        int32_t *status, const float *part, int KS, const float *bias, bool after_kernel,
                        cudaStream_t s);
// counts[e] += 1 for every given id (ids [T][k]); out-of-range ids (and, with
// debug, an expert repeated within a token) set MOE_ERR_DEVICE_BOUNDS.
cudaError_t launch_ids_histogram(const int32_t *ids, int T, int E, int k, int32_t *counts, int32_t *status, int debug,
                                 cudaStream_t s);
cudaError_t launch_scatter(const int32_t *topk_id, int T, int E, int k, int BN, int S, const int32_t *counts,
                           int32_t *offsets, int32_t *perm, int32_t *inv, int32_t *blockmap, int32_t *n_tiles,
                           int max_tiles, int BN2, int32_t *blockmap2, int32_t *n_tiles2, int max_tiles2,
                           int32_t *status, int debug, int32_t *qctr, cudaStream_t s);

// experts_simt.cu (CUDA-core grouped GEMMs, tiles of SIMT_ROWS rows)
constexpr int SIMT_ROWS = 32;
cudaError_t launch_gateup_simt(const uint16_t *x, int T, int H, int I, int E, int k, const int32_t *perm,
                               const int32_t *blockmap, const int32_t *n_tiles, int max_tiles, ExpertPtrs w,
                               uint16_t *h, cudaStream_t s);
cudaError_t launch_down_simt(const uint16_t *h, int T, int H, int I, int E, int k, const int32_t *blockmap,
                             const int32_t *n_tiles, int max_tiles, ExpertPtrs w, uint16_t *y, cudaStream_t s);

// combine.cu
// shared_gate: [H] fp32 or null; x: the layer's expert input (read only with a gate)
// xnorm (or null): also RMSNorm(out) with eps, bit for bit as launch_rmsnorm
cudaError_t launch_combine(const uint16_t *res, const uint16_t *y, const int32_t *inv, const float *topk_w,
                           const uint16_t *x, const float *shared_gate, int T, int H, int k, int S, uint16_t *out,
                           uint16_t *xnorm, float eps, cudaStream_t s);
cudaError_t launch_rmsnorm(const uint16_t *r, int T, int H, float eps, uint16_t *x, cudaStream_t s);
cudaError_t launch_dequant(const uint32_t *q, const uint16_t *sc, const uint16_t *b, int rows, int K, int G,
                           uint16_t *w, cudaStream_t s);

// decode.cu (T == 1: one cooperative launch runs whole layers)
// The decode kernel's scratch: the fp32 router keys and the top-k of the last
// layer run (for inspection), the epoch counter and the tagged exchange
// buffers (decode_tag_words 64-bit words; both zero before the first launch,
// kept between launches), the status word and the optional trace.
struct DecodeScratch {
  float *keys;
  int32_t *topk_id;
  float *topk_w;
  unsigned long long *epoch;
  unsigned long long *tags;
  int32_t *status;
  uint64_t *trace;
  unsigned long long timeout_ns = 1000000000ull;  // limit of every bounded wait
  int withhold = 0;  // test aid (MOE_FLAG_TEST_WITHHOLD): expert 0's key is never published
};
size_t decode_tag_words(int H, int E, int k, int I, int S);
bool decode_supported(int H, int E, int k, int I, int S, int num_sms);
cudaError_t decode_prepare(int H, int E, int k, int I, int S, int num_sms);
cudaError_t launch_decode(const uint16_t *x, const uint16_t *res, int H, int E, int k, int I, int S, int prenorm,
                          float eps, const float *router, const float *bias, ExpertPtrs w, uint16_t *out,
                          const DecodeScratch &sc, int num_sms, int *launches, cudaStream_t s);
// n_layers pre-norm layers on one token, r updated in place: r += MoE_l(RMSNorm(r));
// router/bias/w: host arrays of n_layers (bias may be null, or hold nulls).
cudaError_t launch_decode_stack(uint16_t *r, int n_layers, int H, int E, int k, int I, int S, float eps,
                                const float *const *router, const float *const *bias, const ExpertPtrs *w,
                                const DecodeScratch &sc, int num_sms, int *launches, cudaStream_t s);

}  // namespace moe
