// Tensor-core (tcgen05) grouped expert GEMMs: host-side declarations.
#pragma once
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kernels.h"

#include "moe.h"

namespace moe {

constexpr int TC_ROWS = 128;       // default token rows per block-map tile (gate/up GEMM)
constexpr int TC_DOWN_ROWS = 192;  // token rows per tile of the down GEMM's block map (two accumulators fit)
constexpr int TC_SHORT_ROWS = 64;  // the same map's tile height when experts average few rows

// The driver's cuTensorMapEncodeTiled (null when the driver lacks it).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();

// Dims the tensor-core path handles (H and I multiples of 256); others use
// the CUDA-core kernels.
bool tc_supported(const moe_config &c);
// One-time kernel attributes (dynamic shared memory size); needs a device.
cudaError_t tc_prepare();

// The down GEMM's modes (down_mode): one 128-feature output tile per item
// over blockmap2's taller tiles; two output tiles per item over blockmap;
// two output tiles per item, two items in flight, over blockmap2's short tiles.
enum { TC_DOWN_ONE = 0, TC_DOWN_PAIR = 1, TC_DOWN_PAIR_SHORT = 2 };

// qctr: two work-queue counters (gate/up, down), zero at the launch (the
// scatter kernel of the layer's routing zeroes them).
cudaError_t launch_experts_tc(const moe_plan_t *plan, const uint16_t *x, int T, const int32_t *perm,
                              const int32_t *blockmap, const int32_t *n_tiles, int max_tiles, int down_mode,
                              const int32_t *blockmap2, const int32_t *n_tiles2, int max_tiles2, ExpertPtrs w,
                              uint16_t *h, uint16_t *y, uint16_t *xg, int32_t *qctr, int32_t *status,
                              uint64_t *trace, int *launches, cudaStream_t s);

// Router keys on tensor cores (E % 128 == 0, H % 64 == 0).
bool router_tc_supported(int E, int H);
cudaError_t router_tc_prepare();
// split: workspace for three bf16 copies of the router ([3][E][H]).
// K slices of the router GEMM at T tokens (1, 2, 4 or 8: enough items for
// the SMs), and the fp32 partial-sum buffer a plan for up to Tmax tokens needs.
int router_tc_slices(int T, int E, int H, int num_sms);
size_t router_tc_partial_floats(int Tmax, int E, int H, int num_sms);
// The router's bf16 parts [3][E][H] (hi, mid, lo) from the fp32 router.
cudaError_t launch_router_split(const float *router, int E, int H, uint16_t *split, cudaStream_t s);
// Router keys for T tokens.  split_given: the parts from launch_router_split,
// or null (then they are written into split first).  partial: workspace of
// router_tc_partial_floats floats (16-byte aligned).  *ks_out = the K slices
// used: with 1 the keys (bias added) are in keys; with more, partial holds
// [KS][T][E] fp32 sums that the top-k kernel adds in slice order (+ bias).
// zero (or null): nzero ints the kernel sets to 0 before any of its own work
// (the top-k's histograms, so that no memset sits between the kernels).  The
// kernel starts as a programmatic dependent of the kernel before it in the
// stream and waits for it before touching memory.
// *launches counts the kernels enqueued.
cudaError_t launch_router_tc(const uint16_t *x, int T, int H, const float *router, int E, const float *bias,
                             const uint16_t *split_given, uint16_t *split, float *partial, float *keys,
                             int32_t *status, int32_t *zero, int nzero, int num_sms, int *ks_out, int *launches,
                             cudaStream_t s);
constexpr int ROUTER_TC_MIN_T = 32;  // below this the CUDA-core router is used

}  // namespace moe
