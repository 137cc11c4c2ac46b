// Tensor-core (tcgen05) grouped expert GEMMs: host-side declarations.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include "kernels.h"

#include "moe.h"

namespace moe {

constexpr int TC_ROWS = 128;     // default token rows per block-map tile
constexpr bool TC_READY = false;  // the tcgen05 path is selected by default once built

cudaError_t launch_experts_tc(const moe_plan_t *plan, const uint16_t *x, int T, const int32_t *perm,
                              const int32_t *blockmap, const int32_t *n_tiles, int max_tiles, ExpertPtrs w,
                              uint16_t *h, uint16_t *y, int32_t *status, int *launches, cudaStream_t s);

}  // namespace moe
