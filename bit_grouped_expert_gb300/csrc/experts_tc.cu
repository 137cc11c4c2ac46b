// Tensor-core grouped expert GEMMs (tcgen05): not built yet.
#include "common.cuh"
#include "tc.h"

namespace moe {

cudaError_t launch_experts_tc(const moe_plan_t *, const uint16_t *, int, const int32_t *, const int32_t *,
                              const int32_t *, int, ExpertPtrs, uint16_t *, uint16_t *, int32_t *, int *,
                              cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace moe
