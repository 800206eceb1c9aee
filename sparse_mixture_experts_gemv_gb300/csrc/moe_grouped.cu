// Grouped (prefill) path of the MoE layer -- placeholder until the tensor-core kernels land.
#include "moe_internal.h"

namespace moe {
cudaError_t grouped_prepare(moe_layer*) { return cudaSuccess; }
void grouped_release(moe_layer*) {}
cudaError_t launch_grouped(moe_layer*, const uint16_t*, uint16_t*, int, const float*, cudaStream_t) {
  return cudaErrorNotSupported;
}
}  // namespace moe
