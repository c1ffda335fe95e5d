// placeholder until the tensor-core kernel lands
#include "qwm_internal.cuh"
namespace qwm {
bool attend_mma_supported(const qwm_ctx*) { return false; }
cudaError_t launch_attend_mma(const qwm_ctx*, const void*, int64_t, float, void*, cudaStream_t) {
  return cudaErrorNotSupported;
}
}  // namespace qwm
