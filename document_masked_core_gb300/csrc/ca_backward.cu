// Backward core attention (placeholder until the tcgen05 kernels land).
#include "ca_sm100.cuh"

namespace ca {
cudaError_t launch_backward(const ca_plan *, const void *, const void *, const void *, const void *, const float *,
                            const void *, void *, void *, void *, void *, cudaStream_t) {
    return cudaErrorNotSupported;
}
}  // namespace ca
