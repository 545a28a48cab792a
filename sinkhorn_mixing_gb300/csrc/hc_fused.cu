// hc_fused.cu -- fused path (not yet enabled: every shape takes the general
// kernels).
#include "hc_fused.h"

namespace hc {

bool fused_supported(int, int64_t, const DeviceInfo &) { return false; }

cudaError_t launch_fused(int64_t, int, int64_t, int, float, float, const uint16_t *,
                         const float *, const float *, const float *, float *, float *, float *,
                         float *, uint16_t *, const DeviceInfo &, cudaStream_t) {
    return cudaErrorNotSupported;
}

}  // namespace hc
