// hc_fused.h -- the fused mix projection + Sinkhorn + collapse path
// (tensor-core projection, thread-block clusters), behind hc_mixes_pre and
// hc_mixes.  Not part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "hc_internal.h"

namespace hc {

// True when the fused kernel handles this (hc, d) on the current device.
bool fused_supported(int hc, int64_t d, const DeviceInfo &di);

// pre == nullptr selects the projection-only mode (hc_mixes): only `mixes`
// is written.  Otherwise pre, post, comb and y are written, and mixes when
// it is not null.
cudaError_t launch_fused(int64_t n, int hc, int64_t d, int iters, float eps, float norm_eps,
                         const uint16_t *x, const float *w, const float *scale,
                         const float *base, float *mixes, float *pre, float *post, float *comb,
                         uint16_t *y, const DeviceInfo &di, cudaStream_t s);

// launch_fused with the RMSNorm of the collapse (weight rms_w [d], rms_eps)
// applied before y is written: y = bf16((bf16(sum_j pre_j x_j) rms_w) r), r
// the RMS factor of the binary32 collapse over all d channels.
cudaError_t launch_fused_norm(int64_t n, int hc, int64_t d, int iters, float eps, float norm_eps,
                              const uint16_t *x, const float *w, const float *scale,
                              const float *base, float *mixes, float *pre, float *post,
                              float *comb, uint16_t *y, const float *rms_w, float rms_eps,
                              const DeviceInfo &di, cudaStream_t s);

// hc_post of the previous sublayer followed by hc_mixes_pre on its result,
// in one launch: x_next = hc_post(out, residual, post_in, comb_in) is written
// (x_next may be residual itself), and pre, post, comb, y (and mixes when not
// null) are those of hc_mixes_pre on x_next.  Same shapes as launch_fused.
cudaError_t launch_fused_post(int64_t n, int hc, int64_t d, const uint16_t *out,
                              const uint16_t *residual, const float *post_in,
                              const float *comb_in, uint16_t *x_next, int iters, float eps,
                              float norm_eps, const float *w, const float *scale,
                              const float *base, float *mixes, float *pre, float *post,
                              float *comb, uint16_t *y, const DeviceInfo &di, cudaStream_t s);

}  // namespace hc
