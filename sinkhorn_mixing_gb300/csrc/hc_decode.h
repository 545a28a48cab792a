// hc_decode.h -- the few-token (decode) path behind hc_mixes_pre and
// hc_mixes: one launch spreads up to 16 tokens per 16-CTA cluster over every
// cluster the device holds.  Not part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "hc_internal.h"

namespace hc {

// True when the decode kernel handles n tokens of this (hc, d) on the
// current device.
bool decode_supported(int64_t n, int hc, int64_t d, const DeviceInfo &di);

// pre == nullptr selects the projection-only mode (hc_mixes): only `mixes`
// is written.  Otherwise pre, post, comb and y are written, and mixes when
// it is not null; with rms_w the collapsed rows are RMS-normalised
// (y = (yc / sqrt(mean yc^2 + rms_eps)) * rms_w).
cudaError_t launch_decode(int64_t n, int hc, int64_t d, int iters, float eps, float norm_eps,
                          const uint16_t *x, const float *w, const float *scale,
                          const float *base, float *mixes, float *pre, float *post,
                          float *comb, uint16_t *y, const float *rms_w, float rms_eps,
                          const DeviceInfo &di, cudaStream_t s);

// hc_post of the previous sublayer followed by hc_mixes_pre on its result,
// in one launch (the decode shapes): x_next = hc_post(out, residual,
// post_in, comb_in) is written (x_next may be residual itself), and pre,
// post, comb, y (and mixes when not null) are those of hc_mixes_pre on x_next.
cudaError_t launch_decode_post(int64_t n, int hc, int64_t d, const uint16_t *out,
                               const uint16_t *residual, const float *post_in,
                               const float *comb_in, uint16_t *x_next, int iters, float eps,
                               float norm_eps, const float *w, const float *scale,
                               const float *base, float *mixes, float *pre, float *post,
                               float *comb, uint16_t *y, const DeviceInfo &di, cudaStream_t s);

}  // namespace hc
