// hc_internal.h -- launchers behind the C ABI (not part of the public ABI).
// Arguments are already validated by hc_abi.cu when these are called.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace hc {

struct DeviceInfo {
    int device;
    int sms;
    unsigned long long ctx;  // unique id of the CUDA context the values below belong to
    unsigned int *err_word;  // device address of this device's error word
};

// Unique id (cuCtxGetId) of the calling thread's current CUDA context, or 0
// when none is current.  Ids are never reused within a process, so a cache
// keyed on it is rebuilt after the device's context is destroyed and
// recreated (cudaDeviceReset), when module addresses and function attributes
// are new.
unsigned long long current_context_id();

// Current device's SM count and error-word address, cached per device and
// context.  Per-device kernel set-up elsewhere compares its recorded ctx with
// DeviceInfo::ctx and redoes itself when they differ.
cudaError_t device_info(DeviceInfo *out);

// Path override for tests and diagnosis, read from the environment at each
// call: HCMIX_PATH=general forces the three-kernel path, HCMIX_PATH=ffma the
// same path with the CUDA-core projection, HCMIX_PATH=fused skips the decode
// kernel; unset (or anything else) chooses by shape.
enum ForcedPath { kPathAuto = 0, kPathGeneral = 1, kPathFused = 2, kPathFfma = 3 };
ForcedPath forced_path();

// Programmatic dependent launch for the small-batch kernels (k_decode,
// k_post): launched with the programmatic-stream-serialization attribute,
// such a kernel may start while the kernel before it on the stream is still
// running; its first instruction waits (griddepcontrol.wait) until that
// kernel has completed and its memory is visible, so no input is read early,
// and it then lets the kernel after it start (launch_dependents).  What
// overlaps is the launch and scheduling of one kernel with the tail of the
// other.  HCMIX_PDL=0 in the environment turns it off (read at each call).
bool overlap_launches();

// The driver's cuTensorMapEncodeTiled, or nullptr when it is unavailable.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();

// Adds k to the process-wide count of enqueued kernels (hc_launch_count).
void count_launches(int k);

// cudaGetLastError() after a launch, counting the launch when it succeeded.
inline cudaError_t launched(int k = 1) {
    const cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess) count_launches(k);
    return e;
}

cudaError_t launch_mixes(int64_t n, int hc, int64_t d, float norm_eps, const uint16_t *x,
                         const float *w, float *mixes, const DeviceInfo &di, cudaStream_t s);

// The general path's projection: launch_mixtc when it takes the shape, else
// launch_mixes.  wconv (nullable, 16-byte aligned, mixtc_wconv_bytes(hc, d)
// bytes) is device scratch for W converted to the tensor core's hi/lo rows.
cudaError_t launch_projection(int64_t n, int hc, int64_t d, float norm_eps, const uint16_t *x,
                              const float *w, float *mixes, uint16_t *wconv,
                              const DeviceInfo &di, cudaStream_t s);

// Tensor-core projection with W streamed (hc_mixtc.cu): hc in {4, 8} and
// hc*d a multiple of 64.  With wconv (hc = 8 only) W is converted once into
// it and loaded from there; without, the kernel converts it stage by stage.
bool mixtc_supported(int hc, int64_t d, const DeviceInfo &di);
size_t mixtc_wconv_bytes(int hc, int64_t d);  // 0 where no conversion pass is used
cudaError_t launch_mixtc(int64_t n, int hc, int64_t d, float norm_eps, const uint16_t *x,
                         const float *w, float *mixes, uint16_t *wconv, const DeviceInfo &di,
                         cudaStream_t s);

cudaError_t launch_split_sinkhorn(int64_t n, int hc, int iters, float eps, const float *mixes,
                                  const float *scale, const float *base, float *pre,
                                  float *post, float *comb, const DeviceInfo &di,
                                  cudaStream_t s);

cudaError_t launch_pre(int64_t n, int hc, int64_t d, const uint16_t *x, const float *pre,
                       uint16_t *y, const DeviceInfo &di, cudaStream_t s);

// Collapse + RMSNorm (out_c = y_c / sqrt(mean(y^2) + eps) * g_c), one row
// per CTA at a time (rows beyond 2^20 taken in a grid stride); the collapsed
// row is kept in shared memory up to 96 KB, else in y itself.
cudaError_t launch_pre_norm(int64_t n, int hc, int64_t d, const uint16_t *x, const float *pre,
                            const float *g, float eps, uint16_t *y, const DeviceInfo &di,
                            cudaStream_t s);

cudaError_t launch_post(int64_t n, int hc, int64_t d, const uint16_t *out,
                        const uint16_t *res, const float *post, const float *comb, uint16_t *y,
                        const DeviceInfo &di, cudaStream_t s);

// Diagnostic (hc_selftest.cu): one CTA whose bounded wait can only time out.
cudaError_t launch_wait_timeout(uint64_t limit_ns, const DeviceInfo &di, cudaStream_t s);

}  // namespace hc
