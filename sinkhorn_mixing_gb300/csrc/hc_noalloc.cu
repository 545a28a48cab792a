// hc_noalloc.cu -- hc_mixes_pre_noalloc: the general three-kernel path of
// hc_mixes_pre (tensor-core projection -> split/Sinkhorn -> collapse) with its
// mix-number scratch held in a fixed device array compiled into the library,
// for callers that cannot allocate device memory.
//
// Who needs this: code that runs where cudaMalloc is not allowed or not
// available -- inside a region being captured into a CUDA graph by a framework
// that forbids allocation there, inside a custom allocator's own callbacks, in
// plugins hosted by an engine that owns all device memory and hands out only
// input/output buffers, or in real-time loops that must not touch the
// allocator.  Such callers pass only their inputs and outputs.
//
// The scratch array is a file-scope __device__ variable: every GPU that loads
// the library holds its HC_NOALLOC_SCRATCH_FLOATS floats (4 MiB) until the
// process exits.  All calls share it, so calls that overlap on the GPU (on
// different streams, or on the same device from different threads without
// ordering) race on it.  Each call writes every element it later reads, so no
// part of it has to start at zero and nothing is cleared between calls.
#include <mutex>

#include "../../include/hcmix.h"
#include "hc_internal.h"

namespace hc {
namespace {

static __device__ __align__(256) float g_mix_scratch[HC_NOALLOC_SCRATCH_FLOATS];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
float *g_scratch_ptr[kMaxDevices];
unsigned long long g_scratch_ctx[kMaxDevices];

// Device address of the scratch array on the current device.  In host code
// the array's name is only a host-side stand-in, so the address must come
// from cudaGetSymbolAddress, with that device current.  It is looked up once
// per device and CUDA context (di.ctx, unique in the process): after a
// cudaDeviceReset the module is loaded anew and the address is looked up
// again.
cudaError_t scratch_on_current_device(const DeviceInfo &di, float **out) {
    if (di.device < 0 || di.device >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_scratch_ptr[di.device] == nullptr || di.ctx == 0 ||
        g_scratch_ctx[di.device] != di.ctx) {
        void *p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_mix_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_ptr[di.device] = static_cast<float *>(p);
        g_scratch_ctx[di.device] = di.ctx;
    }
    *out = g_scratch_ptr[di.device];
    return cudaSuccess;
}

bool al16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool finite_nonneg(float v) { return v >= 0.0f && v < __builtin_inff(); }

struct Span {
    uintptr_t lo, hi;
};
Span span(const void *p, uint64_t bytes) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
    return Span{a, a + (uintptr_t)bytes};
}
bool overlap(const Span &a, const Span &b) { return a.lo < b.hi && b.lo < a.hi; }

}  // namespace
}  // namespace hc

extern "C" hc_status hc_mixes_pre_noalloc(int64_t n, int hc, int64_t d, int iters, float eps,
                                          float norm_eps, const uint16_t *x, const float *w_mix,
                                          const float *hc_scale, const float *hc_base, float *pre,
                                          float *post, float *comb, uint16_t *y,
                                          hc_stream_t stream) {
    if (n < 0 || d <= 0) return HC_ERR_INVALID_ARG;
    if (hc != 4 && hc != 8) return HC_ERR_UNSUPPORTED;
    if (d % 8 != 0) return HC_ERR_MISALIGNED;
    if (d > (int64_t(1) << 24)) return HC_ERR_UNSUPPORTED;
    if (iters < 1 || !hc::finite_nonneg(eps) || !hc::finite_nonneg(norm_eps))
        return HC_ERR_INVALID_ARG;
    const int64_t mix = (int64_t)(2 + hc) * hc;
    // the fixed scratch holds n * mix_hc floats at most
    if (n > (int64_t)HC_NOALLOC_SCRATCH_FLOATS / mix) return HC_ERR_UNSUPPORTED;
    if (n == 0) return HC_OK;
    const void *ptrs[] = {x, w_mix, hc_scale, hc_base, pre, post, comb, y};
    for (const void *p : ptrs)
        if (p == nullptr) return HC_ERR_INVALID_ARG;
    for (const void *p : ptrs)
        if (!hc::al16(p)) return HC_ERR_MISALIGNED;
    const uint64_t F = (uint64_t)hc * d;
    const hc::Span outs[] = {hc::span(pre, n * hc * 4ull), hc::span(post, n * hc * 4ull),
                             hc::span(comb, n * (uint64_t)hc * hc * 4ull),
                             hc::span(y, (uint64_t)n * d * 2)};
    const hc::Span ins[] = {hc::span(x, n * F * 2), hc::span(w_mix, mix * F * 4),
                            hc::span(hc_scale, 12), hc::span(hc_base, mix * 4)};
    for (int a = 0; a < 4; ++a) {
        for (int b = a + 1; b < 4; ++b)
            if (hc::overlap(outs[a], outs[b])) return HC_ERR_INVALID_ARG;
        for (const hc::Span &b : ins)
            if (hc::overlap(outs[a], b)) return HC_ERR_INVALID_ARG;
    }
    hc::DeviceInfo di;
    if (hc::device_info(&di) != cudaSuccess) return HC_ERR_CUDA;
    float *scratch = nullptr;
    if (hc::scratch_on_current_device(di, &scratch) != cudaSuccess) return HC_ERR_CUDA;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // the projection hc_mixes_pre's general path uses (tensor cores where
    // they take the shape), with W converted inside the kernel: no scratch
    // beyond the mix numbers
    cudaError_t e = hc::launch_projection(n, hc, d, norm_eps, x, w_mix, scratch, nullptr, di, s);
    if (e == cudaSuccess)
        e = hc::launch_split_sinkhorn(n, hc, iters, eps, scratch, hc_scale, hc_base, pre, post,
                                      comb, di, s);
    if (e == cudaSuccess) e = hc::launch_pre(n, hc, d, x, pre, y, di, s);
    return e == cudaSuccess ? HC_OK : HC_ERR_CUDA;
}
