// hc_abi.cu -- the extern "C" entry points of libhcmix.so: host-side argument
// validation, path selection and launch.  Nothing here allocates memory.
#include <math.h>
#include <stdlib.h>
#include <string.h>
#include <atomic>
#include <mutex>

#include "../../include/hcmix.h"
#include "hc_decode.h"
#include "hc_fused.h"
#include "hc_internal.h"

namespace hc {

// Per-device error word: kernels with bounded waits set bits here instead of
// trapping.  Read and cleared through hc_device_error().
__device__ unsigned int g_err_word;

namespace {
std::atomic<uint64_t> g_launches{0};
constexpr int kMaxDevices = 64;
std::mutex g_mu;
DeviceInfo g_info[kMaxDevices];
bool g_have[kMaxDevices];
}  // namespace

void count_launches(int k) { g_launches.fetch_add((uint64_t)k, std::memory_order_relaxed); }

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}

bool overlap_launches() {
    const char *e = getenv("HCMIX_PDL");
    return e == nullptr || strcmp(e, "0") != 0;
}

ForcedPath forced_path() {
    const char *e = getenv("HCMIX_PATH");
    if (e == nullptr) return kPathAuto;
    if (strcmp(e, "general") == 0) return kPathGeneral;
    if (strcmp(e, "fused") == 0) return kPathFused;
    if (strcmp(e, "ffma") == 0) return kPathFfma;
    return kPathAuto;
}

// The projection of the general path: tensor cores when they take the shape.
cudaError_t launch_projection(int64_t n, int hc, int64_t d, float norm_eps, const uint16_t *x,
                              const float *w, float *mixes, uint16_t *wconv,
                              const DeviceInfo &di, cudaStream_t s) {
    if (mixtc_supported(hc, d, di))
        return launch_mixtc(n, hc, d, norm_eps, x, w, mixes, wconv, di, s);
    return launch_mixes(n, hc, d, norm_eps, x, w, mixes, di, s);
}

unsigned long long current_context_id() {
    static PFN_cuCtxGetCurrent_v4000 get_cur = nullptr;
    static PFN_cuCtxGetId_v12000 get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 4000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_cur = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(f);
        f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(f);
    });
    if (get_cur == nullptr || get_id == nullptr) return 0;
    CUcontext c = nullptr;
    if (get_cur(&c) != CUDA_SUCCESS || c == nullptr) return 0;
    unsigned long long id = 0;
    return get_id(c, &id) == CUDA_SUCCESS ? id : 0;
}

cudaError_t device_info(DeviceInfo *out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    const unsigned long long ctx = current_context_id();
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_have[dev] || ctx == 0 || g_info[dev].ctx != ctx) {
        DeviceInfo di;
        di.device = dev;
        e = cudaDeviceGetAttribute(&di.sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        void *p = nullptr;
        // (also makes the device's primary context current when it was not)
        e = cudaGetSymbolAddress(&p, g_err_word);
        if (e != cudaSuccess) return e;
        di.err_word = static_cast<unsigned int *>(p);
        di.ctx = current_context_id();
        g_info[dev] = di;
        g_have[dev] = true;
    }
    *out = g_info[dev];
    return cudaSuccess;
}

}  // namespace hc

namespace {

bool al16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct Range {
    uintptr_t lo, hi;
};
Range rng(const void *p, uint64_t bytes) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
    return Range{a, a + (uintptr_t)bytes};
}
bool overlap(const Range &a, const Range &b) {
    return a.lo < b.hi && b.lo < a.hi && a.hi > a.lo && b.hi > b.lo;
}

bool finite_nonneg(float v) { return v >= 0.0f && v < INFINITY; }

// Shape checks shared by the entry points that take d.
hc_status check_shape(int64_t n, int hc, int64_t d) {
    if (n < 0 || d <= 0) return HC_ERR_INVALID_ARG;
    if (hc != 4 && hc != 8) return HC_ERR_UNSUPPORTED;
    if (d % 8 != 0) return HC_ERR_MISALIGNED;
    // keep every byte count well inside int64: n <= 2^40, d <= 2^24
    if (n > (int64_t(1) << 40) || d > (int64_t(1) << 24)) return HC_ERR_UNSUPPORTED;
    return HC_OK;
}

hc_status check_hc_n(int64_t n, int hc) {
    if (n < 0) return HC_ERR_INVALID_ARG;
    if (hc != 4 && hc != 8) return HC_ERR_UNSUPPORTED;
    if (n > (int64_t(1) << 40)) return HC_ERR_UNSUPPORTED;
    return HC_OK;
}

hc_status ptrs_ok(std::initializer_list<const void *> ps) {
    for (const void *p : ps)
        if (p == nullptr) return HC_ERR_INVALID_ARG;
    for (const void *p : ps)
        if (!al16(p)) return HC_ERR_MISALIGNED;
    return HC_OK;
}

// Every output range must be disjoint from every other listed range.
bool disjoint(std::initializer_list<Range> outs, std::initializer_list<Range> ins) {
    for (auto a = outs.begin(); a != outs.end(); ++a) {
        for (auto b = a + 1; b != outs.end(); ++b)
            if (overlap(*a, *b)) return false;
        for (const Range &b : ins)
            if (overlap(*a, b)) return false;
    }
    return true;
}

hc_status from_cuda(cudaError_t e) { return e == cudaSuccess ? HC_OK : HC_ERR_CUDA; }

}  // namespace

extern "C" {

const char *hc_status_string(hc_status s) {
    switch (s) {
        case HC_OK: return "HC_OK: success";
        case HC_ERR_INVALID_ARG:
            return "HC_ERR_INVALID_ARG: null pointer, negative size, bad iters/eps, "
                   "overlapping buffers or workspace too small";
        case HC_ERR_UNSUPPORTED: return "HC_ERR_UNSUPPORTED: hc must be 4 or 8; sizes too large";
        case HC_ERR_MISALIGNED:
            return "HC_ERR_MISALIGNED: d must be a multiple of 8 and pointers 16-byte aligned";
        case HC_ERR_CUDA: return "HC_ERR_CUDA: a CUDA runtime call or kernel launch failed";
    }
    return "unknown hc_status";
}

int hc_abi_version(void) { return HCMIX_ABI_VERSION; }

uint64_t hc_launch_count(void) { return hc::g_launches.load(std::memory_order_relaxed); }

namespace {
uint64_t round256(uint64_t b) { return (b + 255u) / 256u * 256u; }
// bytes of the workspace's first part: the mix numbers when mixes is NULL
uint64_t mix_part_bytes(int64_t n, int hc) { return round256((uint64_t)n * ((2 + hc) * hc) * 4u); }
}  // namespace

size_t hc_workspace_bytes(int64_t n, int hc, int64_t d) {
    if (check_shape(n, hc, d) != HC_OK || n == 0) return 0;
    return (size_t)(mix_part_bytes(n, hc) + round256(hc::mixtc_wconv_bytes(hc, d)));
}

// Token count from which hc_mixes takes the streamed-W tensor-core kernel
// rather than the fused kernel's projection-only mode (d = 1024..5120).
constexpr int64_t kFusedProjectionTokens = 16384;

hc_status hc_mixes(int64_t n, int hc, int64_t d, float norm_eps, const uint16_t *x,
                   const float *w_mix, float *mixes, hc_stream_t stream) {
    hc_status st = check_shape(n, hc, d);
    if (st != HC_OK) return st;
    if (!finite_nonneg(norm_eps)) return HC_ERR_INVALID_ARG;
    if (n == 0) return HC_OK;
    if ((st = ptrs_ok({x, w_mix, mixes})) != HC_OK) return st;
    const int mix = (2 + hc) * hc;
    const uint64_t F = (uint64_t)hc * d;
    if (!disjoint({rng(mixes, (uint64_t)n * mix * 4)},
                  {rng(x, (uint64_t)n * F * 2), rng(w_mix, (uint64_t)mix * F * 4)}))
        return HC_ERR_INVALID_ARG;
    hc::DeviceInfo di;
    cudaError_t e = hc::device_info(&di);
    if (e != cudaSuccess) return HC_ERR_CUDA;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (hc::decode_supported(n, hc, d, di)) {
        return from_cuda(hc::launch_decode(n, hc, d, /*iters=*/1, /*eps=*/0.0f, norm_eps, x,
                                           w_mix, nullptr, nullptr, mixes, nullptr, nullptr,
                                           nullptr, nullptr, nullptr, 0.0f, di, s));
    }
    // The projection alone: the fused kernel (W resident in its clusters'
    // shared memory, 112 SMs) up to kFusedProjectionTokens; past one wave of
    // 128-token units the tensor-core kernel with W streamed, on every SM, is
    // faster (65,536 tokens, d = 5120: 515 against 608 us).  The fused
    // kernel's gain is its collapse, which the projection alone does not have.
    if (hc::fused_supported(hc, d, di) &&
        (n < kFusedProjectionTokens || hc::forced_path() == hc::kPathFused ||
         !hc::mixtc_supported(hc, d, di))) {
        return from_cuda(hc::launch_fused(n, hc, d, /*iters=*/1, /*eps=*/0.0f, norm_eps, x,
                                          w_mix, nullptr, nullptr, mixes, nullptr, nullptr,
                                          nullptr, nullptr, di, s));
    }
    return from_cuda(hc::launch_projection(n, hc, d, norm_eps, x, w_mix, mixes, nullptr, di, s));
}

hc_status hc_split_sinkhorn(int64_t n, int hc, int iters, float eps, const float *mixes,
                            const float *hc_scale, const float *hc_base, float *pre,
                            float *post, float *comb, hc_stream_t stream) {
    hc_status st = check_hc_n(n, hc);
    if (st != HC_OK) return st;
    if (iters < 1 || !finite_nonneg(eps)) return HC_ERR_INVALID_ARG;
    if (n == 0) return HC_OK;
    if ((st = ptrs_ok({mixes, hc_scale, hc_base, pre, post, comb})) != HC_OK) return st;
    const uint64_t mix = (uint64_t)(2 + hc) * hc;
    if (!disjoint({rng(pre, n * hc * 4ull), rng(post, n * hc * 4ull),
                   rng(comb, n * (uint64_t)hc * hc * 4ull)},
                  {rng(mixes, n * mix * 4ull), rng(hc_scale, 12), rng(hc_base, mix * 4)}))
        return HC_ERR_INVALID_ARG;
    hc::DeviceInfo di;
    if (hc::device_info(&di) != cudaSuccess) return HC_ERR_CUDA;
    return from_cuda(hc::launch_split_sinkhorn(n, hc, iters, eps, mixes, hc_scale, hc_base, pre,
                                               post, comb, di,
                                               reinterpret_cast<cudaStream_t>(stream)));
}

hc_status hc_pre(int64_t n, int hc, int64_t d, const uint16_t *x, const float *pre, uint16_t *y,
                 hc_stream_t stream) {
    hc_status st = check_shape(n, hc, d);
    if (st != HC_OK) return st;
    if (n == 0) return HC_OK;
    if ((st = ptrs_ok({x, pre, y})) != HC_OK) return st;
    if (!disjoint({rng(y, (uint64_t)n * d * 2)},
                  {rng(x, (uint64_t)n * hc * d * 2), rng(pre, (uint64_t)n * hc * 4)}))
        return HC_ERR_INVALID_ARG;
    hc::DeviceInfo di;
    if (hc::device_info(&di) != cudaSuccess) return HC_ERR_CUDA;
    return from_cuda(
        hc::launch_pre(n, hc, d, x, pre, y, di, reinterpret_cast<cudaStream_t>(stream)));
}

hc_status hc_post(int64_t n, int hc, int64_t d, const uint16_t *out, const uint16_t *residual,
                  const float *post, const float *comb, uint16_t *y, hc_stream_t stream) {
    hc_status st = check_shape(n, hc, d);
    if (st != HC_OK) return st;
    if (n == 0) return HC_OK;
    if ((st = ptrs_ok({out, residual, post, comb, y})) != HC_OK) return st;
    const uint64_t ybytes = (uint64_t)n * hc * d * 2;
    const Range ry = rng(y, ybytes), rr = rng(residual, ybytes);
    const bool in_place = (const void *)y == (const void *)residual;
    if (!in_place && overlap(ry, rr)) return HC_ERR_INVALID_ARG;
    if (!disjoint({ry}, {rng(out, (uint64_t)n * d * 2), rng(post, (uint64_t)n * hc * 4),
                         rng(comb, (uint64_t)n * hc * hc * 4)}))
        return HC_ERR_INVALID_ARG;
    hc::DeviceInfo di;
    if (hc::device_info(&di) != cudaSuccess) return HC_ERR_CUDA;
    return from_cuda(hc::launch_post(n, hc, d, out, residual, post, comb, y, di,
                                     reinterpret_cast<cudaStream_t>(stream)));
}

namespace {

// hc_mixes_pre, and hc_mixes_pre_norm when rms_w is not null.
hc_status mixes_pre_impl(int64_t n, int hc, int64_t d, int iters, float eps, float norm_eps,
                         const uint16_t *x, const float *w_mix, const float *hc_scale,
                         const float *hc_base, const float *rms_w, float rms_eps, float *mixes,
                         float *pre, float *post, float *comb, uint16_t *y, void *workspace,
                         size_t workspace_bytes, hc_stream_t stream) {
    hc_status st = check_shape(n, hc, d);
    if (st != HC_OK) return st;
    if (iters < 1 || !finite_nonneg(eps) || !finite_nonneg(norm_eps)) return HC_ERR_INVALID_ARG;
    if (rms_w != nullptr && !finite_nonneg(rms_eps)) return HC_ERR_INVALID_ARG;
    if (n == 0) return HC_OK;
    if ((st = ptrs_ok({x, w_mix, hc_scale, hc_base, pre, post, comb, y})) != HC_OK) return st;
    if (rms_w != nullptr && !al16(rms_w)) return HC_ERR_MISALIGNED;
    if (mixes != nullptr && !al16(mixes)) return HC_ERR_MISALIGNED;
    const uint64_t mix = (uint64_t)(2 + hc) * hc, F = (uint64_t)hc * d;
    const Range rmix = mixes ? rng(mixes, n * mix * 4) : Range{0, 0};
    const Range rrms = rms_w ? rng(rms_w, (uint64_t)d * 4) : Range{0, 0};
    if (!disjoint({rmix, rng(pre, n * hc * 4ull), rng(post, n * hc * 4ull),
                   rng(comb, n * (uint64_t)hc * hc * 4ull), rng(y, (uint64_t)n * d * 2)},
                  {rng(x, n * F * 2), rng(w_mix, mix * F * 4), rng(hc_scale, 12),
                   rng(hc_base, mix * 4), rrms}))
        return HC_ERR_INVALID_ARG;
    // Without `mixes` the general path keeps the mix numbers in the workspace
    // between its stages; the decode and fused paths read no workspace.  The
    // status a missing or unusable workspace gives on the general path, or
    // HC_OK when it is usable.
    float *m = mixes;
    hc_status ws_status = HC_OK;
    if (m == nullptr) {
        if (workspace == nullptr || workspace_bytes < mix_part_bytes(n, hc)) {
            ws_status = HC_ERR_INVALID_ARG;
        } else if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) {
            ws_status = HC_ERR_MISALIGNED;
        } else if (!disjoint({rng(workspace, workspace_bytes)},
                             {rng(pre, n * hc * 4ull), rng(post, n * hc * 4ull),
                              rng(comb, n * (uint64_t)hc * hc * 4ull),
                              rng(y, (uint64_t)n * d * 2), rng(x, n * F * 2),
                              rng(w_mix, mix * F * 4), rng(hc_scale, 12),
                              rng(hc_base, mix * 4), rrms})) {
            ws_status = HC_ERR_INVALID_ARG;
        } else {
            m = static_cast<float *>(workspace);
        }
        // Shapes that only the general path takes are settled here, before
        // any CUDA call; the others once the path is known.
        if (ws_status != HC_OK && !(hc == 4 && d % 256 == 0 && d <= 5120)) return ws_status;
    }
    hc::DeviceInfo di;
    if (hc::device_info(&di) != cudaSuccess) return HC_ERR_CUDA;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (hc::decode_supported(n, hc, d, di)) {
        return from_cuda(hc::launch_decode(n, hc, d, iters, eps, norm_eps, x, w_mix, hc_scale,
                                           hc_base, mixes, pre, post, comb, y, rms_w, rms_eps,
                                           di, s));
    }
    if (hc::fused_supported(hc, d, di)) {
        // With the RMSNorm: the same kernel with the norm folded into the
        // collapse (its statistic from the copies' Gram matrix, so no second
        // pass over the rows).
        return from_cuda(rms_w == nullptr
                             ? hc::launch_fused(n, hc, d, iters, eps, norm_eps, x, w_mix, hc_scale,
                                                hc_base, mixes, pre, post, comb, y, di, s)
                             : hc::launch_fused_norm(n, hc, d, iters, eps, norm_eps, x, w_mix,
                                                     hc_scale, hc_base, mixes, pre, post, comb, y,
                                                     rms_w, rms_eps, di, s));
    }
    // General path: three kernels, the mix numbers passing through m.  A
    // workspace with room past the mix numbers (hc_workspace_bytes) also
    // takes the converted W; one that is smaller, misaligned or overlapping
    // is simply not used for it.
    if (ws_status != HC_OK) return ws_status;
    uint16_t *wconv = nullptr;
    const uint64_t wcb = hc::mixtc_wconv_bytes(hc, d);
    if (wcb != 0 && workspace != nullptr &&
        (reinterpret_cast<uintptr_t>(workspace) & 255u) == 0) {
        const uint64_t off = mixes == nullptr ? mix_part_bytes(n, hc) : 0;
        if (workspace_bytes >= off + wcb) {
            uint16_t *cand = reinterpret_cast<uint16_t *>(static_cast<uint8_t *>(workspace) + off);
            if (disjoint({rng(cand, wcb)},
                         {rng(pre, n * hc * 4ull), rng(post, n * hc * 4ull),
                          rng(comb, n * (uint64_t)hc * hc * 4ull), rng(y, (uint64_t)n * d * 2),
                          rng(x, n * F * 2), rng(w_mix, mix * F * 4), rng(hc_scale, 12),
                          rng(hc_base, mix * 4), rrms, rng(m, n * mix * 4)}))
                wconv = cand;
        }
    }
    cudaError_t e = hc::launch_projection(n, hc, d, norm_eps, x, w_mix, m, wconv, di, s);
    if (e == cudaSuccess)
        e = hc::launch_split_sinkhorn(n, hc, iters, eps, m, hc_scale, hc_base, pre, post, comb,
                                      di, s);
    if (e == cudaSuccess)
        e = rms_w == nullptr ? hc::launch_pre(n, hc, d, x, pre, y, di, s)
                             : hc::launch_pre_norm(n, hc, d, x, pre, rms_w, rms_eps, y, di, s);
    return from_cuda(e);
}

}  // namespace

hc_status hc_mixes_pre(int64_t n, int hc, int64_t d, int iters, float eps, float norm_eps,
                       const uint16_t *x, const float *w_mix, const float *hc_scale,
                       const float *hc_base, float *mixes, float *pre, float *post, float *comb,
                       uint16_t *y, void *workspace, size_t workspace_bytes,
                       hc_stream_t stream) {
    return mixes_pre_impl(n, hc, d, iters, eps, norm_eps, x, w_mix, hc_scale, hc_base, nullptr,
                          0.0f, mixes, pre, post, comb, y, workspace, workspace_bytes, stream);
}

hc_status hc_mixes_pre_norm(int64_t n, int hc, int64_t d, int iters, float eps, float norm_eps,
                            const uint16_t *x, const float *w_mix, const float *hc_scale,
                            const float *hc_base, const float *rms_weight, float rms_eps,
                            float *mixes, float *pre, float *post, float *comb, uint16_t *y,
                            void *workspace, size_t workspace_bytes, hc_stream_t stream) {
    if (rms_weight == nullptr) return HC_ERR_INVALID_ARG;
    return mixes_pre_impl(n, hc, d, iters, eps, norm_eps, x, w_mix, hc_scale, hc_base,
                          rms_weight, rms_eps, mixes, pre, post, comb, y, workspace,
                          workspace_bytes, stream);
}

hc_status hc_post_mixes_pre(int64_t n, int hc, int64_t d, const uint16_t *out,
                            const uint16_t *residual, const float *post, const float *comb,
                            uint16_t *x_next, int iters, float eps, float norm_eps,
                            const float *w_mix, const float *hc_scale, const float *hc_base,
                            float *mixes, float *pre_next, float *post_next, float *comb_next,
                            uint16_t *y_next, void *workspace, size_t workspace_bytes,
                            hc_stream_t stream) {
    hc_status st = check_shape(n, hc, d);
    if (st != HC_OK) return st;
    if (iters < 1 || !finite_nonneg(eps) || !finite_nonneg(norm_eps)) return HC_ERR_INVALID_ARG;
    if (n == 0) return HC_OK;
    if ((st = ptrs_ok({out, residual, post, comb, x_next, w_mix, hc_scale, hc_base, pre_next,
                       post_next, comb_next, y_next})) != HC_OK)
        return st;
    if (mixes != nullptr && !al16(mixes)) return HC_ERR_MISALIGNED;
    const uint64_t mix = (uint64_t)(2 + hc) * hc, F = (uint64_t)hc * d;
    const uint64_t xbytes = (uint64_t)n * F * 2;
    const Range rx = rng(x_next, xbytes), rres = rng(residual, xbytes);
    const bool in_place = (const void *)x_next == (const void *)residual;
    if (!in_place && overlap(rx, rres)) return HC_ERR_INVALID_ARG;
    const Range rmix = mixes ? rng(mixes, n * mix * 4) : Range{0, 0};
    // every output disjoint from every other and from every input (x_next may
    // be the residual itself)
    if (!disjoint({rx, rmix, rng(pre_next, n * hc * 4ull), rng(post_next, n * hc * 4ull),
                   rng(comb_next, n * (uint64_t)hc * hc * 4ull), rng(y_next, (uint64_t)n * d * 2)},
                  {rng(out, (uint64_t)n * d * 2), rng(post, n * hc * 4ull),
                   rng(comb, n * (uint64_t)hc * hc * 4ull), rng(w_mix, mix * F * 4),
                   rng(hc_scale, 12), rng(hc_base, mix * 4)}))
        return HC_ERR_INVALID_ARG;
    if (!disjoint({rmix, rng(pre_next, n * hc * 4ull), rng(post_next, n * hc * 4ull),
                   rng(comb_next, n * (uint64_t)hc * hc * 4ull), rng(y_next, (uint64_t)n * d * 2)},
                  {rres}))
        return HC_ERR_INVALID_ARG;
    hc::DeviceInfo di;
    if (hc::device_info(&di) != cudaSuccess) return HC_ERR_CUDA;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (hc::fused_supported(hc, d, di) && !hc::decode_supported(n, hc, d, di)) {
        // one launch: the ring streams the residual; the new stream goes to
        // x_next and is projected, normalised and collapsed on the way
        return from_cuda(hc::launch_fused_post(n, hc, d, out, residual, post, comb, x_next,
                                               iters, eps, norm_eps, w_mix, hc_scale, hc_base,
                                               mixes, pre_next, post_next, comb_next, y_next, di,
                                               s));
    }
    if (hc::decode_supported(n, hc, d, di)) {
        // few tokens: the decode kernel forms the new stream from the
        // residual and output slices it loads, writes it, and goes on
        return from_cuda(hc::launch_decode_post(n, hc, d, out, residual, post, comb, x_next, iters,
                                                eps, norm_eps, w_mix, hc_scale, hc_base, mixes,
                                                pre_next, post_next, comb_next, y_next, di, s));
    }
    // other shapes: hc_post, then hc_mixes_pre on its result.
    // hc_mixes_pre's workspace rule is checked here, before the first launch:
    // its general path keeps the mix numbers in the workspace.
    if (mixes == nullptr && !hc::decode_supported(n, hc, d, di) &&
        !hc::fused_supported(hc, d, di)) {
        if (workspace == nullptr || workspace_bytes < mix_part_bytes(n, hc))
            return HC_ERR_INVALID_ARG;
        if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return HC_ERR_MISALIGNED;
        if (!disjoint({rng(workspace, workspace_bytes)},
                      {rx, rres, rng(out, (uint64_t)n * d * 2), rng(post, n * hc * 4ull),
                       rng(comb, n * (uint64_t)hc * hc * 4ull), rng(w_mix, mix * F * 4),
                       rng(hc_scale, 12), rng(hc_base, mix * 4), rng(pre_next, n * hc * 4ull),
                       rng(post_next, n * hc * 4ull), rng(comb_next, n * (uint64_t)hc * hc * 4ull),
                       rng(y_next, (uint64_t)n * d * 2)}))
            return HC_ERR_INVALID_ARG;
    }
    const cudaError_t e = hc::launch_post(n, hc, d, out, residual, post, comb, x_next, di, s);
    if (e != cudaSuccess) return HC_ERR_CUDA;
    return mixes_pre_impl(n, hc, d, iters, eps, norm_eps, x_next, w_mix, hc_scale, hc_base,
                          nullptr, 0.0f, mixes, pre_next, post_next, comb_next, y_next, workspace,
                          workspace_bytes, stream);
}

hc_status hc_selftest_wait_timeout(uint64_t limit_ns, hc_stream_t stream) {
    if (limit_ns < 1 || limit_ns > 1000000000ull) return HC_ERR_INVALID_ARG;
    hc::DeviceInfo di;
    if (hc::device_info(&di) != cudaSuccess) return HC_ERR_CUDA;
    return from_cuda(
        hc::launch_wait_timeout(limit_ns, di, reinterpret_cast<cudaStream_t>(stream)));
}

hc_status hc_device_error(unsigned int *flags, int clear) {
    if (cudaDeviceSynchronize() != cudaSuccess) return HC_ERR_CUDA;
    unsigned int v = 0;
    if (cudaMemcpyFromSymbol(&v, hc::g_err_word, sizeof v) != cudaSuccess) return HC_ERR_CUDA;
    if (flags) *flags = v;
    if (clear) {
        const unsigned int z = 0;
        if (cudaMemcpyToSymbol(hc::g_err_word, &z, sizeof z) != cudaSuccess) return HC_ERR_CUDA;
    }
    return HC_OK;
}

}  // extern "C"
