// hc_common.cuh -- device helpers shared by the HC mixing kernels.
//
// bf16 <-> binary32 conversion, 16-byte streaming loads and stores, and the
// per-token split + Sinkhorn normalisation ("Reading weights" page, pre
// formula and the hc_split_sinkhorn kernel), written once so that the
// standalone and the fused kernels compute identical coefficients.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace hc {

// Error word bits (per device, read by hc_device_error).
constexpr unsigned int kErrWaitTimeout = 1u;
constexpr unsigned int kErrSmemLayout = 2u;  // shared memory base off its 1024-byte boundary

// Programmatic dependent launch (see overlap_launches): wait until the
// kernel before this one on the stream has completed and its memory is
// visible (a no-op when this kernel was launched without the attribute),
// then let the kernel after this one start launching.
__device__ __forceinline__ void griddep_wait_then_release() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------- bf16

// Two bf16 values packed in a 32-bit word -> two floats (exact).
__device__ __forceinline__ float bf16lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16hi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }

// Two floats -> two bf16 (round to nearest even), a in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
}

// 8 bf16 in a uint4 -> 8 floats.
__device__ __forceinline__ void unpack8(const uint4 &v, float f[8]) {
    f[0] = bf16lo(v.x); f[1] = bf16hi(v.x);
    f[2] = bf16lo(v.y); f[3] = bf16hi(v.y);
    f[4] = bf16lo(v.z); f[5] = bf16hi(v.z);
    f[6] = bf16lo(v.w); f[7] = bf16hi(v.w);
}

__device__ __forceinline__ uint4 pack8(const float f[8]) {
    uint4 v;
    v.x = pack_bf16x2(f[0], f[1]);
    v.y = pack_bf16x2(f[2], f[3]);
    v.z = pack_bf16x2(f[4], f[5]);
    v.w = pack_bf16x2(f[6], f[7]);
    return v;
}

// Packed pairs of binary32 in one 64-bit register (lo in the low half) and
// the two-wide FMA on them: d = a * b + d per half, each rounded once.
__device__ __forceinline__ uint64_t pack2(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void unpack2(uint64_t v, float &lo, float &hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ void ffma2(uint64_t &d, uint64_t a, uint64_t b) {
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(d) : "l"(a), "l"(b));
}
__device__ __forceinline__ uint64_t fmul2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ float sum2(uint64_t v) {
    float lo, hi;
    unpack2(v, lo, hi);
    return lo + hi;
}
// The two bf16 of a 32-bit word as a packed pair of binary32 (exact).
__device__ __forceinline__ uint64_t bf16x2_to_f32x2(uint32_t u) {
    return pack2(bf16lo(u), bf16hi(u));
}

// Streaming (evict-first) 16-byte global load/store.  Plain coherent loads:
// safe also when the same kernel later writes the location (in-place post).
__device__ __forceinline__ uint4 ld_stream(const uint4 *p) { return __ldcs(p); }
__device__ __forceinline__ void st_stream(uint4 *p, const uint4 &v) { __stcs(p, v); }

// ------------------------------------------------- split + Sinkhorn

// 1/x for finite, positive, normal x: the hardware approximation refined by one
// Newton-Raphson step for the reciprocal, r' = r + r*(1 - x*r), which brings it
// to about 1 ulp.  (The correctly rounded division is a long subroutine; on the
// per-token critical path of the fused kernel it cost ~25x more.)
__device__ __forceinline__ float rcp_refined(float x) {
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return fmaf(r, fmaf(-x, r, 1.0f), r);
}

// sigmoid(z) = 1 / (1 + e^-z), with the exponential of -|z| only (never
// overflows): sigmoid(z) = 1/(1+e) for z >= 0 and e/(1+e) for z < 0, e = e^-|z|.
__device__ __forceinline__ float sigmoidf_(float z) {
    const float e = expf(-fabsf(z));
    const float r = rcp_refined(1.0f + e);
    return z >= 0.f ? r : e * r;
}

// pre and post of one token ("Reading weights" page, pre formula and the
// hc_split_sinkhorn kernel):
//   pre_j  = sigmoid(m_j s0 + b_j) + eps
//   post_j = 2 sigmoid(m_{HC+j} s1 + b_{HC+j})
template <int HC, typename MixFn, typename BaseFn>
__device__ __forceinline__ void split_pre_post(MixFn m, BaseFn base, float s0, float s1, float eps,
                                               float pre[HC], float post[HC]) {
#pragma unroll
    for (int j = 0; j < HC; ++j) pre[j] = sigmoidf_(fmaf(m(j), s0, base(j))) + eps;
#pragma unroll
    for (int j = 0; j < HC; ++j) post[j] = 2.0f * sigmoidf_(fmaf(m(HC + j), s1, base(HC + j)));
}

// Pairwise sum of v[0..N) (N a power of two): ((v0 + v1) + (v2 + v3)) + ...
// A shorter dependency chain than the sum in index order, which the
// Sinkhorn steps below are bound by.
template <int N>
__device__ __forceinline__ float pair_sum(const float (&v)[N]) {
    static_assert((N & (N - 1)) == 0, "a power of two");
    float t[N];
#pragma unroll
    for (int i = 0; i < N; ++i) t[i] = v[i];
#pragma unroll
    for (int h = N / 2; h >= 1; h /= 2)
#pragma unroll
        for (int i = 0; i < h; ++i) t[i] = t[2 * i] + t[2 * i + 1];
    return t[0];
}

// comb of one token (same kernel on the same page): with
//   L_jk = m_{2HC+j HC+k} s2 + b_{2HC+j HC+k}   (row j, column k)
// C = row softmax of L (max-subtracted, plain row sum) + eps; a column step;
// then (iters-1) x (row step, column step), each step dividing by (sum + eps).
// Rows and columns are summed pairwise (pair_sum).
template <int HC, typename MixFn, typename BaseFn>
__device__ __forceinline__ void sinkhorn_comb(MixFn m, BaseFn base, float s2, int iters, float eps,
                                              float C[HC][HC]) {
#pragma unroll
    for (int j = 0; j < HC; ++j)
#pragma unroll
        for (int k = 0; k < HC; ++k)
            C[j][k] = fmaf(m(2 * HC + j * HC + k), s2, base(2 * HC + j * HC + k));
#pragma unroll
    for (int j = 0; j < HC; ++j) {
        float mx = C[j][0];
#pragma unroll
        for (int k = 1; k < HC; ++k) mx = fmaxf(mx, C[j][k]);
        float e[HC];
#pragma unroll
        for (int k = 0; k < HC; ++k) e[k] = C[j][k] = expf(C[j][k] - mx);
        const float inv = rcp_refined(pair_sum(e));  // >= 1: the row maximum contributes e^0
#pragma unroll
        for (int k = 0; k < HC; ++k) C[j][k] = fmaf(C[j][k], inv, eps);
    }
    auto row_step = [&]() {
#pragma unroll
        for (int j = 0; j < HC; ++j) {
            const float inv = rcp_refined(pair_sum(C[j]) + eps);
#pragma unroll
            for (int k = 0; k < HC; ++k) C[j][k] *= inv;
        }
    };
    auto col_step = [&]() {
#pragma unroll
        for (int k = 0; k < HC; ++k) {
            float c[HC];
#pragma unroll
            for (int j = 0; j < HC; ++j) c[j] = C[j][k];
            const float inv = rcp_refined(pair_sum(c) + eps);
#pragma unroll
            for (int j = 0; j < HC; ++j) C[j][k] *= inv;
        }
    };
    col_step();
    for (int it = 1; it < iters; ++it) {
        row_step();
        col_step();
    }
}

// One token: m = its (2+HC)*HC mix numbers, s0..s2 = hc_scale, base = hc_base.
template <int HC, typename MixFn, typename BaseFn>
__device__ __forceinline__ void split_sinkhorn_token(MixFn m, BaseFn base, float s0, float s1,
                                                     float s2, int iters, float eps,
                                                     float pre[HC], float post[HC],
                                                     float C[HC][HC]) {
    split_pre_post<HC>(m, base, s0, s1, eps, pre, post);
    sinkhorn_comb<HC>(m, base, s2, iters, eps, C);
}

}  // namespace hc
