// hc_norm.cu -- the RMSNorm the block applies to the sublayer input, on the
// collapse output of hc_pre (attn_norm / ffn_norm, named on the
// "Hyper-connections" page without its body; the standard form is taken):
// out_c = (y_c * r) * g_c with r = 1/sqrt(mean_c y_c^2 + eps), y the bf16
// collapse, the mean of squares in fp32.
//
//   k_pre_norm       the collapse followed by the RMSNorm, one CTA per token
//
// It reduces the squares in a fixed order, so repeated calls give the same
// bits.  (The decode and fused kernels apply the norm inside their own
// launches.)
#include "hc_common.cuh"
#include "hc_internal.h"

namespace hc {
namespace {

// --------------------------------------------------------- k_pre_norm
// Collapse followed by the RMSNorm of the sublayer input, one row per CTA at
// a time: the collapse of the whole row (same arithmetic and order as k_pre)
// is rounded to bf16 and kept, the mean of its squares is reduced in a fixed
// order, and out_c = (y_c * r) * g_c is written, with
// r = 1/sqrt(mean(y^2) + eps).  The collapsed row is kept in shared memory
// (kSmemRow) or, for rows too wide for it, in the output row itself; either
// way each thread reads back only the vectors it wrote.
template <int HC, bool kSmemRow>
__global__ void __launch_bounds__(256) k_pre_norm(int64_t n, int64_t nv, float eps,
                                                  const uint4 *__restrict__ x,
                                                  const float *__restrict__ pre,
                                                  const float *__restrict__ g, uint4 *__restrict__ y) {
    extern __shared__ uint4 ys_smem[];  // the row's nv collapsed vectors (kSmemRow)
    __shared__ float red[8];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int64_t t = blockIdx.x; t < n; t += gridDim.x) {
        uint4 *yt = y + t * nv;
        uint4 *ys = kSmemRow ? ys_smem : yt;
        float p[HC];
#pragma unroll
        for (int q = 0; q < HC / 4; ++q) {
            const float4 v = __ldg(reinterpret_cast<const float4 *>(pre + t * HC) + q);
            p[4 * q] = v.x, p[4 * q + 1] = v.y, p[4 * q + 2] = v.z, p[4 * q + 3] = v.w;
        }
        const uint4 *xt = x + t * HC * nv;
        float ss = 0.f;
        for (int64_t v = threadIdx.x; v < nv; v += blockDim.x) {
            uint4 r[HC];
#pragma unroll
            for (int j = 0; j < HC; ++j) r[j] = ld_stream(xt + j * nv + v);
            float acc[8], f[8];
            unpack8(r[0], f);
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[e] = p[0] * f[e];
#pragma unroll
            for (int j = 1; j < HC; ++j) {
                unpack8(r[j], f);
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[e] = fmaf(p[j], f[e], acc[e]);
            }
            const uint4 yv = pack8(acc);
            ys[v] = yv;
            unpack8(yv, f);
#pragma unroll
            for (int e = 0; e < 8; ++e) ss = fmaf(f[e], f[e], ss);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, off);
        if (lane == 0) red[warp] = ss;
        __syncthreads();
        float tot = 0.f;
#pragma unroll
        for (int w = 0; w < 8; ++w) tot += red[w];
        const float r = rsqrtf(tot / (float)(nv * 8) + eps);
        for (int64_t v = threadIdx.x; v < nv; v += blockDim.x) {
            float f[8], o[8];
            unpack8(ys[v], f);
            const float4 g0 = __ldg(reinterpret_cast<const float4 *>(g) + 2 * v);
            const float4 g1 = __ldg(reinterpret_cast<const float4 *>(g) + 2 * v + 1);
            const float gv[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
#pragma unroll
            for (int e = 0; e < 8; ++e) o[e] = (f[e] * r) * gv[e];
            st_stream(yt + v, pack8(o));
        }
        __syncthreads();  // red[] and the shared row are reused by the next row
    }
}

// rows per launch grid: one CTA per row up to this many rows, then a stride
constexpr int64_t kMaxRowGrid = int64_t(1) << 20;
// collapsed rows up to this size stay in shared memory (two CTAs per SM)
constexpr size_t kMaxSmemRow = 96 * 1024;

}  // namespace

cudaError_t launch_pre_norm(int64_t n, int hc, int64_t d, const uint16_t *x, const float *pre,
                            const float *g, float eps, uint16_t *y, const DeviceInfo &,
                            cudaStream_t s) {
    const int64_t nv = d / 8;
    const size_t row = (size_t)nv * 16;
    const unsigned grid = (unsigned)(n < kMaxRowGrid ? n : kMaxRowGrid);
    const uint4 *xv = reinterpret_cast<const uint4 *>(x);
    uint4 *yv = reinterpret_cast<uint4 *>(y);
    if (row > kMaxSmemRow) {
        if (hc == 4)
            k_pre_norm<4, false><<<grid, 256, 0, s>>>(n, nv, eps, xv, pre, g, yv);
        else
            k_pre_norm<8, false><<<grid, 256, 0, s>>>(n, nv, eps, xv, pre, g, yv);
        return launched();
    }
    if (row > 48 * 1024) {
        const cudaError_t e = hc == 4
            ? cudaFuncSetAttribute(k_pre_norm<4, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   (int)row)
            : cudaFuncSetAttribute(k_pre_norm<8, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   (int)row);
        if (e != cudaSuccess) return e;
    }
    if (hc == 4)
        k_pre_norm<4, true><<<grid, 256, row, s>>>(n, nv, eps, xv, pre, g, yv);
    else
        k_pre_norm<8, true><<<grid, 256, row, s>>>(n, nv, eps, xv, pre, g, yv);
    return launched();
}

}  // namespace hc
