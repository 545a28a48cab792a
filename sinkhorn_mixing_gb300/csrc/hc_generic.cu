// hc_generic.cu -- the general HC mixing kernels (any supported hc and d).
//
//   k_mixes          mix projection + RMS statistic ("Mix projection" page)
//   k_split_sinkhorn split + Sinkhorn, one thread per token ("Reading weights")
//   k_pre            collapse y = sum_j pre_j x_j (Block.hc_pre)
//   k_post           expansion y_k = post_k out + sum_j comb_jk r_j (Block.hc_post)
//
// k_pre and k_post are HBM streams: a warp owns one (token, channel segment)
// unit at a time, keeps the token's coefficients in registers, and moves the
// copies in 16-byte vectors with several loads in flight per lane.
#include "hc_common.cuh"
#include "hc_internal.h"

namespace hc {
namespace {

// ------------------------------------------------------------ k_mixes
// One CTA per 32 tokens; 256 threads = 32 tokens x 8 output groups.  The
// feature axis is walked in chunks of 64: the chunk of x is widened to fp32
// and the matching 64 columns of W are staged in shared memory.  Thread
// (tok, g) accumulates mix numbers i = g, g+8, ... of token tok and the
// squares of features k = g, g+8, ... of the chunk.
template <int HC>
__global__ void __launch_bounds__(256) k_mixes(int64_t n, int64_t F, float norm_eps,
                                               const uint16_t *__restrict__ x,
                                               const float *__restrict__ w,
                                               float *__restrict__ mixes) {
    constexpr int MIX = (2 + HC) * HC;
    constexpr int TM = 32, KC = 64, G = 8, NO = MIX / G;
    static_assert(MIX % G == 0, "mix count must split over the groups");
    __shared__ float xs[TM][KC + 1];
    __shared__ float ws[MIX][KC + 1];
    const int tid = threadIdx.x, tok = tid / G, g = tid % G;
    const int64_t t0 = (int64_t)blockIdx.x * TM;
    float acc[NO];
#pragma unroll
    for (int o = 0; o < NO; ++o) acc[o] = 0.0f;
    float ss = 0.0f;

    for (int64_t k0 = 0; k0 < F; k0 += KC) {
        {
            const int row = tid / 8, part = tid % 8;
            const int64_t t = t0 + row, k = k0 + part * 8;
            float f[8];
            if (t < n && k < F) {
                unpack8(*reinterpret_cast<const uint4 *>(x + t * F + k), f);
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) f[e] = 0.0f;
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) xs[row][part * 8 + e] = f[e];
        }
        for (int idx = tid; idx < MIX * KC / 4; idx += 256) {
            const int i = idx / (KC / 4), q = idx % (KC / 4);
            const int64_t k = k0 + q * 4;
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (k < F) v = __ldg(reinterpret_cast<const float4 *>(w + (int64_t)i * F + k));
            ws[i][q * 4 + 0] = v.x;
            ws[i][q * 4 + 1] = v.y;
            ws[i][q * 4 + 2] = v.z;
            ws[i][q * 4 + 3] = v.w;
        }
        __syncthreads();
#pragma unroll 8
        for (int k = 0; k < KC; ++k) {
            const float xv = xs[tok][k];
#pragma unroll
            for (int o = 0; o < NO; ++o) acc[o] = fmaf(xv, ws[g + o * G][k], acc[o]);
        }
#pragma unroll
        for (int k = g; k < KC; k += G) {
            const float xv = xs[tok][k];
            ss = fmaf(xv, xv, ss);
        }
        __syncthreads();
    }
#pragma unroll
    for (int off = G / 2; off > 0; off >>= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, off);
    const float r = rsqrtf(ss / (float)F + norm_eps);
    const int64_t t = t0 + tok;
    if (t < n) {
#pragma unroll
        for (int o = 0; o < NO; ++o) mixes[t * MIX + g + o * G] = acc[o] * r;
    }
}

// --------------------------------------------------- k_split_sinkhorn
template <int HC>
__global__ void __launch_bounds__(128) k_split_sinkhorn(int64_t n, int iters, float eps,
                                                        const float *__restrict__ mixes,
                                                        const float *__restrict__ scale,
                                                        const float *__restrict__ base,
                                                        float *__restrict__ pre,
                                                        float *__restrict__ post,
                                                        float *__restrict__ comb) {
    constexpr int MIX = (2 + HC) * HC;
    const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= n) return;
    float m[MIX];
    const float4 *src = reinterpret_cast<const float4 *>(mixes + t * MIX);
#pragma unroll
    for (int q = 0; q < MIX / 4; ++q) {
        const float4 v = __ldg(src + q);
        m[4 * q + 0] = v.x;
        m[4 * q + 1] = v.y;
        m[4 * q + 2] = v.z;
        m[4 * q + 3] = v.w;
    }
    float p[HC], po[HC], C[HC][HC];
    split_sinkhorn_token<HC>([&](int i) { return m[i]; }, [&](int i) { return __ldg(base + i); },
                             __ldg(scale + 0), __ldg(scale + 1), __ldg(scale + 2), iters, eps, p,
                             po, C);
#pragma unroll
    for (int q = 0; q < HC / 4; ++q) {
        reinterpret_cast<float4 *>(pre + t * HC)[q] =
            make_float4(p[4 * q], p[4 * q + 1], p[4 * q + 2], p[4 * q + 3]);
        reinterpret_cast<float4 *>(post + t * HC)[q] =
            make_float4(po[4 * q], po[4 * q + 1], po[4 * q + 2], po[4 * q + 3]);
    }
#pragma unroll
    for (int j = 0; j < HC; ++j)
#pragma unroll
        for (int q = 0; q < HC / 4; ++q)
            reinterpret_cast<float4 *>(comb + (t * HC + j) * HC)[q] =
                make_float4(C[j][4 * q], C[j][4 * q + 1], C[j][4 * q + 2], C[j][4 * q + 3]);
}

// ------------------------------------------------------ stream units
// A unit is (token t, vector segment s) covering 16-byte vectors
// [s*seg, min(nv, (s+1)*seg)) of each of the token's rows.
struct Units {
    int64_t nv;    // vectors per row (d / 8)
    int64_t seg;   // vectors per segment
    int64_t nseg;  // segments per token
};

// ---------------------------------------------------------------- k_pre
template <int HC, int U>
__global__ void __launch_bounds__(256) k_pre(int64_t n, Units un, const uint4 *__restrict__ x,
                                             const float *__restrict__ pre,
                                             uint4 *__restrict__ y) {
    const int lane = threadIdx.x & 31;
    const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const int64_t units = n * un.nseg;
    for (int64_t u = warp; u < units; u += nwarps) {
        const int64_t t = u / un.nseg, s = u % un.nseg;
        const int64_t v0 = s * un.seg, v1 = min(un.nv, v0 + un.seg);
        float p[HC];
#pragma unroll
        for (int q = 0; q < HC / 4; ++q) {
            const float4 v = __ldg(reinterpret_cast<const float4 *>(pre + t * HC) + q);
            p[4 * q] = v.x, p[4 * q + 1] = v.y, p[4 * q + 2] = v.z, p[4 * q + 3] = v.w;
        }
        const uint4 *xt = x + t * HC * un.nv;
        uint4 *yt = y + t * un.nv;
        for (int64_t vb = v0 + lane; vb < v1; vb += 32 * U) {
            uint4 r[U][HC];
#pragma unroll
            for (int a = 0; a < U; ++a) {
                const int64_t v = vb + 32 * a;
                if (v < v1) {
#pragma unroll
                    for (int j = 0; j < HC; ++j) r[a][j] = ld_stream(xt + j * un.nv + v);
                }
            }
#pragma unroll
            for (int a = 0; a < U; ++a) {
                const int64_t v = vb + 32 * a;
                if (v < v1) {
                    float acc[8], f[8];
                    unpack8(r[a][0], f);
#pragma unroll
                    for (int e = 0; e < 8; ++e) acc[e] = p[0] * f[e];
#pragma unroll
                    for (int j = 1; j < HC; ++j) {
                        unpack8(r[a][j], f);
#pragma unroll
                        for (int e = 0; e < 8; ++e) acc[e] = fmaf(p[j], f[e], acc[e]);
                    }
                    st_stream(yt + v, pack8(acc));
                }
            }
        }
    }
}

// --------------------------------------------------------------- k_post
// residual may equal y (in place): each lane loads every copy of a vector
// before it stores any copy of that vector, and vectors are lane-private.
template <int HC, int U>
__global__ void __launch_bounds__(256) k_post(int64_t n, Units un, const uint4 *__restrict__ out,
                                              const uint4 *res, const float *__restrict__ post,
                                              const float *__restrict__ comb, uint4 *y) {
    griddep_wait_then_release();
    const int lane = threadIdx.x & 31;
    const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const int64_t units = n * un.nseg;
    for (int64_t u = warp; u < units; u += nwarps) {
        const int64_t t = u / un.nseg, s = u % un.nseg;
        const int64_t v0 = s * un.seg, v1 = min(un.nv, v0 + un.seg);
        float po[HC], cm[HC][HC];
#pragma unroll
        for (int q = 0; q < HC / 4; ++q) {
            const float4 v = __ldg(reinterpret_cast<const float4 *>(post + t * HC) + q);
            po[4 * q] = v.x, po[4 * q + 1] = v.y, po[4 * q + 2] = v.z, po[4 * q + 3] = v.w;
        }
#pragma unroll
        for (int j = 0; j < HC; ++j)
#pragma unroll
            for (int q = 0; q < HC / 4; ++q) {
                const float4 v =
                    __ldg(reinterpret_cast<const float4 *>(comb + (t * HC + j) * HC) + q);
                cm[j][4 * q] = v.x, cm[j][4 * q + 1] = v.y;
                cm[j][4 * q + 2] = v.z, cm[j][4 * q + 3] = v.w;
            }
        const uint4 *ot = out + t * un.nv;
        const uint4 *rt = res + t * HC * un.nv;
        uint4 *yt = y + t * HC * un.nv;
        for (int64_t vb = v0 + lane; vb < v1; vb += 32 * U) {
            uint4 o[U], r[U][HC];
#pragma unroll
            for (int a = 0; a < U; ++a) {
                const int64_t v = vb + 32 * a;
                if (v < v1) {
                    o[a] = ld_stream(ot + v);
#pragma unroll
                    for (int j = 0; j < HC; ++j) r[a][j] = ld_stream(rt + j * un.nv + v);
                }
            }
#pragma unroll
            for (int a = 0; a < U; ++a) {
                const int64_t v = vb + 32 * a;
                if (v < v1) {
                    float of[8], rf[HC][8];
                    unpack8(o[a], of);
#pragma unroll
                    for (int j = 0; j < HC; ++j) unpack8(r[a][j], rf[j]);
#pragma unroll
                    for (int k = 0; k < HC; ++k) {
                        float acc[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            float s2 = po[k] * of[e];
#pragma unroll
                            for (int j = 0; j < HC; ++j) s2 = fmaf(cm[j][k], rf[j][e], s2);
                            acc[e] = s2;
                        }
                        st_stream(yt + k * un.nv + v, pack8(acc));
                    }
                }
            }
        }
    }
}

// ------------------------------------------------------ k_post_shared
// k_post for large hc (8): the token's post and comb live in a per-warp slot
// of shared memory and are read as broadcasts, instead of 72 registers per
// lane, so that two CTAs fit on an SM (with them in registers the kernel
// needed 187 registers and ran one CTA per SM).  Same arithmetic and order
// as k_post.
template <int HC>
__global__ void __launch_bounds__(256, 2) k_post_shared(int64_t n, Units un,
                                                         const uint4 *__restrict__ out,
                                                         const uint4 *res,
                                                         const float *__restrict__ post,
                                                         const float *__restrict__ comb, uint4 *y) {
    __shared__ float coef[8][HC * HC + HC];  // per warp: comb [j][k], then post [k]
    griddep_wait_then_release();
    const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
    const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const int64_t units = n * un.nseg;
    float *cf = coef[wib];
    for (int64_t u = warp; u < units; u += nwarps) {
        const int64_t t = u / un.nseg, s = u % un.nseg;
        const int64_t v0 = s * un.seg, v1 = min(un.nv, v0 + un.seg);
        __syncwarp();
        for (int q = lane; q < HC * HC; q += 32) cf[q] = __ldg(comb + t * HC * HC + q);
        if (lane < HC) cf[HC * HC + lane] = __ldg(post + t * HC + lane);
        __syncwarp();
        const uint4 *ot = out + t * un.nv;
        const uint4 *rt = res + t * HC * un.nv;
        uint4 *yt = y + t * HC * un.nv;
        for (int64_t v = v0 + lane; v < v1; v += 32) {
            uint4 o = ld_stream(ot + v), r[HC];
#pragma unroll
            for (int j = 0; j < HC; ++j) r[j] = ld_stream(rt + j * un.nv + v);
            float of[8], rf[HC][8];
            unpack8(o, of);
#pragma unroll
            for (int j = 0; j < HC; ++j) unpack8(r[j], rf[j]);
#pragma unroll
            for (int k = 0; k < HC; ++k) {
                const float pk = cf[HC * HC + k];
                float acc[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[e] = pk * of[e];
#pragma unroll
                for (int j = 0; j < HC; ++j) {
                    const float c = cf[j * HC + k];
#pragma unroll
                    for (int e = 0; e < 8; ++e) acc[e] = fmaf(c, rf[j][e], acc[e]);
                }
                st_stream(yt + k * un.nv + v, pack8(acc));
            }
        }
    }
}

// Split each token's nv vectors into segments so that there are enough
// warp units to fill the GPU when n is small.
Units make_units(int64_t n, int64_t nv, int sms) {
    const int64_t target = (int64_t)sms * 32;  // warp units wanted
    int64_t nseg = (target + n - 1) / n;
    const int64_t max_seg = (nv + 31) / 32;
    if (nseg < 1) nseg = 1;
    if (nseg > max_seg) nseg = max_seg;
    int64_t seg = (nv + nseg - 1) / nseg;
    seg = (seg + 31) / 32 * 32;
    Units u;
    u.nv = nv;
    u.seg = seg;
    u.nseg = (nv + seg - 1) / seg;
    return u;
}

int64_t stream_grid(int64_t units, int sms, int blocks_per_sm) {
    const int64_t want = (units + 7) / 8;  // 8 warps per 256-thread block
    const int64_t cap = (int64_t)sms * blocks_per_sm;
    return want < cap ? want : cap;
}

}  // namespace

cudaError_t launch_mixes(int64_t n, int hc, int64_t d, float norm_eps, const uint16_t *x,
                         const float *w, float *mixes, const DeviceInfo &, cudaStream_t s) {
    const int64_t F = (int64_t)hc * d;
    const dim3 grid((unsigned)((n + 31) / 32));
    if (hc == 4)
        k_mixes<4><<<grid, 256, 0, s>>>(n, F, norm_eps, x, w, mixes);
    else
        k_mixes<8><<<grid, 256, 0, s>>>(n, F, norm_eps, x, w, mixes);
    return launched();
}

cudaError_t launch_split_sinkhorn(int64_t n, int hc, int iters, float eps, const float *mixes,
                                  const float *scale, const float *base, float *pre,
                                  float *post, float *comb, const DeviceInfo &, cudaStream_t s) {
    const dim3 grid((unsigned)((n + 127) / 128));
    if (hc == 4)
        k_split_sinkhorn<4><<<grid, 128, 0, s>>>(n, iters, eps, mixes, scale, base, pre, post,
                                                 comb);
    else
        k_split_sinkhorn<8><<<grid, 128, 0, s>>>(n, iters, eps, mixes, scale, base, pre, post,
                                                 comb);
    return launched();
}

cudaError_t launch_pre(int64_t n, int hc, int64_t d, const uint16_t *x, const float *pre,
                       uint16_t *y, const DeviceInfo &di, cudaStream_t s) {
    const Units un = make_units(n, d / 8, di.sms);
    const dim3 grid((unsigned)stream_grid(n * un.nseg, di.sms, 4));
    const uint4 *xv = reinterpret_cast<const uint4 *>(x);
    uint4 *yv = reinterpret_cast<uint4 *>(y);
    if (hc == 4)
        k_pre<4, 2><<<grid, 256, 0, s>>>(n, un, xv, pre, yv);
    else
        k_pre<8, 1><<<grid, 256, 0, s>>>(n, un, xv, pre, yv);
    return launched();
}

cudaError_t launch_post(int64_t n, int hc, int64_t d, const uint16_t *out,
                        const uint16_t *res, const float *post, const float *comb, uint16_t *y,
                        const DeviceInfo &di, cudaStream_t s) {
    const Units un = make_units(n, d / 8, di.sms);
    const dim3 grid((unsigned)stream_grid(n * un.nseg, di.sms, 4));
    const uint4 *ov = reinterpret_cast<const uint4 *>(out);
    const uint4 *rv = reinterpret_cast<const uint4 *>(res);
    uint4 *yv = reinterpret_cast<uint4 *>(y);
    // with programmatic dependent launch (overlap_launches)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(256);
    cfg.stream = s;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = overlap_launches() ? 1 : 0;
    const cudaError_t e =
        hc == 4 ? cudaLaunchKernelEx(&cfg, k_post<4, 2>, n, un, ov, rv, post, comb, yv)
                : cudaLaunchKernelEx(&cfg, k_post_shared<8>, n, un, ov, rv, post, comb, yv);
    if (e != cudaSuccess) return e;
    return launched();
}

}  // namespace hc
