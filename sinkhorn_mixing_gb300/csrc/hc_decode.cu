// hc_decode.cu -- RMS statistic + mix projection + split/Sinkhorn + collapse
// for a few tokens (decode), hc = 4, on sm_103a ("Mix projection" page:
// formula for m, Block.hc_mixes, Block.hc_pre; "Reading weights" page:
// hc_split_sinkhorn).
//
// Work decomposition
//   * A cluster of 16 CTAs (one per SM) takes up to 16 consecutive tokens,
//     and one launch holds as many clusters as the device co-schedules: 64
//     tokens run on 7 clusters (112 SMs) instead of one.
//   * CTA r of a cluster owns channels [r*w, (r+1)*w) of every copy
//     (w = d/16) and keeps its slice of W_mix (fp32, 24 x 4 x w) and of its
//     tokens' x (bf16, tokens x 4 x w) in shared memory.
//   * The slices arrive by asynchronous copies: W's before the wait for the
//     kernel in front (W is a parameter), x's after it; the projection
//     starts when all are in.
//   * Partial mix numbers and sums of squares on CUDA cores (packed
//     two-wide fma): warp (g, h) takes tokens 4g..4g+3 and mixes 6h..6h+5
//     (and the squares of token 4g+h) over all 4w features, each lane the
//     feature pairs 64 apart starting at 2*lane; the 32 lanes' partials are
//     then summed in lane order through shared memory.
//   * Each CTA sends its 25 partial numbers per token (24 mixes, sum of
//     squares) to the token's owner, CTA t of the cluster for its token t,
//     with asynchronous 4-byte stores whose bytes complete the owner's
//     barrier.  The owner sums the 16 records in CTA order, forms r, m and
//     pre and sends pre to all 16 CTAs the same way; beside it, warp 15 of
//     the owner CTA (one the collapse of up to 14 tokens leaves idle) runs
//     the Sinkhorn for comb from the mix numbers the owner left in shared
//     memory.
//   * Every CTA collapses its own w channels of the cluster's tokens from the
//     x slice it holds, so x is read from memory once.
//
// Every wait is bounded: a wait that exceeds the time limit sets the CTA's
// abort flag and bit 0 of the device error word, and the CTA runs to the
// teardown (no trap; no CTA leaves its cluster while another may still
// address its shared memory).
#include <cuda.h>

#include <mutex>

#include "hc_common.cuh"
#include "hc_decode.h"
#include "hc_ptx.cuh"

namespace hc {
namespace {

using namespace ptx;

constexpr int kCluster = 16;
constexpr int kMix = 24;
constexpr int kMaxTok = 16;           // tokens per cluster, one owner CTA each
constexpr int kRecVals = kMix + 1;    // per (sender, token): 24 mixes + sum of squares
constexpr int kRecStride = 28;        // floats between two senders' records
constexpr int kWarps = 16;            // warp (g, h): tokens 4g.., mixes 6h..
constexpr int kThreads = kWarps * 32;
constexpr int kPartVals = 28;         // per warp: 4 tokens x 6 mixes + slots for 4 sums of squares
constexpr int kPartStride = 33;       // lanes per partial value, padded: no bank conflicts
constexpr int kMaxW = 320;            // channels per CTA (d <= 5120)

struct DecodeParams {
    int n;
    int d;
    int w;     // channels per CTA, d / 16
    int tpc;   // tokens per cluster
    int iters;
    int mixes_only;
    float eps;
    float norm_eps;
    float F;
    const uint16_t *x;
    const float *w_mix;
    const float *scale;
    const float *base;
    float *mixes;
    float *pre;
    float *post;
    float *comb;
    uint16_t *y;
    unsigned int *err;
    const float *rms_w;  // RMSNorm weight of the sublayer input, or null
    float rms_eps;
    // hc_post of the previous sublayer in front (null out: none): x is its
    // residual stream, and the kernel works on x_next = hc_post(out, x,
    // post_in, comb_in), which it also writes (x_next may be x itself)
    const uint16_t *out;
    const float *post_in;
    const float *comb_in;
    uint16_t *x_next;
};

__host__ __device__ constexpr int round4(int t) { return (t + 3) & ~3; }

// 16-byte asynchronous copy global -> shared (cached in L2 only).
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
// Wait until all of this thread's copy groups are in.
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.wait_group 0;" ::: "memory");
}

// W slice [24][4w] fp32, later reused for the lanes' partials
__host__ __device__ constexpr size_t wreg_bytes(int w) {
    return (size_t)kMix * 4 * w * 4 > (size_t)kWarps * kPartVals * kPartStride * 4
               ? (size_t)kMix * 4 * w * 4
               : (size_t)kWarps * kPartVals * kPartStride * 4;
}
// x slice [round4(tpc)][4w] bf16
__host__ __device__ constexpr size_t xreg_bytes(int w, int tpc) {
    return (size_t)round4(tpc) * 4 * w * 2;
}
// the previous sublayer's output slice [round4(tpc)][w] bf16 (with hc_post in front)
__host__ __device__ constexpr size_t oreg_bytes(int w, int tpc) {
    return (size_t)round4(tpc) * w * 2;
}
__host__ __device__ constexpr size_t smem_bytes(int w, int tpc) {
    return wreg_bytes(w) + xreg_bytes(w, tpc) + oreg_bytes(w, tpc) + kCluster * kRecStride * 4 +
           kMaxTok * 4 * 4 +
           kCluster * kMaxTok * 4 + 32 * 4 + 4 * 8 + 16;
}

__global__ void __launch_bounds__(kThreads, 1) k_decode(const DecodeParams p) {
    extern __shared__ __align__(16) uint8_t smem[];
    const int w = p.w, nf = 4 * w;
    const size_t wreg = wreg_bytes(w);
    float *ws = reinterpret_cast<float *>(smem);    // [24][nf]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rank = (int)(blockIdx.x % kCluster);
    const int64_t F = 4LL * p.d;
    float *part = ws;                               // [16 warps][28][33], after the projection
    uint16_t *xs = reinterpret_cast<uint16_t *>(smem + wreg);  // [round4(tpc)][nf]
    uint16_t *osh = reinterpret_cast<uint16_t *>(smem + wreg + xreg_bytes(w, p.tpc));  // [tpc][w]
    float *recv = reinterpret_cast<float *>(smem + wreg + xreg_bytes(w, p.tpc) +
                                            oreg_bytes(w, p.tpc));  // [16][28]
    float *preb = recv + kCluster * kRecStride;     // [16][4]: pre of the cluster's tokens
    float *normp = preb + kMaxTok * 4;              // [16 senders][16 tokens]: partial sums of y^2
    float *msh = normp + kCluster * kMaxTok;        // [24 (+8)]: the owned token's mix numbers
    uint64_t *bars = reinterpret_cast<uint64_t *>(msh + 32);
    int *abort_word = reinterpret_cast<int *>(bars + 4);
    volatile int *abort = abort_word;
    const int64_t tok0 = (int64_t)(blockIdx.x / kCluster) * p.tpc;
    const int tv = (int)((int64_t)p.n - tok0 < p.tpc ? (int64_t)p.n - tok0 : p.tpc);
    const bool mixes_only = p.mixes_only != 0;
    const uint32_t bRecv = su32(bars), bPre = su32(bars + 1), bNorm = su32(bars + 2);
    const uint32_t bMix = su32(bars + 3);  // msh holds the owned token's mix numbers
    constexpr int kWarpComb = kWarps - 1;  // runs the owned token's Sinkhorn
    const bool norm = p.rms_w != nullptr && !mixes_only;

    // Each barrier completes once: recv when the 16 records of this CTA's
    // token are in (owners only), pre when pre of all tv tokens is in, norm
    // (with the RMSNorm) when every CTA's partial sum of y^2 of every token is,
    // mix when the owner has put its token's mix numbers in msh.  All of it
    // comes from the launch parameters, so it is done first, and the cluster
    // arrival (a release) comes before any copy is in flight: a release waits
    // for this thread's earlier memory operations, the copies included.
    if (threadIdx.x == 0) {
        *abort_word = 0;
        mbar_init(bRecv, 1);
        mbar_init(bPre, 1);
        mbar_init(bNorm, 1);
        mbar_init(bMix, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        if (rank < tv) mbar_expect_tx(bRecv, kCluster * kRecVals * 4);
        if (!mixes_only) mbar_expect_tx(bPre, (uint32_t)tv * 16);
        if (norm) mbar_expect_tx(bNorm, (uint32_t)(kCluster * tv * 4));
    }
    cluster_arrive();  // waited for before the first remote store

    // The W slice (row i, copy j -> W[i][j*d + r*w ...], w floats), before
    // the wait for the kernel in front: W_mix is a parameter, not an
    // activation, so its copies overlap that kernel's tail (with programmatic
    // dependent launch) and everything the kernel in front writes is read
    // only after the wait.  Rows by warp, 16-byte pieces by lane: no division
    // in the index math.
    for (int j = 0; j < 4; ++j) {
        const int wv = w / 4;
        for (int i = warp; i < kMix; i += kWarps) {
            const float *src = p.w_mix + (int64_t)i * F + (int64_t)j * p.d + rank * w;
            const uint32_t dst = su32(ws + i * nf + j * w);
            for (int q = lane; q < wv; q += 32) cp_async16(dst + 16 * q, src + 4 * q);
        }
    }
    cp_async_commit();
    griddep_wait_then_release();

    // The x slice (token t, copy j -> x[tok0+t][j][r*w ...]) follows as
    // asynchronous copies.  Rows up to the next multiple of 4 tokens are zero.
    const bool post_in_front = p.out != nullptr;
    if (post_in_front) {
        // With hc_post in front the new stream needs all four copies of a
        // channel at once: one group takes the residual slice (all copies)
        // and the output slice.
        const int xv = w / 8, tz = round4(tv);
        for (int e = warp; e < 5 * tz; e += kWarps) {
            const int t = e / 5, j = e % 5;  // j < 4: copy j of the residual; 4: out
            uint16_t *dst = j < 4 ? xs + t * nf + j * w : osh + t * w;
            if (t < tv) {
                const uint16_t *src = j < 4 ? p.x + ((tok0 + t) * 4 + j) * (int64_t)p.d + rank * w
                                            : p.out + (tok0 + t) * (int64_t)p.d + rank * w;
                for (int q = lane; q < xv; q += 32) cp_async16(su32(dst + 8 * q), src + 8 * q);
            } else {
                for (int q = lane; q < xv; q += 32)
                    *reinterpret_cast<uint4 *>(dst + 8 * q) = make_uint4(0u, 0u, 0u, 0u);
            }
        }
        cp_async_commit();
        cp_async_wait_all();
        __syncthreads();  // the residual and output slices (and W) are in
        // hc_post ("Mix projection" page, Block.hc_post), in the order of
        // k_post: x'_k = post_k out + sum_i comb[i][k] x_i, rounded to bf16,
        // written over the residual in shared memory (all four copies of a
        // vector are read before any is written) and to x_next
        for (int e = threadIdx.x; e < tv * xv; e += kThreads) {
            const int t = e / xv, v = e % xv;
            const int64_t tok = tok0 + t;
            float po[4], cm[4][4];
            const float4 pv = __ldg(reinterpret_cast<const float4 *>(p.post_in) + tok);
            po[0] = pv.x, po[1] = pv.y, po[2] = pv.z, po[3] = pv.w;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float4 cv = __ldg(reinterpret_cast<const float4 *>(p.comb_in) + tok * 4 + i);
                cm[i][0] = cv.x, cm[i][1] = cv.y, cm[i][2] = cv.z, cm[i][3] = cv.w;
            }
            float of[8], rf[4][8];
            unpack8(*reinterpret_cast<const uint4 *>(osh + t * w + 8 * v), of);
#pragma unroll
            for (int i = 0; i < 4; ++i)
                unpack8(*reinterpret_cast<const uint4 *>(xs + t * nf + i * w + 8 * v), rf[i]);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                float acc[8];
#pragma unroll
                for (int e2 = 0; e2 < 8; ++e2) {
                    float s2 = po[k] * of[e2];
#pragma unroll
                    for (int i = 0; i < 4; ++i) s2 = fmaf(cm[i][k], rf[i][e2], s2);
                    acc[e2] = s2;
                }
                const uint4 nv = pack8(acc);
                *reinterpret_cast<uint4 *>(xs + t * nf + k * w + 8 * v) = nv;
                st_stream(reinterpret_cast<uint4 *>(p.x_next + (tok * 4 + k) * (int64_t)p.d +
                                                    rank * w + 8 * v),
                          nv);
            }
        }
    } else {
        const int xv = w / 8, tz = round4(tv);
        for (int j = 0; j < 4; ++j) {
            for (int t = warp; t < tz; t += kWarps) {
                uint16_t *dst = xs + t * nf + j * w;
                if (t < tv) {
                    const uint16_t *src = p.x + ((tok0 + t) * 4 + j) * (int64_t)p.d + rank * w;
                    for (int q = lane; q < xv; q += 32) cp_async16(su32(dst + 8 * q), src + 8 * q);
                } else {
                    for (int q = lane; q < xv; q += 32)
                        *reinterpret_cast<uint4 *>(dst + 8 * q) = make_uint4(0u, 0u, 0u, 0u);
                }
            }
        }
        cp_async_commit();
    }

    // Partial mix numbers of tokens 4g..4g+3 and the sum of squares of token
    // 4g+h, as pairs (even feature, odd feature) summed at the end.  One wait
    // for every copy group, then no barrier until the projection is done, so
    // that the warps drift apart and one warp's shared-memory loads overlap
    // another's FMAs (with a barrier per copy they ran in lockstep: loads,
    // then FMAs).
    const int g = warp >> 2, h = warp & 3;
    const bool active = 4 * g < tv;
    uint64_t acc[4][6], ssq = 0;
#pragma unroll
    for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int k = 0; k < 6; ++k) acc[u][k] = 0;
    cp_async_wait_all();
    __syncthreads();  // every thread's copies are in
    if (active) {
        for (int j = 0; j < 4; ++j) {
            // unrolled, so that the loads of several feature blocks are in
            // flight together (the loop is bound by shared-memory latency)
#pragma unroll 5
            for (int f = j * w + 2 * lane; f < (j + 1) * w; f += 64) {
                uint64_t wv[6];
#pragma unroll
                for (int k = 0; k < 6; ++k)
                    wv[k] = *reinterpret_cast<const uint64_t *>(ws + (6 * h + k) * nf + f);
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const uint32_t xx =
                        *reinterpret_cast<const uint32_t *>(xs + (4 * g + u) * nf + f);
                    const uint64_t xp = pack2(bf16lo(xx), bf16hi(xx));
#pragma unroll
                    for (int k = 0; k < 6; ++k) ffma2(acc[u][k], xp, wv[k]);
                    if (u == h) ffma2(ssq, xp, xp);
                }
            }
        }
    }
    __syncthreads();  // W is no longer read: its space takes the partials
    if (active) {
        float *pw = part + warp * kPartVals * kPartStride;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
#pragma unroll
            for (int k = 0; k < 6; ++k) pw[(u * 6 + k) * kPartStride + lane] = sum2(acc[u][k]);
        }
        pw[(24 + h) * kPartStride + lane] = sum2(ssq);
    }
    __syncthreads();
    cluster_wait();  // every CTA's barriers exist and are armed

    // Sum each value over the 32 lanes in lane order and send it to the
    // owner of its token: record slot [rank][mix] (slot 24: sum of squares).
    for (int e = threadIdx.x; e < kWarps * kPartVals; e += kThreads) {
        const int ww = e / kPartVals, v = e % kPartVals;
        const int hh = ww & 3;
        const int u = v < 24 ? v / 6 : v - 24;
        const int t = 4 * (ww >> 2) + u;
        if (t >= tv || (v >= 24 && hh != u)) continue;  // token u's squares: warp h = u
        const int slot = v < 24 ? 6 * hh + v % 6 : kMix;
        const float *src = part + (ww * kPartVals + v) * kPartStride;
        float s = 0.f;
#pragma unroll 8
        for (int l = 0; l < 32; ++l) s += src[l];
        st_async_f32(mapa(su32(recv + rank * kRecStride + slot), (uint32_t)t), s,
                     mapa(bRecv, (uint32_t)t));
    }
    __syncthreads();  // the partials are read: their space may take the collapsed rows

    if (rank < tv && warp == 0) {
        // Owner of token tok0 + rank: lane k < 25 sums value k of the 16
        // records in CTA order.
        if (__all_sync(0xFFFFFFFFu, wait_bar<true>(bRecv, 0, abort, p.err))) {
            float v = 0.f;
            if (lane < kRecVals)
                for (int s2 = 0; s2 < kCluster; ++s2) v += recv[s2 * kRecStride + lane];
            const float ssum = __shfl_sync(0xFFFFFFFFu, v, kMix);
            const float r = rsqrtf(ssum / p.F + p.norm_eps);
            const float m = v * r;
            const int64_t t = tok0 + rank;
            if (p.mixes != nullptr && lane < kMix) p.mixes[t * kMix + lane] = m;
            if (!mixes_only) {
                // the mix numbers to the Sinkhorn warp first, so that comb
                // is computed beside the split and the pre broadcast
                if (lane < kMix) msh[lane] = m;
                __syncwarp();
                if (lane == 0) mbar_arrive(bMix);
                float mm[kMix], bse[kMix];
#pragma unroll
                for (int k = 0; k < kMix; ++k) {
                    mm[k] = __shfl_sync(0xFFFFFFFFu, m, k);
                    bse[k] = __ldg(p.base + k);
                }
                const float s0 = __ldg(p.scale + 0), s1 = __ldg(p.scale + 1);
                float pr[4], po[4];
                split_pre_post<4>([&](int k) { return mm[k]; }, [&](int k) { return bse[k]; },
                                  s0, s1, p.eps, pr, po);
                // pre to every CTA of the cluster, then comb off the collapse's path
                if (lane < kCluster)
                    st_async_v4(mapa(su32(preb + rank * 4), (uint32_t)lane), pr[0], pr[1], pr[2],
                                pr[3], mapa(bPre, (uint32_t)lane));
                if (lane == 0) {
                    reinterpret_cast<float4 *>(p.pre)[t] = make_float4(pr[0], pr[1], pr[2], pr[3]);
                    reinterpret_cast<float4 *>(p.post)[t] =
                        make_float4(po[0], po[1], po[2], po[3]);
                }
            }
        }
    } else if (!mixes_only && warp > 0) {
        if (warp == kWarpComb && rank < tv) {
            // comb of the owned token, on one lane (spread over 16 lanes, one
            // entry each with shuffle row and column sums, it measured
            // slower: a shuffle costs more than the other rows' steps it
            // saves), beside the owner warp's split and pre broadcast; then
            // this warp's share of the collapse as usual
            if (__all_sync(0xFFFFFFFFu, wait_bar<false>(bMix, 0, abort, p.err)) && lane == 0) {
                float Cm[4][4];
                sinkhorn_comb<4>([&](int k) { return msh[k]; }, [&](int k) { return __ldg(p.base + k); },
                                 __ldg(p.scale + 2), p.iters, p.eps, Cm);
                const int64_t t = tok0 + rank;
#pragma unroll
                for (int jj = 0; jj < 4; ++jj)
                    reinterpret_cast<float4 *>(p.comb)[t * 4 + jj] =
                        make_float4(Cm[jj][0], Cm[jj][1], Cm[jj][2], Cm[jj][3]);
            }
            __syncwarp();
        }
        // Collapse y = sum_j pre_j x_j of this CTA's channels, warps 1..15,
        // one token per warp at a time.  With the RMSNorm the rows are kept
        // in shared memory (bf16), the warp's partial sum of y^2 goes to every
        // CTA of the cluster, and the rows are scaled once all 16 are in.
        if (__all_sync(0xFFFFFFFFu, wait_bar<true>(bPre, 0, abort, p.err))) {
            const int xv = w / 8;
            uint4 *ybuf = reinterpret_cast<uint4 *>(ws);  // [16 tokens][xv]
            for (int t = warp - 1; t < tv; t += kWarps - 1) {
                const float4 pr = reinterpret_cast<const float4 *>(preb)[t];
                const uint16_t *xt = xs + t * nf;
                uint4 *yt = reinterpret_cast<uint4 *>(p.y + (tok0 + t) * (int64_t)p.d + rank * w);
                float ss = 0.f;
                for (int q = lane; q < xv; q += 32) {
                    float acc8[8], f8[8];
                    unpack8(reinterpret_cast<const uint4 *>(xt)[q], f8);
#pragma unroll
                    for (int e = 0; e < 8; ++e) acc8[e] = pr.x * f8[e];
                    unpack8(reinterpret_cast<const uint4 *>(xt + w)[q], f8);
#pragma unroll
                    for (int e = 0; e < 8; ++e) acc8[e] = fmaf(pr.y, f8[e], acc8[e]);
                    unpack8(reinterpret_cast<const uint4 *>(xt + 2 * w)[q], f8);
#pragma unroll
                    for (int e = 0; e < 8; ++e) acc8[e] = fmaf(pr.z, f8[e], acc8[e]);
                    unpack8(reinterpret_cast<const uint4 *>(xt + 3 * w)[q], f8);
#pragma unroll
                    for (int e = 0; e < 8; ++e) acc8[e] = fmaf(pr.w, f8[e], acc8[e]);
                    const uint4 yv = pack8(acc8);
                    if (!norm) {
                        st_stream(yt + q, yv);
                    } else {
                        ybuf[t * xv + q] = yv;
                        unpack8(yv, f8);
#pragma unroll
                        for (int e = 0; e < 8; ++e) ss = fmaf(f8[e], f8[e], ss);
                    }
                }
                if (norm) {
#pragma unroll
                    for (int off = 16; off > 0; off >>= 1)
                        ss += __shfl_xor_sync(0xFFFFFFFFu, ss, off);
                    if (lane < kCluster)
                        st_async_f32(mapa(su32(normp + rank * kMaxTok + t), (uint32_t)lane), ss,
                                     mapa(bNorm, (uint32_t)lane));
                }
            }
            if (norm &&
                __all_sync(0xFFFFFFFFu, wait_bar<true>(bNorm, 0, abort, p.err))) {
                for (int t = warp - 1; t < tv; t += kWarps - 1) {
                    float tot = 0.f;
                    for (int s2 = 0; s2 < kCluster; ++s2) tot += normp[s2 * kMaxTok + t];
                    const float r = rsqrtf(tot / (float)p.d + p.rms_eps);
                    uint4 *yt =
                        reinterpret_cast<uint4 *>(p.y + (tok0 + t) * (int64_t)p.d + rank * w);
                    const float4 *gw = reinterpret_cast<const float4 *>(p.rms_w + rank * w);
                    for (int q = lane; q < xv; q += 32) {
                        float f8[8], o8[8];
                        unpack8(ybuf[t * xv + q], f8);
                        const float4 g0 = __ldg(gw + 2 * q), g1 = __ldg(gw + 2 * q + 1);
                        const float gv[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
#pragma unroll
                        for (int e = 0; e < 8; ++e) o8[e] = (f8[e] * r) * gv[e];
                        st_stream(yt + q, pack8(o8));
                    }
                }
            }
        }
    }

    // A CTA that took a store from another CTA waited for it above, so no
    // store is still in flight toward a CTA that passes this barrier: the
    // barrier needs no release (pending global stores need not drain).
    __syncwarp();
    __syncthreads();
    asm volatile("barrier.cluster.arrive.relaxed.aligned;\n\t"
                 "barrier.cluster.wait.aligned;" ::: "memory");
}

// ---------------------------------------------------------------- host

struct DevState {
    bool init = false;
    unsigned long long ctx = 0;  // the context the set-up below was done in
    bool ok = false;
    int max_clusters = 0;
};
std::mutex g_dmu;
DevState g_dec[64];

const DevState &dec_state(const DeviceInfo &di) {
    std::lock_guard<std::mutex> lk(g_dmu);
    DevState &st = g_dec[di.device];
    if (st.init && st.ctx == di.ctx) return st;
    st = DevState();
    st.init = true;
    st.ctx = di.ctx;
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, di.device) != cudaSuccess) return st;
    if (prop.major != 10 || prop.minor != 3) return st;  // built for sm_103a only
    const size_t smem = smem_bytes(kMaxW, kMaxTok);
    if (cudaFuncSetAttribute(k_decode, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
            cudaSuccess ||
        cudaFuncSetAttribute(k_decode, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) !=
            cudaSuccess) {
        cudaGetLastError();
        return st;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(kCluster);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = kCluster;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int nc = 0;
    if (cudaOccupancyMaxActiveClusters(&nc, (void *)k_decode, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return st;
    }
    st.max_clusters = nc;
    st.ok = nc > 0;
    return st;
}

}  // namespace

bool decode_supported(int64_t n, int hc, int64_t d, const DeviceInfo &di) {
    if (hc != 4 || n < 1 || d % (kCluster * 16) != 0 || d > (int64_t)kCluster * kMaxW) return false;
    if (forced_path() != kPathAuto) return false;
    const DevState &st = dec_state(di);
    return st.ok && n <= (int64_t)kMaxTok * st.max_clusters;
}

namespace {

cudaError_t launch_decode_impl(int64_t n, int hc, int64_t d, int iters, float eps, float norm_eps,
                               const uint16_t *x, const float *w, const float *scale,
                               const float *base, float *mixes, float *pre, float *post,
                               float *comb, uint16_t *y, const float *rms_w, float rms_eps,
                               const uint16_t *out, const float *post_in, const float *comb_in,
                               uint16_t *x_next, const DeviceInfo &di, cudaStream_t s) {
    const DevState &st = dec_state(di);
    if (!st.ok || hc != 4 || n < 1 || n > (int64_t)kMaxTok * st.max_clusters)
        return cudaErrorNotSupported;
    DecodeParams p;
    p.n = (int)n;
    p.d = (int)d;
    p.w = (int)(d / kCluster);
    p.tpc = (int)((n + st.max_clusters - 1) / st.max_clusters);
    p.iters = iters;
    p.mixes_only = pre == nullptr ? 1 : 0;
    p.eps = eps;
    p.norm_eps = norm_eps;
    p.F = (float)(4 * d);
    p.x = x;
    p.w_mix = w;
    p.scale = scale;
    p.base = base;
    p.mixes = mixes;
    p.pre = pre;
    p.post = post;
    p.comb = comb;
    p.y = y;
    p.err = di.err_word;
    p.rms_w = rms_w;
    p.rms_eps = rms_eps;
    p.out = out;
    p.post_in = post_in;
    p.comb_in = comb_in;
    p.x_next = x_next;
    const int nclusters = (int)((n + p.tpc - 1) / p.tpc);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(nclusters * kCluster));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem_bytes(p.w, p.tpc);
    cfg.stream = s;
    // 16-CTA clusters, with programmatic dependent launch (overlap_launches)
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kCluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = overlap_launches() ? 2 : 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, k_decode, p);
    if (e != cudaSuccess) return e;
    return launched();
}

}  // namespace

cudaError_t launch_decode(int64_t n, int hc, int64_t d, int iters, float eps, float norm_eps,
                          const uint16_t *x, const float *w, const float *scale,
                          const float *base, float *mixes, float *pre, float *post,
                          float *comb, uint16_t *y, const float *rms_w, float rms_eps,
                          const DeviceInfo &di, cudaStream_t s) {
    return launch_decode_impl(n, hc, d, iters, eps, norm_eps, x, w, scale, base, mixes, pre, post,
                              comb, y, rms_w, rms_eps, nullptr, nullptr, nullptr, nullptr, di, s);
}

cudaError_t launch_decode_post(int64_t n, int hc, int64_t d, const uint16_t *out,
                               const uint16_t *residual, const float *post_in,
                               const float *comb_in, uint16_t *x_next, int iters, float eps,
                               float norm_eps, const float *w, const float *scale,
                               const float *base, float *mixes, float *pre, float *post,
                               float *comb, uint16_t *y, const DeviceInfo &di, cudaStream_t s) {
    if (pre == nullptr) return cudaErrorNotSupported;
    return launch_decode_impl(n, hc, d, iters, eps, norm_eps, residual, w, scale, base, mixes, pre,
                              post, comb, y, nullptr, 0.f, out, post_in, comb_in, x_next, di, s);
}

}  // namespace hc
