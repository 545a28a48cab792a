// hc_mixtc.cu -- RMS statistic + mix projection on the tensor cores for any
// token count, hc in {4, 8}, with W_mix streamed rather than resident
// ("Mix projection" page: the formula for m, Block.hc_mixes).
//
// Work decomposition
//   * Persistent CTAs, one per SM, take units of kTPU consecutive 128-token
//     tiles in turn.  A unit's feature axis is walked in stages of 64
//     features: TMA brings each tile's x sub-tile [128 tokens x 64]
//     (128-byte swizzled, K-major) and one W sub-tile [mix x 64] (fp32 rows)
//     into a ring of kStages slots.  An SM's intake of W is what bounds the
//     kernel at hc = 8 (W is 13 MB, read from L2 once per unit), so there a
//     unit is two tiles sharing every W stage.
//   * 4 convert warps split the W sub-tile into bf16 hi rows (bf16(W)) and lo
//     rows (bf16(W - hi)) in the swizzled K-major layout the tensor core
//     reads.  At hc = 8 that conversion is a fifth of the kernel's shared-
//     memory traffic, so when the caller provides room, k_convert_w writes
//     the hi/lo rows to global memory once per call and the kernel (PRE)
//     loads them by TMA, already swizzled, with a deeper ring.
//   * Per stage and tile, 4 tcgen05.mma (M = 128 tokens, N = 2*mix rows of hi
//     and lo, K = 16) accumulate x.(W_hi + W_lo) in TMEM (binary32).  bf16 x is exact
//     and hi + lo carries ~16 mantissa bits of W.  The tensor core's own
//     accumulation loses about one binary32 unit per step in one direction, so
//     a unit's feature axis is cut into parts of kPart stages (256 MMA steps):
//     each part accumulates in TMEM and the epilogue adds the parts in
//     binary32 registers (round to nearest); with one tile per unit two TMEM
//     buffers let the MMAs go on during the read-out.  One chain over 40,960
//     features was off by 1.4e-4 relative.
//   * 4 square warps add x^2 per token from the same sub-tiles.
//   * 4 epilogue warps per tile (one per TMEM lane quadrant, 32 tokens each)
//     read the accumulators, add hi and lo, scale by r = 1/sqrt(mean x^2 +
//     eps) and write the mix numbers.
// Every wait is bounded; a timeout sets the CTA's abort flag and bit 0 of the
// device error word, and all roles run to the teardown (no trap; TMEM and
// in-flight copies are always waited for).
#include <cuda.h>

#include <mutex>

#include "hc_common.cuh"
#include "hc_internal.h"
#include "hc_ptx.cuh"

namespace hc {
namespace {

using namespace ptx;

constexpr int kTok = 128;                // tokens per tile (MMA M)
constexpr int kK = 64;                   // features per stage
constexpr int kXBytes = kTok * kK * 2;   // x sub-tile, 16 KB
constexpr int kPart = 64;                // stages per tensor-core accumulation chain
// warp roles: 0 producer, 1 MMA, 2..5 squares (32 tokens of every tile each),
// 6, 7 and the two after the epilogue warps convert W, 8.. epilogue (4 per
// tile of a unit, one per TMEM lane quadrant)
constexpr int kWarpProducer = 0;
constexpr int kWarpMma = 1;
constexpr int kWarpSq0 = 2;
constexpr int kWarpEpi0 = 8;

template <int HC, bool PRE = false>
struct Cfg {
    static constexpr int kMix = (2 + HC) * HC;      // 24 or 80
    static constexpr int kNW = 2 * kMix;            // B rows: hi then lo
    static constexpr int kTPU = HC == 8 ? 2 : 1;    // tiles per unit
    static constexpr int kAccBufs = kTPU == 1 ? 2 : 1;
    static constexpr int kStages = HC == 8 ? (PRE ? 4 : 3) : 6;
    static constexpr int kWfBytes = kMix * kK * 4;  // fp32 W sub-tile
    static constexpr int kWbBytes = kNW * kK * 2;   // bf16 hi/lo sub-tile
    static constexpr int kXStage = kTPU * kXBytes;  // x sub-tiles of a stage
    static constexpr int kTmemCols = HC == 8 ? 512 : 128;
    static constexpr int kWarps = 10 + 4 * kTPU;
    static constexpr int kThreads = kWarps * 32;
    // tcgen05 instruction descriptor: D f32, A/B bf16, K-major, N = kNW, M = 128
    static constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) |
                                       ((uint32_t)(kNW >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
    static_assert(kNW % 16 == 0 && kNW <= 256, "MMA N");
    static_assert(kAccBufs * kTPU * kNW <= kTmemCols, "accumulators fit in TMEM");
    static_assert(kWbBytes % 1024 == 0 && kWfBytes % 1024 == 0, "swizzle atoms and TMA alignment");
    __host__ __device__ static constexpr bool is_convert(int w) {
        return w == 6 || w == 7 || w == kWarpEpi0 + 4 * kTPU || w == kWarpEpi0 + 4 * kTPU + 1;
    }
    __host__ __device__ static constexpr int convert_index(int w) {
        return w < kWarpEpi0 ? w - 6 : w - (kWarpEpi0 + 4 * kTPU) + 2;
    }
};

struct MixParams {
    int64_t n;
    int F;
    int nk;         // stages per unit, F / 64
    int num_tiles;
    int num_units;
    float norm_eps;
    float *mixes;
    unsigned int *err;
};

template <int HC, bool PRE>
__host__ __device__ constexpr size_t ring_bytes() {
    using C = Cfg<HC, PRE>;
    return (size_t)C::kStages * (C::kXStage + C::kWbBytes + (PRE ? 0 : C::kWfBytes));
}

// barrier indices
template <int HC, bool PRE>
struct Bars {
    static constexpr int S = Cfg<HC, PRE>::kStages;
    static constexpr int A = Cfg<HC, PRE>::kAccBufs;
    static constexpr int full(int s) { return s; }
    static constexpr int conv(int s) { return S + s; }
    static constexpr int empty(int s) { return 2 * S + s; }
    static constexpr int acc_full(int b) { return 3 * S + b; }
    static constexpr int acc_empty(int b) { return 3 * S + A + b; }
    static constexpr int sq_full(int b) { return 3 * S + 2 * A + b; }
    static constexpr int sq_empty(int b) { return 3 * S + 2 * A + 2 + b; }
    static constexpr int drain = 3 * S + 2 * A + 4;
    static constexpr int count = drain + 1;
};

template <int HC, bool PRE>
__host__ __device__ constexpr size_t smem_bytes() {
    return 1024 /* alignment slack */ + ring_bytes<HC, PRE>() + 2 * Cfg<HC, PRE>::kTPU * kTok * 4 +
           Bars<HC, PRE>::count * 8 + 16;
}

// W fp32 [kMix][F] -> the B rows of every 64-feature stage, bf16, unswizzled:
// wc[kc][r][64] with r < kMix the hi rows bf16(W) and r = kMix + i the lo rows
// bf16(W - hi) -- the same numbers the convert warps write into shared memory.
template <int HC>
__global__ void __launch_bounds__(256) k_convert_w(int F, const float *__restrict__ w,
                                                   uint4 *__restrict__ wc) {
    constexpr int kMix = Cfg<HC>::kMix;
    const int64_t total = (int64_t)(F / kK) * kMix * 8;  // (stage, row, 8-feature piece)
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total;
         e += (int64_t)gridDim.x * blockDim.x) {
        const int q = (int)(e & 7);
        const int64_t rest = e >> 3;
        const int i = (int)(rest % kMix);
        const int64_t kc = rest / kMix;
        const float4 *src = reinterpret_cast<const float4 *>(w + (int64_t)i * F + kc * kK + q * 8);
        const float4 a = __ldg(src), b2 = __ldg(src + 1);
        const float v[8] = {a.x, a.y, a.z, a.w, b2.x, b2.y, b2.z, b2.w};
        float lo[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) lo[u] = v[u] - __bfloat162float(__float2bfloat16_rn(v[u]));
        uint4 hv, lv;
        hv.x = pack_bf16x2(v[0], v[1]);
        hv.y = pack_bf16x2(v[2], v[3]);
        hv.z = pack_bf16x2(v[4], v[5]);
        hv.w = pack_bf16x2(v[6], v[7]);
        lv.x = pack_bf16x2(lo[0], lo[1]);
        lv.y = pack_bf16x2(lo[2], lo[3]);
        lv.z = pack_bf16x2(lo[4], lo[5]);
        lv.w = pack_bf16x2(lo[6], lo[7]);
        uint4 *st = wc + kc * (2 * kMix) * 8;  // stage kc: 2*kMix rows of 8 pieces
        st[i * 8 + q] = hv;
        st[(kMix + i) * 8 + q] = lv;
    }
}

template <int HC, bool PRE>
__global__ void __launch_bounds__(Cfg<HC, PRE>::kThreads, 1)
    k_mixtc(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
            const MixParams p) {
    using C = Cfg<HC, PRE>;
    using B = Bars<HC, PRE>;
    constexpr int S = C::kStages;
    constexpr int TPU = C::kTPU;
    constexpr int AB = C::kAccBufs;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint8_t *xr = base;                               // [S][TPU][128 x 64] bf16, swizzled
    uint8_t *wb = xr + (size_t)S * C::kXStage;        // [S][kNW x 64] bf16, swizzled
    float *wf = reinterpret_cast<float *>(wb + (size_t)S * C::kWbBytes);  // [S][kMix][64], !PRE
    float *sq = wf + (PRE ? 0 : (size_t)S * C::kMix * kK);  // [2][TPU][128]
    uint64_t *bars = reinterpret_cast<uint64_t *>(sq + 2 * TPU * kTok);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + B::count);
    int *abort_word = reinterpret_cast<int *>(tmem_slot + 1);
    volatile int *abort = abort_word;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int U = (int)blockIdx.x < p.num_units
                      ? (p.num_units - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x
                      : 0;
    auto bar = [&](int i) { return su32(bars + i); };

    if (threadIdx.x == 0) {
        *abort_word = 0;
        for (int s = 0; s < S; ++s) {
            mbar_init(bar(B::full(s)), 1);
            mbar_init(bar(B::conv(s)), 4);
            mbar_init(bar(B::empty(s)), 5);  // MMA commit + 4 square warps
        }
        for (int b = 0; b < AB; ++b) {
            mbar_init(bar(B::acc_full(b)), 1);
            mbar_init(bar(B::acc_empty(b)), 4 * TPU);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar(B::sq_full(b)), 4);
            mbar_init(bar(B::sq_empty(b)), 4 * TPU);
        }
        mbar_init(bar(B::drain), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == kWarpMma) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         su32(tmem_slot)),
                     "r"(C::kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == kWarpProducer) {
        if (lane == 0) {
            int last_use[S];
            for (int s = 0; s < S; ++s) last_use[s] = -1;
            bool ok = true;
            uint32_t q = 0;
            for (int it = 0; it < U && ok; ++it) {
                const int unit = (int)blockIdx.x + it * (int)gridDim.x;
                for (int kc = 0; kc < p.nk; ++kc, ++q) {
                    const int slot = (int)(q % S);
                    const uint32_t use = q / S;
                    if (!wait_bar<false>(bar(B::empty(slot)), (use & 1) ^ 1, abort, p.err)) {
                        ok = false;
                        break;
                    }
                    mbar_expect_tx(bar(B::full(slot)),
                                   (uint32_t)(C::kXStage + (PRE ? C::kWbBytes : C::kWfBytes)));
                    // a unit's second tile past the last token reads zeros
#pragma unroll
                    for (int v = 0; v < TPU; ++v)
                        tma_load_2d(su32(xr + (size_t)slot * C::kXStage + v * kXBytes), &tm_x,
                                    kc * kK, (unit * TPU + v) * kTok, bar(B::full(slot)));
                    if (PRE)  // the stage's hi/lo rows, swizzled on the way in
                        tma_load_2d(su32(wb + (size_t)slot * C::kWbBytes), &tm_w, 0, kc * C::kNW,
                                    bar(B::full(slot)));
                    else
                        tma_load_2d(su32(wf + (size_t)slot * C::kMix * kK), &tm_w, kc * kK, 0,
                                    bar(B::full(slot)));
                    last_use[slot] = (int)use;
                }
            }
            // no TMA may still be writing this CTA's shared memory at exit
            for (int s = 0; s < S; ++s)
                if (last_use[s] >= 0)
                    wait_bar<false>(bar(B::full(s)), (uint32_t)last_use[s] & 1, abort, p.err);
        }
    } else if (warp == kWarpMma) {
        if (lane == 0) {
            bool ok = true;
            uint32_t q = 0, gp = 0;  // stage and accumulation-part counters
            for (int it = 0; it < U && ok; ++it) {
                for (int k0 = 0; k0 < p.nk && ok; k0 += kPart, ++gp) {
                    const int b = (int)(gp % AB);
                    if (!wait_bar<false>(bar(B::acc_empty(b)), ((gp / AB) & 1) ^ 1, abort, p.err))
                        break;
                    tc_fence_after();
                    const int k1 = k0 + kPart < p.nk ? k0 + kPart : p.nk;
                    for (int kc = k0; kc < k1; ++kc, ++q) {
                        const int slot = (int)(q % S);
                        const uint32_t par = (q / S) & 1;
                        if (!wait_bar<false>(bar(B::full(slot)), par, abort, p.err) ||
                            (!PRE && !wait_bar<false>(bar(B::conv(slot)), par, abort, p.err))) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t b0 = su32(wb + (size_t)slot * C::kWbBytes);
#pragma unroll
                        for (int v = 0; v < TPU; ++v) {
                            const uint32_t a0 = su32(xr + (size_t)slot * C::kXStage + v * kXBytes);
                            const uint32_t d_tmem = tmem + (uint32_t)((b * TPU + v) * C::kNW);
#pragma unroll
                            for (int k = 0; k < 4; ++k)
                                mma_bf16(d_tmem, sw128_desc(a0 + 32 * k), sw128_desc(b0 + 32 * k),
                                         C::kIdesc, ((kc - k0) | k) != 0);
                        }
                        mma_commit(bar(B::empty(slot)));
                    }
                    if (!ok) break;
                    mma_commit(bar(B::acc_full(b)));
                }
            }
            // all issued MMAs complete before TMEM is freed
            mma_commit(bar(B::drain));
            wait_bar<false>(bar(B::drain), 0, abort, p.err);
        }
    } else if (C::is_convert(warp) && !PRE) {
        // W sub-tile (fp32 rows of 64) -> bf16 hi rows 0..kMix-1 and lo rows
        // kMix..2kMix-1, 8 features per 16-byte chunk, swizzled K-major.
        const int ci = C::convert_index(warp) * 32 + lane;
        uint32_t q = 0;
        bool ok = true;
        for (int it = 0; it < U && ok; ++it) {
            for (int kc = 0; kc < p.nk; ++kc, ++q) {
                const int slot = (int)(q % S);
                if (!__all_sync(0xFFFFFFFFu, wait_bar<false>(bar(B::full(slot)), (q / S) & 1,
                                                             abort, p.err))) {
                    ok = false;
                    break;
                }
                const float *src = wf + (size_t)slot * C::kMix * kK;
                uint8_t *dst = wb + (size_t)slot * C::kWbBytes;
                for (int e = ci; e < C::kMix * 8; e += 128) {
                    const int i = e >> 3, c = e & 7;
                    const float4 a = *reinterpret_cast<const float4 *>(src + i * kK + 8 * c);
                    const float4 b2 = *reinterpret_cast<const float4 *>(src + i * kK + 8 * c + 4);
                    float v[8] = {a.x, a.y, a.z, a.w, b2.x, b2.y, b2.z, b2.w}, lo[8];
#pragma unroll
                    for (int u = 0; u < 8; ++u)
                        lo[u] = v[u] - __bfloat162float(__float2bfloat16_rn(v[u]));
                    uint4 hv, lv;
                    hv.x = pack_bf16x2(v[0], v[1]);
                    hv.y = pack_bf16x2(v[2], v[3]);
                    hv.z = pack_bf16x2(v[4], v[5]);
                    hv.w = pack_bf16x2(v[6], v[7]);
                    lv.x = pack_bf16x2(lo[0], lo[1]);
                    lv.y = pack_bf16x2(lo[2], lo[3]);
                    lv.z = pack_bf16x2(lo[4], lo[5]);
                    lv.w = pack_bf16x2(lo[6], lo[7]);
                    const int rl = C::kMix + i;
                    *reinterpret_cast<uint4 *>(dst + (i >> 3) * 1024 + (i & 7) * 128 +
                                               ((c ^ (i & 7)) << 4)) = hv;
                    *reinterpret_cast<uint4 *>(dst + (rl >> 3) * 1024 + (rl & 7) * 128 +
                                               ((c ^ (rl & 7)) << 4)) = lv;
                }
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(B::conv(slot)));
            }
        }
    } else if (warp >= kWarpSq0 && warp < kWarpSq0 + 4) {
        // Sums of squares: warp 2+g takes tokens 32g..32g+31 of every tile of
        // the unit, lane = token, chunks in swizzle order so 8 consecutive
        // lanes hit 8 bank groups.
        const int i = 32 * (warp - kWarpSq0) + lane;
        uint32_t q = 0;
        bool ok = true;
        for (int it = 0; it < U && ok; ++it) {
            const int bs = it & 1;
            const uint32_t use = (uint32_t)(it >> 1);
            float ss[TPU];
#pragma unroll
            for (int v = 0; v < TPU; ++v) ss[v] = 0.f;
            for (int kc = 0; kc < p.nk; ++kc, ++q) {
                const int slot = (int)(q % S);
                if (!__all_sync(0xFFFFFFFFu, wait_bar<false>(bar(B::full(slot)), (q / S) & 1,
                                                             abort, p.err))) {
                    ok = false;
                    break;
                }
#pragma unroll
                for (int v = 0; v < TPU; ++v) {
                    const uint32_t row = su32(xr + (size_t)slot * C::kXStage + v * kXBytes) +
                                         (i >> 3) * 1024 + (i & 7) * 128;
#pragma unroll
                    for (int m = 0; m < 8; ++m) {
                        float f[8];
                        unpack8(lds128(row + ((m ^ (i & 7)) << 4)), f);
#pragma unroll
                        for (int e = 0; e < 8; ++e) ss[v] = fmaf(f[e], f[e], ss[v]);
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(B::empty(slot)));
            }
            if (!ok) break;
            if (!__all_sync(0xFFFFFFFFu,
                            wait_bar<false>(bar(B::sq_empty(bs)), (use & 1) ^ 1, abort, p.err)))
                break;
#pragma unroll
            for (int v = 0; v < TPU; ++v) sq[(bs * TPU + v) * kTok + i] = ss[v];
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B::sq_full(bs)));
        }
    } else if (warp >= kWarpEpi0 && warp < kWarpEpi0 + 4 * TPU) {
        // Tile v of the unit, TMEM lanes 32*(warp % 4).. = its tokens; the
        // parts of the unit are added in registers, then scaled by r and
        // written.
        const int v = (warp - kWarpEpi0) >> 2;
        const int i = 32 * (warp & 3) + lane;
        const uint32_t tlane = (uint32_t)((warp & 3) * 32) << 16;
        uint32_t gp = 0;
        bool ok = true;
        for (int it = 0; it < U && ok; ++it) {
            const int unit = (int)blockIdx.x + it * (int)gridDim.x;
            float m[C::kMix];
#pragma unroll
            for (int k = 0; k < C::kMix; ++k) m[k] = 0.f;
            for (int k0 = 0; k0 < p.nk; k0 += kPart, ++gp) {
                const int b = (int)(gp % AB);
                if (!__all_sync(0xFFFFFFFFu, wait_bar<false>(bar(B::acc_full(b)), (gp / AB) & 1,
                                                             abort, p.err))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t taddr = tmem + tlane + (uint32_t)((b * TPU + v) * C::kNW);
#pragma unroll
                for (int g = 0; g < C::kMix / 8; ++g) {
                    float hi[8], lo[8];
                    tmem_ld8(taddr + 8 * g, hi);
                    tmem_ld8(taddr + C::kMix + 8 * g, lo);
                    tmem_ld_wait();
#pragma unroll
                    for (int e = 0; e < 8; ++e) m[8 * g + e] += hi[e] + lo[e];
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(B::acc_empty(b)));
            }
            if (!ok) break;
            const uint32_t use = (uint32_t)(it >> 1);
            const int bs = it & 1;
            if (!__all_sync(0xFFFFFFFFu, wait_bar<false>(bar(B::sq_full(bs)), use & 1, abort, p.err)))
                break;
            const float r = rsqrtf(sq[(bs * TPU + v) * kTok + i] / (float)p.F + p.norm_eps);
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B::sq_empty(bs)));
            const int64_t t = ((int64_t)unit * TPU + v) * kTok + i;
            if (t < p.n) {
                float4 *dst = reinterpret_cast<float4 *>(p.mixes + t * C::kMix);
#pragma unroll
                for (int q4 = 0; q4 < C::kMix / 4; ++q4)
                    dst[q4] = make_float4(m[4 * q4] * r, m[4 * q4 + 1] * r, m[4 * q4 + 2] * r,
                                          m[4 * q4 + 3] * r);
            }
        }
    }

    // ------------------------------------------------------------ teardown
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kWarpMma) {
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(C::kTmemCols)
                     : "memory");
    }
}

// ---------------------------------------------------------------- host

struct DevState {
    bool init = false;
    unsigned long long ctx = 0;  // the context the set-up below was done in
    bool ok = false;
};
std::mutex g_mmu;
DevState g_mix[64];

template <int HC, bool PRE>
bool set_attrs() {
    return cudaFuncSetAttribute(k_mixtc<HC, PRE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)smem_bytes<HC, PRE>()) == cudaSuccess;
}

const DevState &mix_state(const DeviceInfo &di) {
    std::lock_guard<std::mutex> lk(g_mmu);
    DevState &st = g_mix[di.device];
    if (st.init && st.ctx == di.ctx) return st;
    st = DevState();
    st.init = true;
    st.ctx = di.ctx;
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, di.device) != cudaSuccess) return st;
    if (prop.major != 10 || prop.minor != 3) return st;  // built for sm_103a only
    if (tensor_map_encoder() == nullptr) return st;
    if (!set_attrs<4, false>() || !set_attrs<8, false>() || !set_attrs<8, true>()) {
        cudaGetLastError();
        return st;
    }
    st.ok = true;
    return st;
}

template <int HC>
cudaError_t launch(int64_t n, int64_t d, float norm_eps, const uint16_t *x, const float *w,
                   float *mixes, uint16_t *wconv, const DeviceInfo &di, cudaStream_t s) {
    constexpr int MIX = (2 + HC) * HC;
    constexpr bool kCanPre = HC == 8;  // where the conversion is worth a pass of its own
    const int64_t F = (int64_t)HC * d;
    const bool pre = kCanPre && wconv != nullptr;
    CUtensorMap tm_x, tm_w;
    {
        // x as [n rows][F] bf16; one box = 64 features of 128 tokens, swizzled
        const cuuint64_t gdim[2] = {(cuuint64_t)F, (cuuint64_t)n};
        const cuuint64_t gstride[1] = {(cuuint64_t)F * 2};
        const cuuint32_t box[2] = {kK, kTok};
        const cuuint32_t es[2] = {1, 1};
        if (tensor_map_encoder()(&tm_x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                                 const_cast<uint16_t *>(x), gdim, gstride, box, es,
                                 CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                 CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                 CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    if (pre) {
        // converted W as [(F/64) * 2 mix rows][64] bf16; one box = one stage's
        // hi and lo rows, 128-byte swizzled like x
        const cuuint64_t gdim[2] = {(cuuint64_t)kK, (cuuint64_t)(F / kK) * 2 * MIX};
        const cuuint64_t gstride[1] = {(cuuint64_t)kK * 2};
        const cuuint32_t box[2] = {kK, (cuuint32_t)(2 * MIX)};
        const cuuint32_t es[2] = {1, 1};
        if (tensor_map_encoder()(&tm_w, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, wconv, gdim, gstride,
                                 box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                 CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                 CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    } else {
        // W as [mix rows][F] fp32; one box = 64 features of every row
        const cuuint64_t gdim[2] = {(cuuint64_t)F, (cuuint64_t)MIX};
        const cuuint64_t gstride[1] = {(cuuint64_t)F * 4};
        const cuuint32_t box[2] = {kK, (cuuint32_t)MIX};
        const cuuint32_t es[2] = {1, 1};
        if (tensor_map_encoder()(&tm_w, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2,
                                 const_cast<float *>(w), gdim, gstride, box, es,
                                 CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                                 CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                 CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    MixParams p;
    p.n = n;
    p.F = (int)F;
    p.nk = (int)(F / kK);
    p.num_tiles = (int)((n + kTok - 1) / kTok);
    p.num_units = (p.num_tiles + Cfg<HC>::kTPU - 1) / Cfg<HC>::kTPU;
    p.norm_eps = norm_eps;
    p.mixes = mixes;
    p.err = di.err_word;
    const int grid = p.num_units < di.sms ? p.num_units : di.sms;
    if (pre) {
        if constexpr (kCanPre) {
            const int64_t items = (F / kK) * MIX * 8;
            const int64_t cgrid = (items + 255) / 256 < (int64_t)di.sms * 8
                                      ? (items + 255) / 256 : (int64_t)di.sms * 8;
            k_convert_w<HC><<<(unsigned)cgrid, 256, 0, s>>>((int)F, w,
                                                           reinterpret_cast<uint4 *>(wconv));
            k_mixtc<HC, true><<<grid, Cfg<HC, true>::kThreads, smem_bytes<HC, true>(), s>>>(
                tm_x, tm_w, p);
            return launched(2);
        }
    }
    k_mixtc<HC, false><<<grid, Cfg<HC, false>::kThreads, smem_bytes<HC, false>(), s>>>(tm_x,
                                                                                       tm_w, p);
    return launched();
}

}  // namespace

bool mixtc_supported(int hc, int64_t d, const DeviceInfo &di) {
    if (hc != 4 && hc != 8) return false;
    if (((int64_t)hc * d) % kK != 0 || (int64_t)hc * d > (int64_t)1 << 30) return false;
    if (forced_path() == kPathFfma) return false;
    return mix_state(di).ok;
}

size_t mixtc_wconv_bytes(int hc, int64_t d) {
    return hc == 8 ? (size_t)4 * (size_t)((2 + hc) * hc) * (size_t)(hc * d) : 0;
}

cudaError_t launch_mixtc(int64_t n, int hc, int64_t d, float norm_eps, const uint16_t *x,
                         const float *w, float *mixes, uint16_t *wconv, const DeviceInfo &di,
                         cudaStream_t s) {
    if (!mix_state(di).ok || n < 1 || n >= ((int64_t)1 << 31)) return cudaErrorNotSupported;
    return hc == 4 ? launch<4>(n, d, norm_eps, x, w, mixes, nullptr, di, s)
                   : launch<8>(n, d, norm_eps, x, w, mixes, wconv, di, s);
}

}  // namespace hc
