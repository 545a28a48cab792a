// hc_fused.cu -- fused RMS statistic + mix projection + split/Sinkhorn +
// collapse for hc = 4 on sm_103a ("Mix projection" page: formula for m,
// Block.hc_mixes, Block.hc_pre; "Reading weights" page: hc_split_sinkhorn).
//
// Work decomposition
//   * A cluster of 16 CTAs (one per SM) is persistent over 64-token tiles.
//     CTA r owns channels [r*w, (r+1)*w) of every copy (w = d/16), i.e.
//     4*w of the F = 4*d features of each token.
//   * The CTA keeps its slice of W_mix resident in shared memory for the whole
//     kernel, split into bf16 hi + lo rows (48 rows = 24 hi, 24 lo), in the
//     128-byte-swizzled K-major layout the tensor core reads.
//   * x streams through an 8-stage ring of [64 tokens x 64 features] TMA
//     boxes.  Per box: 4 tcgen05.mma (M=128 rows of which the 64 tokens are
//     the first half, N=48, K=16) accumulate x.(W_hi + W_lo) in TMEM
//     (binary32), and one of 4 "square" warps adds the box's x^2 per token.
//   * At the end of a tile each CTA sends its 24 partial mix numbers and
//     partial sum of squares per token to the token's owner CTA (4 tokens per
//     CTA) through distributed shared memory.  The owner reduces the 16
//     partials in a fixed order, forms r and m, runs the split + Sinkhorn for
//     its tokens, writes pre/post/comb (and m), and broadcasts pre back to
//     all 16 CTAs.
//   * The collapse y = sum_j pre_j x_j re-reads the tile's x slice through
//     the same ring (the boxes were read a few microseconds earlier and come
//     from L2) and writes y.
//   The ring order per CTA is P(0), P(1), C(0), P(2), C(1), ... where P(t)
//   are the projection boxes of tile t and C(t) its collapse boxes, so the
//   collapse of a tile overlaps the projection of the next one.  Every ring
//   consumer (MMA thread, square warps, collapse warps) walks every stage in
//   this order and releases it, using the data only of its own stages.
//
// Every wait is bounded: a wait that exceeds kTimeoutNs sets the CTA's abort
// flag and bit 0 of the device error word, and all roles then run to the
// common teardown (no trap, TMEM always freed, no CTA leaves its cluster
// while others may still address its shared memory).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "hc_common.cuh"
#include "hc_fused.h"

namespace hc {
namespace {

constexpr int kCluster = 16;        // CTAs per cluster
constexpr int kTM = 64;             // tokens per tile
constexpr int kMix = 24;            // (2 + 4) * 4
constexpr int kNW = 48;             // B rows: 24 hi + 24 lo
constexpr int kStages = 8;          // x ring depth
constexpr int kStageBytes = kTM * 128;   // one [64 x 64] bf16 box
constexpr int kWChunkBytes = kNW * 128;  // one [48 x 64] bf16 chunk of W
constexpr int kOwn = kTM / kCluster;     // tokens owned per CTA per tile
constexpr int kRec = 28;                 // floats per partial record (24 + ssq + pad)
constexpr int kThreads = 416;
constexpr int kTmemCols = 128;
constexpr uint64_t kTimeoutNs = 1000000000ull;  // 1 s

// warp roles
constexpr int kWarpProducer = 0;
constexpr int kWarpMma = 1;
constexpr int kWarpSq0 = 2;   // 2..5: sums of squares, warp 2+j takes copy j
constexpr int kWarpEpi0 = 8;  // 8, 9: TMEM read-out (lanes 0..63), records to the owners
constexpr int kWarpOwner = 12;  // reduces the records of this CTA's tokens, Sinkhorn
// collapse warps: 6, 7, 10, 11

// tcgen05 instruction descriptor: D f32, A/B bf16, both K-major, N=48, M=128.
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(kNW >> 3) << 17) |
                            ((uint32_t)(128 >> 4) << 24);

struct FusedParams {
    int64_t n;
    int d;
    int ncc;        // 64-channel chunks per CTA slice (w / 64)
    int nkc;        // K boxes per CTA per tile (4 * ncc)
    int num_tiles;
    int iters;
    int mixes_only;
    float eps;
    float norm_eps;
    float F;
    const float *w;
    const float *scale;
    const float *base;
    float *mixes;
    float *pre;
    float *post;
    float *comb;
    uint16_t *y;
    unsigned int *err;
};

// ------------------------------------------------------------ PTX helpers

__device__ __forceinline__ uint32_t su32(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ uint64_t gtimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar, uint32_t count = 1) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(count)
                 : "memory");
}

// Arrive on a barrier of another CTA of the cluster (address from mapa).
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(
                     cluster_addr)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ bool mbar_try_cluster(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait for the phase of `bar` with the given parity.  Returns false
// (and raises the abort flag) on timeout or when the CTA is already aborting.
template <bool kClusterScope>
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int *abort,
                                         unsigned int *err) {
    if (kClusterScope ? mbar_try_cluster(bar, parity) : mbar_try(bar, parity)) return true;
    const uint64_t t0 = gtimer();
    while (true) {
        if (kClusterScope ? mbar_try_cluster(bar, parity) : mbar_try(bar, parity)) return true;
        if (*abort) return false;
        if (gtimer() - t0 > kTimeoutNs) {
            *abort = 1;
            atomicOr(err, kErrWaitTimeout);
            return false;
        }
    }
}

__device__ __forceinline__ uint32_t mapa(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}

__device__ __forceinline__ void st_cluster_v4(uint32_t addr, float a, float b, float c, float d) {
    asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(a), "f"(b),
                 "f"(c), "f"(d)
                 : "memory");
}

__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::
                     : "memory");
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int c0, int c1,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
        : "memory");
}

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups
// 1024 bytes apart, descriptor version 1.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) |
           ((uint64_t)(1024 >> 4) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(kIdesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float v[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_ld_wait() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr));
    return v;
}

// ---------------------------------------------------------------- layout

struct Smem {
    uint8_t *w;       // nkc chunks of [48 x 64] bf16, swizzled
    uint8_t *ring;    // kStages boxes of [64 x 64] bf16, swizzled
    float *recv;      // [2][kCluster][kOwn][kRec]   partials received as owner
    float *pre;       // [2][kTM][4]                 pre of the tile's tokens
    float *sq;        // [2][4][kTM]                 partial sums of squares
    float *stage;     // [kOwn][4]                   pre of the owned tokens
    uint64_t *bar;    // barriers, see below
    uint32_t *tmem;   // TMEM base address written by tcgen05.alloc
    int *abort;
};

// barrier indices
__host__ __device__ constexpr int bFull(int s) { return s; }
__host__ __device__ constexpr int bEmpty(int s) { return kStages + s; }
__host__ __device__ constexpr int bAccFull(int b) { return 2 * kStages + b; }
__host__ __device__ constexpr int bAccEmpty(int b) { return 2 * kStages + 2 + b; }
__host__ __device__ constexpr int bSqFull(int b) { return 2 * kStages + 4 + b; }
__host__ __device__ constexpr int bSqEmpty(int b) { return 2 * kStages + 6 + b; }
__host__ __device__ constexpr int bRecvFull(int b) { return 2 * kStages + 8 + b; }
__host__ __device__ constexpr int bRecvFree(int b) { return 2 * kStages + 10 + b; }
__host__ __device__ constexpr int bPreFull(int b) { return 2 * kStages + 12 + b; }
constexpr int kMmaDrain = 2 * kStages + 14;
// Every ring consumer walks every stage in order and releases it once: the
// MMA thread (1, through tcgen05.commit for P boxes), the 4 square warps and,
// unless only the mix numbers are wanted, the 4 collapse warps.  Because no
// consumer skips a stage, each waiter has seen the slot's previous phase and
// the parity of the phase it waits for is unambiguous.
constexpr int kEmptyArrivalsFull = 9;
constexpr int kEmptyArrivalsMixes = 5;
constexpr int kNumBars = 2 * kStages + 15;

__host__ __device__ constexpr size_t smem_bytes(int nkc) {
    return 1024 /* alignment slack */ + (size_t)nkc * kWChunkBytes +
           (size_t)kStages * kStageBytes + 2 * kCluster * kOwn * kRec * 4 + 2 * kTM * 4 * 4 +
           2 * 4 * kTM * 4 + kOwn * 4 * 4 + kNumBars * 8 + 16;
}

__device__ __forceinline__ Smem carve(uint8_t *raw, int nkc) {
    uintptr_t a = (reinterpret_cast<uintptr_t>(raw) + 1023) & ~(uintptr_t)1023;
    uint8_t *p = reinterpret_cast<uint8_t *>(a);
    Smem s;
    s.w = p;
    p += (size_t)nkc * kWChunkBytes;
    s.ring = p;
    p += kStages * kStageBytes;
    s.recv = reinterpret_cast<float *>(p);
    p += 2 * kCluster * kOwn * kRec * 4;
    s.pre = reinterpret_cast<float *>(p);
    p += 2 * kTM * 4 * 4;
    s.sq = reinterpret_cast<float *>(p);
    p += 2 * 4 * kTM * 4;
    s.stage = reinterpret_cast<float *>(p);
    p += kOwn * 4 * 4;
    s.bar = reinterpret_cast<uint64_t *>(p);
    p += kNumBars * 8;
    s.tmem = reinterpret_cast<uint32_t *>(p);
    s.abort = reinterpret_cast<int *>(p + 4);
    return s;
}

// Feature index (within the token's F) of K box kc = cc*4 + j of CTA `rank`.
__device__ __forceinline__ int box_feature(int kc, int rank, const FusedParams &p) {
    const int cc = kc >> 2, j = kc & 3;
    return j * p.d + rank * (p.ncc * 64) + cc * 64;
}

// ---------------------------------------------------------------- kernel

__global__ void __launch_bounds__(kThreads, 1)
    k_fused(const __grid_constant__ CUtensorMap tmap, const FusedParams p) {
    extern __shared__ uint8_t smem_raw[];
    const Smem sm = carve(smem_raw, p.nkc);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rank = (int)(blockIdx.x % kCluster);
    const int cluster = (int)(blockIdx.x / kCluster);
    const int nclusters = (int)(gridDim.x / kCluster);
    const int nkc = p.nkc;
    const bool mixes_only = p.mixes_only != 0;
    const int T = cluster < p.num_tiles ? (p.num_tiles - cluster + nclusters - 1) / nclusters : 0;
    volatile int *abort = sm.abort;
    auto bar = [&](int i) { return su32(sm.bar + i); };

    // ------------------------------------------------------------ set-up
    if (threadIdx.x == 0) {
        *abort = 0;
        for (int s = 0; s < kStages; ++s) {
            mbar_init(bar(bFull(s)), 1);
            mbar_init(bar(bEmpty(s)), mixes_only ? kEmptyArrivalsMixes : kEmptyArrivalsFull);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar(bAccFull(b)), 1);
            mbar_init(bar(bAccEmpty(b)), 2);
            mbar_init(bar(bSqFull(b)), 4);
            mbar_init(bar(bSqEmpty(b)), 2);
            mbar_init(bar(bRecvFull(b)), kCluster * kOwn);
            mbar_init(bar(bRecvFree(b)), kCluster);
            mbar_init(bar(bPreFull(b)), kCluster);
        }
        mbar_init(bar(kMmaDrain), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == kWarpMma) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         su32(sm.tmem)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    if (warp == kWarpProducer && lane == 0)
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap))
                     : "memory");
    // W slice -> bf16 hi/lo rows in the swizzled K-major layout.  Row nr < 24
    // holds hi(W[nr]), row 24 + i holds lo(W[i]) = bf16(W - hi).
    {
        const int total = kNW * nkc * 8;
        const int64_t F = 4LL * p.d;
        for (int idx = threadIdx.x; idx < total; idx += kThreads) {
            const int q = idx & 7, rest = idx >> 3;
            const int nr = rest % kNW, kc = rest / kNW;
            const int i = nr % kMix;
            const bool lo = nr >= kMix;
            const float4 *src = reinterpret_cast<const float4 *>(
                p.w + (int64_t)i * F + box_feature(kc, rank, p) + q * 8);
            const float4 a = __ldg(src), b2 = __ldg(src + 1);
            float v[8] = {a.x, a.y, a.z, a.w, b2.x, b2.y, b2.z, b2.w};
            if (lo) {
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    v[e] = v[e] - __bfloat162float(__float2bfloat16_rn(v[e]));
            }
            uint4 o;
            o.x = pack_bf16x2(v[0], v[1]);
            o.y = pack_bf16x2(v[2], v[3]);
            o.z = pack_bf16x2(v[4], v[5]);
            o.w = pack_bf16x2(v[6], v[7]);
            uint8_t *dst = sm.w + (size_t)kc * kWChunkBytes + (nr >> 3) * 1024 + (nr & 7) * 128 +
                           ((q ^ (nr & 7)) << 4);
            *reinterpret_cast<uint4 *>(dst) = o;
        }
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    cluster_sync_all();  // every CTA's barriers exist before any remote arrive
    const uint32_t tmem = *sm.tmem;

    // ------------------------------------------------------------ roles
    if (warp == kWarpProducer) {
        if (lane == 0) {
            uint32_t q = 0;
            int last_use[kStages];
#pragma unroll
            for (int s = 0; s < kStages; ++s) last_use[s] = -1;
            bool ok = true;
            for (int it = 0; it <= T && ok; ++it) {
                for (int part = 0; part < 2 && ok; ++part) {
                    int tt;
                    if (part == 0) {
                        if (it >= T) continue;
                        tt = it;
                    } else {
                        if (mixes_only || it < 1) continue;
                        tt = it - 1;
                    }
                    const int tile = cluster + tt * nclusters;
                    for (int kc = 0; kc < nkc; ++kc, ++q) {
                        const int slot = (int)(q % kStages);
                        const uint32_t use = q / kStages;
                        if (!wait_bar<false>(bar(bEmpty(slot)), (use & 1) ^ 1, abort, p.err)) {
                            ok = false;
                            break;
                        }
                        mbar_expect_tx(bar(bFull(slot)), kStageBytes);
                        tma_load_2d(su32(sm.ring + slot * kStageBytes), &tmap,
                                    box_feature(kc, rank, p), tile * kTM, bar(bFull(slot)));
                        last_use[slot] = (int)use;
                    }
                }
            }
            // no TMA may still be writing this CTA's shared memory at exit
            for (int s = 0; s < kStages; ++s)
                if (last_use[s] >= 0)
                    wait_bar<false>(bar(bFull(s)), (uint32_t)last_use[s] & 1, abort, p.err);
        }
    } else if (warp == kWarpMma) {
        // Walks every ring stage in order: P boxes feed the tensor core, C
        // boxes are only acknowledged (wait for the load, then release).
        if (lane == 0) {
            uint32_t q = 0;
            bool ok = true;
            for (int it = 0; it <= T && ok; ++it) {
                if (it < T) {
                    const int b = it & 1;
                    const uint32_t use = (uint32_t)(it >> 1);
                    if (!wait_bar<false>(bar(bAccEmpty(b)), (use & 1) ^ 1, abort, p.err)) break;
                    tc_fence_after();
                    const uint32_t d_tmem = tmem + (uint32_t)(b * 64);
                    for (int kc = 0; kc < nkc; ++kc, ++q) {
                        const int slot = (int)(q % kStages);
                        if (!wait_bar<false>(bar(bFull(slot)), (q / kStages) & 1, abort, p.err)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t a0 = su32(sm.ring + slot * kStageBytes);
                        const uint32_t b0 = su32(sm.w + (size_t)kc * kWChunkBytes);
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            mma_bf16(d_tmem, sw128_desc(a0 + 32 * k), sw128_desc(b0 + 32 * k),
                                     (kc | k) != 0);
                        mma_commit(bar(bEmpty(slot)));
                    }
                    if (!ok) break;
                    mma_commit(bar(bAccFull(b)));
                }
                if (!mixes_only && it >= 1) {
                    for (int kc = 0; kc < nkc; ++kc, ++q) {
                        const int slot = (int)(q % kStages);
                        if (!wait_bar<false>(bar(bFull(slot)), (q / kStages) & 1, abort, p.err)) {
                            ok = false;
                            break;
                        }
                        mbar_arrive(bar(bEmpty(slot)));
                    }
                }
            }
            // all issued MMAs complete before TMEM is freed
            mma_commit(bar(kMmaDrain));
            wait_bar<false>(bar(kMmaDrain), 0, abort, p.err);
        }
    } else if (warp >= kWarpSq0 && warp < kWarpSq0 + 4) {
        // Sums of squares: warp 2+j uses the P boxes of copy j (lane l
        // accumulates tokens l and l+32 of the tile) and acknowledges every
        // other stage of the ring.
        const int j = warp - kWarpSq0;
        uint32_t q = 0;
        bool ok = true;
        for (int it = 0; it <= T && ok; ++it) {
            if (it < T) {
                const int b = it & 1;
                const uint32_t use = (uint32_t)(it >> 1);
                float s0 = 0.f, s1 = 0.f;
                for (int kc = 0; kc < nkc; ++kc, ++q) {
                    const int slot = (int)(q % kStages);
                    if (!__all_sync(0xFFFFFFFFu, wait_bar<false>(bar(bFull(slot)),
                                                                 (q / kStages) & 1, abort, p.err))) {
                        ok = false;
                        break;
                    }
                    if ((kc & 3) == j) {
                        const uint32_t base = su32(sm.ring + slot * kStageBytes);
#pragma unroll
                        for (int c = 0; c < 8; ++c) {
                            float f[8];
                            // chunk c ^ (row & 7): the same 8 chunks of the row, and
                            // 8 consecutive lanes touch 8 different bank groups
                            unpack8(lds128(base + lane * 128 + ((c ^ (lane & 7)) << 4)), f);
#pragma unroll
                            for (int e = 0; e < 8; ++e) s0 = fmaf(f[e], f[e], s0);
                            unpack8(lds128(base + (lane + 32) * 128 + ((c ^ (lane & 7)) << 4)), f);
#pragma unroll
                            for (int e = 0; e < 8; ++e) s1 = fmaf(f[e], f[e], s1);
                        }
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(bEmpty(slot)));
                }
                if (!ok) break;
                if (!__all_sync(0xFFFFFFFFu,
                                wait_bar<false>(bar(bSqEmpty(b)), (use & 1) ^ 1, abort, p.err)))
                    break;
                sm.sq[(b * 4 + j) * kTM + lane] = s0;
                sm.sq[(b * 4 + j) * kTM + lane + 32] = s1;
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(bSqFull(b)));
            }
            if (!mixes_only && it >= 1) {
                for (int kc = 0; kc < nkc; ++kc, ++q) {
                    const int slot = (int)(q % kStages);
                    if (!__all_sync(0xFFFFFFFFu, wait_bar<false>(bar(bFull(slot)),
                                                                 (q / kStages) & 1, abort, p.err))) {
                        ok = false;
                        break;
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(bEmpty(slot)));
                }
            }
        }
    } else if (warp == kWarpEpi0 || warp == kWarpEpi0 + 1) {
        // TMEM lanes 32*(warp%4) .. +31 = tokens of the tile
        const int i = (warp - kWarpEpi0) * 32 + lane;
        const int owner = i / kOwn, u = i % kOwn;
        for (int it = 0; it < T; ++it) {
            const int b = it & 1;
            const uint32_t use = (uint32_t)(it >> 1);
            const int tile = cluster + it * nclusters;
            if (!__all_sync(0xFFFFFFFFu, wait_bar<false>(bar(bAccFull(b)), use & 1, abort, p.err)))
                break;
            tc_fence_after();
            float acc[48];
            const uint32_t taddr = tmem + ((uint32_t)((warp & 3) * 32) << 16) + (uint32_t)(b * 64);
            tmem_ld16(taddr, acc);
            tmem_ld16(taddr + 16, acc + 16);
            tmem_ld16(taddr + 32, acc + 32);
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(bAccEmpty(b)));
            if (!__all_sync(0xFFFFFFFFu, wait_bar<false>(bar(bSqFull(b)), use & 1, abort, p.err)))
                break;
            float ss = 0.f;
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) ss += sm.sq[(b * 4 + jj) * kTM + i];
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(bSqEmpty(b)));
            // the owner's record slot for this tile parity must be free
            if (!__all_sync(0xFFFFFFFFu,
                            wait_bar<true>(bar(bRecvFree(b)), (use & 1) ^ 1, abort, p.err)))
                break;
            const uint32_t rec =
                mapa(su32(sm.recv + ((b * kCluster + rank) * kOwn + u) * kRec), (uint32_t)owner);
#pragma unroll
            for (int v = 0; v < 6; ++v)
                st_cluster_v4(rec + 16 * v, acc[4 * v] + acc[24 + 4 * v],
                              acc[4 * v + 1] + acc[24 + 4 * v + 1],
                              acc[4 * v + 2] + acc[24 + 4 * v + 2],
                              acc[4 * v + 3] + acc[24 + 4 * v + 3]);
            st_cluster_v4(rec + 96, ss, 0.f, 0.f, 0.f);
            mbar_arrive_remote(mapa(bar(bRecvFull(b)), (uint32_t)owner));

        }
    } else if (warp == kWarpOwner) {
        // Owner of tokens rank*kOwn + u (u < kOwn) of every tile: lanes u < kOwn
        // reduce the 16 records of their token in a fixed order, form r and m,
        // run split + Sinkhorn; lanes 0..15 then release the record slots and
        // deliver pre to CTA `lane`, one release-ordered arrive each.
        float bse[kMix], s0 = 0.f, s1 = 0.f, s2 = 0.f;
        if (!mixes_only && lane < kOwn) {
#pragma unroll
            for (int k = 0; k < kMix; ++k) bse[k] = __ldg(p.base + k);
            s0 = __ldg(p.scale + 0);
            s1 = __ldg(p.scale + 1);
            s2 = __ldg(p.scale + 2);
        }
        for (int it = 0; it < T; ++it) {
            const int b = it & 1;
            const uint32_t use = (uint32_t)(it >> 1);
            const int tile = cluster + it * nclusters;
            if (!__all_sync(0xFFFFFFFFu,
                            wait_bar<true>(bar(bRecvFull(b)), use & 1, abort, p.err)))
                break;
            float m[kMix];
            float ssum = 0.f;
            if (lane < kOwn) {
#pragma unroll
                for (int k = 0; k < kMix; ++k) m[k] = 0.f;
                for (int src = 0; src < kCluster; ++src) {
                    const float4 *r4 = reinterpret_cast<const float4 *>(
                        sm.recv + ((b * kCluster + src) * kOwn + lane) * kRec);
#pragma unroll
                    for (int v = 0; v < 6; ++v) {
                        const float4 t4 = r4[v];
                        m[4 * v] += t4.x;
                        m[4 * v + 1] += t4.y;
                        m[4 * v + 2] += t4.z;
                        m[4 * v + 3] += t4.w;
                    }
                    ssum += r4[6].x;
                }
            }
            __syncwarp();
            // all records of this parity read: release them to every sender
            if (lane < kCluster) mbar_arrive_remote(mapa(bar(bRecvFree(b)), (uint32_t)lane));
            if (lane < kOwn) {
                const float r = rsqrtf(ssum / p.F + p.norm_eps);
#pragma unroll
                for (int k = 0; k < kMix; ++k) m[k] *= r;
                const int64_t t = (int64_t)tile * kTM + rank * kOwn + lane;
                if (t < p.n && p.mixes != nullptr) {
                    float4 *dst = reinterpret_cast<float4 *>(p.mixes + t * kMix);
#pragma unroll
                    for (int v = 0; v < 6; ++v)
                        dst[v] = make_float4(m[4 * v], m[4 * v + 1], m[4 * v + 2], m[4 * v + 3]);
                }
                if (!mixes_only) {
                    float pr[4], po[4], Cm[4][4];
                    split_sinkhorn_token<4>([&](int k) { return m[k]; },
                                            [&](int k) { return bse[k]; }, s0, s1, s2, p.iters,
                                            p.eps, pr, po, Cm);
                    if (t < p.n) {
                        reinterpret_cast<float4 *>(p.pre)[t] =
                            make_float4(pr[0], pr[1], pr[2], pr[3]);
                        reinterpret_cast<float4 *>(p.post)[t] =
                            make_float4(po[0], po[1], po[2], po[3]);
#pragma unroll
                        for (int jj = 0; jj < 4; ++jj)
                            reinterpret_cast<float4 *>(p.comb)[t * 4 + jj] =
                                make_float4(Cm[jj][0], Cm[jj][1], Cm[jj][2], Cm[jj][3]);
                    }
                    reinterpret_cast<float4 *>(sm.stage)[lane] =
                        make_float4(pr[0], pr[1], pr[2], pr[3]);
                }
            }
            __syncwarp();
            if (!mixes_only && lane < kCluster) {
                const uint32_t pa = su32(sm.pre + (b * kTM + rank * kOwn) * 4);
#pragma unroll
                for (int u = 0; u < kOwn; ++u) {
                    const float4 v4 = reinterpret_cast<const float4 *>(sm.stage)[u];
                    st_cluster_v4(mapa(pa + 16 * u, (uint32_t)lane), v4.x, v4.y, v4.z, v4.w);
                }
                mbar_arrive_remote(mapa(bar(bPreFull(b)), (uint32_t)lane));
            }
            __syncwarp();
        }
    } else if (!mixes_only) {
        // Collapse warps 6, 7, 10, 11 -> cw 0..3, 16 tokens each.  They
        // acknowledge the P boxes and use the C boxes, 4 copies at a time.
        const int cw = warp < kWarpEpi0 ? warp - 6 : warp - 8;
        const int w = p.ncc * 64;
        uint32_t q = 0;
        bool ok = true;
        for (int it = 0; it <= T && ok; ++it) {
            if (it < T) {
                for (int kc = 0; kc < nkc; ++kc, ++q) {
                    const int slot = (int)(q % kStages);
                    if (!__all_sync(0xFFFFFFFFu, wait_bar<false>(bar(bFull(slot)),
                                                                 (q / kStages) & 1, abort, p.err))) {
                        ok = false;
                        break;
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(bEmpty(slot)));
                }
                if (!ok) break;
            }
            if (it < 1) continue;
            const int tt = it - 1;
            const int b = tt & 1;
            const uint32_t use = (uint32_t)(tt >> 1);
            const int tile = cluster + tt * nclusters;
            if (!__all_sync(0xFFFFFFFFu, wait_bar<true>(bar(bPreFull(b)), use & 1, abort, p.err)))
                break;
            for (int cc = 0; cc < p.ncc && ok; ++cc, q += 4) {
                int slot[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint32_t qj = q + j;
                    slot[j] = (int)(qj % kStages);
                    if (ok && !wait_bar<false>(bar(bFull(slot[j])), (qj / kStages) & 1, abort,
                                               p.err))
                        ok = false;
                }
                ok = __all_sync(0xFFFFFFFFu, ok);
                if (!ok) break;
#pragma unroll
                for (int uu = 0; uu < 4; ++uu) {
                    const int i = 16 * cw + 4 * uu + (lane >> 3);
                    const int mch = lane & 7;
                    const float4 pr = *reinterpret_cast<const float4 *>(sm.pre + (b * kTM + i) * 4);
                    const uint32_t off = i * 128 + ((mch ^ (i & 7)) << 4);
                    float acc[8], f[8];
                    unpack8(lds128(su32(sm.ring + slot[0] * kStageBytes) + off), f);
#pragma unroll
                    for (int e = 0; e < 8; ++e) acc[e] = pr.x * f[e];
                    unpack8(lds128(su32(sm.ring + slot[1] * kStageBytes) + off), f);
#pragma unroll
                    for (int e = 0; e < 8; ++e) acc[e] = fmaf(pr.y, f[e], acc[e]);
                    unpack8(lds128(su32(sm.ring + slot[2] * kStageBytes) + off), f);
#pragma unroll
                    for (int e = 0; e < 8; ++e) acc[e] = fmaf(pr.z, f[e], acc[e]);
                    unpack8(lds128(su32(sm.ring + slot[3] * kStageBytes) + off), f);
#pragma unroll
                    for (int e = 0; e < 8; ++e) acc[e] = fmaf(pr.w, f[e], acc[e]);
                    const int64_t t = (int64_t)tile * kTM + i;
                    if (t < p.n)
                        st_stream(reinterpret_cast<uint4 *>(p.y + t * p.d + rank * w + cc * 64 +
                                                            mch * 8),
                                  pack8(acc));
                }
                __syncwarp();
                if (lane == 0) {
#pragma unroll
                    for (int j = 0; j < 4; ++j) mbar_arrive(bar(bEmpty(slot[j])));
                }
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
                     "r"(kTmemCols)
                     : "memory");
    }
    cluster_sync_all();  // no CTA leaves while another may address its smem
}

// ---------------------------------------------------------------- host

struct DevState {
    bool init = false;
    bool ok = false;
    int max_clusters = 0;
};
std::mutex g_fmu;
DevState g_dev[64];

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

const DevState &dev_state(const DeviceInfo &di) {
    std::lock_guard<std::mutex> lk(g_fmu);
    DevState &st = g_dev[di.device];
    if (st.init) return st;
    st.init = true;
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, di.device) != cudaSuccess) return st;
    if (prop.major != 10 || prop.minor != 3) return st;  // built for sm_103a only
    if (encode_fn() == nullptr) return st;
    const size_t smem = smem_bytes(4 * 5);
    if (cudaFuncSetAttribute(k_fused, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem) != cudaSuccess)
        return st;
    if (cudaFuncSetAttribute(k_fused, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) !=
        cudaSuccess)
        return st;
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
    if (cudaOccupancyMaxActiveClusters(&nc, k_fused, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return st;
    }
    st.max_clusters = nc;
    st.ok = nc > 0;
    return st;
}

bool path_forced_general() {
    const char *e = getenv("HCMIX_PATH");
    return e != nullptr && e[0] == 'g';
}

}  // namespace

bool fused_supported(int hc, int64_t d, const DeviceInfo &di) {
    if (hc != 4 || d % (kCluster * 64) != 0 || d < 2 * kCluster * 64 || d > 5 * kCluster * 64)
        return false;
    if (path_forced_general()) return false;
    return dev_state(di).ok;
}

cudaError_t launch_fused(int64_t n, int hc, int64_t d, int iters, float eps, float norm_eps,
                         const uint16_t *x, const float *w, const float *scale,
                         const float *base, float *mixes, float *pre, float *post, float *comb,
                         uint16_t *y, const DeviceInfo &di, cudaStream_t s) {
    const DevState &st = dev_state(di);
    if (!st.ok || hc != 4 || n >= (int64_t(1) << 31)) return cudaErrorNotSupported;
    const int64_t F = 4 * d;
    CUtensorMap tmap;
    const cuuint64_t gdim[2] = {(cuuint64_t)F, (cuuint64_t)n};
    const cuuint64_t gstride[1] = {(cuuint64_t)(F * 2)};
    const cuuint32_t box[2] = {64, kTM};
    const cuuint32_t estride[2] = {1, 1};
    CUresult r = encode_fn()(&tmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                             const_cast<uint16_t *>(x), gdim, gstride, box, estride,
                             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                             CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    FusedParams p;
    p.n = n;
    p.d = (int)d;
    p.ncc = (int)(d / (kCluster * 64));
    p.nkc = 4 * p.ncc;
    p.num_tiles = (int)((n + kTM - 1) / kTM);
    p.iters = iters;
    p.mixes_only = pre == nullptr ? 1 : 0;
    p.eps = eps;
    p.norm_eps = norm_eps;
    p.F = (float)F;
    p.w = w;
    p.scale = scale;
    p.base = base;
    p.mixes = mixes;
    p.pre = pre;
    p.post = post;
    p.comb = comb;
    p.y = y;
    p.err = di.err_word;
    const int nclusters = p.num_tiles < st.max_clusters ? p.num_tiles : st.max_clusters;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(nclusters * kCluster));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem_bytes(p.nkc);
    cfg.stream = s;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = kCluster;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, k_fused, tmap, p);
    if (e != cudaSuccess) return e;
    return launched();
}

}  // namespace hc
