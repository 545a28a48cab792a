// hc_fused.cu -- fused RMS statistic + mix projection + split/Sinkhorn +
// collapse for hc = 4 on sm_103a ("Mix projection" page: formula for m,
// Block.hc_mixes, Block.hc_pre; "Reading weights" page: hc_split_sinkhorn).
//
// Work decomposition
//   * A cluster of 16 CTAs (one per SM) is persistent over 64-token tiles.
//     CTA r owns, in every copy, the 64-channel chunks cc*16 + r (cc <
//     d/1024), i.e. 4*d/16 of the F = 4*d features of each token.  So at
//     each stage the cluster reads 2 KB contiguous of every (token, copy) row
//     (contiguous 640-byte blocks per CTA put the CTAs' 128-byte pieces of a
//     row 640 bytes apart).
//   * The CTA keeps its slice of W_mix resident in shared memory for the whole
//     kernel, split into bf16 hi + lo rows (48 rows = 24 hi, 24 lo), in the
//     128-byte-swizzled K-major layout the tensor core reads.
//   * x streams through a 3-slot ring: one TMA operation per (tile, 64-channel
//     chunk) brings that chunk of all 4 copies of the tile's 64 tokens (4
//     swizzled [64 x 64] sub-tiles, 32 KB).  Few, large TMA operations matter:
//     the per-CTA rate of TMA operations, not their size, bounds the bandwidth
//     of small boxes; three slots keep two loads in flight while the third is
//     consumed.  Per sub-tile, 4 tcgen05.mma (M=128 rows of which the 64 tokens
//     are the first half, N=48, K=16) accumulate x.(W_hi + W_lo) in TMEM
//     (binary32); 4 square warps add x^2 per token.
//   * At the end of a tile each CTA sends its 24 partial mix numbers and
//     partial sum of squares per token to the token's owner CTA (4 tokens per
//     CTA) with asynchronous distributed-shared-memory stores whose bytes
//     complete the owner's barrier; the owner hands the buffer back with a
//     relaxed remote arrive (a release-ordered one waits for the SM's memory
//     traffic and cost microseconds per tile).  The owner warp reduces the 16
//     records in a fixed order, forms r and m, computes pre (and then post and
//     the Sinkhorn comb) and writes them out.
//   * The owner CTA also collapses its own tokens: y = sum_j pre_j x_j over
//     all d channels of its 4 tokens, re-reading their rows with 16-byte loads
//     (the bytes were fetched from HBM by the cluster's TMA a few microseconds
//     earlier and are served by L2).  pre never leaves the CTA.
//   Every consumer of the ring (MMA thread, 4 square warps) waits on and
//   releases every stage in order, so each wait is for the phase right after
//   one it has already seen.
//
// Two variants of the same kernel (template flags):
//   * POST (hc_post_mixes_pre): hc_post of the previous sublayer in front.
//     The ring streams the residual; 8 post warps (20 warps in all) rewrite
//     each stage in place into the new stream (post_k out + sum_j comb[j][k]
//     x_j, in hc_post's order), which the MMA and the squares then read; the
//     MMA thread stores each rewritten stage to x_next with one TMA store
//     from the slot and, at a tile's last stage, waits for the stores to
//     complete before the tile's records may leave (the collapse re-reads
//     x_next).
//   * NORM (hc_mixes_pre_norm): the RMSNorm of the collapse.  The square
//     warps also sum the ten entries G_jk = sum_c x_jc x_kc of each row's
//     copies and store them, with the row's sum of squares, into the owners'
//     records; the owner forms the
//     collapse's sum of squares as pre^T G pre, so its RMS factor is known
//     before the collapse writes y = bf16((bf16(sum_j pre_j x_j) g) r).
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
#include "hc_ptx.cuh"

namespace hc {
namespace {

using namespace ptx;

constexpr int kCluster = 16;             // CTAs per cluster
constexpr int kTM = 64;                  // tokens per tile
constexpr int kMix = 24;                 // (2 + 4) * 4
constexpr int kNW = 48;                  // B rows: 24 hi + 24 lo
constexpr int kSlots = 3;                // x ring depth (one 64-channel chunk of a tile per slot)
constexpr int kSubBytes = kTM * 128;     // one swizzled [64 tokens x 64 channels] sub-tile
constexpr int kStageBytes = 4 * kSubBytes;  // the 4 copies' sub-tiles of one chunk
constexpr int kWChunkBytes = kNW * 128;  // one [48 x 64] bf16 chunk of W
constexpr int kOwn = kTM / kCluster;     // tokens owned per CTA per tile
// floats per partial record: 24 mix partials, the sum of squares, and with
// the RMSNorm the 10 entries G_jk (j <= k) of the copies' Gram matrix
constexpr int kRec = 36;
constexpr int kGram = 10;
// bytes of records one owner receives per tile: 16 senders x 4 tokens x
// record bytes per sender and token: 6 x 16 (mixes) + 16 (sum of squares,
// padded), or with the RMSNorm 6 x 16 (mixes, from the read-out warps) +
// 3 x 16 (sum of squares and Gram entries, padded, from the square warps)
__host__ __device__ constexpr uint32_t recv_tx(bool norm) {
    return kCluster * kOwn * (norm ? 9 * 16 : 7 * 16);
}
constexpr int kMaxNcc = 5;               // w <= 320 channels per CTA (d <= 5120)
constexpr int kTmemCols = 128;
// The producer runs at most kLag tiles ahead of this CTA's collapse, which
// re-reads every tile from L2 and so needs it to still be there.
constexpr int kLag = 3;
constexpr int kColDoneBufs = 4;  // > kLag: the awaited phase is unambiguous
static_assert(kColDoneBufs > kLag, "pre staging and col_done must outlive the lag");

// warp roles.  hc_mixes_pre: 16 warps (512 threads, 128 registers each);
// with POST (hc_post in front) 20 warps (96 registers: 5 warps per SM
// sub-partition), 8 of them computing the new stream.
constexpr int kWarpProducer = 0;
constexpr int kWarpMma = 1;      // lane 0 issues the MMAs (and with POST the x_next stores)
constexpr int kWarpEpi0 = 8;     // 8, 9: TMEM read-out (lanes 0..63), records to owners
constexpr int kWarpOwner = 12;   // reduces the records of this CTA's tokens, Sinkhorn
constexpr int kCollapseWarps = 7;
constexpr int kCollapseThreads = kCollapseWarps * 32;
// The wide layout (POST, and NORM whose square warps also sum the Gram
// entries) has 20 warps and 8 square warps; the plain one 16 and 4.
template <bool POST, bool NORM = false>
struct Roles {
    static constexpr bool kWide = POST || NORM;
    static constexpr int kWarps = kWide ? 20 : 16;
    static constexpr int kThreads = kWarps * 32;
    // square warps (with POST: post warps): 2..5, or 2..7, 10, 11
    static constexpr int kSqWarps = kWide ? 8 : 4;
    __host__ __device__ static constexpr int sq_index(int w) {
        return (w >= 2 && w < (kWide ? 8 : 6)) ? w - 2 : (kWide && (w == 10 || w == 11)) ? w - 4 : -1;
    }
    // collapse warps: 6, 7, 10, 11, 13, 14, 15, or 13..19
    __host__ __device__ static constexpr int col_index(int w) {
        return kWide ? (w >= 13 && w < 20 ? w - 13 : -1)
                     : (w == 6 ? 0 : w == 7 ? 1 : w == 10 ? 2 : w == 11 ? 3
                                                  : (w >= 13 && w < 16 ? w - 9 : -1));
    }
    // Ring consumers: the MMA commit and the square warps; with POST the MMA
    // commit and the MMA thread once the slot's TMA store has read it (the
    // post warps are done with a slot when they arrive on post_done, before
    // either of those reads it).
    static constexpr int kEmptyArrivals = POST ? 2 : 1 + kSqWarps;
    // sq_full: the square warps, and with POST the MMA thread once the
    // tile's new stream is written and visible (the epilogue waits for it
    // before the tile's records go out, and so before any collapse re-reads)
    static constexpr int kSqFullArrivals = kSqWarps + (POST ? 1 : 0);
    // lanes per token row in the square warps: a lane covers 8 / kLanesPerRow
    // 16-byte pieces (8 channels each) of each copy
    static constexpr int kLanesPerRow = kWide ? 4 : 2;
    static constexpr int kPieces = 8 / kLanesPerRow;
};
constexpr int kThreadsPlain = Roles<false>::kThreads;
constexpr int kThreadsWide = Roles<true>::kThreads;
static_assert(Roles<false, true>::kThreads == kThreadsWide, "POST and NORM share a layout");

// tcgen05 instruction descriptor: D f32, A/B bf16, both K-major, N=48, M=128.
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(kNW >> 3) << 17) |
                            ((uint32_t)(128 >> 4) << 24);

struct FusedParams {
    int64_t n;
    int d;
    int ncc;        // 64-channel sub-tiles per copy per CTA (w / 64)
    int num_tiles;
    int iters;
    int mixes_only;
    float eps;
    float norm_eps;
    float F;
    const uint16_t *x;
    const float *w;
    const float *scale;
    const float *base;
    float *mixes;
    float *pre;
    float *post;
    float *comb;
    uint16_t *y;
    unsigned int *err;
    // hc_post of the previous sublayer (POST variant only): the ring streams
    // the residual, and the stream x that the projection, the squares and
    // the collapse see is x_next = hc_post(out, residual, post_in, comb_in)
    const uint16_t *out;
    const float *post_in;
    const float *comb_in;
    uint16_t *x_next;
    // RMSNorm of the sublayer input (NORM variant only): y is written as
    // RMSNorm(y) with weight rms_w [d]
    const float *rms_w;
    float rms_eps;
};

__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap *map, int c0, int c1,
                                            int c2, int c3, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar)
        : "memory");
}

// TMA store of a [64 x 64] x 4 box from shared memory, and the bulk-group
// bookkeeping that tells when it has read the slot / written memory.
__device__ __forceinline__ void tma_store_4d(const CUtensorMap *map, int c0, int c1, int c2,
                                             int c3, uint32_t src) {
    asm volatile(
        "cp.async.bulk.tensor.4d.global.shared::cta.bulk_group [%0, {%1, %2, %3, %4}], [%5];" ::"l"(
            reinterpret_cast<uint64_t>(map)),
        "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(src)
        : "memory");
}
__device__ __forceinline__ void bulk_commit() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
template <int N>
__device__ __forceinline__ void bulk_wait() {
    asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}
// L2 prefetch of a [64 x 64] box of a 2-D tensor
__device__ __forceinline__ void tma_prefetch_2d(const CUtensorMap *map, int c0, int c1) {
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(c0), "r"(c1)
                 : "memory");
}

// ---------------------------------------------------------------- layout

struct Smem {
    uint8_t *ring;    // kSlots stages of 4 sub-tiles [64 x 64] bf16 (one per copy), swizzled
    uint8_t *w;       // 4*ncc chunks of [48 x 64] bf16, swizzled, chunk = copy*ncc + cc
    float *recv;      // [kCluster][kOwn][kRec]      partials received as owner
    float *sq;        // [2][kTM]                    this CTA's partial sums of squares
    float *stage;     // [kColDoneBufs][kOwn][8]     pre (and the RMS factor) of the owned tokens, by tile % 4
    uint64_t *bar;    // barriers, see below
    uint32_t *tmem;   // TMEM base address written by tcgen05.alloc
    int *abort;
};

// barrier indices
__host__ __device__ constexpr int bFull(int s) { return s; }
__host__ __device__ constexpr int bEmpty(int s) { return kSlots + s; }
__host__ __device__ constexpr int bAccFull(int b) { return 2 * kSlots + b; }
__host__ __device__ constexpr int bAccEmpty(int b) { return 2 * kSlots + 2 + b; }
__host__ __device__ constexpr int bSqFull(int b) { return 2 * kSlots + 4 + b; }
__host__ __device__ constexpr int bSqEmpty(int b) { return 2 * kSlots + 6 + b; }
constexpr int kRecvFull = 2 * kSlots + 8;
constexpr int kRecvFree = 2 * kSlots + 9;
__host__ __device__ constexpr int bPreReady(int i) { return 2 * kSlots + 10 + i; }
__host__ __device__ constexpr int bColDone(int i) { return 2 * kSlots + 10 + kColDoneBufs + i; }
constexpr int kMmaDrain = 2 * kSlots + 10 + 2 * kColDoneBufs;
__host__ __device__ constexpr int bPostDone(int s) { return kMmaDrain + 1 + s; }
constexpr int kNumBars = kMmaDrain + 1 + kSlots;

constexpr size_t kRingBytes = (size_t)kSlots * kStageBytes;
constexpr size_t kRecvBytes = (size_t)kCluster * kOwn * kRec * 4;

// The dynamic shared memory of a kernel with no static shared memory starts
// on a 1024-byte boundary (the 128-byte swizzle atoms of the ring and W need
// it); the kernel checks that and does no work if it does not hold.
__host__ __device__ constexpr size_t smem_bytes(int ncc) {
    return kRingBytes + (size_t)4 * ncc * kWChunkBytes + kRecvBytes + 2 * kTM * 4 +
           kColDoneBufs * kOwn * 8 * 4 + kNumBars * 8 + 16;
}

static_assert(smem_bytes(kMaxNcc) <= 232448, "over the 227 KB of shared memory per CTA");

__device__ __forceinline__ Smem carve(uint8_t *raw, int ncc) {
    uint8_t *p = raw;
    Smem s;
    s.ring = p;
    p += kRingBytes;
    // The M=128 operand of the last sub-tile reads 8 KB past the ring (rows
    // 64..127, never used): W, which follows, is at least that large.
    s.w = p;
    p += (size_t)4 * ncc * kWChunkBytes;
    s.recv = reinterpret_cast<float *>(p);
    p += kRecvBytes;
    s.sq = reinterpret_cast<float *>(p);
    p += 2 * kTM * 4;
    s.stage = reinterpret_cast<float *>(p);
    p += kColDoneBufs * kOwn * 8 * 4;
    s.bar = reinterpret_cast<uint64_t *>(p);
    p += kNumBars * 8;
    s.tmem = reinterpret_cast<uint32_t *>(p);
    s.abort = reinterpret_cast<int *>(p + 4);
    return s;
}
static_assert(4 * kWChunkBytes >= kSubBytes, "overrun of the last sub-tile");
static_assert(kStageBytes % 1024 == 0 && kWChunkBytes % 1024 == 0, "swizzle atoms stay aligned");

// First feature (within the token's F) of W chunk kc = copy*ncc + cc of CTA `rank`.
__device__ __forceinline__ int chunk_feature(int kc, int rank, const FusedParams &p) {
    const int j = kc / p.ncc, cc = kc % p.ncc;
    return j * p.d + (cc * kCluster + rank) * 64;
}

// ---------------------------------------------------------------- kernel

// NCC = w / 64 (64-channel sub-tiles per copy per CTA) is a template
// parameter so that all index arithmetic is by constants.
template <int NCC, bool POST, bool NORM>
__global__ void __launch_bounds__(Roles<POST, NORM>::kThreads, 1)
    k_fused(const __grid_constant__ CUtensorMap tmap, const __grid_constant__ CUtensorMap tmap_xn,
            const __grid_constant__ CUtensorMap tmap_out, const FusedParams p) {
    using R = Roles<POST, NORM>;
    constexpr int kThreads = R::kThreads;
    static_assert(!(POST && NORM), "hc_post in front and the RMSNorm behind are separate variants");
    constexpr uint32_t kRecvTx = recv_tx(NORM);
    extern __shared__ uint8_t smem_raw[];
    constexpr int ncc = NCC;
    const Smem sm = carve(smem_raw, ncc);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rank = (int)(blockIdx.x % kCluster);
    const int cluster = (int)(blockIdx.x / kCluster);
    const int nclusters = (int)(gridDim.x / kCluster);
    const bool mixes_only = p.mixes_only != 0;
    // off its 1024-byte boundary the layout would not fit: no tiles then
    const bool aligned = (su32(smem_raw) & 1023u) == 0;
    const int T = cluster < p.num_tiles && aligned
                      ? (p.num_tiles - cluster + nclusters - 1) / nclusters
                      : 0;
    volatile int *abort = sm.abort;
    auto bar = [&](int i) { return su32(sm.bar + i); };

    // ------------------------------------------------------------ set-up
    if (threadIdx.x == 0) {
        *abort = 0;
        if (!aligned) atomicOr(p.err, kErrSmemLayout);
        for (int s = 0; s < kSlots; ++s) {
            mbar_init(bar(bFull(s)), 1);
            mbar_init(bar(bEmpty(s)), R::kEmptyArrivals);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar(bAccFull(b)), 1);
            mbar_init(bar(bAccEmpty(b)), 2);
            mbar_init(bar(bSqFull(b)), R::kSqFullArrivals);
            mbar_init(bar(bSqEmpty(b)), 2);
        }
        mbar_init(bar(kRecvFull), 1);
        mbar_init(bar(kRecvFree), kCluster);
        for (int i = 0; i < kColDoneBufs; ++i) {
            mbar_init(bar(bPreReady(i)), 1);
            mbar_init(bar(bColDone(i)), kCollapseWarps);
        }
        mbar_init(bar(kMmaDrain), 1);
        for (int s = 0; s < kSlots; ++s) mbar_init(bar(bPostDone(s)), R::kSqWarps);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        mbar_expect_tx(bar(kRecvFull), kRecvTx);
        // The first stages' loads go out now, so that their latency overlaps
        // the W set-up below (the ring and W are disjoint).
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap))
                     : "memory");
        for (int q = 0; q < kSlots && q < ncc * T; ++q) {
            mbar_expect_tx(bar(bFull(q)), kStageBytes);
            tma_load_4d(su32(sm.ring + q * kStageBytes), &tmap, 0, (cluster + (q / ncc) * nclusters) * kTM,
                        (q % ncc) * kCluster + rank, 0, bar(bFull(q)));
        }
        // POST: the first tile's sublayer output into L2 (the post warps
        // read it with plain loads, one stage ahead)
        if (POST && T > 0)
            for (int cc = 0; cc < ncc; ++cc)
                tma_prefetch_2d(&tmap_out, (cc * kCluster + rank) * 64, cluster * kTM);
    }
    if (warp == kWarpMma) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         su32(sm.tmem)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    // W slice -> bf16 hi/lo rows in the swizzled K-major layout.  Row i < 24
    // holds hi(W[i]), row 24 + i holds lo(W[i]) = bf16(W - hi).  Each 8-float
    // piece of W is read once for both rows, with kPieces pieces in flight
    // per thread (one piece at a time waited a full L2 round trip each).
    {
        constexpr int kPieces = R::kWide ? 4 : 8;  // 96 registers in the wide layout
        const int nkc = 4 * ncc;
        const int total = kMix * nkc * 8;  // (piece q, row i, chunk kc)
        const int64_t F = 4LL * p.d;
        for (int base = threadIdx.x; base < total; base += kPieces * kThreads) {
            float4 a[kPieces], b2[kPieces];
#pragma unroll
            for (int u = 0; u < kPieces; ++u) {
                const int idx = base + u * kThreads;
                if (idx < total) {
                    const int q = idx & 7, rest = idx >> 3;
                    const int i = rest % kMix, kc = rest / kMix;
                    const float4 *src = reinterpret_cast<const float4 *>(
                        p.w + (int64_t)i * F + chunk_feature(kc, rank, p) + q * 8);
                    a[u] = __ldg(src);
                    b2[u] = __ldg(src + 1);
                }
            }
#pragma unroll
            for (int u = 0; u < kPieces; ++u) {
                const int idx = base + u * kThreads;
                if (idx < total) {
                    const int q = idx & 7, rest = idx >> 3;
                    const int i = rest % kMix, kc = rest / kMix;
                    float v[8] = {a[u].x, a[u].y, a[u].z, a[u].w,
                                  b2[u].x, b2[u].y, b2[u].z, b2[u].w};
                    float lo[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        lo[e] = v[e] - __bfloat162float(__float2bfloat16_rn(v[e]));
                    uint4 h, l;
                    h.x = pack_bf16x2(v[0], v[1]);
                    h.y = pack_bf16x2(v[2], v[3]);
                    h.z = pack_bf16x2(v[4], v[5]);
                    h.w = pack_bf16x2(v[6], v[7]);
                    l.x = pack_bf16x2(lo[0], lo[1]);
                    l.y = pack_bf16x2(lo[2], lo[3]);
                    l.z = pack_bf16x2(lo[4], lo[5]);
                    l.w = pack_bf16x2(lo[6], lo[7]);
                    uint8_t *chunk = sm.w + (size_t)kc * kWChunkBytes;
                    const int rl = kMix + i;
                    *reinterpret_cast<uint4 *>(chunk + (i >> 3) * 1024 + (i & 7) * 128 +
                                               ((q ^ (i & 7)) << 4)) = h;
                    *reinterpret_cast<uint4 *>(chunk + (rl >> 3) * 1024 + (rl & 7) * 128 +
                                               ((q ^ (rl & 7)) << 4)) = l;
                }
            }
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
        // stage q = ncc*it + cc: chunk cc of this CTA's channels, all 4 copies
        if (lane == 0) {
            int last_use[kSlots] = {-1, -1, -1};
            bool ok = true;
            for (int it = 0; it < T && ok; ++it) {
                const int tile = cluster + it * nclusters;
                // Stay at most kLag tiles ahead of this CTA's collapse: it
                // re-reads each tile from L2, which holds it only for a bounded
                // window.  Tile it-kLag uses col_done buffer (it-kLag) % 4; the
                // next tile on that buffer is not loaded yet, so the awaited
                // phase is the only one that can be pending.
                if (!mixes_only && it >= kLag) {
                    const int tw = it - kLag;
                    if (!wait_bar<false>(bar(bColDone(tw % kColDoneBufs)),
                                         (uint32_t)(tw / kColDoneBufs) & 1, abort, p.err))
                        break;
                }
                // POST: the next tile's sublayer output into L2, a tile ahead
                if (POST && it + 1 < T)
                    for (int cc = 0; cc < ncc; ++cc)
                        tma_prefetch_2d(&tmap_out, (cc * kCluster + rank) * 64, (tile + nclusters) * kTM);
                for (int cc = 0; cc < ncc; ++cc) {
                    const uint32_t q = (uint32_t)(ncc * it + cc);
                    const int slot = (int)(q % kSlots);
                    const uint32_t use = q / kSlots;
                    if (q < (uint32_t)kSlots) {  // issued during the set-up
                        last_use[slot] = 0;
                        continue;
                    }
                    if (!wait_bar<false>(bar(bEmpty(slot)), (use & 1) ^ 1, abort, p.err)) {
                        ok = false;
                        break;
                    }
                    mbar_expect_tx(bar(bFull(slot)), kStageBytes);
                    tma_load_4d(su32(sm.ring + slot * kStageBytes), &tmap, 0, tile * kTM,
                                cc * kCluster + rank, 0, bar(bFull(slot)));
                    last_use[slot] = (int)use;
                }
            }
            // no TMA may still be writing this CTA's shared memory at exit
            for (int s = 0; s < kSlots; ++s)
                if (last_use[s] >= 0)
                    wait_bar<false>(bar(bFull(s)), (uint32_t)last_use[s] & 1, abort, p.err);
        }
    } else if (warp == kWarpMma) {
        if (lane == 0) {
            bool ok = true;
            for (int it = 0; it < T && ok; ++it) {
                const int b = it & 1;
                const uint32_t use = (uint32_t)(it >> 1);
                if (!wait_bar<false>(bar(bAccEmpty(b)), (use & 1) ^ 1, abort, p.err)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem + (uint32_t)(b * 64);
                for (int cc = 0; cc < ncc; ++cc) {
                    const uint32_t q = (uint32_t)(ncc * it + cc);
                    const int slot = (int)(q % kSlots);
                    // with POST the square warps first turn the residual stage
                    // into the new stream in place
                    if (!wait_bar<false>(bar(POST ? bPostDone(slot) : bFull(slot)), (q / kSlots) & 1,
                                         abort, p.err)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a0 = su32(sm.ring + slot * kStageBytes);
                    const uint32_t b0 = su32(sm.w + (size_t)cc * kWChunkBytes);
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            mma_bf16(d_tmem, sw128_desc(a0 + j * kSubBytes + 32 * k),
                                     sw128_desc(b0 + j * ncc * kWChunkBytes + 32 * k), kIdesc,
                                     (cc | j | k) != 0);
                    }
                    mma_commit(bar(bEmpty(slot)));
                    if (POST) {
                        // x_next: the rewritten stage goes out by one TMA
                        // store straight from its slot (rows past n are
                        // clipped by the tensor map).  A slot is released once
                        // its store has read it.
                        tma_store_4d(&tmap_xn, 0, (cluster + it * nclusters) * kTM,
                                     cc * kCluster + rank, 0, a0);
                        bulk_commit();
                        if (cc + 1 < ncc) {
                            bulk_wait_read<0>();
                        } else {
                            // The tile's stores are complete and visible
                            // GPU-wide before its sq_full arrival, which the
                            // epilogue awaits before the tile's records leave
                            // for the owners (whose collapse re-reads x_next).
                            bulk_wait<0>();
                            asm volatile("fence.proxy.async.global;" ::: "memory");
                            __threadfence();
                            mbar_arrive(bar(bSqFull(b)));
                        }
                        mbar_arrive(bar(bEmpty(slot)));
                    }
                }
                if (!ok) break;
                mma_commit(bar(bAccFull(b)));
            }
            // nothing may still read this CTA's shared memory at exit
            if (POST) bulk_wait<0>();
            // all issued MMAs complete before TMEM is freed
            mma_commit(bar(kMmaDrain));
            wait_bar<false>(bar(kMmaDrain), 0, abort, p.err);
        }
    } else if (R::sq_index(warp) >= 0) {
        // Sums of squares of every stage: token i of the tile, lanes
        // kLanesPerRow per 128-byte row, kPieces 16-byte pieces each.  With
        // POST these warps first compute the new stream (hc_post) in place.
        constexpr int LP = R::kLanesPerRow, PP = R::kPieces;
        const int i = (32 / LP) * R::sq_index(warp) + lane / LP;
        const int part = lane % LP;  // pieces PP*part .. PP*part + PP-1 of each row
        auto tile_of = [&](uint32_t q) { return cluster + (int)(q / ncc) * nclusters; };
        // POST: the sublayer output's 8*PP channels of this thread's row for
        // stage q, loaded one stage ahead; the token's post and comb per tile
        uint4 onext[PP];
#pragma unroll
        for (int m = 0; m < PP; ++m) onext[m] = make_uint4(0, 0, 0, 0);
        auto prefetch_out = [&](uint32_t q) {
            if (!POST || q >= (uint32_t)(ncc * T)) return;
            const int64_t tok = (int64_t)tile_of(q) * kTM + i;
            if (tok >= p.n) {
#pragma unroll
                for (int m = 0; m < PP; ++m) onext[m] = make_uint4(0, 0, 0, 0);
                return;
            }
            const uint4 *src = reinterpret_cast<const uint4 *>(
                p.out + tok * (int64_t)p.d + (int)(q % ncc) * (kCluster * 64) + rank * 64 +
                8 * PP * part);
#pragma unroll
            for (int m = 0; m < PP; ++m) onext[m] = ld_stream(src + m);
        };
        float po[4] = {0.f, 0.f, 0.f, 0.f}, cmf[4][4];  // the token's post and comb
        prefetch_out(0);
        bool ok = true;
        for (int it = 0; it < T && ok; ++it) {
            const int b = it & 1;
            const uint32_t use = (uint32_t)(it >> 1);
            // One packed accumulator set per 32-channel quarter of the row
            // (pieces 2a, 2a+1), summed in the order (stage, piece, copy) and
            // then as ((q0 + q1) + (q2 + q3)): the same sums whichever lanes
            // hold the quarters, so both variants agree bit for bit.
            uint64_t s2[PP / 2][4];
#pragma unroll
            for (int a2 = 0; a2 < PP / 2; ++a2)
#pragma unroll
                for (int e = 0; e < 4; ++e) s2[a2][e] = 0;
            // NORM: the copies' Gram matrix G_jk = sum_c x_jc x_kc of this
            // thread's channels, entries j <= k in row order, packed pairs
            uint64_t g2[NORM ? kGram : 1];
#pragma unroll
            for (int q2 = 0; q2 < (NORM ? kGram : 1); ++q2) g2[q2] = 0;
            if (POST) {
                const int64_t tok = (int64_t)tile_of((uint32_t)(ncc * it)) * kTM + i;
                float4 pv = make_float4(0.f, 0.f, 0.f, 0.f), cv[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) cv[j] = pv;
                if (tok < p.n) {
                    pv = __ldg(reinterpret_cast<const float4 *>(p.post_in) + tok);
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        cv[j] = __ldg(reinterpret_cast<const float4 *>(p.comb_in) + tok * 4 + j);
                }
                po[0] = pv.x, po[1] = pv.y, po[2] = pv.z, po[3] = pv.w;
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    cmf[j][0] = cv[j].x, cmf[j][1] = cv[j].y, cmf[j][2] = cv[j].z, cmf[j][3] = cv[j].w;
            }
            for (int cc = 0; cc < ncc; ++cc) {
                const uint32_t q = (uint32_t)(ncc * it + cc);
                const int slot = (int)(q % kSlots);
                if (!__all_sync(0xFFFFFFFFu, wait_bar<false>(bar(bFull(slot)), (q / kSlots) & 1,
                                                             abort, p.err))) {
                    ok = false;
                    break;
                }
                const uint32_t base = su32(sm.ring + slot * kStageBytes) + i * 128;
                // 16-byte piece m of copy j of this thread's row, 128-byte
                // swizzle: the lanes of one quarter-warp hit distinct bank groups
                auto piece = [&](int j, int m) -> uint32_t {
                    return base + j * kSubBytes + (((PP * part + m) ^ (i & 7)) << 4);
                };
                if (!POST && !NORM) {
#pragma unroll
                    for (int m = 0; m < PP; ++m)
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const uint4 v = lds128(piece(j, m));
                            const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const uint64_t xp = bf16x2_to_f32x2(wv[e]);
                                ffma2(s2[m / 2][e], xp, xp);
                            }
                        }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(bEmpty(slot)));
                } else if (!POST) {
                    // the same squares in the same order, and the Gram
                    // entries of the piece's four copies
#pragma unroll
                    for (int m = 0; m < PP; ++m) {
                        uint64_t xp[4][4];  // the piece's four copies, packed binary32 pairs
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const uint4 v = lds128(piece(j, m));
                            xp[j][0] = bf16x2_to_f32x2(v.x);
                            xp[j][1] = bf16x2_to_f32x2(v.y);
                            xp[j][2] = bf16x2_to_f32x2(v.z);
                            xp[j][3] = bf16x2_to_f32x2(v.w);
                        }
#pragma unroll
                        for (int j = 0; j < 4; ++j)
#pragma unroll
                            for (int e = 0; e < 4; ++e) ffma2(s2[m / 2][e], xp[j][e], xp[j][e]);
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            int q2 = 0;
#pragma unroll
                            for (int j = 0; j < 4; ++j)
#pragma unroll
                                for (int k = j; k < 4; ++k) ffma2(g2[q2++], xp[j][e], xp[k][e]);
                        }
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(bEmpty(slot)));
                } else {
                    // hc_post ("Mix projection" page, Block.hc_post) of this
                    // thread's channels of the stage, one 8-channel piece at a
                    // time: x'_k = post_k out + sum_j comb[j][k] x_j, the
                    // product first, then the copies j = 0..3 in order (as
                    // hc_post); written back over the residual in the slot
                    // (all four input copies of a piece are read before any is
                    // written).  The MMA thread stores the slot to x_next.
                    uint4 ocur[PP];
#pragma unroll
                    for (int m = 0; m < PP; ++m) ocur[m] = onext[m];
                    prefetch_out(q + 1);
#pragma unroll
                    for (int m = 0; m < PP; ++m) {
                        // the piece's inputs as packed binary32 pairs, once
                        uint64_t xp[4][4], op[4];
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const uint4 v = lds128(piece(j, m));
                            xp[j][0] = bf16x2_to_f32x2(v.x);
                            xp[j][1] = bf16x2_to_f32x2(v.y);
                            xp[j][2] = bf16x2_to_f32x2(v.z);
                            xp[j][3] = bf16x2_to_f32x2(v.w);
                        }
                        op[0] = bf16x2_to_f32x2(ocur[m].x);
                        op[1] = bf16x2_to_f32x2(ocur[m].y);
                        op[2] = bf16x2_to_f32x2(ocur[m].z);
                        op[3] = bf16x2_to_f32x2(ocur[m].w);
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            uint64_t acc2[4];
                            const uint64_t pk = pack2(po[k], po[k]);
#pragma unroll
                            for (int e = 0; e < 4; ++e) acc2[e] = fmul2(pk, op[e]);
#pragma unroll
                            for (int j = 0; j < 4; ++j) {
                                const uint64_t cmk = pack2(cmf[j][k], cmf[j][k]);
#pragma unroll
                                for (int e = 0; e < 4; ++e) ffma2(acc2[e], cmk, xp[j][e]);
                            }
                            uint32_t nw[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                float lo, hi;
                                unpack2(acc2[e], lo, hi);
                                nw[e] = pack_bf16x2(lo, hi);
                                const uint64_t xq = bf16x2_to_f32x2(nw[e]);
                                ffma2(s2[m / 2][e], xq, xq);
                            }
                            sts128(piece(k, m), make_uint4(nw[0], nw[1], nw[2], nw[3]));
                        }
                    }
                    // the new stream in the slot, for the tensor core and the
                    // TMA store (async proxy)
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(bPostDone(slot)));
                }
            }
            if (!ok) break;
            float ss = 0.f;
#pragma unroll
            for (int a2 = 0; a2 < PP / 2; ++a2) {
                const float qs = (sum2(s2[a2][0]) + sum2(s2[a2][1])) +
                                 (sum2(s2[a2][2]) + sum2(s2[a2][3]));
                ss = a2 == 0 ? qs : ss + qs;
            }
#pragma unroll
            for (int sh = 1; sh < LP; sh <<= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, sh);
            // NORM: the row's Gram entries (the same in every lane of the row)
            float gs[NORM ? kGram : 1];
#pragma unroll
            for (int q2 = 0; q2 < (NORM ? kGram : 1); ++q2) {
                gs[q2] = NORM ? sum2(g2[q2]) : 0.f;
#pragma unroll
                for (int sh = 1; sh < LP; sh <<= 1)
                    if (NORM) gs[q2] += __shfl_xor_sync(0xFFFFFFFFu, gs[q2], sh);
            }
            if (!__all_sync(0xFFFFFFFFu,
                            wait_bar<false>(bar(bSqEmpty(b)), (use & 1) ^ 1, abort, p.err)))
                break;
            if (part == 0) sm.sq[b * kTM + i] = ss;
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(bSqFull(b)));
            if (NORM) {
                // the row's sum of squares and Gram entries go straight into
                // its owner's record (floats 24..35), once the owner has read
                // the previous tile's records; their bytes complete its
                // recv_full
                if (!__all_sync(0xFFFFFFFFu, wait_bar<true>(bar(kRecvFree), ((uint32_t)it & 1) ^ 1,
                                                            abort, p.err)))
                    break;
                if (part == 0) {
                    const int owner = i / kOwn, u = i % kOwn;
                    const uint32_t rec =
                        mapa(su32(sm.recv + (rank * kOwn + u) * kRec), (uint32_t)owner);
                    const uint32_t rfull = mapa(bar(kRecvFull), (uint32_t)owner);
                    constexpr int g = NORM ? kGram : 1;  // (indices valid for NORM)
                    // floats 24..35: the sum of squares, G_00..G_33, a pad
                    st_async_v4(rec + 96, ss, gs[0], gs[1 % g], gs[2 % g], rfull);
                    st_async_v4(rec + 112, gs[3 % g], gs[4 % g], gs[5 % g], gs[6 % g], rfull);
                    st_async_v4(rec + 128, gs[7 % g], gs[8 % g], gs[9 % g], 0.f, rfull);
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
            const float ss = sm.sq[b * kTM + i];
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(bSqEmpty(b)));
            // the owner must have read the records of the previous tile
            if (!__all_sync(0xFFFFFFFFu,
                            wait_bar<true>(bar(kRecvFree), ((uint32_t)it & 1) ^ 1, abort, p.err)))
                break;
            const uint32_t rec =
                mapa(su32(sm.recv + (rank * kOwn + u) * kRec), (uint32_t)owner);
            // 7 asynchronous stores; their bytes complete the owner's recv_full
            const uint32_t rfull = mapa(bar(kRecvFull), (uint32_t)owner);
#pragma unroll
            for (int v = 0; v < 6; ++v)
                st_async_v4(rec + 16 * v, acc[4 * v] + acc[24 + 4 * v],
                            acc[4 * v + 1] + acc[24 + 4 * v + 1],
                            acc[4 * v + 2] + acc[24 + 4 * v + 2],
                            acc[4 * v + 3] + acc[24 + 4 * v + 3], rfull);
            // with the RMSNorm the square warps send the sum of squares
            // beside the Gram entries
            if (!NORM) st_async_v4(rec + 96, ss, 0.f, 0.f, 0.f, rfull);
        }
    } else if (warp == kWarpOwner) {
        // Owner of tokens rank*kOwn + u (u < kOwn) of every tile: the 8 lanes
        // 8u..8u+7 reduce the 16 records of token u (lane 8u+q the records of
        // senders q and q+8, then a butterfly over the 8 lanes: a fixed
        // order), lane 8u forms r, m and pre for this CTA's collapse; lanes
        // 16..31 then hand the record buffer back to the 16 senders, and
        // lanes 8u run the Sinkhorn for comb.
        const int u = lane >> 3;
        const bool lead = (lane & 7) == 0;
        float bse[kMix], s0 = 0.f, s1 = 0.f, s2 = 0.f;
        if (!mixes_only && lead) {
#pragma unroll
            for (int k = 0; k < kMix; ++k) bse[k] = __ldg(p.base + k);
            s0 = __ldg(p.scale + 0);
            s1 = __ldg(p.scale + 1);
            s2 = __ldg(p.scale + 2);
        }
        for (int it = 0; it < T; ++it) {
            const int tile = cluster + it * nclusters;
            if (!__all_sync(0xFFFFFFFFu,
                            wait_bar<true>(bar(kRecvFull), (uint32_t)it & 1, abort, p.err)))
                break;
            float m[kMix];
            float ssum = 0.f;
            float G[NORM ? kGram : 1];  // NORM: the token's Gram entries over all d
#pragma unroll
            for (int q2 = 0; q2 < (NORM ? kGram : 1); ++q2) G[q2] = 0.f;
            {
                static_assert(kCluster == 16 && kOwn * 8 == 32, "8 lanes per owned token");
                const float4 *ra = reinterpret_cast<const float4 *>(
                    sm.recv + ((lane & 7) * kOwn + u) * kRec);
                const float4 *rb = reinterpret_cast<const float4 *>(
                    sm.recv + (((lane & 7) + 8) * kOwn + u) * kRec);
#pragma unroll
                for (int v = 0; v < 6; ++v) {
                    const float4 a4 = ra[v], b4 = rb[v];
                    m[4 * v] = a4.x + b4.x;
                    m[4 * v + 1] = a4.y + b4.y;
                    m[4 * v + 2] = a4.z + b4.z;
                    m[4 * v + 3] = a4.w + b4.w;
                }
                const float4 a6 = ra[6], b6 = rb[6];
                ssum = a6.x + b6.x;
                if (NORM) {
                    const float4 a7 = ra[7], b7 = rb[7], a8 = ra[8], b8 = rb[8];
                    const float ga[kGram] = {a6.y, a6.z, a6.w, a7.x, a7.y, a7.z, a7.w, a8.x, a8.y, a8.z};
                    const float gb[kGram] = {b6.y, b6.z, b6.w, b7.x, b7.y, b7.z, b7.w, b8.x, b8.y, b8.z};
#pragma unroll
                    for (int q2 = 0; q2 < (NORM ? kGram : 1); ++q2) G[q2] = ga[q2] + gb[q2];
                }
#pragma unroll
                for (int sh = 1; sh < 8; sh <<= 1) {
#pragma unroll
                    for (int k = 0; k < kMix; ++k) m[k] += __shfl_xor_sync(0xFFFFFFFFu, m[k], sh);
                    ssum += __shfl_xor_sync(0xFFFFFFFFu, ssum, sh);
                    if (NORM) {
#pragma unroll
                        for (int q2 = 0; q2 < (NORM ? kGram : 1); ++q2)
                            G[q2] += __shfl_xor_sync(0xFFFFFFFFu, G[q2], sh);
                    }
                }
            }
            float pr[4], po[4];
            int64_t t = 0;
            if (lead) {
                const float r = rsqrtf(ssum / p.F + p.norm_eps);
#pragma unroll
                for (int k = 0; k < kMix; ++k) m[k] *= r;
                t = (int64_t)tile * kTM + rank * kOwn + u;
                if (t < p.n && p.mixes != nullptr) {
                    float4 *dst = reinterpret_cast<float4 *>(p.mixes + t * kMix);
#pragma unroll
                    for (int v = 0; v < 6; ++v)
                        dst[v] = make_float4(m[4 * v], m[4 * v + 1], m[4 * v + 2], m[4 * v + 3]);
                }
                if (!mixes_only) {
                    // stage[it % 4] was last read by the collapse of tile it-4,
                    // which finished before the producer loaded tile it-1
                    // (the producer stays at most kLag = 3 tiles ahead).
                    split_pre_post<4>([&](int k) { return m[k]; }, [&](int k) { return bse[k]; },
                                      s0, s1, p.eps, pr, po);
                    float rs = 0.f;
                    if (NORM) {
                        // RMSNorm statistic of the collapse y = sum_j pre_j x_j
                        // over all d channels: sum_c y_c^2 = pre^T G pre (of
                        // the binary32 collapse, before its bf16 rounding)
                        float q = 0.f;
                        int q2 = 0;
#pragma unroll
                        for (int j = 0; j < 4; ++j)
#pragma unroll
                            for (int k = j; k < 4; ++k, ++q2)
                                q = fmaf((k == j ? 1.f : 2.f) * pr[j] * pr[k], G[q2 % (NORM ? kGram : 1)], q);
                        rs = rsqrtf(fmaxf(q, 0.f) / (float)p.d + p.rms_eps);
                    }
                    // the collapse weights pre, and with NORM the token's
                    // RMSNorm factor
                    float4 *st4 =
                        reinterpret_cast<float4 *>(sm.stage) + 2 * ((it % kColDoneBufs) * kOwn + u);
                    st4[0] = make_float4(pr[0], pr[1], pr[2], pr[3]);
                    if (NORM) st4[1] = make_float4(rs, 0.f, 0.f, 0.f);
                }
            }
            __syncwarp();
            // pre first: this CTA's collapse waits for it
            if (!mixes_only && lane == 0) mbar_arrive(bar(bPreReady(it % kColDoneBufs)));
            // All records are read (their values are in registers and used
            // above, so no later store can overtake the loads): arm recv_full
            // for the next tile's bytes, then release the buffer to every
            // sender, lanes 16..31 one CTA each.
            if (lane == 0) mbar_expect_tx(bar(kRecvFull), kRecvTx);
            if (lane >= 32 - kCluster)
                mbar_arrive_remote_relaxed(mapa(bar(kRecvFree), (uint32_t)(lane - (32 - kCluster))));
            if (!mixes_only) {
                // then the Sinkhorn for comb, off the collapse's critical path
                if (lead) {
                    float Cm[4][4];
                    sinkhorn_comb<4>([&](int k) { return m[k]; }, [&](int k) { return bse[k]; },
                                     s2, p.iters, p.eps, Cm);
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
                }
            }
            __syncwarp();
        }
    } else if (!mixes_only) {
        // Collapse of this CTA's own tokens rank*kOwn + u (u < kOwn) of every
        // tile, over all d channels: 7 warps, 224 threads.  Output vector
        // o = (token u = o / nv, 8 channels at 8*(o % nv)); 4 vectors in flight
        // per thread, each needing the 4 copies (16-byte loads from L2).
        const int ct = R::col_index(warp) * 32 + lane;
        constexpr int nv = NCC * 8 * kCluster;  // vectors per copy row (d / 8)
        constexpr int nout = kOwn * nv;
        const uint4 *x = reinterpret_cast<const uint4 *>(p.x);
        // NORM: this thread's vectors v = ct + 224 k (8 channels each)
        constexpr int kNormV = NORM ? (nv + kCollapseThreads - 1) / kCollapseThreads : 1;
        for (int it = 0; it < T; ++it) {
            const int tile = cluster + it * nclusters;
            const int ib = it % kColDoneBufs;
            if (!__all_sync(0xFFFFFFFFu, wait_bar<false>(bar(bPreReady(ib)),
                                                         (uint32_t)(it / kColDoneBufs) & 1, abort,
                                                         p.err)))
                break;
            const int64_t tok0 = (int64_t)tile * kTM + rank * kOwn;
            if (NORM) {
                // vector v (8 channels) of all kOwn tokens per step, two
                // tokens' loads in flight at a time (96 registers), so that
                // the weight loaded once for v serves the four of them:
                // y = bf16((bf16(sum_j pre_j x_j) g) r)
#pragma unroll
                for (int k = 0; k < kNormV; ++k) {
                    const int v = ct + k * kCollapseThreads;
                    if (v >= nv) break;
                    const float4 g0 = __ldg(reinterpret_cast<const float4 *>(p.rms_w) + 2 * v);
                    const float4 g1 = __ldg(reinterpret_cast<const float4 *>(p.rms_w) + 2 * v + 1);
                    const float gw[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
#pragma unroll
                    for (int h2 = 0; h2 < kOwn; h2 += 2) {
                        uint4 xv[2][4];
#pragma unroll
                        for (int u = 0; u < 2; ++u) {
                            const int64_t tok = tok0 + h2 + u;
                            if (tok < p.n) {
#pragma unroll
                                for (int j = 0; j < 4; ++j)
                                    xv[u][j] = __ldcs(x + (tok * 4 + j) * nv + v);
                            }
                        }
#pragma unroll
                        for (int u = 0; u < 2; ++u) {
                            const int64_t tok = tok0 + h2 + u;
                            if (tok < p.n) {
                                const float4 *st4 = reinterpret_cast<const float4 *>(sm.stage) +
                                                    2 * (ib * kOwn + h2 + u);
                                const float4 pr = st4[0];
                                const float rs = st4[1].x;
                                float acc[8], f[8];
                                unpack8(xv[u][0], f);
#pragma unroll
                                for (int e = 0; e < 8; ++e) acc[e] = pr.x * f[e];
                                unpack8(xv[u][1], f);
#pragma unroll
                                for (int e = 0; e < 8; ++e) acc[e] = fmaf(pr.y, f[e], acc[e]);
                                unpack8(xv[u][2], f);
#pragma unroll
                                for (int e = 0; e < 8; ++e) acc[e] = fmaf(pr.z, f[e], acc[e]);
                                unpack8(xv[u][3], f);
#pragma unroll
                                for (int e = 0; e < 8; ++e) acc[e] = fmaf(pr.w, f[e], acc[e]);
                                // the collapse in bf16 (as hc_pre writes it),
                                // then the RMSNorm: (y g) r
                                unpack8(pack8(acc), f);
#pragma unroll
                                for (int e = 0; e < 8; ++e) acc[e] = (f[e] * gw[e]) * rs;
                                st_stream(reinterpret_cast<uint4 *>(p.y) + tok * nv + v, pack8(acc));
                            }
                        }
                    }
                }
            } else {
                constexpr int G = POST ? 3 : 4;  // 96 registers with POST
                for (int o0 = ct; o0 < nout; o0 += G * kCollapseThreads) {
                    uint4 xv[G][4];
#pragma unroll
                    for (int g = 0; g < G; ++g) {
                        const int o = o0 + g * kCollapseThreads;
                        const int64_t tok = tok0 + o / nv;
                        if (o < nout && tok < p.n) {
#pragma unroll
                            for (int j = 0; j < 4; ++j)
                                xv[g][j] = __ldcs(x + (tok * 4 + j) * nv + o % nv);
                        }
                    }
#pragma unroll
                    for (int g = 0; g < G; ++g) {
                        const int o = o0 + g * kCollapseThreads;
                        const int64_t tok = tok0 + o / nv;
                        if (o < nout && tok < p.n) {
                            const float4 pr = reinterpret_cast<const float4 *>(
                                sm.stage)[2 * (ib * kOwn + o / nv)];
                            float acc[8], f[8];
                            unpack8(xv[g][0], f);
#pragma unroll
                            for (int e = 0; e < 8; ++e) acc[e] = pr.x * f[e];
                            unpack8(xv[g][1], f);
#pragma unroll
                            for (int e = 0; e < 8; ++e) acc[e] = fmaf(pr.y, f[e], acc[e]);
                            unpack8(xv[g][2], f);
#pragma unroll
                            for (int e = 0; e < 8; ++e) acc[e] = fmaf(pr.z, f[e], acc[e]);
                            unpack8(xv[g][3], f);
#pragma unroll
                            for (int e = 0; e < 8; ++e) acc[e] = fmaf(pr.w, f[e], acc[e]);
                            st_stream(reinterpret_cast<uint4 *>(p.y) + tok * nv + o % nv, pack8(acc));
                        }
                    }
                }
            }
            // this warp is done with tile it (its pre slot and its L2 lines)
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(bColDone(ib)));
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
    unsigned long long ctx = 0;  // the context the set-up below was done in
    bool ok = false;
    int max_clusters[2] = {0, 0};  // co-resident clusters, plain / wide layout
};
std::mutex g_fmu;
DevState g_dev[64];

using FusedKernel = void (*)(CUtensorMap, CUtensorMap, CUtensorMap, FusedParams);

// The instantiation for w = 64 * ncc channels per CTA (post: with the
// previous sublayer's hc_post in front; norm: with the RMSNorm of the
// collapse behind; not both).
template <int NCC>
FusedKernel kernel_ncc(bool post, bool norm) {
    return post ? k_fused<NCC, true, false> : norm ? k_fused<NCC, false, true>
                                                   : k_fused<NCC, false, false>;
}
FusedKernel kernel_for(int ncc, bool post, bool norm = false) {
    switch (ncc) {
        case 1: return kernel_ncc<1>(post, norm);
        case 2: return kernel_ncc<2>(post, norm);
        case 3: return kernel_ncc<3>(post, norm);
        case 4: return kernel_ncc<4>(post, norm);
        default: return kernel_ncc<5>(post, norm);
    }
}

const DevState &dev_state(const DeviceInfo &di) {
    std::lock_guard<std::mutex> lk(g_fmu);
    DevState &st = g_dev[di.device];
    if (st.init && st.ctx == di.ctx) return st;
    st = DevState();
    st.init = true;
    st.ctx = di.ctx;
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, di.device) != cudaSuccess) return st;
    if (prop.major != 10 || prop.minor != 3) return st;  // built for sm_103a only
    if (tensor_map_encoder() == nullptr) return st;
    for (int ncc = 1; ncc <= kMaxNcc; ++ncc)
        for (int v = 0; v < 3; ++v) {  // plain, post, norm
            const FusedKernel k = kernel_for(ncc, v == 1, v == 2);
            if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)smem_bytes(ncc)) != cudaSuccess)
                return st;
            if (cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) !=
                cudaSuccess)
                return st;
        }
    for (int post = 0; post < 2; ++post) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(kCluster);
        cfg.blockDim = dim3(post ? kThreadsWide : kThreadsPlain);
        cfg.dynamicSmemBytes = smem_bytes(kMaxNcc);
        cudaLaunchAttribute attr;
        attr.id = cudaLaunchAttributeClusterDimension;
        attr.val.clusterDim.x = kCluster;
        attr.val.clusterDim.y = 1;
        attr.val.clusterDim.z = 1;
        cfg.attrs = &attr;
        cfg.numAttrs = 1;
        int nc = 0;
        if (cudaOccupancyMaxActiveClusters(&nc, kernel_for(kMaxNcc, post), &cfg) != cudaSuccess) {
            cudaGetLastError();
            return st;
        }
        st.max_clusters[post] = nc;
    }
    st.ok = st.max_clusters[0] > 0 && st.max_clusters[1] > 0;
    return st;
}


}  // namespace

bool fused_supported(int hc, int64_t d, const DeviceInfo &di) {
    if (hc != 4 || d % (kCluster * 64) != 0 || d < kCluster * 64 || d > kMaxNcc * kCluster * 64)
        return false;
    if (forced_path() == kPathGeneral || forced_path() == kPathFfma) return false;
    return dev_state(di).ok;
}

namespace {

// ring_src: the tensor the ring streams (x, or the residual with POST);
// x: the stream the collapse re-reads (x, or x_next with POST).
cudaError_t launch_impl(int64_t n, int64_t d, int iters, float eps, float norm_eps,
                        const uint16_t *ring_src, const uint16_t *x, const float *w,
                        const float *scale, const float *base, float *mixes, float *pre,
                        float *post, float *comb, uint16_t *y, const uint16_t *out,
                        const float *post_in, const float *comb_in, uint16_t *x_next,
                        const float *rms_w, float rms_eps, const DeviceInfo &di,
                        cudaStream_t s) {
    const DevState &st = dev_state(di);
    if (!st.ok || n >= (int64_t(1) << 31)) return cudaErrorNotSupported;
    const bool with_post = out != nullptr, with_norm = rms_w != nullptr;
    if (with_post && with_norm) return cudaErrorNotSupported;
    const int64_t F = 4 * d;
    const int ncc = (int)(d / (kCluster * 64));
    // 4-D view of x: {64 channels, token, 64-channel chunk of a copy, copy};
    // one box = one chunk of all 4 copies of 64 tokens, landing as 4 swizzled
    // sub-tiles.
    CUtensorMap tmap;
    const cuuint64_t gdim[4] = {64, (cuuint64_t)n, (cuuint64_t)(d / 64), 4};
    const cuuint64_t gstride[3] = {(cuuint64_t)(F * 2), 128, (cuuint64_t)(d * 2)};
    const cuuint32_t box[4] = {64, kTM, 1, 4};
    const cuuint32_t estride[4] = {1, 1, 1, 1};
    CUresult r = tensor_map_encoder()(&tmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
                             const_cast<uint16_t *>(ring_src), gdim, gstride, box, estride,
                             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                             CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    // with POST the same view of x_next, for the stores of the rewritten
    // stages, and a 2-D view {channel, token} of the sublayer output, for
    // its L2 prefetches
    CUtensorMap tmap_xn = tmap, tmap_out = tmap;
    if (with_post) {
        r = tensor_map_encoder()(&tmap_xn, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, x_next, gdim,
                                 gstride, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                 CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                 CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
        const cuuint64_t odim[2] = {(cuuint64_t)d, (cuuint64_t)n};
        const cuuint64_t ostride[1] = {(cuuint64_t)(d * 2)};
        const cuuint32_t obox[2] = {64, kTM};
        r = tensor_map_encoder()(&tmap_out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                                 const_cast<uint16_t *>(out), odim, ostride, obox, estride,
                                 CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                                 CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                 CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    }
    FusedParams p;
    p.n = n;
    p.d = (int)d;
    p.ncc = ncc;
    p.num_tiles = (int)((n + kTM - 1) / kTM);
    p.iters = iters;
    p.mixes_only = pre == nullptr ? 1 : 0;
    p.eps = eps;
    p.norm_eps = norm_eps;
    p.F = (float)F;
    p.x = x;
    p.w = w;
    p.scale = scale;
    p.base = base;
    p.mixes = mixes;
    p.pre = pre;
    p.post = post;
    p.comb = comb;
    p.y = y;
    p.err = di.err_word;
    p.out = out;
    p.post_in = post_in;
    p.comb_in = comb_in;
    p.x_next = x_next;
    p.rms_w = rms_w;
    p.rms_eps = rms_eps;
    const int mc = st.max_clusters[with_post || with_norm ? 1 : 0];
    const int nclusters = p.num_tiles < mc ? p.num_tiles : mc;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(nclusters * kCluster));
    cfg.blockDim = dim3(with_post || with_norm ? kThreadsWide : kThreadsPlain);
    cfg.dynamicSmemBytes = smem_bytes(p.ncc);
    cfg.stream = s;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = kCluster;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel_for(p.ncc, with_post, with_norm), tmap, tmap_xn,
                                             tmap_out, p);
    if (e != cudaSuccess) return e;
    return launched();
}

}  // namespace

cudaError_t launch_fused(int64_t n, int hc, int64_t d, int iters, float eps, float norm_eps,
                         const uint16_t *x, const float *w, const float *scale,
                         const float *base, float *mixes, float *pre, float *post, float *comb,
                         uint16_t *y, const DeviceInfo &di, cudaStream_t s) {
    if (hc != 4) return cudaErrorNotSupported;
    return launch_impl(n, d, iters, eps, norm_eps, x, x, w, scale, base, mixes, pre, post, comb,
                       y, nullptr, nullptr, nullptr, nullptr, nullptr, 0.f, di, s);
}

cudaError_t launch_fused_norm(int64_t n, int hc, int64_t d, int iters, float eps, float norm_eps,
                              const uint16_t *x, const float *w, const float *scale,
                              const float *base, float *mixes, float *pre, float *post,
                              float *comb, uint16_t *y, const float *rms_w, float rms_eps,
                              const DeviceInfo &di, cudaStream_t s) {
    if (hc != 4 || pre == nullptr || rms_w == nullptr) return cudaErrorNotSupported;
    return launch_impl(n, d, iters, eps, norm_eps, x, x, w, scale, base, mixes, pre, post, comb,
                       y, nullptr, nullptr, nullptr, nullptr, rms_w, rms_eps, di, s);
}

cudaError_t launch_fused_post(int64_t n, int hc, int64_t d, const uint16_t *out,
                              const uint16_t *residual, const float *post_in,
                              const float *comb_in, uint16_t *x_next, int iters, float eps,
                              float norm_eps, const float *w, const float *scale,
                              const float *base, float *mixes, float *pre, float *post,
                              float *comb, uint16_t *y, const DeviceInfo &di, cudaStream_t s) {
    if (hc != 4 || pre == nullptr) return cudaErrorNotSupported;
    return launch_impl(n, d, iters, eps, norm_eps, residual, x_next, w, scale, base, mixes, pre,
                       post, comb, y, out, post_in, comb_in, x_next, nullptr, 0.f, di, s);
}

}  // namespace hc
