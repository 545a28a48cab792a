/*
 * hcmix.h -- C ABI of libhcmix.so: hyper-connection (HC) residual mixing on
 * NVIDIA GB300 (sm_103a).
 *
 * The operations are those of the "DeepSeek V4.1" model-atlas pages:
 *   hc_mixes           "Mix projection" page: formula for m and Block.hc_mixes
 *   hc_split_sinkhorn  "Reading weights" page: pre formula and the
 *                      hc_split_sinkhorn kernel and its wrapper
 *   hc_pre, hc_post    "Mix projection" page: Block.hc_pre, Block.hc_post
 *   hc_mixes_pre       the first three fused: what one sublayer needs before
 *                      it runs (Block docstring on the same page)
 *   hc_post_mixes_pre  hc_post of one sublayer fused with hc_mixes_pre of the
 *                      next (same docstring)
 *
 * Conventions shared by every entry point
 *   - Every tensor pointer is a DEVICE pointer owned by the caller.  The
 *     library never allocates, frees or retains memory, and keeps no pointer
 *     after a call returns.
 *   - Every call is asynchronous on `stream` (NULL = the legacy default
 *     stream) and returns as soon as its kernels are enqueued.
 *   - n is the flattened token count (the pages view [b, s, ...] tensors as
 *     [n, ...]); hc is the number of residual copies; d the channel width.
 *     F = hc*d features per token and mix_hc = (2+hc)*hc mix numbers.
 *   - bf16 tensors are passed as their 16-bit patterns (uint16_t); float
 *     tensors are IEEE binary32.  All tensors are dense, row-major, with the
 *     layouts stated per function.
 *   - Arguments are validated on the host before anything is enqueued; a
 *     call that returns an error has launched nothing.  n == 0 is a valid
 *     no-op.  Supported: hc in {4, 8}; d > 0 with d % 8 == 0; every pointer
 *     16-byte aligned; iters >= 1; eps >= 0; norm_eps >= 0.
 *   - Outputs must not overlap inputs or each other, except that hc_post may
 *     write y over residual exactly (y == residual).
 *   - The library never aborts, exits or traps.  CUDA launch failures are
 *     returned as HC_ERR_CUDA.  Kernels with bounded internal waits record a
 *     timeout in a per-device error word that hc_device_error() reads.
 *   - Launch overlap (environment variable HCMIX_PDL=0 turns it off): the
 *     decode kernel (hc = 4, d % 256 == 0, d <= 5120, up to 16 tokens per
 *     16-CTA cluster the device co-schedules: 112 on GB300; it serves
 *     hc_mixes, hc_mixes_pre, hc_mixes_pre_norm and hc_post_mixes_pre on
 *     those shapes) and the hc_post kernel are launched with programmatic
 *     dependent launch, so they may start while the kernel enqueued just
 *     before them in the stream is still running.  They read every
 *     activation only after that kernel has completed, but the decode kernel
 *     starts copying its slice of w_mix at once: w_mix must not be written by
 *     the kernel enqueued immediately before the call (weights written by an
 *     earlier kernel, a copy or a memset in between are fine).
 */
#ifndef HCMIX_H
#define HCMIX_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t / CUstream. */
typedef struct CUstream_st *hc_stream_t;

typedef enum hc_status {
    HC_OK = 0,
    HC_ERR_INVALID_ARG = 1,  /* null pointer, negative size, bad iters/eps,
                                overlapping buffers, workspace too small */
    HC_ERR_UNSUPPORTED = 2,  /* hc not in {4, 8}, sizes beyond int64 range */
    HC_ERR_MISALIGNED = 3,   /* d % 8 != 0 or a pointer not 16-byte aligned */
    HC_ERR_CUDA = 4          /* a CUDA runtime call or launch failed */
} hc_status;

#define HCMIX_ABI_VERSION 1

/* Static, NUL-terminated description of a status code.  Never NULL. */
const char *hc_status_string(hc_status s);

/* HCMIX_ABI_VERSION of the built library. */
int hc_abi_version(void);

/*
 * hc_mixes -- mix projection ("Mix projection" page, formula for m):
 *   r_t          = 1 / sqrt( mean_f x_{t,f}^2 + norm_eps )
 *   mixes_{t,i}  = r_t * sum_f x_{t,f} * w_mix_{i,f}
 * with x flattened per token, f = j*d + c.  Accumulation is binary32.
 *   x      [n, hc, d] bf16 (in)
 *   w_mix  [mix_hc, hc*d] float (in) -- the hc_{attn,ffn}_fn parameter
 *   mixes  [n, mix_hc] float (out)
 */
hc_status hc_mixes(int64_t n, int hc, int64_t d, float norm_eps,
                   const uint16_t *x, const float *w_mix, float *mixes,
                   hc_stream_t stream);

/*
 * hc_split_sinkhorn -- split of the mixes and Sinkhorn normalisation
 * ("Reading weights" page, pre formula and the hc_split_sinkhorn kernel):
 *   pre_j   = sigmoid(m_j * s0 + b_j) + eps
 *   post_j  = 2 * sigmoid(m_{hc+j} * s1 + b_{hc+j})
 *   L_{j,k} = m_{2hc+j*hc+k} * s2 + b_{2hc+j*hc+k}
 *   comb    = softmax over k of L, + eps; then a column step; then iters-1
 *             rounds of (row step, column step), where a step divides each
 *             entry by (its row or column sum + eps).
 *   mixes    [n, mix_hc] float (in)
 *   hc_scale [3] float (in) = (s0, s1, s2);  hc_base [mix_hc] float (in) = b
 *   pre, post [n, hc] float (out);  comb [n, hc, hc] float (out), [t, j, k]
 * iters < 1 is rejected (HC_ERR_INVALID_ARG).
 */
hc_status hc_split_sinkhorn(int64_t n, int hc, int iters, float eps,
                            const float *mixes, const float *hc_scale,
                            const float *hc_base, float *pre, float *post,
                            float *comb, hc_stream_t stream);

/*
 * hc_pre -- collapse of the copies ("Mix projection" page, Block.hc_pre):
 *   y_{t,c} = sum_j pre_{t,j} * x_{t,j,c}, binary32 accumulation, stored as
 *   bf16 rounded to nearest-even.
 *   x [n, hc, d] bf16 (in);  pre [n, hc] float (in);  y [n, d] bf16 (out)
 */
hc_status hc_pre(int64_t n, int hc, int64_t d, const uint16_t *x,
                 const float *pre, uint16_t *y, hc_stream_t stream);

/*
 * hc_post -- expansion back to hc copies ("Mix projection" page,
 * Block.hc_post):
 *   y_{t,k,c} = post_{t,k} * out_{t,c} + sum_j comb_{t,j,k} * residual_{t,j,c}
 * (the sum runs over the FIRST comb index), binary32 arithmetic, stored as
 * bf16 rounded to nearest-even.
 *   out [n, d] bf16 (in);  residual [n, hc, d] bf16 (in)
 *   post [n, hc] float (in);  comb [n, hc, hc] float (in)
 *   y [n, hc, d] bf16 (out); y == residual (in place) is allowed.
 */
hc_status hc_post(int64_t n, int hc, int64_t d, const uint16_t *out,
                  const uint16_t *residual, const float *post,
                  const float *comb, uint16_t *y, hc_stream_t stream);

/*
 * hc_mixes_pre -- hc_mixes, hc_split_sinkhorn and hc_pre in one call, i.e.
 * everything a sublayer needs from the stream before it runs (Block
 * docstring, "Mix projection" page).  Results equal those of the three
 * separate calls up to binary32 rounding order.
 *   x [n, hc, d] bf16 (in); w_mix, hc_scale, hc_base as above (in)
 *   mixes [n, mix_hc] float (out, may be NULL)
 *   pre, post [n, hc], comb [n, hc, hc] float (out)
 *   y [n, d] bf16 (out) -- the collapsed sublayer input
 *   workspace: device scratch (nullable), 256-byte aligned, not shared with
 *   another call in flight.  hc_workspace_bytes(n, hc, d) is a size that
 *   serves every path.  What reads it:
 *     - the decode and fused paths (hc = 4 with d % 256 == 0, d <= 5120, on
 *       the shapes and token counts they take) read none of it: NULL, or
 *       any size, is accepted there;
 *     - the general path (every other shape) keeps the mix numbers there
 *       when mixes is NULL: the workspace must then hold at least n * mix_hc
 *       floats (rounded up to 256 bytes), else HC_ERR_INVALID_ARG (or
 *       HC_ERR_MISALIGNED), returned before anything is enqueued;
 *     - at hc = 8 the general path also puts W converted to the tensor
 *       core's bf16 hi/lo rows (4 * mix_hc * hc*d bytes) past the mix numbers
 *       (at its start when mixes is given); a workspace without that room is
 *       accepted and the projection then converts W inside its kernel
 *       (slower, same results bit for bit).
 */
hc_status hc_mixes_pre(int64_t n, int hc, int64_t d, int iters, float eps,
                       float norm_eps, const uint16_t *x, const float *w_mix,
                       const float *hc_scale, const float *hc_base,
                       float *mixes, float *pre, float *post, float *comb,
                       uint16_t *y, void *workspace, size_t workspace_bytes,
                       hc_stream_t stream);

/*
 * hc_mixes_pre_norm -- hc_mixes_pre whose collapsed output is also passed
 * through the RMSNorm the block applies before the sublayer (attn_norm /
 * ffn_norm; named on the pages but not shown, so the standard form is
 * taken): with yc the bf16 collapse of hc_mixes_pre,
 *   y[t][c] = bf16( (yc[t][c] / sqrt(mean_c yc[t][c]^2 + rms_eps)) * rms_weight[c] ).
 *   rms_weight [d] float (in, 16-byte aligned); rms_eps >= 0 (the model uses
 *   1e-20); all other arguments, the workspace rule included, as in
 *   hc_mixes_pre.  y holds the normalised rows; pre/post/comb/mixes are those
 *   of hc_mixes_pre.  rms_weight == NULL is HC_ERR_INVALID_ARG.
 * One launch on every path.  On the fused path (hc = 4, d a multiple of 1024
 * above the decode limit) the mean of squares is that of the binary32
 * collapse before its bf16 rounding (pre^T G pre, G the copies' Gram matrix
 * summed while the tokens stream through), so the factor is known before y
 * is written; it differs from the formula above by far less than one bf16
 * step of y.
 */
hc_status hc_mixes_pre_norm(int64_t n, int hc, int64_t d, int iters, float eps,
                            float norm_eps, const uint16_t *x, const float *w_mix,
                            const float *hc_scale, const float *hc_base,
                            const float *rms_weight, float rms_eps, float *mixes,
                            float *pre, float *post, float *comb, uint16_t *y,
                            void *workspace, size_t workspace_bytes,
                            hc_stream_t stream);

/*
 * hc_post_mixes_pre -- the boundary between two sublayers in one call: the
 * expansion of sublayer s's output back into the stream, then everything the
 * next sublayer needs from that stream ("Mix projection" page, Block
 * docstring: each sublayer sits between hc_pre and hc_post, and the stream
 * hc_post produces is the input of the next sublayer):
 *   x_next = hc_post(out, residual, post, comb)              (sublayer s)
 *   (y_next, pre_next, post_next, comb_next[, mixes])
 *          = hc_mixes_pre(x_next; w_mix, hc_scale, hc_base)   (sublayer s+1)
 * Each sublayer uses the coefficients computed from its own input stream.
 * Results equal those of hc_post followed by hc_mixes_pre: x_next bit for
 * bit; the rest up to binary32 rounding order (bit for bit where both calls
 * take the same projection kernel).  At hc = 4 it is one kernel that reads
 * the residual once -- the new stream is computed in shared memory, stored to
 * x_next and projected from there, which saves re-reading it from HBM -- on
 * the fused path (d a multiple of 1024 up to 5120, more tokens than the
 * decode kernel takes) and on the decode path (up to 16 tokens per 16-CTA
 * cluster the device co-schedules, d a multiple of 256 up to 5120).
 *   out [n, d] bf16;  residual [n, hc, d] bf16;  post [n, hc], comb [n, hc, hc]
 *   float -- sublayer s's output and coefficients (in)
 *   x_next [n, hc, d] bf16 (out) -- the new stream; x_next == residual (in
 *   place) is allowed
 *   w_mix, hc_scale, hc_base -- sublayer s+1's parameters (in)
 *   mixes (out, may be NULL), pre_next, post_next [n, hc], comb_next
 *   [n, hc, hc], y_next [n, d] -- as hc_mixes_pre's outputs on x_next
 *   workspace, workspace_bytes -- as in hc_mixes_pre
 * Every output must be disjoint from every input and from every other output
 * (except x_next == residual); in particular pre_next/post_next/comb_next may
 * not be the buffers that hold post/comb.
 */
hc_status hc_post_mixes_pre(int64_t n, int hc, int64_t d, const uint16_t *out,
                            const uint16_t *residual, const float *post, const float *comb,
                            uint16_t *x_next, int iters, float eps, float norm_eps,
                            const float *w_mix, const float *hc_scale, const float *hc_base,
                            float *mixes, float *pre_next, float *post_next, float *comb_next,
                            uint16_t *y_next, void *workspace, size_t workspace_bytes,
                            hc_stream_t stream);

/* Scratch bytes for hc_mixes_pre(_norm) at these sizes, enough for whichever
 * path the call takes: n * mix_hc floats rounded up to 256 bytes, plus at
 * hc = 8 the converted W (4 * mix_hc * hc*d bytes, rounded up to 256); 0 for
 * n == 0 or invalid sizes.  Paths that read less (the decode and fused paths
 * read nothing) accept a smaller workspace or NULL, as hc_mixes_pre states.
 * Pure host function; the value depends only on its arguments. */
size_t hc_workspace_bytes(int64_t n, int hc, int64_t d);

/*
 * hc_device_error -- reads the error word of the current CUDA device:
 * bit 0 set = a kernel gave up on a bounded wait (its outputs for the
 * affected tile are not valid); bit 1 set = a fused kernel found its shared
 * memory not on a 1024-byte boundary and did no work (its outputs are not
 * valid).  Synchronises the device.  With clear != 0
 * the word is reset to 0 afterwards.  flags may be NULL (then only clears).
 */
hc_status hc_device_error(unsigned int *flags, int clear);

/*
 * hc_selftest_wait_timeout -- diagnostic with no counterpart on the pages:
 * enqueues one CTA that waits, through the same bounded wait the kernels
 * use, on a barrier nothing arrives on, so the wait gives up after
 * limit_ns nanoseconds and sets bit 0 of the error word (read it with
 * hc_device_error).  It shows that a wait that cannot finish ends with a
 * status instead of a hang or a fault, and that the context stays usable.
 * 1 <= limit_ns <= 1e9 (else HC_ERR_INVALID_ARG).
 */
hc_status hc_selftest_wait_timeout(uint64_t limit_ns, hc_stream_t stream);

/* Device floats that libhcmix.so keeps for hc_mixes_pre_noalloc: a fixed
 * array of 4 MiB on every GPU that loads the library, held until exit. */
#define HC_NOALLOC_SCRATCH_FLOATS (1u << 20)

/*
 * hc_mixes_pre_noalloc -- hc_mixes_pre for callers that cannot allocate device
 * memory.  The pages have no counterpart to this entry point; it exists for
 * this library's users only.
 *
 * Some callers may not call cudaMalloc at all: an engine or plugin host that
 * owns every device allocation and hands its plugins only input and output
 * buffers, a framework capturing a region into a CUDA graph where allocation
 * is forbidden, an allocator's own callbacks, or a real-time loop that must
 * never reach the allocator.  hc_mixes_pre needs a workspace for the mix
 * numbers when the caller does not want them and the shape takes its general
 * path; this call keeps them instead in a fixed array compiled into the
 * library (HC_NOALLOC_SCRATCH_FLOATS floats), and otherwise runs what
 * hc_mixes_pre's general path runs with mixes == NULL: the projection (on the
 * tensor cores where they take the shape, converting W inside the kernel,
 * else on the CUDA cores), split/Sinkhorn, and the collapse.  Its results
 * equal those of hc_mixes_pre on that path; on the decode and fused paths
 * hc_mixes_pre agrees with it within the library's tolerances.
 *
 * Arguments, layouts and validation are those of hc_mixes_pre without mixes
 * and workspace.  n * (2+hc)*hc must not exceed HC_NOALLOC_SCRATCH_FLOATS
 * (43,690 tokens at hc = 4, 13,107 at hc = 8); larger n is rejected with
 * HC_ERR_UNSUPPORTED before anything is enqueued.  The call allocates and
 * frees nothing.
 *
 * The first call on a device (and the first after the device's context was
 * recreated, e.g. by cudaDeviceReset) looks up the device address of the array
 * on the current device (cudaGetSymbolAddress), so make that first call before
 * any stream capture.  All calls share the one array per device: calls that
 * overlap on the GPU (different streams, or unordered work from different
 * threads) race on it and must be ordered by the caller.  Each call writes
 * every scratch element it reads, so nothing needs clearing between calls.
 */
hc_status hc_mixes_pre_noalloc(int64_t n, int hc, int64_t d, int iters, float eps,
                               float norm_eps, const uint16_t *x, const float *w_mix,
                               const float *hc_scale, const float *hc_base, float *pre,
                               float *post, float *comb, uint16_t *y, hc_stream_t stream);

/* Number of kernels this library has enqueued in this process (all devices,
 * all threads) since it was loaded.  Host-only counter for diagnostics. */
uint64_t hc_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* HCMIX_H */
