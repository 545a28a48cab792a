/*
 * hc_oracle.c -- float64 CPU oracle for hyper-connection (HC) residual mixing.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, obviously correct
 * statement of what the GPU path computes.  Only the test suite, the smoke
 * check and the benchmark's CPU-baseline leg load it.  It shares no code,
 * header, table or constant with the CUDA library: the two meet only through
 * the seeded input generators.
 *
 * Sources (all on the "DeepSeek V4.1" model-atlas pages):
 *   - "Mix projection" page, the formula for m and the code of Block.hc_mixes:
 *     m = x^f W_mix^T / sqrt(mean((x^f)^2) + norm_eps),
 *     one statistic per token over all hc*d features, x^f = x.flatten(2), so
 *     feature f = j*d + c for copy j and channel c.
 *   - "Reading weights" page, the pre formula and the hc_split_sinkhorn kernel:
 *     pre/post sigmoids, then a row softmax plus eps,
 *     a column normalisation and iters-1 rounds of row-then-column
 *     normalisation, every later denominator being (sum + eps).
 *   - "Mix projection" page, the code of Block.hc_pre and Block.hc_post.
 *   - The RMSNorm the block applies to hc_pre's output (attn_norm / ffn_norm)
 *     is named but not shown on the pages: the standard form is taken (see
 *     orc_hc_rmsnorm).
 *
 * Arithmetic: every step in double.  bf16 inputs are decoded exactly; bf16
 * outputs are rounded once, directly from the double value, to nearest-even.
 * Loops are plain and in the order the pages state them; the only
 * parallelism is an optional OpenMP loop over independent tokens, which does
 * not change any result.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------ bf16 */

/* Exact decode: a bf16 value is the upper half of an IEEE binary32. */
double orc_bf16_to_double(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Round a double to the nearest bf16, ties to even, in one step (no detour
 * through binary32, which would round twice).  bf16 has the exponent range of
 * binary32 and 8 significant bits, so the spacing of representable values
 * near |v| is 2^(e-7) for 2^e <= |v| < 2^(e+1), e >= -126, and 2^-133 in the
 * subnormal range. */
uint16_t orc_double_to_bf16(double v)
{
    if (isnan(v))
        return (uint16_t)(signbit(v) ? 0xFFC0u : 0x7FC0u);
    int neg = signbit(v) ? 1 : 0;
    double a = fabs(v);
    if (isinf(a))
        return (uint16_t)(neg ? 0xFF80u : 0x7F80u);
    if (a == 0.0)
        return (uint16_t)(neg ? 0x8000u : 0x0000u);
    int e;
    (void)frexp(a, &e);          /* a = m * 2^e, 0.5 <= m < 1 */
    int lead = e - 1;            /* a in [2^lead, 2^(lead+1)) */
    if (lead < -126)
        lead = -126;             /* subnormal spacing */
    double q = ldexp(1.0, lead - 7);
    double t = a / q;            /* exact: scaling by a power of two */
    double fl = floor(t);
    double frac = t - fl;        /* exact for t < 2^53 */
    if (frac > 0.5 || (frac == 0.5 && fmod(fl, 2.0) != 0.0))
        fl += 1.0;
    double r = fl * q;
    if (r >= ldexp(1.0, 128))    /* beyond the largest finite bf16 */
        return (uint16_t)(neg ? 0xFF80u : 0x7F80u);
    float f = (float)r;          /* exact: r is a bf16 value */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    uint16_t bits = (uint16_t)(u >> 16);
    return (uint16_t)(bits | (neg ? 0x8000u : 0u));
}

/* Elementwise form of orc_double_to_bf16 over an array of m values. */
void orc_round_bf16_array(int64_t m, const double *v, uint16_t *out)
{
    for (int64_t i = 0; i < m; ++i)
        out[i] = orc_double_to_bf16(v[i]);
}

/* ---------------------------------------------------------- hc_mixes */

/* Mix projection ("Mix projection" page, formula for m; Block.hc_mixes):
 *   r_t        = 1 / sqrt( (1/F) * sum_f x_{t,f}^2 + norm_eps )
 *   mixes_{t,i} = ( sum_f x_{t,f} * W_{i,f} ) * r_t
 * x:     [n, hc, d] bf16 bits, feature f = j*d + c
 * w:     [mix_hc, F] binary32, F = hc*d, mix_hc = (2+hc)*hc
 * mixes: [n, mix_hc] double (out)
 * rms_inv: [n] double (out, may be NULL) -- r_t */
void orc_hc_mixes(int64_t n, int hc, int64_t d, double norm_eps,
                  const uint16_t *x, const float *w, double *mixes,
                  double *rms_inv)
{
    const int64_t F = (int64_t)hc * d;
    const int mix_hc = (2 + hc) * hc;
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < n; ++t) {
        const uint16_t *xt = x + t * F;
        double ss = 0.0;
        for (int64_t f = 0; f < F; ++f) {
            double v = orc_bf16_to_double(xt[f]);
            ss += v * v;
        }
        double r = 1.0 / sqrt(ss / (double)F + norm_eps);
        if (rms_inv)
            rms_inv[t] = r;
        for (int i = 0; i < mix_hc; ++i) {
            const float *wi = w + (int64_t)i * F;
            double acc = 0.0;
            for (int64_t f = 0; f < F; ++f)
                acc += orc_bf16_to_double(xt[f]) * (double)wi[f];
            mixes[t * mix_hc + i] = acc * r;
        }
    }
}

/* ------------------------------------------------ hc_split_sinkhorn */

static double sigmoid(double z) { return 1.0 / (1.0 + exp(-z)); }

/* Split of the mixes and Sinkhorn normalisation ("Reading weights" page,
 * pre formula and the hc_split_sinkhorn kernel).  Per token, with
 * s = hc_scale[0..2] and b = hc_base[0..mix_hc):
 *   pre_j  = sigmoid(m_j * s0 + b_j) + eps                     j < hc
 *   post_j = 2 * sigmoid(m_{hc+j} * s1 + b_{hc+j})              j < hc
 *   L_{j,k} = m_{2hc + j*hc + k} * s2 + b_{2hc + j*hc + k}      row j, column k
 *   C = softmax over k of L (max-subtracted, divided by the plain row sum), + eps
 *   C_{j,k} /= (sum_j' C_{j',k} + eps)                           column step
 *   repeat iters-1 times:
 *     C_{j,k} /= (sum_k' C_{j,k'} + eps)                         row step
 *     C_{j,k} /= (sum_j' C_{j',k} + eps)                         column step
 * mixes: [n, mix_hc] double; pre, post: [n, hc]; comb: [n, hc, hc] (row j,
 * column k, row-major).  iters >= 1.  hc <= 16. */
void orc_hc_split_sinkhorn(int64_t n, int hc, int iters, double eps,
                           const double *mixes, const float *hc_scale,
                           const float *hc_base, double *pre, double *post,
                           double *comb)
{
    const int mix_hc = (2 + hc) * hc;
    const double s0 = hc_scale[0], s1 = hc_scale[1], s2 = hc_scale[2];
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < n; ++t) {
        const double *m = mixes + t * mix_hc;
        double C[16][16];
        for (int j = 0; j < hc; ++j)
            pre[t * hc + j] = sigmoid(m[j] * s0 + (double)hc_base[j]) + eps;
        for (int j = 0; j < hc; ++j)
            post[t * hc + j] =
                2.0 * sigmoid(m[hc + j] * s1 + (double)hc_base[hc + j]);
        for (int j = 0; j < hc; ++j)
            for (int k = 0; k < hc; ++k)
                C[j][k] = m[2 * hc + j * hc + k] * s2 +
                          (double)hc_base[2 * hc + j * hc + k];

        /* row softmax, then + eps (no eps in this denominator) */
        for (int j = 0; j < hc; ++j) {
            double mx = C[j][0];
            for (int k = 1; k < hc; ++k)
                if (C[j][k] > mx)
                    mx = C[j][k];
            double s = 0.0;
            for (int k = 0; k < hc; ++k) {
                C[j][k] = exp(C[j][k] - mx);
                s += C[j][k];
            }
            for (int k = 0; k < hc; ++k)
                C[j][k] = C[j][k] / s + eps;
        }
        /* column step */
        for (int k = 0; k < hc; ++k) {
            double s = 0.0;
            for (int j = 0; j < hc; ++j)
                s += C[j][k];
            for (int j = 0; j < hc; ++j)
                C[j][k] = C[j][k] / (s + eps);
        }
        for (int it = 1; it < iters; ++it) {
            /* row step */
            for (int j = 0; j < hc; ++j) {
                double s = 0.0;
                for (int k = 0; k < hc; ++k)
                    s += C[j][k];
                for (int k = 0; k < hc; ++k)
                    C[j][k] = C[j][k] / (s + eps);
            }
            /* column step */
            for (int k = 0; k < hc; ++k) {
                double s = 0.0;
                for (int j = 0; j < hc; ++j)
                    s += C[j][k];
                for (int j = 0; j < hc; ++j)
                    C[j][k] = C[j][k] / (s + eps);
            }
        }
        for (int j = 0; j < hc; ++j)
            for (int k = 0; k < hc; ++k)
                comb[(t * hc + j) * hc + k] = C[j][k];
    }
}

/* ------------------------------------------------------------ hc_pre */

/* Collapse of the copies ("Mix projection" page, Block.hc_pre):
 *   y_{t,c} = sum_j pre_{t,j} * x_{t,j,c}, stored in bf16.
 * x: [n, hc, d] bf16 bits; pre: [n, hc] double;
 * y: [n, d] double (out, may be NULL); y_bf16: [n, d] bits (out, may be NULL);
 * mag: [n, d] double (out, may be NULL) -- sum_j |pre_j * x_{j,c}|, the scale
 *      of the terms, used by tests to bound the binary32 evaluation error. */
void orc_hc_pre(int64_t n, int hc, int64_t d, const uint16_t *x,
                const double *pre, double *y, uint16_t *y_bf16, double *mag)
{
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < n; ++t) {
        for (int64_t c = 0; c < d; ++c) {
            double acc = 0.0, am = 0.0;
            for (int j = 0; j < hc; ++j) {
                double term =
                    pre[t * hc + j] * orc_bf16_to_double(x[(t * hc + j) * d + c]);
                acc += term;
                am += fabs(term);
            }
            if (y)
                y[t * d + c] = acc;
            if (y_bf16)
                y_bf16[t * d + c] = orc_double_to_bf16(acc);
            if (mag)
                mag[t * d + c] = am;
        }
    }
}

/* ----------------------------------------------------------- hc_post */

/* Expansion back to hc copies ("Mix projection" page, Block.hc_post):
 *   y_{t,k,c} = post_{t,k} * out_{t,c} + sum_j comb_{t,j,k} * res_{t,j,c}
 * The sum runs over the FIRST comb index j (comb.unsqueeze(-1) times
 * residual.unsqueeze(-2), summed over the copy axis of the residual).
 * out: [n, d] bf16 bits; res: [n, hc, d] bf16 bits; post: [n, hc] double;
 * comb: [n, hc, hc] double; y: [n, hc, d] double (may be NULL);
 * y_bf16: [n, hc, d] bits (may be NULL); mag: [n, hc, d] (may be NULL). */
/*
 * RMSNorm of the collapsed sublayer input (the block's attn_norm / ffn_norm
 * applied to hc_pre's output).  Its body is not on the pages; the plain
 * standard form is taken: with y the bf16 collapse output decoded exactly,
 *   out_c = y_c * g_c / sqrt(mean_c(y_c^2) + eps),
 * rounded once to bf16 (nearest-even).  out (double) and out_bf16 may be NULL.
 */
void orc_hc_rmsnorm(int64_t n, int64_t d, const uint16_t *y, const float *g, double eps,
                    double *out, uint16_t *out_bf16)
{
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < n; ++t) {
        double ss = 0.0;
        for (int64_t c = 0; c < d; ++c) {
            const double v = orc_bf16_to_double(y[t * d + c]);
            ss += v * v;
        }
        const double inv = 1.0 / sqrt(ss / (double)d + eps);
        for (int64_t c = 0; c < d; ++c) {
            const double v = orc_bf16_to_double(y[t * d + c]) * (double)g[c] * inv;
            if (out)
                out[t * d + c] = v;
            if (out_bf16)
                out_bf16[t * d + c] = orc_double_to_bf16(v);
        }
    }
}

void orc_hc_post(int64_t n, int hc, int64_t d, const uint16_t *out,
                 const uint16_t *res, const double *post, const double *comb,
                 double *y, uint16_t *y_bf16, double *mag)
{
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < n; ++t) {
        for (int k = 0; k < hc; ++k) {
            for (int64_t c = 0; c < d; ++c) {
                double term0 = post[t * hc + k] * orc_bf16_to_double(out[t * d + c]);
                double acc = term0, am = fabs(term0);
                for (int j = 0; j < hc; ++j) {
                    double term = comb[(t * hc + j) * hc + k] *
                                  orc_bf16_to_double(res[(t * hc + j) * d + c]);
                    acc += term;
                    am += fabs(term);
                }
                int64_t o = (t * hc + k) * d + c;
                if (y)
                    y[o] = acc;
                if (y_bf16)
                    y_bf16[o] = orc_double_to_bf16(acc);
                if (mag)
                    mag[o] = am;
            }
        }
    }
}

/* Threads the OpenMP loops above use (1 without OpenMP). */
int orc_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void orc_set_num_threads(int k)
{
#ifdef _OPENMP
    if (k > 0)
        omp_set_num_threads(k);
#else
    (void)k;
#endif
}
