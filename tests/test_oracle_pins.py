"""Pins for the float64 oracle: checks against facts that do not come from the
oracle itself -- closed forms, invariants, special cases that reduce to a
library routine, and an independent formulation of the 2x2 Sinkhorn iteration.

Each group names the statement on the "DeepSeek V4.1" pages that it pins and
the plausible mistakes it would catch.
"""
import json
import math
import os

import numpy as np
import pytest
import scipy.optimize
import scipy.special
import torch

import oracle
from sinkhorn_mixing_gb300 import inputs

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
EPS = 1e-6


def rng(seed):
    return np.random.default_rng(seed)


def bf16_of(a):
    """bf16 bit patterns of float values (torch's RNE cast from float32)."""
    t = torch.tensor(np.asarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


# ------------------------------------------------------------- bf16 rounding

def test_bf16_decode_roundtrip_all_patterns():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    vals = oracle.bf16_bits_to_f64(bits)
    finite = ~np.isnan(vals)
    back = oracle.f64_to_bf16_bits(vals[finite])
    assert np.array_equal(back, bits[finite])


def test_bf16_round_matches_torch_on_binary32_values():
    # For values that are exactly binary32, one rounding to bf16 is what
    # torch's float32 -> bfloat16 cast does (round to nearest even).
    r = rng(1)
    mags = np.concatenate([
        r.standard_normal(20000),
        r.standard_normal(5000) * 1e-38,      # subnormal range
        r.standard_normal(5000) * 1e30,
        (1 + r.integers(0, 1 << 16, 5000) * 2.0 ** -16),  # many exact ties
    ]).astype(np.float32)
    ours = oracle.f64_to_bf16_bits(mags.astype(np.float64))
    assert np.array_equal(ours, bf16_of(mags))


def test_bf16_round_ties_overflow_and_no_double_rounding():
    f = oracle.f64_to_bf16_bits
    one = 0x3F80
    assert f([1.0 + 2.0 ** -8])[0] == one            # tie -> even (down)
    assert f([1.0 + 3 * 2.0 ** -8])[0] == one + 2    # tie -> even (up)
    # just above a tie: a detour through binary32 would land on the tie and
    # round down; one rounding from double must round up.
    assert f([1.0 + 2.0 ** -8 + 2.0 ** -40])[0] == one + 1
    assert f([-(1.0 + 2.0 ** -8 + 2.0 ** -40)])[0] == 0x8000 | (one + 1)
    big = (2 - 2.0 ** -7) * 2.0 ** 127                 # largest finite bf16
    assert f([big])[0] == 0x7F7F
    assert f([big + 2.0 ** 119])[0] == 0x7F80          # halfway -> even = inf
    assert f([2.0 ** -133])[0] == 0x0001               # smallest subnormal
    assert f([2.0 ** -134])[0] == 0x0000               # tie -> even (zero)
    assert f([3 * 2.0 ** -135])[0] == 0x0001
    assert f([-0.0])[0] == 0x8000


# ----------------------------------------------------------------- hc_mixes
# Mix projection page: m = x^f W^T / sqrt(mean((x^f)^2) + eps), x^f = x.flatten(2).

@pytest.mark.parametrize("a,norm_eps", [(0.75, 1e-20), (-1.5, 1e-20), (0.5, 0.75)])
def test_mixes_constant_stream_closed_form(a, norm_eps):
    # x_f = a for every f: mean(x^2) = a^2, so m_i = a * sum_f W_if / sqrt(a^2 + eps).
    # With a = 0.5, eps = 0.75 the root is exactly 1.  Catches: sum instead of
    # mean, eps outside the root, a missing root, a wrong W axis.
    hc, d, n = 4, 16, 2
    F = hc * d
    w = rng(2).standard_normal((24, F)).astype(np.float32)
    x = np.full((n, hc, d), bf16_of([a])[0], dtype=np.uint16)
    m = oracle.hc_mixes(x, w, norm_eps)
    want = a * w.astype(np.float64).sum(axis=1) / math.sqrt(a * a + norm_eps)
    np.testing.assert_allclose(m, np.broadcast_to(want, m.shape), rtol=1e-13,
                               atol=1e-13)


def test_mixes_one_hot_rows_pin_feature_layout():
    # Entries +-1/2 give mean(x^2) = 1/4 and r = 2 exactly.  W row i one-hot
    # at f_i = j_i * d + c_i must return 2 * x[t, j_i, c_i]: pins f = j*d + c
    # (flatten of [hc, d]) and the row order of W.
    hc, d, n = 4, 8, 3
    r = rng(3)
    signs = r.choice([-0.5, 0.5], size=(n, hc, d))
    x = bf16_of(signs).reshape(n, hc, d)
    js = r.integers(0, hc, 24)
    cs = r.integers(0, d, 24)
    w = np.zeros((24, hc * d), dtype=np.float32)
    w[np.arange(24), js * d + cs] = 1.0
    m = oracle.hc_mixes(x, w, 1e-20)
    assert np.array_equal(m, 2.0 * signs[:, js, cs])


@pytest.mark.parametrize("k", [-3, 5])
def test_mixes_invariant_to_power_of_two_scaling(k):
    hc, d, n = 4, 32, 4
    r = rng(4)
    xf = r.standard_normal((n, hc, d)).astype(np.float32)
    x1 = bf16_of(xf)
    x2 = bf16_of(oracle.bf16_bits_to_f64(x1) * 2.0 ** k)   # exact rescale
    w = (r.standard_normal((24, hc * d)) / math.sqrt(hc * d)).astype(np.float32)
    np.testing.assert_allclose(oracle.hc_mixes(x2, w), oracle.hc_mixes(x1, w),
                               rtol=1e-12, atol=1e-14)


def test_mixes_zero_token():
    x = np.zeros((2, 4, 8), dtype=np.uint16)
    w = rng(5).standard_normal((24, 32)).astype(np.float32)
    m, rinv = oracle.hc_mixes(x, w, 1e-20, return_rms_inv=True)
    assert np.all(m == 0.0)
    np.testing.assert_allclose(rinv, 1e10, rtol=1e-15)


def test_mixes_match_library_matmul_and_norm():
    hc, d, n = 8, 24, 5
    r = rng(6)
    x = bf16_of(r.standard_normal((n, hc, d)) * 3).reshape(n, hc, d)
    X = oracle.bf16_bits_to_f64(x).reshape(n, hc * d)
    w = r.standard_normal(((2 + hc) * hc, hc * d)).astype(np.float32)
    want = (X @ w.astype(np.float64).T) * (math.sqrt(hc * d) /
                                           np.linalg.norm(X, axis=1))[:, None]
    np.testing.assert_allclose(oracle.hc_mixes(x, w, 0.0), want, rtol=1e-12,
                               atol=1e-12)


# ------------------------------------------------------- hc_split_sinkhorn
# Reading weights page: pre/post sigmoids and the Sinkhorn normalisation.

def _split_inputs(hc, n, seed, base_std=1.0, s=(0.7, 1.3, 2.9), mix_std=1.0):
    r = rng(seed)
    mix_hc = (2 + hc) * hc
    mixes = r.standard_normal((n, mix_hc)) * mix_std
    base = (r.standard_normal(mix_hc) * base_std).astype(np.float32)
    scale = np.array(s, dtype=np.float32)
    return mixes, scale, base


def _logits(mixes, scale, base, hc):
    return (mixes[:, 2 * hc:] * np.float64(scale[2]) +
            base[2 * hc:].astype(np.float64)).reshape(-1, hc, hc)


def test_pre_post_closed_form_and_scale_indices():
    # pre uses hc_scale[0] and base[0:hc]; post uses hc_scale[1], base[hc:2hc]
    # and a factor 2; eps is added to pre only.  Distinct scales catch a
    # swapped index.
    hc, n = 4, 64
    mixes, scale, base = _split_inputs(hc, n, 7)
    pre, post, _ = oracle.hc_split_sinkhorn(mixes, scale, base, hc, 20, EPS)
    b = base.astype(np.float64)
    want_pre = scipy.special.expit(mixes[:, :hc] * np.float64(scale[0]) + b[:hc]) + EPS
    want_post = 2 * scipy.special.expit(mixes[:, hc:2 * hc] * np.float64(scale[1]) +
                                        b[hc:2 * hc])
    np.testing.assert_allclose(pre, want_pre, rtol=1e-14, atol=1e-16)
    np.testing.assert_allclose(post, want_post, rtol=1e-14, atol=1e-16)


@pytest.mark.parametrize("hc", [4, 8])
def test_coefficient_ranges(hc):
    mixes, scale, base = _split_inputs(hc, 256, 8, base_std=2.0)
    pre, post, comb = oracle.hc_split_sinkhorn(mixes, scale, base, hc, 20, EPS)
    assert np.all(pre > EPS) and np.all(pre < 1 + EPS)
    assert np.all(post > 0) and np.all(post < 2)
    assert np.all(comb > 0)


@pytest.mark.parametrize("hc", [2, 4, 8])
def test_one_iteration_is_row_softmax_plus_eps_then_column_step(hc):
    # iters = 1: softmax over the LAST index (row j, column k), + eps with no
    # eps in the softmax denominator, then one column step with (sum + eps).
    mixes, scale, base = _split_inputs(hc, 32, 9, base_std=2.0)
    _, _, comb = oracle.hc_split_sinkhorn(mixes, scale, base, hc, 1, EPS)
    A = scipy.special.softmax(_logits(mixes, scale, base, hc), axis=-1) + EPS
    want = A / (A.sum(axis=-2, keepdims=True) + EPS)
    np.testing.assert_allclose(comb, want, rtol=1e-13, atol=1e-18)


def _cross_ratios(C):
    hc = C.shape[-1]
    out = []
    for j in range(hc):
        for j2 in range(j + 1, hc):
            for k in range(hc):
                for k2 in range(k + 1, hc):
                    out.append(C[:, j, k] * C[:, j2, k2] /
                               (C[:, j, k2] * C[:, j2, k]))
    return np.stack(out, axis=1)


@pytest.mark.parametrize("iters", [1, 2, 7, 20, 50])
def test_sinkhorn_steps_are_diagonal_scalings(iters):
    # Every normalisation multiplies whole rows or columns by positive
    # factors, so all cross-ratios equal those of A = softmax(L) + eps.
    hc = 4
    mixes, scale, base = _split_inputs(hc, 64, 10, base_std=2.0)
    _, _, comb = oracle.hc_split_sinkhorn(mixes, scale, base, hc, iters, EPS)
    A = scipy.special.softmax(_logits(mixes, scale, base, hc), axis=-1) + EPS
    np.testing.assert_allclose(_cross_ratios(comb), _cross_ratios(A), rtol=1e-10)


@pytest.mark.parametrize("iters", [2, 20])
def test_last_step_is_a_column_step_with_eps(iters):
    # After the final column step, column sums are S/(S+eps) < 1 for the
    # previous column sums S; for moderate logits S is O(1).
    hc = 4
    mixes, scale, base = _split_inputs(hc, 128, 11, s=(1.0, 1.0, 0.5), base_std=0.5)
    _, _, comb = oracle.hc_split_sinkhorn(mixes, scale, base, hc, iters, EPS)
    cs = comb.sum(axis=-2)
    assert np.all(cs < 1.0) and np.all(cs > 1.0 - 4 * EPS)


def test_hc2_converges_to_closed_form_doubly_stochastic_limit():
    # For a positive 2x2 A = [[a, b], [c, d]] the doubly stochastic scaling is
    # [[t, 1-t], [1-t, t]], t = sqrt(ad) / (sqrt(ad) + sqrt(bc)).  With +eps in
    # every denominator the fixed point has all row and column sums equal to
    # 1 - eps, i.e. (1 - eps) times that matrix.
    hc = 2
    mixes, scale, base = _split_inputs(hc, 64, 12, base_std=1.0, s=(0.7, 1.3, 1.0))
    _, _, comb = oracle.hc_split_sinkhorn(mixes, scale, base, hc, 2000, EPS)
    A = scipy.special.softmax(_logits(mixes, scale, base, hc), axis=-1) + EPS
    a, b, c, d = A[:, 0, 0], A[:, 0, 1], A[:, 1, 0], A[:, 1, 1]
    t = np.sqrt(a * d) / (np.sqrt(a * d) + np.sqrt(b * c))
    want = (1 - EPS) * np.stack([np.stack([t, 1 - t], -1),
                                 np.stack([1 - t, t], -1)], -2)
    np.testing.assert_allclose(comb, want, rtol=0, atol=1e-12)


def _doubly_stochastic_scaling(A):
    """D1 A D2 with unit row and column sums, by root finding on the log
    scalings (scipy's hybrid Powell method) -- not by alternating scaling."""
    hc = A.shape[0]

    def resid(z):
        u, v = z[:hc], np.concatenate([z[hc:], [0.0]])
        M = np.exp(u)[:, None] * A * np.exp(v)[None, :]
        return np.concatenate([M.sum(1) - 1, (M.sum(0) - 1)[:-1]])

    sol = scipy.optimize.root(resid, np.zeros(2 * hc - 1), method="hybr",
                              options=dict(xtol=1e-14))
    assert np.max(np.abs(resid(sol.x))) < 1e-13
    u, v = sol.x[:hc], np.concatenate([sol.x[hc:], [0.0]])
    return np.exp(u)[:, None] * A * np.exp(v)[None, :]


def test_hc4_converges_to_scaled_doubly_stochastic_matrix():
    hc = 4
    mixes, scale, base = _split_inputs(hc, 16, 13, base_std=1.0, s=(1, 1, 1.0))
    _, _, comb = oracle.hc_split_sinkhorn(mixes, scale, base, hc, 3000, EPS)
    A = scipy.special.softmax(_logits(mixes, scale, base, hc), axis=-1) + EPS
    for i in range(len(A)):
        want = (1 - EPS) * _doubly_stochastic_scaling(A[i])
        np.testing.assert_allclose(comb[i], want, rtol=0, atol=1e-10)


@pytest.mark.parametrize("iters", [1, 2, 3, 20])
@pytest.mark.parametrize("eps", [0.0, EPS, 1e-2])
def test_uniform_logits_follow_scalar_recurrence(iters, eps):
    # Constant logits: A = 1/hc + eps everywhere and every normalisation maps
    # the common value c to c / (hc*c + eps); there are 2*iters - 1 of them.
    hc = 4
    mixes = np.zeros((3, 24))
    mixes[:, :8] = rng(14).standard_normal((3, 8))
    base = np.zeros(24, dtype=np.float32)
    base[8:] = 0.3
    _, _, comb = oracle.hc_split_sinkhorn(mixes, np.array([1, 1, 1.7], np.float32),
                                          base, hc, iters, eps)
    c = 1.0 / hc + eps
    for _ in range(2 * iters - 1):
        c = c / (hc * c + eps)
    np.testing.assert_allclose(comb, c, rtol=1e-14)


@pytest.mark.parametrize("iters", [1, 2, 3, 5, 12])
def test_hc2_matches_column_odds_recurrence(iters):
    # Independent formulation of the 2x2 iteration at eps = 0, in terms of the
    # column odds p = C00/C10, q = C01/C11.  A column step leaves the odds
    # unchanged; a row step multiplies both by r1/r0 (the ratio of row sums).
    # The logits are chosen so that the iteration is far from converged, so
    # the test fixes the number and the order of the steps.
    hc = 2
    L = np.array([[[5.0, 0.0], [1.0, 4.5]], [[0.3, 2.0], [3.0, -1.0]],
                  [[6.0, -2.0], [-3.0, 5.5]]])
    n = len(L)
    mixes = np.zeros((n, 8))
    mixes[:, 4:] = L.reshape(n, 4)
    _, _, comb = oracle.hc_split_sinkhorn(mixes, np.ones(3, np.float32),
                                          np.zeros(8, np.float32), hc, iters, 0.0)
    A = scipy.special.softmax(L, axis=-1)
    p = A[:, 0, 0] / A[:, 1, 0]
    q = A[:, 0, 1] / A[:, 1, 1]
    for _ in range(iters - 1):
        x, y = p / (1 + p), q / (1 + q)
        ratio = (2 - x - y) / (x + y)
        p, q = p * ratio, q * ratio
    x, y = p / (1 + p), q / (1 + q)
    want = np.stack([np.stack([x, y], -1), np.stack([1 - x, 1 - y], -1)], -2)
    np.testing.assert_allclose(comb, want, rtol=1e-12, atol=1e-15)
    if iters >= 3:
        # far from converged: row sums still visibly off 1
        assert np.max(np.abs(comb.sum(-1) - 1)) > 1e-3


def test_row_sum_deviation_shrinks_with_iterations_on_extreme_logits():
    # Sinkhorn-Knopp row sums converge, but slowly at logit spreads of about
    # +-40 (hc = 8, base variance 5, scale U(2, 8)); the aggregate deviation
    # must not grow from 1 to 20 to 50 iterations.
    wl = inputs.WORKLOADS["stress"]
    hc = wl.hc
    p = inputs.make_params(wl)
    mixes = rng(15).standard_normal((2000, wl.mix_hc))
    dev = []
    for it in (1, 20, 50):
        _, _, comb = oracle.hc_split_sinkhorn(mixes, p["hc_scale"].numpy(),
                                              p["hc_base"].numpy(), hc, it, EPS)
        dev.append(np.mean(np.abs(comb.sum(-1) - 1)))
        assert np.max(np.abs(comb.sum(-2) - 1)) < (1e-3 if it >= 2 else 1.0)
    assert dev[0] >= dev[1] >= dev[2]


def test_moderate_logits_reach_unit_row_and_column_sums_in_20_iterations():
    hc = 4
    mixes, scale, base = _split_inputs(hc, 512, 16, s=(1, 1, 0.5), base_std=0.5)
    _, _, comb = oracle.hc_split_sinkhorn(mixes, scale, base, hc, 20, EPS)
    assert np.max(np.abs(comb.sum(-1) - 1)) < 1e-3
    assert np.max(np.abs(comb.sum(-2) - 1)) < 1e-3


def test_zero_token_coefficients_depend_on_base_only():
    hc, d = 4, 16
    x = np.zeros((2, hc, d), dtype=np.uint16)
    w = rng(17).standard_normal((24, hc * d)).astype(np.float32)
    base = rng(18).standard_normal(24).astype(np.float32)
    base[8:] = -0.7
    scale = np.array([1.1, 0.9, 3.0], np.float32)
    pre, post, comb = oracle.hc_split_sinkhorn(oracle.hc_mixes(x, w), scale, base,
                                               hc, 20, EPS)
    b = base.astype(np.float64)
    np.testing.assert_allclose(pre, np.broadcast_to(scipy.special.expit(b[:4]) + EPS,
                                                    pre.shape), rtol=1e-15)
    np.testing.assert_allclose(post, np.broadcast_to(2 * scipy.special.expit(b[4:8]),
                                                     post.shape), rtol=1e-15)
    c = 1.0 / hc + EPS
    for _ in range(39):
        c = c / (hc * c + EPS)
    np.testing.assert_allclose(comb, c, rtol=1e-14)


# ------------------------------------------------------------------ hc_pre
# Mix projection page, Block.hc_pre: y = sum_j pre_j * x_j, cast to bf16.

def _stream(n, hc, d, seed, scale=1.0):
    return bf16_of(rng(seed).standard_normal((n, hc, d)) * scale).reshape(n, hc, d)


def test_pre_equal_weights_is_mean_of_copies():
    n, hc, d = 4, 4, 32
    x = _stream(n, hc, d, 19)
    y, yb, _ = oracle.hc_pre(x, np.full((n, hc), 0.25))
    X = oracle.bf16_bits_to_f64(x)
    assert np.array_equal(y, X.mean(axis=1))
    y3, _, _ = oracle.hc_pre(x, np.full((n, hc), 0.3))
    np.testing.assert_allclose(y3, 0.3 * hc * X.mean(axis=1), rtol=1e-14, atol=1e-15)
    assert np.array_equal(yb, oracle.f64_to_bf16_bits(X.mean(axis=1)))


def test_pre_one_hot_weights_select_a_copy():
    n, hc, d = 3, 4, 16
    x = _stream(n, hc, d, 20)
    for j in range(hc):
        p = np.zeros((n, hc))
        p[:, j] = 1.0
        _, yb, _ = oracle.hc_pre(x, p)
        assert np.array_equal(yb, x[:, j, :])


def test_pre_matches_einsum():
    n, hc, d = 5, 8, 24
    x = _stream(n, hc, d, 21)
    p = rng(22).uniform(0, 1, (n, hc))
    y, _, mag = oracle.hc_pre(x, p)
    X = oracle.bf16_bits_to_f64(x)
    np.testing.assert_allclose(y, np.einsum("tj,tjc->tc", p, X), rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(mag, np.einsum("tj,tjc->tc", p, np.abs(X)), rtol=1e-13)


# ----------------------------------------------------------------- hc_post
# Mix projection page, Block.hc_post: y_k = post_k * out + sum_j comb[j, k] * r_j.

def test_post_identity_comb_returns_residual():
    n, hc, d = 3, 4, 16
    res = _stream(n, hc, d, 23)
    out = _stream(n, 1, d, 24).reshape(n, d)
    _, yb, _ = oracle.hc_post(out, res, np.zeros((n, hc)),
                              np.broadcast_to(np.eye(hc), (n, hc, hc)))
    assert np.array_equal(yb, res)


@pytest.mark.parametrize("hc", [4, 8])
def test_post_permutation_comb_pins_the_summed_index(hc):
    # comb[j, (j+1) % hc] = 1: the sum over the first index gives
    # y_k = r_{k-1}; summing over the second index would give r_{k+1}.
    n, d = 2, 8
    res = _stream(n, hc, d, 25)
    out = _stream(n, 1, d, 26).reshape(n, d)
    P = np.zeros((hc, hc))
    P[np.arange(hc), (np.arange(hc) + 1) % hc] = 1.0
    _, yb, _ = oracle.hc_post(out, res, np.zeros((n, hc)), np.broadcast_to(P, (n, hc, hc)))
    assert np.array_equal(yb, res[:, (np.arange(hc) - 1) % hc, :])


def test_post_zero_comb_scales_output():
    n, hc, d = 2, 4, 16
    res = _stream(n, hc, d, 27)
    out = _stream(n, 1, d, 28).reshape(n, d)
    post = np.array([[0.5, 1.0, 2.0, 0.25], [1.0, 0.125, 4.0, 1.0]])
    _, yb, _ = oracle.hc_post(out, res, post, np.zeros((n, hc, hc)))
    want = bf16_of(oracle.bf16_bits_to_f64(out)[:, None, :] * post[:, :, None])
    assert np.array_equal(yb, want.reshape(n, hc, d))


def test_post_matches_einsum():
    n, hc, d = 4, 4, 24
    res = _stream(n, hc, d, 29)
    out = _stream(n, 1, d, 30).reshape(n, d)
    post = rng(31).uniform(0, 2, (n, hc))
    comb = rng(32).uniform(0, 1, (n, hc, hc))
    y, _, _ = oracle.hc_post(out, res, post, comb)
    R = oracle.bf16_bits_to_f64(res)
    O = oracle.bf16_bits_to_f64(out)
    want = post[:, :, None] * O[:, None, :] + np.einsum("tjk,tjc->tkc", comb, R)
    np.testing.assert_allclose(y, want, rtol=1e-13, atol=1e-14)


# ------------------------------------------------------------ whole chain

def _fp32_restatement(x, w, scale, base, out, res, hc, iters, eps, norm_eps):
    """The pages' PyTorch statements in float32 on the CPU (torch ops), with the
    Sinkhorn steps as the kernel's comments state them."""
    xf = x.flatten(1).float()
    rs = torch.rsqrt(xf.square().mean(-1, keepdim=True) + norm_eps)
    mixes = torch.nn.functional.linear(xf, w) * rs
    pre = torch.sigmoid(mixes[:, :hc] * scale[0] + base[:hc]) + eps
    post = 2 * torch.sigmoid(mixes[:, hc:2 * hc] * scale[1] + base[hc:2 * hc])
    comb = (mixes[:, 2 * hc:] * scale[2] + base[2 * hc:]).view(-1, hc, hc)
    comb = comb.softmax(-1) + eps
    comb = comb / (comb.sum(-2, keepdim=True) + eps)
    for _ in range(iters - 1):
        comb = comb / (comb.sum(-1, keepdim=True) + eps)
        comb = comb / (comb.sum(-2, keepdim=True) + eps)
    y_pre = torch.sum(pre.unsqueeze(-1) * x.float(), dim=1).to(x.dtype)
    y_post = (post.unsqueeze(-1) * out.unsqueeze(-2) +
              torch.sum(comb.unsqueeze(-1) * res.unsqueeze(-2), dim=1)).type_as(out)
    return mixes, pre, post, comb, y_pre, y_post


def test_chain_fp32_restatement_agrees_with_oracle_on_tiny_workload():
    wl = inputs.WORKLOADS["tiny"]
    s = inputs.make_streams(wl)
    p = inputs.make_params(wl)
    ref = oracle.chain(inputs.bf16_bits(s["x"]), p["w"].numpy(), p["hc_scale"].numpy(),
                       p["hc_base"].numpy(), inputs.bf16_bits(s["out"]),
                       inputs.bf16_bits(s["residual"]), 20, wl.eps, wl.norm_eps)
    m, pre, post, comb, y_pre, y_post = _fp32_restatement(
        s["x"], p["w"], p["hc_scale"], p["hc_base"], s["out"], s["residual"],
        wl.hc, 20, wl.eps, wl.norm_eps)
    np.testing.assert_allclose(m.numpy(), ref["mixes"], rtol=1e-5, atol=1e-5)
    np.testing.assert_allclose(pre.numpy(), ref["pre"], atol=1e-5)
    np.testing.assert_allclose(post.numpy(), ref["post"], atol=1e-5)
    np.testing.assert_allclose(comb.numpy(), ref["comb"], atol=1e-5)
    for got, want in ((y_pre, ref["y_pre"]), (y_post, ref["y_post"])):
        g = got.float().numpy().astype(np.float64)
        np.testing.assert_allclose(g, want, rtol=2 ** -7, atol=1e-3)


# -------------------------------------------------------- printed constants

def test_printed_constants_and_parameter_counts():
    with open(os.path.join(GOLDEN, "constants.json")) as f:
        k = {key: v["value"] for key, v in json.load(f).items() if key[0] != "_"}
    wl = inputs.WORKLOADS["decode"]
    assert (wl.hc, wl.d, wl.iters[0], wl.eps, wl.norm_eps) == (
        k["hc_mult"], k["dim"], k["hc_sinkhorn_iters"], k["hc_eps"], k["norm_eps"])
    assert wl.mix_hc == k["mix_hc"] and wl.F == k["flat_features"]
    assert inputs.make_params(wl)["w"].numel() == k["w_mix_params"]
    assert wl.hc + 1 == k["pre_params_per_instance"]  # hc offsets + one scale


# ---------------------------------------------------- RMSNorm of the collapse
# The block normalises hc_pre's output before the sublayer (attn_norm /
# ffn_norm); the pages name it but do not show it, so the oracle takes the
# standard form out = y * g / sqrt(mean(y^2) + eps).  These pins would catch a
# sum in place of the mean, a missing square root, a dropped weight or eps,
# or a normalisation over the wrong axis.

def test_rmsnorm_constant_row_with_unit_weight_is_its_sign():
    y = bf16_of(np.array([[3.0] * 16, [-0.25] * 16]))
    out, bits = oracle.hc_rmsnorm(y, np.ones(16, np.float32))
    assert np.all(bits[0] == bf16_of([1.0])[0]) and np.all(bits[1] == bf16_of([-1.0])[0])
    np.testing.assert_allclose(out, [[1.0] * 16, [-1.0] * 16], rtol=1e-15)


def test_rmsnorm_unit_weight_output_has_unit_mean_square():
    y = bf16_of(rng(61).normal(0, 3, (5, 384)))
    out, _ = oracle.hc_rmsnorm(y, np.ones(384, np.float32))
    np.testing.assert_allclose((out ** 2).mean(axis=1), 1.0, rtol=1e-12)


def test_rmsnorm_power_of_two_scaling_invariance():
    # mean of squares scales by 4^k, so the output is unchanged (eps 1e-20 is
    # far below binary64 resolution here)
    v = rng(62).normal(0, 1, (3, 256))
    g = rng(63).uniform(0.5, 2.0, 256).astype(np.float32)
    a = oracle.hc_rmsnorm(bf16_of(v), g)[1]
    b = oracle.hc_rmsnorm(bf16_of(v * 8.0), g)[1]
    c = oracle.hc_rmsnorm(bf16_of(v / 64.0), g)[1]
    assert np.array_equal(a, b) and np.array_equal(a, c)


def test_rmsnorm_is_linear_in_the_weight_and_per_channel():
    v = bf16_of(rng(64).normal(0, 1, (2, 128)))
    g = rng(65).uniform(0.5, 2.0, 128).astype(np.float32)
    base, _ = oracle.hc_rmsnorm(v, g)
    twice, _ = oracle.hc_rmsnorm(v, (2.0 * g).astype(np.float32))
    np.testing.assert_array_equal(twice, 2.0 * base)
    # a weight of zero on one channel zeroes exactly that channel
    g0 = g.copy()
    g0[17] = 0.0
    z, _ = oracle.hc_rmsnorm(v, g0)
    assert np.all(z[:, 17] == 0.0)
    np.testing.assert_array_equal(np.delete(z, 17, axis=1), np.delete(base, 17, axis=1))


def test_rmsnorm_normalises_each_token_separately():
    v = rng(66).normal(0, 1, (2, 64))
    both, _ = oracle.hc_rmsnorm(bf16_of(np.stack([v[0], 1000 * v[1]])), np.ones(64, np.float32))
    one, _ = oracle.hc_rmsnorm(bf16_of(v[:1]), np.ones(64, np.float32))
    np.testing.assert_array_equal(both[0], one[0])


def test_rmsnorm_zero_row_and_eps():
    z = np.zeros((1, 32), np.uint16)
    out, bits = oracle.hc_rmsnorm(z, np.ones(32, np.float32))
    assert np.all(out == 0.0) and np.all(bits == 0)
    # a tiny row meets eps: y = 2^-60 everywhere, eps = 2^-100 * 3 ->
    # out = 2^-60 / sqrt(2^-120 + 3 * 2^-100) = 2^-60 / (2^-50 sqrt(3 + 2^-20))
    y = bf16_of(np.full((1, 32), 2.0 ** -60))
    out, _ = oracle.hc_rmsnorm(y, np.ones(32, np.float32), eps=3 * 2.0 ** -100)
    np.testing.assert_allclose(out, 2.0 ** -10 / math.sqrt(3 + 2.0 ** -20), rtol=1e-14)
