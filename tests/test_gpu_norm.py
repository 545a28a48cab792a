"""hc_mixes_pre_norm: hc_mixes_pre whose collapsed output is also passed
through the RMSNorm of the sublayer input.  Checked against the oracle stage
by stage: the coefficients as for hc_mixes_pre, the normalised rows against
the oracle's RMSNorm of the same call's collapse (one rounding apart) and of
the oracle's own collapse."""
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import compare
from sinkhorn_mixing_gb300 import inputs
from parity import bits, check_mixes_all, check_norm_all, check_split_all, oracle_mixes

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def hc():
    from sinkhorn_mixing_gb300 import build
    build.build()
    import sinkhorn_mixing_gb300 as m
    m.hc_device_error(clear=True)
    yield m
    torch.cuda.synchronize()
    assert m.hc_device_error(clear=True) == 0


def np64(t):
    return t.detach().cpu().double().numpy()


def case(n, H, d, seed, scale_lo=0.1, scale_hi=10.0):
    g = torch.Generator(device="cuda").manual_seed(seed)
    x = torch.randn((n, H, d), device="cuda", generator=g)
    s = torch.exp(torch.empty((n, 1, 1), device="cuda").uniform_(
        np.log(scale_lo), np.log(scale_hi), generator=g))
    x = (x * s).to(torch.bfloat16)
    mix = (2 + H) * H
    w = torch.randn((mix, H * d), device="cuda", generator=g) / (H * d) ** 0.5
    sc = torch.rand(3, device="cuda", generator=g) * 1.5 + 0.5
    base = torch.randn(mix, device="cuda", generator=g)
    rw = torch.rand(d, device="cuda", generator=g) * 1.5 + 0.25
    return x, w, sc, base, rw


def key_diff(a_bits, b_bits):
    return np.abs(compare.bf16_key(a_bits) - compare.bf16_key(b_bits))


@pytest.mark.parametrize("n,H,d", [(5, 4, 64), (64, 4, 5120), (37, 4, 2304), (300, 8, 1024),
                                   (1000, 4, 5120), (129, 4, 1024), (200, 4, 2048),
                                   (500, 4, 3072), (333, 4, 4096)])
def test_norm_matches_oracle(hc, n, H, d):
    x, w, sc, base, rw = case(n, H, d, 3 * n + d + H)
    y, pre, post, comb, m = hc.hc_mixes_pre_norm(x, w, sc, base, rw, 20, want_mixes=True)
    torch.cuda.synchronize()
    xb = inputs.bf16_bits(x)
    compare.check_mixes(np64(m), oracle.hc_mixes(xb, w.cpu().numpy()))
    o_pre, o_post, o_comb = oracle.hc_split_sinkhorn(np64(m), sc.cpu().numpy(),
                                                     base.cpu().numpy(), H, 20, 1e-6)
    compare.check_abs(np64(pre), o_pre, 1e-5, "pre")
    compare.check_abs(np64(post), o_post, 1e-5, "post")
    compare.check_abs(np64(comb), o_comb, 1e-5, "comb")
    # the oracle's collapse with the GPU's pre, normalised by the oracle; the
    # GPU's collapse may differ from it by one bf16 step or, where the H
    # terms cancel, by H binary32 roundings of their magnitude (as in the
    # collapse's own check), and the norm factor scales that difference
    _, yc_bits, mag = oracle.hc_pre(xb, np64(pre))
    g = rw.cpu().numpy().astype(np.float64)
    out_want, want_bits = oracle.hc_rmsnorm(yc_bits, rw.cpu().numpy())
    yc = oracle.bf16_bits_to_f64(yc_bits)
    inv = 1.0 / np.sqrt((yc ** 2).mean(axis=1, keepdims=True) + 1e-20)
    got = oracle.bf16_bits_to_f64(inputs.bf16_bits(y))
    allowed = (np.abs(g) * inv * (compare.bf16_ulp(yc) + H * 2.0 ** -24 * mag) +
               compare.bf16_ulp(out_want) + 1e-5 * np.abs(out_want))
    err = np.abs(got - out_want)
    assert np.all(err <= allowed), float((err / allowed).max())
    # away from cancellation the rows agree to the bf16 step
    assert np.mean(key_diff(inputs.bf16_bits(y), want_bits) <= 1) > 0.999


@pytest.mark.parametrize("path", ["general", "auto"])
@pytest.mark.parametrize("n,H,d", [(64, 4, 5120), (300, 8, 1024), (1000, 4, 5120)])
def test_norm_is_rmsnorm_of_the_same_collapse(hc, n, H, d, path):
    # the same path without the norm gives the collapse the norm was applied
    # to; normalising it in float64 must land within one bf16 step
    x, w, sc, base, rw = case(n, H, d, 17 + H)
    old = os.environ.get("HCMIX_PATH")
    os.environ["HCMIX_PATH"] = path
    try:
        y = hc.hc_mixes_pre_norm(x, w, sc, base, rw)[0]
        yc = hc.hc_mixes_pre(x, w, sc, base)[0]
        torch.cuda.synchronize()
    finally:
        if old is None:
            os.environ.pop("HCMIX_PATH", None)
        else:
            os.environ["HCMIX_PATH"] = old
    _, want = oracle.hc_rmsnorm(inputs.bf16_bits(yc), rw.cpu().numpy())
    assert key_diff(inputs.bf16_bits(y), want).max() <= 1


def test_norm_workspace_and_errors(hc):
    n, H, d = 40, 4, 1024
    x, w, sc, base, rw = case(n, H, d, 5)
    a = hc.hc_mixes_pre_norm(x, w, sc, base, rw, want_mixes=True)
    b = hc.hc_mixes_pre_norm(x, w, sc, base, rw)   # workspace path, no mixes output
    torch.cuda.synchronize()
    for u, v in zip(a[:4], b[:4]):
        assert torch.equal(u, v)
    before = hc.hc_launch_count()
    with pytest.raises(ValueError):
        hc.hc_mixes_pre_norm(x, w, sc, base, rw[:-8])
    assert hc.hc_launch_count() == before


def test_norm_deterministic_and_guarded(hc):
    n, H, d = 200, 4, 2048
    x, w, sc, base, rw = case(n, H, d, 8)
    pad = 64
    buf = torch.full((n * d + 2 * pad,), 77, dtype=torch.bfloat16, device="cuda")
    y = buf[pad:pad + n * d].view(n, d)
    hc.hc_mixes_pre_norm(x, w, sc, base, rw, y=y)
    first = y.clone()
    hc.hc_mixes_pre_norm(x, w, sc, base, rw, y=y)
    torch.cuda.synchronize()
    assert torch.equal(first.view(torch.int16), y.view(torch.int16))
    assert torch.all(buf[:pad] == 77) and torch.all(buf[-pad:] == 77)


def test_norm_wide_rows_kept_in_the_output(hc):
    # d = 50,176: a collapsed row (98 KB) is too wide for shared memory and is
    # kept in y between the two passes
    n, H, d = 3, 4, 50176
    x, w, sc, base, rw = case(n, H, d, 41)
    y, pre, post, comb, m = hc.hc_mixes_pre_norm(x, w, sc, base, rw, 20, want_mixes=True)
    torch.cuda.synchronize()
    xb = inputs.bf16_bits(x)
    compare.check_mixes(np64(m), oracle.hc_mixes(xb, w.cpu().numpy()))
    _, yc_bits, mag = oracle.hc_pre(xb, np64(pre))
    out_want, want_bits = oracle.hc_rmsnorm(yc_bits, rw.cpu().numpy())
    yc = oracle.bf16_bits_to_f64(yc_bits)
    inv = 1.0 / np.sqrt((yc ** 2).mean(axis=1, keepdims=True) + 1e-20)
    got = oracle.bf16_bits_to_f64(inputs.bf16_bits(y))
    g = rw.cpu().numpy().astype(np.float64)
    allowed = (np.abs(g) * inv * (compare.bf16_ulp(yc) + H * 2.0 ** -24 * mag) +
               compare.bf16_ulp(out_want) + 1e-5 * np.abs(out_want))
    assert np.all(np.abs(got - out_want) <= allowed)
    assert np.mean(key_diff(inputs.bf16_bits(y), want_bits) <= 1) > 0.999


@pytest.mark.parametrize("d", [8, 1024])
def test_norm_rows_beyond_one_launch_grid(hc, d):
    # 2^20 + 5 rows: the norm kernels take one row per CTA up to 2^20 rows and
    # the rest in a grid stride (d = 8: general path; d = 1024: the fused
    # kernel followed by the row pass)
    n, H = (1 << 20) + 5, 4
    g = torch.Generator(device="cuda").manual_seed(d)
    x = torch.randn((n, H, d), device="cuda", generator=g, dtype=torch.bfloat16)
    w = torch.randn(((2 + H) * H, H * d), device="cuda", generator=g) / (H * d) ** 0.5
    sc = torch.rand(3, device="cuda", generator=g) + 0.5
    base = torch.randn((2 + H) * H, device="cuda", generator=g)
    rw = torch.rand(d, device="cuda", generator=g) + 0.25
    y = hc.hc_mixes_pre_norm(x, w, sc, base, rw)[0]
    yc = hc.hc_mixes_pre(x, w, sc, base)[0]
    torch.cuda.synchronize()
    idx = np.unique(np.concatenate([np.arange(4), np.arange((1 << 20) - 4, n),
                                    np.random.default_rng(d).integers(0, n, 200)]))
    _, want = oracle.hc_rmsnorm(inputs.bf16_bits(yc[idx]), rw.cpu().numpy())
    assert key_diff(inputs.bf16_bits(y[idx]), want).max() <= 1


def test_fused_norm_is_one_launch_and_matches_the_oracle_on_every_token(hc):
    # 40,000 tokens at d = 5120 on the fused path: the RMSNorm is folded into
    # the collapse (its statistic from the copies' Gram matrix), one launch;
    # every token against the oracle, stage by stage
    n, H, d = 40000, 4, 5120
    x, w, sc, base, rw = case(n, H, d, 99)
    before = hc.hc_launch_count()
    y, pre, post, comb, m = hc.hc_mixes_pre_norm(x, w, sc, base, rw, 20, want_mixes=True)
    torch.cuda.synchronize()
    assert hc.hc_launch_count() - before == 1
    xb = bits(x)
    check_mixes_all(np64(m), oracle_mixes(None, xb, w.cpu().numpy(), 1e-20))
    check_split_all(np64(m), np64(pre), np64(post), np64(comb), sc.cpu().numpy(),
                    base.cpu().numpy(), H, 20, 1e-6)
    check_norm_all(bits(y), xb, np64(pre), rw.cpu().numpy(), H,
                   what="fused normalised y (40,000 tokens)")


def test_fused_norm_coefficients_equal_the_plain_call(hc):
    # the norm changes only y: mixes, pre, post and comb are bit for bit
    # those of hc_mixes_pre (same squares, same order)
    n, H, d = 3000, 4, 5120
    x, w, sc, base, rw = case(n, H, d, 7)
    y1, pre1, post1, comb1, m1 = hc.hc_mixes_pre_norm(x, w, sc, base, rw, 20, want_mixes=True)
    y0, pre0, post0, comb0, m0 = hc.hc_mixes_pre(x, w, sc, base, 20, want_mixes=True)
    torch.cuda.synchronize()
    for a, b in ((pre1, pre0), (post1, post0), (comb1, comb0), (m1, m0)):
        assert torch.equal(a, b)
