"""hc_post_mixes_pre: the boundary between two sublayers in one call
(hc_post of sublayer s, then hc_mixes_pre of sublayer s+1 on the new stream).

It must equal the two separate calls -- the new stream bit for bit, the rest
bit for bit too where both take the same projection kernel -- on the fused
path (one kernel) and on every other path (the two calls inside), in place
or not; and it must match the float64 oracle stage by stage on every token of
a many-tile case."""
import os

import numpy as np
import pytest
import torch

from sinkhorn_mixing_gb300 import inputs
from parity import (check_mixes_all, check_post_all, check_pre_all, check_split_all, bits,
                    np64, oracle_mixes)

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


def case(n, H, d, seed):
    """Sublayer s's output, stream and coefficients; sublayer s+1's parameters
    (the argument order of hc_post_mixes_pre)."""
    g = torch.Generator(device="cuda").manual_seed(seed)
    mix = (2 + H) * H
    res = (torch.randn((n, H, d), device="cuda", generator=g) *
           torch.exp(torch.empty((n, 1, 1), device="cuda").uniform_(
               np.log(0.1), np.log(10.0), generator=g))).to(torch.bfloat16)
    out = torch.randn((n, d), device="cuda", generator=g).to(torch.bfloat16)
    post = torch.rand((n, H), device="cuda", generator=g) * 2
    comb = torch.rand((n, H, H), device="cuda", generator=g)
    comb = comb / comb.sum(1, keepdim=True)
    w = torch.randn((mix, H * d), device="cuda", generator=g) / (H * d) ** 0.5
    sc = torch.rand(3, device="cuda", generator=g) * 1.5 + 0.5
    base = torch.randn(mix, device="cuda", generator=g)
    return out, res, post, comb, w, sc, base


def separate(hc, out, res, post, comb, w, sc, base):
    x1 = hc.hc_post(out, res, post, comb)
    y, pre, post1, comb1, m = hc.hc_mixes_pre(x1, w, sc, base, want_mixes=True)
    return x1, y, pre, post1, comb1, m


def with_path(path):
    old = os.environ.get("HCMIX_PATH")
    if path is None:
        os.environ.pop("HCMIX_PATH", None)
    else:
        os.environ["HCMIX_PATH"] = path
    return old


def restore(old):
    if old is None:
        os.environ.pop("HCMIX_PATH", None)
    else:
        os.environ["HCMIX_PATH"] = old


@pytest.mark.parametrize("n,H,d,path,fused", [
    (200, 4, 5120, None, True),       # the fused kernel
    (3000, 4, 5120, None, True),
    (129, 4, 1024, None, True),
    (1000, 4, 3072, None, True),
    (70, 4, 2048, "fused", True),     # the fused kernel below the decode limit
    (33, 4, 5120, None, True),        # the decode kernel with hc_post in front
    (1, 4, 5120, None, True),
    (64, 4, 2048, None, True),
    (112, 4, 5120, None, True),       # 16 tokens on each of 7 clusters
    (37, 4, 2304, None, True),        # w = 144: a channel slice not a multiple of 64
    (300, 4, 136, None, False),       # hc_post, then the general path
    (150, 8, 1024, None, False),      # hc=8: hc_post, then the general path
])
def test_equals_hc_post_then_hc_mixes_pre(hc, n, H, d, path, fused):
    old = with_path(path)
    try:
        args = case(n, H, d, seed=n + d + H)
        before = hc.hc_launch_count()
        want = separate(hc, *args)
        sep_launches = hc.hc_launch_count() - before
        before = hc.hc_launch_count()
        got = hc.hc_post_mixes_pre(*args, want_mixes=True)
        torch.cuda.synchronize()
        assert hc.hc_launch_count() - before == (1 if fused else sep_launches)
    finally:
        restore(old)
    names = ("x_next", "y", "pre", "post", "comb", "mixes")
    for nm, a, b in zip(names, got, want):
        assert torch.equal(a, b), nm


@pytest.mark.parametrize("n", [777, 50])  # the fused kernel; the decode kernel
def test_in_place_and_without_mixes(hc, n):
    out, res, post, comb, w, sc, base = case(n, 4, 5120, seed=5)
    want = separate(hc, out, res.clone(), post, comb, w, sc, base)
    x_next, y, pre, post1, comb1, m = hc.hc_post_mixes_pre(out, res, post, comb, w, sc, base,
                                                           x_next=res)
    torch.cuda.synchronize()
    assert m is None
    assert x_next.data_ptr() == res.data_ptr()
    for a, b in zip((res, y, pre, post1, comb1), want[:5]):
        assert torch.equal(a, b)


def test_two_sublayers_chained(hc):
    # attention then FFN sublayer of one block, each with its own parameters:
    # mixes_pre(A) -> post_mixes_pre(A -> F) -> post(F), against the four
    # separate calls
    wl = inputs.WORKLOADS["prefill"]
    s = inputs.make_streams(wl, n=2048, device="cuda")
    s2 = inputs.make_streams(wl, n=2048, device="cuda", seed_offset=1)
    pa = inputs.make_params(wl, 0, device="cuda")
    pf = inputs.make_params(wl, 1, device="cuda")
    x, out_a, out_f = s["x"], s["out"], s2["out"]
    ya, prea, posta, comba, _ = hc.hc_mixes_pre(x, pa["w"], pa["hc_scale"], pa["hc_base"])
    x1, yf, pref, postf, combf, _ = hc.hc_post_mixes_pre(out_a, x, posta, comba, pf["w"],
                                                         pf["hc_scale"], pf["hc_base"])
    x2 = hc.hc_post(out_f, x1, postf, combf)
    x1s = hc.hc_post(out_a, x, posta, comba)
    yfs, prefs, postfs, combfs, _ = hc.hc_mixes_pre(x1s, pf["w"], pf["hc_scale"], pf["hc_base"])
    x2s = hc.hc_post(out_f, x1s, postfs, combfs)
    torch.cuda.synchronize()
    for a, b in ((x1, x1s), (yf, yfs), (pref, prefs), (postf, postfs), (combf, combfs),
                 (x2, x2s)):
        assert torch.equal(a, b)


def test_every_token_against_the_oracle(hc):
    # 40,000 tokens (625 tiles over every cluster), stage parity on every
    # token: the new stream against the oracle's hc_post; the mix numbers
    # against the oracle's projection of that stream; pre/post/comb against
    # the oracle's split + Sinkhorn of the call's own mix numbers; y against
    # the oracle's collapse with the call's own pre
    n = 40000
    out, res, post, comb, w, sc, base = case(n, 4, 5120, seed=77)
    x1, y, pre, post1, comb1, m = hc.hc_post_mixes_pre(out, res, post, comb, w, sc, base,
                                                       want_mixes=True)
    torch.cuda.synchronize()
    xb = bits(x1)
    check_post_all(xb, bits(out), bits(res), np64(post), np64(comb), 4,
                   "post_mixes_pre x_next (40,000 tokens)")
    check_mixes_all(np64(m), oracle_mixes(None, xb, w.cpu().numpy(), 1e-20))
    check_split_all(np64(m), np64(pre), np64(post1), np64(comb1), sc.cpu().numpy(),
                    base.cpu().numpy(), 4, 20, 1e-6)
    check_pre_all(bits(y), xb, np64(pre), 4, "post_mixes_pre y (40,000 tokens)")


def test_overlapping_buffers_are_rejected_before_any_launch(hc):
    out, res, post, comb, w, sc, base = case(64, 4, 1024, seed=1)
    before = hc.hc_launch_count()
    with pytest.raises(hc.HcError):  # the new coefficients on top of the old ones
        hc.hc_post_mixes_pre(out, res, post, comb, w, sc, base, pre=post)
    with pytest.raises(hc.HcError):  # x_next partly over the residual
        buf = torch.empty((65, 4, 1024), dtype=torch.bfloat16, device="cuda")
        buf[:64].copy_(res)
        hc.hc_post_mixes_pre(out, buf[:64], post, comb, w, sc, base, x_next=buf[1:65])
    assert hc.hc_launch_count() == before


def test_decode_boundary_against_the_oracle(hc):
    # the decode kernel with hc_post in front, 112 tokens (16 on each of 7
    # clusters), stage parity on every token
    n = 112
    out, res, post, comb, w, sc, base = case(n, 4, 5120, seed=91)
    before = hc.hc_launch_count()
    x1, y, pre, post1, comb1, m = hc.hc_post_mixes_pre(out, res, post, comb, w, sc, base,
                                                       want_mixes=True)
    torch.cuda.synchronize()
    assert hc.hc_launch_count() - before == 1
    xb = bits(x1)
    check_post_all(xb, bits(out), bits(res), np64(post), np64(comb), 4,
                   "decode boundary x_next (112 tokens)")
    check_mixes_all(np64(m), oracle_mixes(None, xb, w.cpu().numpy(), 1e-20))
    check_split_all(np64(m), np64(pre), np64(post1), np64(comb1), sc.cpu().numpy(),
                    base.cpu().numpy(), 4, 20, 1e-6)
    check_pre_all(bits(y), xb, np64(pre), 4, "decode boundary y (112 tokens)")
