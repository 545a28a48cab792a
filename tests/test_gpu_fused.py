"""The fused tensor-core path of hc_mixes_pre / hc_mixes (hc=4, d a multiple
of 1024 in [1024, 5120]): it is the path taken (one launch per call), it
matches the oracle stage by stage on ragged and multi-tile token counts, and
it agrees with the general three-kernel path on the same inputs."""
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import compare
from sinkhorn_mixing_gb300 import inputs
from parity import check_mixes_all, check_pre_all, check_split_all, oracle_mixes

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def fused_path_only():
    """Small token counts would otherwise take the decode kernel."""
    old = os.environ.get("HCMIX_PATH")
    os.environ["HCMIX_PATH"] = "fused"
    yield
    if old is None:
        os.environ.pop("HCMIX_PATH", None)
    else:
        os.environ["HCMIX_PATH"] = old


@pytest.fixture(scope="module")
def hc():
    from sinkhorn_mixing_gb300 import build
    build.build()
    import sinkhorn_mixing_gb300 as m
    m.hc_device_error(clear=True)
    yield m
    torch.cuda.synchronize()
    assert m.hc_device_error(clear=True) == 0


def bits(t):
    return inputs.bf16_bits(t)


def np64(t):
    return t.detach().cpu().double().numpy()


def case(n, d, seed, scale_lo=0.1, scale_hi=10.0):
    g = torch.Generator(device="cuda").manual_seed(seed)
    x = torch.randn((n, 4, d), device="cuda", generator=g)
    s = torch.exp(torch.empty((n, 1, 1), device="cuda").uniform_(
        np.log(scale_lo), np.log(scale_hi), generator=g))
    x = (x * s).to(torch.bfloat16)
    w = torch.randn((24, 4 * d), device="cuda", generator=g) / (4 * d) ** 0.5
    sc = torch.rand(3, device="cuda", generator=g) * 1.5 + 0.5
    base = torch.randn(24, device="cuda", generator=g)
    return x, w, sc, base


def check_all(x, w, sc, base, y, pre, post, comb, m, iters=20, idx=None):
    n = x.shape[0]
    idx = np.arange(n) if idx is None else idx
    xb = bits(x[idx])
    compare.check_mixes(np64(m)[idx], oracle.hc_mixes(xb, w.cpu().numpy()))
    o_pre, o_post, o_comb = oracle.hc_split_sinkhorn(np64(m)[idx], sc.cpu().numpy(),
                                                     base.cpu().numpy(), 4, iters, 1e-6)
    compare.check_abs(np64(pre)[idx], o_pre, 1e-5, "pre")
    compare.check_abs(np64(post)[idx], o_post, 1e-5, "post")
    compare.check_abs(np64(comb)[idx], o_comb, 1e-5, "comb")
    want, _, mag = oracle.hc_pre(xb, np64(pre)[idx])
    return compare.check_bf16(bits(y[idx]), want, mag, 4, "y")


@pytest.mark.parametrize("n,d", [(64, 5120), (1, 5120), (70, 5120), (200, 2048),
                                 (129, 3072), (1000, 4096), (100, 1024), (3000, 5120)])
def test_fused_small_and_ragged(hc, n, d):
    x, w, sc, base = case(n, d, seed=n + d)
    before = hc.hc_launch_count()
    y, pre, post, comb, m = hc.hc_mixes_pre(x, w, sc, base, want_mixes=True)
    torch.cuda.synchronize()
    assert hc.hc_launch_count() - before == 1, "fused path not taken"
    assert hc.hc_device_error(clear=False) == 0
    check_all(x, w, sc, base, y, pre, post, comb, m)


def test_fused_mixes_only_entry(hc):
    x, w, sc, base = case(300, 5120, seed=5)
    before = hc.hc_launch_count()
    m = hc.hc_mixes(x, w)
    torch.cuda.synchronize()
    assert hc.hc_launch_count() - before == 1
    compare.check_mixes(np64(m), oracle.hc_mixes(bits(x), w.cpu().numpy()))


@pytest.mark.parametrize("iters", [1, 20, 50])
def test_fused_many_tiles_every_token(hc, iters):
    # 625 tiles over every cluster: every tile, round and owner is compared
    n = 40000
    x, w, sc, base = case(n, 5120, seed=iters, scale_lo=1e-3, scale_hi=1e3)
    y, pre, post, comb, m = hc.hc_mixes_pre(x, w, sc, base, iters, want_mixes=True)
    torch.cuda.synchronize()
    xb = bits(x)
    check_mixes_all(np64(m), oracle_mixes(None, xb, w.cpu().numpy(), 1e-20))
    check_split_all(np64(m), np64(pre), np64(post), np64(comb), sc.cpu().numpy(),
                    base.cpu().numpy(), 4, iters, 1e-6)
    check_pre_all(bits(y), xb, np64(pre), 4, "fused y (40,000 tokens, iters %d)" % iters)


@pytest.mark.parametrize("n", [33, 300, 4096])
def test_fused_and_decode_paths_take_a_null_workspace(hc, n):
    # the decode (33 tokens) and fused (300, 4096 tokens) paths read no
    # workspace: the C ABI accepts NULL there, with the same results as the
    # binding's call (which passes a workspace)
    import ctypes
    from sinkhorn_mixing_gb300 import binding
    os.environ.pop("HCMIX_PATH", None)  # the shape decides
    x, w, sc, base = case(n, 5120, seed=n)
    want = hc.hc_mixes_pre(x, w, sc, base)
    pre = torch.empty((n, 4), device="cuda")
    post = torch.empty((n, 4), device="cuda")
    comb = torch.empty((n, 4, 4), device="cuda")
    y = torch.empty((n, 5120), dtype=torch.bfloat16, device="cuda")
    P = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    st = binding.lib().hc_mixes_pre(n, 4, 5120, 20, 1e-6, 1e-20, P(x), P(w), P(sc), P(base),
                                    None, P(pre), P(post), P(comb), P(y), None, 0,
                                    ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, binding.status_string(st)
    torch.cuda.synchronize()
    for a, b in zip((y, pre, post, comb), want[:4]):
        assert torch.equal(a, b)


def test_fused_agrees_with_general_path(hc):
    x, w, sc, base = case(777, 5120, seed=9)
    a = hc.hc_mixes_pre(x, w, sc, base, want_mixes=True)
    os.environ["HCMIX_PATH"] = "general"
    try:
        before = hc.hc_launch_count()
        b = hc.hc_mixes_pre(x, w, sc, base, want_mixes=True)
        torch.cuda.synchronize()
        assert hc.hc_launch_count() - before == 3
    finally:
        os.environ["HCMIX_PATH"] = "fused"
    ya, pa, qa, ca, ma = a
    yb, pb, qb, cb, mb = b
    torch.testing.assert_close(ma, mb, rtol=1e-4, atol=1e-4)
    torch.testing.assert_close(pa, pb, rtol=0, atol=1e-4)
    torch.testing.assert_close(ca, cb, rtol=0, atol=1e-4)
    # y differs only where pre differs in the last bits: compare via the oracle
    want, _, mag = oracle.hc_pre(bits(x), np64(pa))
    compare.check_bf16(bits(ya), want, mag, 4, "fused y")


def test_fused_repeated_calls_are_deterministic(hc):
    x, w, sc, base = case(512, 5120, seed=3)
    r1 = hc.hc_mixes_pre(x, w, sc, base, want_mixes=True)
    r2 = hc.hc_mixes_pre(x, w, sc, base, want_mixes=True)
    torch.cuda.synchronize()
    for u, v in zip(r1, r2):
        assert torch.equal(u, v)
