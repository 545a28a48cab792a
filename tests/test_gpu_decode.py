"""The few-token (decode) path of hc_mixes_pre / hc_mixes (hc=4, d a multiple
of 256 up to 5120, up to 16 tokens per cluster): it is the path taken (one
launch per call), it matches the oracle stage by stage, and it agrees with
the other paths on the same inputs."""
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import compare
from sinkhorn_mixing_gb300 import inputs

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


def run(hc, x, w, sc, base, iters=20):
    n, _, d = x.shape
    pre = torch.empty((n, 4), device="cuda")
    post = torch.empty((n, 4), device="cuda")
    comb = torch.empty((n, 4, 4), device="cuda")
    y = torch.empty((n, d), dtype=torch.bfloat16, device="cuda")
    m = torch.empty((n, 24), device="cuda")
    before = hc.hc_launch_count()
    hc.hc_mixes_pre(x, w, sc, base, iters, pre=pre, post=post, comb=comb, y=y, mixes=m)
    torch.cuda.synchronize()
    launches = hc.hc_launch_count() - before
    return y, pre, post, comb, m, launches


def check_all(x, w, sc, base, y, pre, post, comb, m, iters=20):
    xb = inputs.bf16_bits(x)
    compare.check_mixes(np64(m), oracle.hc_mixes(xb, w.cpu().numpy()))
    o_pre, o_post, o_comb = oracle.hc_split_sinkhorn(np64(m), sc.cpu().numpy(),
                                                     base.cpu().numpy(), 4, iters, 1e-6)
    compare.check_abs(np64(pre), o_pre, 1e-5, "pre")
    compare.check_abs(np64(post), o_post, 1e-5, "post")
    compare.check_abs(np64(comb), o_comb, 1e-5, "comb")
    want, _, mag = oracle.hc_pre(xb, np64(pre))
    return compare.check_bf16(inputs.bf16_bits(y), want, mag, 4, "y")


@pytest.mark.parametrize("n,d", [(1, 5120), (3, 5120), (16, 5120), (17, 5120), (64, 5120),
                                 (100, 5120), (112, 5120), (64, 4096), (37, 2304),
                                 (64, 1024), (5, 256)])
def test_decode_matches_oracle(hc, n, d):
    x, w, sc, base = case(n, d, 11 * n + d)
    y, pre, post, comb, m, launches = run(hc, x, w, sc, base)
    assert launches == 1, "decode path not taken"
    check_all(x, w, sc, base, y, pre, post, comb, m)


@pytest.mark.parametrize("iters", [1, 50])
def test_decode_iters(hc, iters):
    x, w, sc, base = case(64, 5120, 5 + iters, 1e-3, 1e3)
    y, pre, post, comb, m, launches = run(hc, x, w, sc, base, iters)
    assert launches == 1
    check_all(x, w, sc, base, y, pre, post, comb, m, iters)


def test_decode_mixes_only_entry(hc):
    x, w, _, _ = case(64, 5120, 3)
    m = torch.empty((64, 24), device="cuda")
    before = hc.hc_launch_count()
    hc.hc_mixes(x, w, mixes=m)
    torch.cuda.synchronize()
    assert hc.hc_launch_count() - before == 1
    compare.check_mixes(np64(m), oracle.hc_mixes(inputs.bf16_bits(x), w.cpu().numpy()))


def test_decode_without_mixes_output(hc):
    n, d = 40, 5120
    x, w, sc, base = case(n, d, 8)
    pre = torch.empty((n, 4), device="cuda")
    post = torch.empty((n, 4), device="cuda")
    comb = torch.empty((n, 4, 4), device="cuda")
    y = torch.empty((n, d), dtype=torch.bfloat16, device="cuda")
    wsp = torch.empty(hc.hc_workspace_bytes(n, 4, d), dtype=torch.uint8, device="cuda")
    hc.hc_mixes_pre(x, w, sc, base, pre=pre, post=post, comb=comb, y=y, workspace=wsp)
    y2, pre2, post2, comb2, _, _ = run(hc, x, w, sc, base)
    assert torch.equal(pre, pre2) and torch.equal(comb, comb2) and torch.equal(post, post2)
    assert torch.equal(y.view(torch.int16), y2.view(torch.int16))


@pytest.mark.parametrize("path", ["fused", "general"])
def test_decode_agrees_with_other_paths(hc, path):
    n, d = 64, 5120
    x, w, sc, base = case(n, d, 21)
    y, pre, post, comb, m, _ = run(hc, x, w, sc, base)
    os.environ["HCMIX_PATH"] = path
    try:
        y2, pre2, post2, comb2, m2, launches = run(hc, x, w, sc, base)
    finally:
        del os.environ["HCMIX_PATH"]
    assert launches == (1 if path == "fused" else 3)
    compare.check_mixes(np64(m), np64(m2).astype(np.float64))
    for a, b in ((pre, pre2), (post, post2), (comb, comb2)):
        assert float((a - b).abs().max()) < 2e-5
    # y = sum_j pre_j x_j: the paths' pre differ by < 2e-5, and each y is
    # rounded to bf16 once, so |y - y2| <= 2^-8 (|y| + |y2|) + 2e-5 sum_j |x_j|
    dp = float(torch.maximum((pre - pre2).abs().max(), torch.tensor(0.0, device="cuda")))
    bound = (2.0 ** -8 * (y.float().abs() + y2.float().abs()) +
             (dp + 1e-7) * x.float().abs().sum(dim=1))
    assert bool(((y.float() - y2.float()).abs() <= bound).all())


@pytest.mark.parametrize("iters", [1, 20, 50])
def test_decode_coefficients_equal_the_split_kernel_on_its_own_mixes(hc, iters):
    # The decode kernel's owner lane must give bit for bit what the
    # one-token-per-thread split kernel gives for the same mix numbers (the
    # same operations on the same values, in the same order).  Large logit
    # scales reach the eps-dominated corners.
    n, d = 64, 5120
    x, w, sc, base = case(n, d, 40 + iters)
    sc = sc * 20
    y, pre, post, comb, m, launches = run(hc, x, w, sc, base, iters=iters)
    assert launches == 1
    pre2, post2, comb2 = hc.hc_split_sinkhorn(m, sc, base, 4, iters, 1e-6)
    torch.cuda.synchronize()
    for a, b in ((pre, pre2), (post, post2), (comb, comb2)):
        assert torch.equal(a.view(torch.int32), b.view(torch.int32))


def test_decode_repeated_calls_are_deterministic(hc):
    x, w, sc, base = case(100, 5120, 4)
    a = run(hc, x, w, sc, base)
    b = run(hc, x, w, sc, base)
    for u, v in zip(a[:5], b[:5]):
        assert torch.equal(u.view(torch.int32) if u.dtype == torch.float32 else u.view(torch.int16),
                           v.view(torch.int32) if v.dtype == torch.float32 else v.view(torch.int16))


def test_decode_under_cuda_graph_replay(hc):
    n, d = 64, 5120
    x, w, sc, base = case(n, d, 9)
    pre = torch.empty((n, 4), device="cuda")
    post = torch.empty((n, 4), device="cuda")
    comb = torch.empty((n, 4, 4), device="cuda")
    y = torch.empty((n, d), dtype=torch.bfloat16, device="cuda")
    m = torch.empty((n, 24), device="cuda")
    call = lambda: hc.hc_mixes_pre(x, w, sc, base, pre=pre, post=post, comb=comb, y=y, mixes=m)
    call()
    torch.cuda.synchronize()
    ref = [t.clone() for t in (y, pre, post, comb, m)]
    for t in (y, pre, post, comb, m):
        t.zero_()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            call()
    torch.cuda.synchronize()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    for a, b in zip((y, pre, post, comb, m), ref):
        assert torch.equal(a, b)


@pytest.mark.parametrize("graph", [False, True])
def test_chained_sublayers_equal_with_and_without_launch_overlap(hc, graph):
    # Each kernel of the chain reads what the one before it wrote (x -> pre,
    # post, comb -> the new x -> ...).  With programmatic dependent launch a
    # kernel may start while its predecessor runs; it must still read only
    # after it, so the chain ends on the same bits as with the launches
    # serialised (HCMIX_PDL=0), eagerly and replayed from a CUDA graph.
    n, d = 64, 5120
    x0, w, sc, base = case(n, d, 31)
    g = torch.Generator(device="cuda").manual_seed(32)
    outs = [torch.randn((n, d), device="cuda", generator=g).to(torch.bfloat16) for _ in range(6)]

    def chain(x):
        for out in outs:
            y, pre, post, comb, _ = hc.hc_mixes_pre(x, w, sc, base)
            x = hc.hc_post(out + y, x, post, comb)
        return x

    results = []
    for flag in ("1", "0"):
        old = os.environ.get("HCMIX_PDL")
        os.environ["HCMIX_PDL"] = flag
        try:
            if graph:
                xs = x0.clone()
                side = torch.cuda.Stream()
                side.wait_stream(torch.cuda.current_stream())
                with torch.cuda.stream(side):
                    chain(xs)  # warm-up outside the capture
                    torch.cuda.synchronize()
                    gr = torch.cuda.CUDAGraph()
                    with torch.cuda.graph(gr, stream=side):
                        xr = chain(xs)
                    gr.replay()
                torch.cuda.synchronize()
                results.append(xr.clone())
            else:
                results.append(chain(x0.clone()))
                torch.cuda.synchronize()
        finally:
            if old is None:
                os.environ.pop("HCMIX_PDL", None)
            else:
                os.environ["HCMIX_PDL"] = old
    assert torch.equal(results[0].view(torch.int16), results[1].view(torch.int16))


def test_new_weights_are_read_after_an_intervening_write(hc):
    # The decode kernel copies its W slice before it waits for the kernel in
    # front of it.  Weights rewritten on the stream before the call, with
    # other work in between as the header requires, must still be the ones
    # it uses.
    n, d = 64, 5120
    x, w, sc, base = case(n, d, 41)
    first = run(hc, x, w, sc, base)
    g = torch.Generator(device="cuda").manual_seed(42)
    w.mul_(-0.5).add_(torch.randn(w.shape, device="cuda", generator=g) / (4 * d) ** 0.5)
    scratch = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    scratch.zero_()
    y, pre, post, comb, m, launches = run(hc, x, w, sc, base)
    assert launches == 1, "decode path not taken"
    assert not torch.equal(m, first[4])
    check_all(x, w, sc, base, y, pre, post, comb, m)
