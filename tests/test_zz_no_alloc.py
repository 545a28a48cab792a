"""hc_mixes_pre_noalloc: the entry point for callers that cannot allocate
device memory (plugin hosts that own all allocations, graph-capture regions,
allocator callbacks, real-time loops).  It keeps the mix numbers in a fixed
array inside the library instead of a caller workspace.

Called here through the C ABI (ctypes on libhcmix.so) and checked against the
existing hc_mixes_pre on the same inputs, on two calls in a row with
different inputs so that the reuse of the shared array is exercised.  This
file is collected last on purpose; it runs alone or after the other tests.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from oracle import compare
from sinkhorn_mixing_gb300 import inputs
from parity import check_mixes_all, check_pre_all, check_split_all, oracle_mixes

pytestmark = pytest.mark.gpu

OK, UNSUPPORTED = 0, 2


@pytest.fixture(scope="module")
def L():
    from sinkhorn_mixing_gb300 import binding, build
    build.build()
    lib = binding.lib()
    P, i64, i32, f32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float
    lib.hc_mixes_pre_noalloc.argtypes = [i64, i32, i64, i32, f32, f32, P, P, P, P, P, P, P, P, P]
    lib.hc_mixes_pre_noalloc.restype = i32
    return lib


def ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def case(n, hc, d, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    mix = (2 + hc) * hc
    x = torch.randn((n, hc, d), device="cuda", generator=g).to(torch.bfloat16)
    w = torch.randn((mix, hc * d), device="cuda", generator=g) / (hc * d) ** 0.5
    sc = torch.rand(3, device="cuda", generator=g) * 1.5 + 0.5
    base = torch.randn(mix, device="cuda", generator=g)
    return x, w, sc, base


def noalloc(L, x, w, sc, base, iters=20, eps=1e-6, norm_eps=1e-20):
    n, hc, d = x.shape
    pre = torch.empty((n, hc), device="cuda")
    post = torch.empty((n, hc), device="cuda")
    comb = torch.empty((n, hc, hc), device="cuda")
    y = torch.empty((n, d), dtype=torch.bfloat16, device="cuda")
    st = L.hc_mixes_pre_noalloc(n, hc, d, iters, eps, norm_eps, ptr(x), ptr(w), ptr(sc),
                                ptr(base), ptr(pre), ptr(post), ptr(comb), ptr(y),
                                ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == OK, st
    return y, pre, post, comb


@pytest.mark.parametrize("path", ["general", "ffma"])
@pytest.mark.parametrize("n,hc,d", [(37, 4, 64), (300, 8, 5120), (500, 4, 5120)])
def test_noalloc_equals_hc_mixes_pre_on_the_general_path(L, n, hc, d, path):
    # the no-allocation entry runs hc_mixes_pre's general three-kernel path
    # (tensor-core projection, or the CUDA-core one when the path is pinned to
    # it); hc_mixes_pre pinned to the same path gives identical results
    import os
    import sinkhorn_mixing_gb300 as m
    old = os.environ.get("HCMIX_PATH")
    os.environ["HCMIX_PATH"] = path
    try:
        for call, seed in enumerate((1, 2)):
            x, w, sc, base = case(n, hc, d, seed + 10 * hc)
            got = noalloc(L, x, w, sc, base)
            want = m.hc_mixes_pre(x, w, sc, base)[:4]
            torch.cuda.synchronize()
            for a, b in zip(got, want):
                assert torch.equal(a, b), "call %d differs" % call
    finally:
        if old is None:
            os.environ.pop("HCMIX_PATH", None)
        else:
            os.environ["HCMIX_PATH"] = old


def test_noalloc_matches_fused_entry_point_within_tolerance(L):
    # at hc=4, d=5120 hc_mixes_pre takes the fused tensor-core kernel; the
    # coefficients agree within the tolerance used between the two paths and
    # y is within 1 bf16 ulp of the oracle's collapse with the call's own pre
    import sinkhorn_mixing_gb300 as m
    for seed in (3, 4):
        x, w, sc, base = case(500, 4, 5120, seed)
        y, pre, post, comb = noalloc(L, x, w, sc, base)
        y2, pre2, post2, comb2, _ = m.hc_mixes_pre(x, w, sc, base)
        torch.cuda.synchronize()
        torch.testing.assert_close(pre, pre2, rtol=0, atol=1e-4)
        torch.testing.assert_close(post, post2, rtol=0, atol=1e-4)
        torch.testing.assert_close(comb, comb2, rtol=0, atol=1e-4)
        want, _, mag = oracle.hc_pre(inputs.bf16_bits(x), pre.cpu().double().numpy())
        compare.check_bf16(inputs.bf16_bits(y), want, mag, 4, "noalloc y")


def test_noalloc_every_token_against_the_oracle(L):
    # 40,000 tokens (hc=4, d=5120, within the fixed scratch), two calls in a
    # row with different inputs.  Stage parity on every token: the mix numbers
    # of the same projection kernel (hc_mixes on the general path) against the
    # oracle's, the call's pre/post/comb against the oracle's split + Sinkhorn
    # of those mix numbers, and y against the oracle's collapse with the
    # call's own pre.
    import os
    import sinkhorn_mixing_gb300 as m
    n = 40000
    old = os.environ.get("HCMIX_PATH")
    try:
        for seed in (21, 22):
            x, w, sc, base = case(n, 4, 5120, seed)
            y, pre, post, comb = noalloc(L, x, w, sc, base)
            os.environ["HCMIX_PATH"] = "general"
            mix = m.hc_mixes(x, w)
            # the same kernels as the call's own stages: its coefficients follow
            pre2, post2, comb2 = m.hc_split_sinkhorn(mix, sc, base)
            torch.cuda.synchronize()
            for a, b in ((pre, pre2), (post, post2), (comb, comb2)):
                assert torch.equal(a, b)
            xb = inputs.bf16_bits(x)
            f64 = lambda t: t.cpu().double().numpy()  # noqa: E731
            check_mixes_all(f64(mix), oracle_mixes(None, xb, w.cpu().numpy(), 1e-20))
            check_split_all(f64(mix), f64(pre), f64(post), f64(comb), sc.cpu().numpy(),
                            base.cpu().numpy(), 4, 20, 1e-6)
            check_pre_all(inputs.bf16_bits(y), xb, f64(pre), 4, "noalloc y (call %d)" % seed)
    finally:
        if old is None:
            os.environ.pop("HCMIX_PATH", None)
        else:
            os.environ["HCMIX_PATH"] = old


def test_noalloc_rejects_sizes_beyond_its_scratch(L):
    import sinkhorn_mixing_gb300 as m
    cap = (1 << 20) // 24  # tokens at hc = 4
    before = m.hc_launch_count()
    fake = ctypes.c_void_p(1 << 20)
    st = L.hc_mixes_pre_noalloc(cap + 1, 4, 64, 20, 1e-6, 1e-20, *([fake] * 8), None)
    assert st == UNSUPPORTED
    assert m.hc_launch_count() == before
