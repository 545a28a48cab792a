"""The tensor-core projection with W streamed (the general path's projection
for hc in {4, 8}): it matches the oracle on one tile, ragged tiles and several
tiles per CTA, and it agrees with the CUDA-core projection."""
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


@pytest.fixture
def path():
    old = os.environ.get("HCMIX_PATH")

    def set_path(v):
        if v is None:
            os.environ.pop("HCMIX_PATH", None)
        else:
            os.environ["HCMIX_PATH"] = v
    yield set_path
    set_path(old)


def case(n, H, d, seed, scale_lo=0.1, scale_hi=10.0):
    g = torch.Generator(device="cuda").manual_seed(seed)
    x = torch.randn((n, H, d), device="cuda", generator=g)
    s = torch.exp(torch.empty((n, 1, 1), device="cuda").uniform_(
        np.log(scale_lo), np.log(scale_hi), generator=g))
    x = (x * s).to(torch.bfloat16)
    mix = (2 + H) * H
    w = torch.randn((mix, H * d), device="cuda", generator=g) / (H * d) ** 0.5
    return x, w


def np64(t):
    return t.detach().cpu().double().numpy()


@pytest.mark.parametrize("H,n,d", [(8, 1, 5120), (8, 300, 5120), (8, 129, 1024),
                                   (4, 200, 2048), (4, 5, 64), (4, 1000, 5120),
                                   (8, 40000, 256)])
def test_projection_matches_oracle(hc, path, H, n, d):
    path("general")
    x, w = case(n, H, d, 7 * n + d + H)
    m = torch.empty((n, (2 + H) * H), device="cuda")
    before = hc.hc_launch_count()
    hc.hc_mixes(x, w, mixes=m)
    torch.cuda.synchronize()
    assert hc.hc_launch_count() - before == 1
    idx = np.arange(n) if n <= 1200 else np.unique(np.concatenate(
        [np.arange(8), np.arange(n - 8, n), np.random.default_rng(1).integers(0, n, 300)]))
    compare.check_mixes(np64(m)[idx], oracle.hc_mixes(inputs.bf16_bits(x[idx]),
                                                      w.cpu().numpy()))


@pytest.mark.parametrize("H,n,d", [(8, 500, 5120), (4, 333, 2048)])
def test_projection_agrees_with_cuda_core_projection(hc, path, H, n, d):
    x, w = case(n, H, d, 3 + H)
    path("general")
    a = hc.hc_mixes(x, w)
    path("ffma")
    b = hc.hc_mixes(x, w)
    torch.cuda.synchronize()
    compare.check_mixes(np64(a), np64(b))


def test_hc8_mixes_pre_through_tensor_projection(hc, path):
    # hc = 8, stress-like logits: the three-kernel path with the tensor-core
    # projection, checked stage by stage against the oracle
    n, H, d = 257, 8, 5120
    x, w = case(n, H, d, 99, 1e-3, 1e3)
    g = torch.Generator(device="cuda").manual_seed(5)
    sc = torch.rand(3, device="cuda", generator=g) * 6 + 2
    base = torch.randn(80, device="cuda", generator=g) * 5 ** 0.5
    before = hc.hc_launch_count()
    y, pre, post, comb, m = hc.hc_mixes_pre(x, w, sc, base, 20, want_mixes=True)
    torch.cuda.synchronize()
    # W conversion, projection, split/Sinkhorn, collapse
    assert hc.hc_launch_count() - before == 4
    xb = inputs.bf16_bits(x)
    compare.check_mixes(np64(m), oracle.hc_mixes(xb, w.cpu().numpy()))
    o_pre, o_post, o_comb = oracle.hc_split_sinkhorn(np64(m), sc.cpu().numpy(),
                                                     base.cpu().numpy(), 8, 20, 1e-6)
    compare.check_abs(np64(pre), o_pre, 1e-5, "pre")
    compare.check_abs(np64(post), o_post, 1e-5, "post")
    compare.check_abs(np64(comb), o_comb, 1e-5, "comb")
    want, _, mag = oracle.hc_pre(xb, np64(pre))
    compare.check_bf16(inputs.bf16_bits(y), want, mag, 8, "y")


@pytest.mark.parametrize("n", [4096, 16384, 20000])
def test_projection_only_dispatch_by_token_count(hc, path, n):
    # hc_mixes alone takes the fused kernel below 16,384 tokens and the
    # streamed-W tensor-core kernel from there on; both agree with the oracle
    H, d = 4, 1024
    x, w = case(n, H, d, 11 + n)
    path(None)
    auto = hc.hc_mixes(x, w)
    path("fused" if n < 16384 else "general")
    pinned = hc.hc_mixes(x, w)
    torch.cuda.synchronize()
    assert torch.equal(auto.view(torch.int32), pinned.view(torch.int32))
    idx = np.unique(np.concatenate([np.arange(4), np.arange(n - 4, n),
                                    np.random.default_rng(n).integers(0, n, 200)]))
    compare.check_mixes(np64(auto)[idx], oracle.hc_mixes(inputs.bf16_bits(x[idx]),
                                                         w.cpu().numpy()))


def test_bench_projection_mode_agrees_across_kernels(hc):
    # `bench.py --projection` times hc_mixes on the CUDA-core kernel, the
    # streamed-W tensor-core kernel and the fused kernel's projection-only
    # mode; on a 4,096-token case each is one launch and all agree with the
    # CUDA-core result to the mixes tolerance
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--projection",
                        "--tokens", "4096", "--steps", "2", "--warmup", "3"],
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    proj = line["projection"]
    assert set(proj) == {"ffma", "general", "fused"}
    for name, rec in proj.items():
        assert rec["launches_per_call"] == 1, name
        assert rec["us_per_launch"] > 0
        assert rec["max_rel_diff_vs_ffma"] <= 1e-4, (name, rec["max_rel_diff_vs_ffma"])



@pytest.mark.parametrize("n,d", [(300, 5120), (129, 1024), (5, 64), (3, 8)])
def test_hc8_projection_from_converted_w_is_bit_identical(hc, path, n, d):
    # with room in the workspace W is converted once into it and the kernel
    # loads it from there; without, the kernel converts each stage itself:
    # the tensor core sees the same numbers in the same order
    path(None)
    H = 8
    x, w = case(n, H, d, 23 + n)
    g = torch.Generator(device="cuda").manual_seed(3)
    sc = torch.rand(3, device="cuda", generator=g) + 0.5
    base = torch.randn(80, device="cuda", generator=g)
    need = hc.hc_workspace_bytes(n, H, d)
    small = (n * 80 * 4 + 255) // 256 * 256
    assert need > small
    outs = []
    for wsb in (need, small):
        ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
        before = hc.hc_launch_count()
        r = hc.hc_mixes_pre(x, w, sc, base, workspace=ws)
        m = torch.empty((n, 80), device="cuda")
        hc.hc_mixes_pre(x, w, sc, base, mixes=m, workspace=ws)
        torch.cuda.synchronize()
        outs.append((r, m, hc.hc_launch_count() - before))
    (r1, m1, l1), (r2, m2, l2) = outs
    assert l1 == 2 * 4 and l2 == 2 * 3  # converted W: 4 launches per call, else 3
    assert torch.equal(m1.view(torch.int32), m2.view(torch.int32))
    for a, b in zip(r1[:4], r2[:4]):
        assert torch.equal(a.view(torch.int16) if a.dtype == torch.bfloat16 else a.view(torch.int32),
                           b.view(torch.int16) if b.dtype == torch.bfloat16 else b.view(torch.int32))
    compare.check_mixes(np64(m1), oracle.hc_mixes(inputs.bf16_bits(x), w.cpu().numpy()))
