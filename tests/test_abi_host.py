"""Host-side tests of the C ABI: the library builds for sm_103a, loads, exports
every entry point that include/hcmix.h declares, and rejects bad arguments
with the documented status codes before touching any GPU.  The device
pointers used here are fake addresses: validation never dereferences them, and
every call below returns before the first CUDA runtime call."""
import ctypes
import math
import os
import re
import shutil

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "hcmix.h")

OK, INVALID, UNSUPPORTED, MISALIGNED, CUDA = 0, 1, 2, 3, 4

pytestmark = pytest.mark.skipif(shutil.which("nvcc") is None and
                                not os.path.exists("/usr/local/cuda/bin/nvcc"),
                                reason="nvcc not available")


@pytest.fixture(scope="module")
def L():
    from sinkhorn_mixing_gb300 import build
    build.build()
    from sinkhorn_mixing_gb300 import binding
    return binding.lib()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(hc_[a-z_0-9]+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for want in ("hc_mixes", "hc_split_sinkhorn", "hc_pre", "hc_post", "hc_mixes_pre",
                 "hc_workspace_bytes", "hc_status_string", "hc_abi_version",
                 "hc_device_error"):
        assert want in names


def test_library_exports_every_declared_symbol(L):
    for name in declared_functions():
        assert hasattr(L, name), name
    assert L.hc_abi_version() == 1


def test_status_strings(L):
    for s in range(5):
        assert L.hc_status_string(s).decode().startswith("HC_")
    assert L.hc_status_string(99) is not None


A = 1 << 20          # a 16-byte aligned fake device address
GAP = 1 << 36        # spacing that keeps the fake buffers disjoint


def fake(i, off=0):
    return ctypes.c_void_p(A + i * GAP + off)


def _gpu_present():
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:  # pragma: no cover
        return False


# Calls whose arguments pass validation go on to their first CUDA call.  With
# no GPU that call fails (HC_ERR_CUDA) and nothing runs; on a machine with a
# GPU they would launch kernels on the fake addresses, so they are made only
# where no GPU is present.
NO_GPU = not _gpu_present()


def post_call(L, n=4, hc=4, d=64, out=None, res=None, post=None, comb=None, y=None):
    args = [fake(0) if out is None else out, fake(1) if res is None else res,
            fake(2) if post is None else post, fake(3) if comb is None else comb,
            fake(4) if y is None else y]
    return L.hc_post(n, hc, d, *args, None)


def test_shape_checks(L):
    assert post_call(L, n=-1) == INVALID
    assert post_call(L, d=0) == INVALID
    assert post_call(L, hc=3) == UNSUPPORTED
    assert post_call(L, hc=16) == UNSUPPORTED
    assert post_call(L, d=12) == MISALIGNED
    assert post_call(L, n=1 << 41) == UNSUPPORTED
    # n == 0 is a no-op, even with null pointers
    assert L.hc_post(0, 4, 64, None, None, None, None, None, None) == OK
    assert L.hc_pre(0, 4, 64, None, None, None, None) == OK
    assert L.hc_mixes(0, 4, 64, 1e-20, None, None, None, None) == OK
    assert L.hc_split_sinkhorn(0, 4, 20, 1e-6, None, None, None, None, None, None, None) == OK


def test_pointer_checks(L):
    assert post_call(L, out=ctypes.c_void_p(0)) == INVALID
    assert post_call(L, comb=fake(3, 4)) == MISALIGNED
    assert post_call(L, y=fake(4, 8)) == MISALIGNED
    assert L.hc_pre(4, 4, 64, fake(0), None, fake(2), None) == INVALID


def test_overlap_checks(L):
    # y overlapping out (but not identical to residual) is rejected
    assert post_call(L, y=fake(0, 16)) == INVALID
    # y partially overlapping residual is rejected; y == residual is allowed
    # and proceeds to the first CUDA call (which fails without a GPU)
    assert post_call(L, y=fake(1, 16)) == INVALID
    if NO_GPU:
        assert post_call(L, y=fake(1)) == CUDA
    # hc_pre output on top of its input
    assert L.hc_pre(4, 4, 64, fake(0), fake(1), fake(0, 32), None) == INVALID


def test_scalar_checks(L):
    f = L.hc_split_sinkhorn
    args = [fake(i) for i in range(6)]
    assert f(4, 4, 0, 1e-6, *args, None) == INVALID          # iters < 1
    assert f(4, 4, -3, 1e-6, *args, None) == INVALID
    assert f(4, 4, 20, -1e-6, *args, None) == INVALID        # eps < 0
    assert f(4, 4, 20, math.nan, *args, None) == INVALID
    assert f(4, 4, 20, math.inf, *args, None) == INVALID
    assert f(4, 5, 20, 1e-6, *args, None) == UNSUPPORTED
    assert L.hc_mixes(4, 4, 64, -1.0, fake(0), fake(1), fake(2), None) == INVALID
    assert L.hc_mixes(4, 4, 64, math.nan, fake(0), fake(1), fake(2), None) == INVALID


def mixes_pre_call(L, n=4, hc=4, d=64, iters=20, mixes=None, ws=None, wsb=0):
    ptrs = [fake(i) for i in range(4)]  # x, w, scale, base
    outs = [mixes, fake(5), fake(6), fake(7), fake(8)]  # mixes, pre, post, comb, y
    return L.hc_mixes_pre(n, hc, d, iters, 1e-6, 1e-20, *ptrs, *outs, ws, wsb, None)


def test_workspace_rules(L):
    n, hc, d = 4, 4, 64
    need = L.hc_workspace_bytes(n, hc, d)
    assert need == 512  # 4 tokens x 24 floats = 384 bytes, rounded up to 256
    assert L.hc_workspace_bytes(0, 4, 64) == 0
    assert L.hc_workspace_bytes(4, 3, 64) == 0
    # at hc = 8 it also holds W converted to the tensor core's hi/lo rows
    # (2 * 80 rows x hc*d bf16), past the mix numbers
    assert L.hc_workspace_bytes(65536, 8, 5120) == 65536 * 80 * 4 + 4 * 80 * 8 * 5120
    assert L.hc_workspace_bytes(4, 8, 64) == 1280 + 4 * 80 * 512
    # a workspace for the mix numbers alone is still accepted (W is then
    # converted inside the projection kernel)
    if NO_GPU:
        assert mixes_pre_call(L, hc=8, ws=fake(9), wsb=1280) == CUDA
    assert mixes_pre_call(L, hc=8, ws=fake(9), wsb=1279) == INVALID
    # no mixes and no workspace -> rejected before any CUDA call
    assert mixes_pre_call(L) == INVALID
    assert mixes_pre_call(L, ws=fake(9), wsb=need - 1) == INVALID
    assert mixes_pre_call(L, ws=fake(9, 16), wsb=need) == MISALIGNED
    assert mixes_pre_call(L, ws=fake(5), wsb=need) == INVALID      # overlaps pre
    assert mixes_pre_call(L, iters=0, mixes=fake(4)) == INVALID
    assert mixes_pre_call(L, mixes=fake(4, 4)) == MISALIGNED
    if NO_GPU:
        # valid arguments reach the first CUDA call
        assert mixes_pre_call(L, ws=fake(9), wsb=need) == CUDA
        # shapes the decode or fused path may take read no workspace: without
        # one (or with one too small for the mix numbers) they pass
        # validation; the general path's need is checked once the path is known
        assert mixes_pre_call(L, d=5120) == CUDA
        assert mixes_pre_call(L, d=1024, ws=fake(9), wsb=16) == CUDA
        assert mixes_pre_call(L, d=256) == CUDA


def post_mixes_pre_call(L, n=4, hc=4, d=64, iters=20, x_next=None, pre=None, mixes=None, ws=None,
                        wsb=0):
    # out, residual, post, comb | x_next | w, scale, base | mixes, pre, post', comb', y
    args = [fake(0), fake(1), fake(2), fake(3), fake(4) if x_next is None else x_next, iters,
            1e-6, 1e-20, fake(5), fake(6), fake(7), mixes, fake(8) if pre is None else pre,
            fake(9), fake(10), fake(11), ws, wsb, None]
    return L.hc_post_mixes_pre(n, hc, d, *args)


def test_post_mixes_pre_validation(L):
    # n == 0 is a no-op even with null pointers
    assert L.hc_post_mixes_pre(0, 4, 64, *([None] * 5), 20, 1e-6, 1e-20, *([None] * 8), None, 0,
                               None) == OK
    assert post_mixes_pre_call(L, hc=3) == UNSUPPORTED
    assert post_mixes_pre_call(L, d=12) == MISALIGNED
    assert post_mixes_pre_call(L, iters=0) == INVALID
    assert post_mixes_pre_call(L, x_next=ctypes.c_void_p(0)) == INVALID
    assert post_mixes_pre_call(L, pre=fake(8, 4)) == MISALIGNED
    assert post_mixes_pre_call(L, mixes=fake(12, 8)) == MISALIGNED
    # x_next partly over the residual; the new coefficients over the old ones;
    # an output over the sublayer output
    assert post_mixes_pre_call(L, x_next=fake(1, 16)) == INVALID
    assert post_mixes_pre_call(L, pre=fake(2)) == INVALID
    assert post_mixes_pre_call(L, pre=fake(0, 32)) == INVALID
    # pre_next over the residual, with x_next in place
    assert post_mixes_pre_call(L, x_next=fake(1), pre=fake(1, 64)) == INVALID
    if NO_GPU:
        # in place (x_next == residual) passes validation
        assert post_mixes_pre_call(L, x_next=fake(1)) == CUDA
