"""Thin Python binding of libhcmix.so (argument marshalling only).

Every function has the name of the C entry point it calls and does nothing
but check tensor dtypes/devices/contiguity, allocate missing outputs with
torch (as the reference wrapper does with ``new_empty``), and pass raw device
pointers plus the current CUDA stream.  All arithmetic runs in the library's
kernels; there is no fallback path: if the library is missing or a call
fails, an exception is raised.

Leading dimensions are flattened to the token count n, as the pages' wrapper
views ``[b, s, ...]`` tensors as ``[n, ...]``; outputs keep the caller's
leading dimensions.
"""
import ctypes
import functools
import os
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libhcmix.so")

HC_OK = 0
_lib = None


class HcError(RuntimeError):
    """A non-OK hc_status returned by the library."""

    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__("%s: %s" % (what, status_string(status)))


def lib():
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                "libhcmix.so is not built (%s); run `python -m "
                "sinkhorn_mixing_gb300.build`" % LIB_PATH)
        L = ctypes.CDLL(LIB_PATH)
        P, i64, i32, f32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float
        L.hc_status_string.argtypes = [i32]
        L.hc_status_string.restype = ctypes.c_char_p
        L.hc_abi_version.restype = i32
        L.hc_mixes.argtypes = [i64, i32, i64, f32, P, P, P, P]
        L.hc_split_sinkhorn.argtypes = [i64, i32, i32, f32, P, P, P, P, P, P, P]
        L.hc_pre.argtypes = [i64, i32, i64, P, P, P, P]
        L.hc_post.argtypes = [i64, i32, i64, P, P, P, P, P, P]
        L.hc_mixes_pre.argtypes = [i64, i32, i64, i32, f32, f32, P, P, P, P, P, P, P, P, P, P,
                                   ctypes.c_size_t, P]
        L.hc_mixes_pre_norm.argtypes = [i64, i32, i64, i32, f32, f32, P, P, P, P, P, f32, P, P,
                                        P, P, P, P, ctypes.c_size_t, P]
        L.hc_post_mixes_pre.argtypes = [i64, i32, i64, P, P, P, P, P, i32, f32, f32, P, P, P, P,
                                        P, P, P, P, P, ctypes.c_size_t, P]
        L.hc_workspace_bytes.argtypes = [i64, i32, i64]
        L.hc_workspace_bytes.restype = ctypes.c_size_t
        L.hc_device_error.argtypes = [ctypes.POINTER(ctypes.c_uint), i32]
        L.hc_launch_count.restype = ctypes.c_uint64
        L.hc_selftest_wait_timeout.argtypes = [ctypes.c_uint64, P]
        L.hc_selftest_wait_timeout.restype = i32
        for f in ("hc_mixes", "hc_split_sinkhorn", "hc_pre", "hc_post", "hc_mixes_pre",
                  "hc_mixes_pre_norm", "hc_post_mixes_pre", "hc_device_error"):
            getattr(L, f).restype = i32
        _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().hc_status_string(int(status)).decode()


def _check(status: int, what: str):
    if status != HC_OK:
        raise HcError(status, what)


def _ptr(t: Optional[torch.Tensor]):
    # a plain int (or None for NULL): ctypes converts it for c_void_p arguments
    return None if t is None else t.data_ptr()


# The raw handle of the current stream without building a Stream object
# (a few microseconds per call on the decode path); public API otherwise.
_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(dev: torch.device, stream) -> int:
    if stream is not None:
        return stream.cuda_stream
    if _raw_stream is not None:
        return _raw_stream(dev.index)
    return torch.cuda.current_stream(dev).cuda_stream


def _call(dev: torch.device, fn, *args):
    """fn(*args) with `dev` as the current device, switching (and back) only
    when it is not already current."""
    cur = torch.cuda.current_device()
    if cur == dev.index:
        return fn(*args)
    torch.cuda.set_device(dev.index)
    try:
        return fn(*args)
    finally:
        torch.cuda.set_device(cur)


def _need(t: torch.Tensor, name: str, dtype, dev=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor" % name)
    if t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if dev is not None and t.get_device() != dev.index:
        raise ValueError("%s is on %s, expected %s" % (name, t.device, dev))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    return t


def _out(t, name, shape, dtype, dev):
    if t is None:
        return torch.empty(shape, dtype=dtype, device=dev)
    _need(t, name, dtype, dev)
    if tuple(t.shape) != tuple(shape):
        raise ValueError("%s must have shape %s, got %s" % (name, tuple(shape), tuple(t.shape)))
    return t


def _stream_dims(x: torch.Tensor):
    if x.dim() < 2:
        raise ValueError("x must be [..., hc, d]")
    lead = tuple(x.shape[:-2])
    hc, d = int(x.shape[-2]), int(x.shape[-1])
    n = 1
    for s in lead:
        n *= int(s)
    return lead, n, hc, d


def abi_version() -> int:
    return int(lib().hc_abi_version())


@functools.lru_cache(maxsize=256)
def hc_workspace_bytes(n: int, hc: int, d: int) -> int:
    # a pure function of its arguments (hcmix.h), so it is asked once per shape
    return int(lib().hc_workspace_bytes(int(n), int(hc), int(d)))


def hc_mixes(x, w_mix, norm_eps: float = 1e-20, mixes=None, stream=None):
    """x [..., hc, d] bf16, w_mix [(2+hc)*hc, hc*d] fp32 -> mixes [..., mix_hc] fp32."""
    _need(x, "x", torch.bfloat16)
    dev = x.device
    lead, n, hc, d = _stream_dims(x)
    _need(w_mix, "w_mix", torch.float32, dev)
    mix = (2 + hc) * hc
    mixes = _out(mixes, "mixes", lead + (mix,), torch.float32, dev)
    _check(_call(dev, lib().hc_mixes, n, hc, d, float(norm_eps), _ptr(x), _ptr(w_mix),
                 _ptr(mixes), _stream(dev, stream)), "hc_mixes")
    return mixes


def hc_split_sinkhorn(mixes, hc_scale, hc_base, hc_mult: int = 4, sinkhorn_iters: int = 20,
                      eps: float = 1e-6, pre=None, post=None, comb=None, stream=None):
    """mixes [..., (2+hc)*hc] fp32 -> pre [..., hc], post [..., hc], comb [..., hc, hc]."""
    _need(mixes, "mixes", torch.float32)
    dev = mixes.device
    hc = int(hc_mult)
    mix = (2 + hc) * hc
    if mixes.shape[-1] != mix:
        raise ValueError("mixes last dim must be %d" % mix)
    lead = tuple(mixes.shape[:-1])
    n = mixes.numel() // mix
    _need(hc_scale, "hc_scale", torch.float32, dev)
    _need(hc_base, "hc_base", torch.float32, dev)
    pre = _out(pre, "pre", lead + (hc,), torch.float32, dev)
    post = _out(post, "post", lead + (hc,), torch.float32, dev)
    comb = _out(comb, "comb", lead + (hc, hc), torch.float32, dev)
    _check(_call(dev, lib().hc_split_sinkhorn, n, hc, int(sinkhorn_iters), float(eps),
                 _ptr(mixes), _ptr(hc_scale), _ptr(hc_base), _ptr(pre), _ptr(post), _ptr(comb),
                 _stream(dev, stream)), "hc_split_sinkhorn")
    return pre, post, comb


def hc_pre(x, pre, y=None, stream=None):
    """x [..., hc, d] bf16, pre [..., hc] fp32 -> y [..., d] bf16."""
    _need(x, "x", torch.bfloat16)
    dev = x.device
    lead, n, hc, d = _stream_dims(x)
    _need(pre, "pre", torch.float32, dev)
    if pre.numel() != n * hc:
        raise ValueError("pre must hold n*hc values")
    y = _out(y, "y", lead + (d,), torch.bfloat16, dev)
    _check(_call(dev, lib().hc_pre, n, hc, d, _ptr(x), _ptr(pre), _ptr(y), _stream(dev, stream)),
           "hc_pre")
    return y


def hc_post(out, residual, post, comb, y=None, stream=None):
    """out [..., d] bf16, residual [..., hc, d] bf16, post [..., hc], comb [..., hc, hc]
    -> y [..., hc, d] bf16 (y may be residual itself)."""
    _need(residual, "residual", torch.bfloat16)
    dev = residual.device
    lead, n, hc, d = _stream_dims(residual)
    _need(out, "out", torch.bfloat16, dev)
    if out.numel() != n * d:
        raise ValueError("out must hold n*d values")
    _need(post, "post", torch.float32, dev)
    _need(comb, "comb", torch.float32, dev)
    if post.numel() != n * hc or comb.numel() != n * hc * hc:
        raise ValueError("post/comb sizes do not match residual")
    y = _out(y, "y", lead + (hc, d), torch.bfloat16, dev)
    _check(_call(dev, lib().hc_post, n, hc, d, _ptr(out), _ptr(residual), _ptr(post), _ptr(comb),
                 _ptr(y), _stream(dev, stream)), "hc_post")
    return y


def hc_mixes_pre(x, w_mix, hc_scale, hc_base, sinkhorn_iters: int = 20, eps: float = 1e-6,
                 norm_eps: float = 1e-20, want_mixes: bool = False, mixes=None, pre=None,
                 post=None, comb=None, y=None, workspace=None, stream=None):
    """Fused mix projection + split/Sinkhorn + collapse.
    Returns (y, pre, post, comb, mixes-or-None)."""
    _need(x, "x", torch.bfloat16)
    dev = x.device
    lead, n, hc, d = _stream_dims(x)
    mix = (2 + hc) * hc
    _need(w_mix, "w_mix", torch.float32, dev)
    _need(hc_scale, "hc_scale", torch.float32, dev)
    _need(hc_base, "hc_base", torch.float32, dev)
    if want_mixes or mixes is not None:
        mixes = _out(mixes, "mixes", lead + (mix,), torch.float32, dev)
    pre = _out(pre, "pre", lead + (hc,), torch.float32, dev)
    post = _out(post, "post", lead + (hc,), torch.float32, dev)
    comb = _out(comb, "comb", lead + (hc, hc), torch.float32, dev)
    y = _out(y, "y", lead + (d,), torch.bfloat16, dev)
    wbytes = 0
    if mixes is None or hc == 8:
        # the mix numbers when not returned; at hc = 8 also W converted for
        # the tensor-core projection (hcmix.h, hc_workspace_bytes)
        wbytes = hc_workspace_bytes(n, hc, d)
        if workspace is None and wbytes:
            workspace = torch.empty(wbytes, dtype=torch.uint8, device=dev)
    if workspace is not None:
        _need(workspace, "workspace", torch.uint8, dev)
        wbytes = workspace.numel()
    _check(_call(dev, lib().hc_mixes_pre, n, hc, d, int(sinkhorn_iters), float(eps),
                 float(norm_eps), _ptr(x), _ptr(w_mix), _ptr(hc_scale), _ptr(hc_base),
                 _ptr(mixes), _ptr(pre), _ptr(post), _ptr(comb), _ptr(y), _ptr(workspace), wbytes,
                 _stream(dev, stream)), "hc_mixes_pre")
    return y, pre, post, comb, mixes


def hc_mixes_pre_norm(x, w_mix, hc_scale, hc_base, rms_weight, sinkhorn_iters: int = 20,
                      eps: float = 1e-6, norm_eps: float = 1e-20, rms_eps: float = 1e-20,
                      want_mixes: bool = False, mixes=None, pre=None, post=None, comb=None, y=None,
                      workspace=None, stream=None):
    """hc_mixes_pre whose collapsed output y is also RMS-normalised with
    rms_weight [d].  Returns (y, pre, post, comb, mixes-or-None)."""
    _need(x, "x", torch.bfloat16)
    dev = x.device
    lead, n, hc, d = _stream_dims(x)
    mix = (2 + hc) * hc
    _need(w_mix, "w_mix", torch.float32, dev)
    _need(hc_scale, "hc_scale", torch.float32, dev)
    _need(hc_base, "hc_base", torch.float32, dev)
    _need(rms_weight, "rms_weight", torch.float32, dev)
    if tuple(rms_weight.shape) != (d,):
        raise ValueError("rms_weight must have shape (%d,)" % d)
    if want_mixes or mixes is not None:
        mixes = _out(mixes, "mixes", lead + (mix,), torch.float32, dev)
    pre = _out(pre, "pre", lead + (hc,), torch.float32, dev)
    post = _out(post, "post", lead + (hc,), torch.float32, dev)
    comb = _out(comb, "comb", lead + (hc, hc), torch.float32, dev)
    y = _out(y, "y", lead + (d,), torch.bfloat16, dev)
    wbytes = 0
    if mixes is None or hc == 8:
        wbytes = hc_workspace_bytes(n, hc, d)
        if workspace is None and wbytes:
            workspace = torch.empty(wbytes, dtype=torch.uint8, device=dev)
    if workspace is not None:
        _need(workspace, "workspace", torch.uint8, dev)
        wbytes = workspace.numel()
    _check(_call(dev, lib().hc_mixes_pre_norm, n, hc, d, int(sinkhorn_iters), float(eps),
                 float(norm_eps), _ptr(x), _ptr(w_mix), _ptr(hc_scale), _ptr(hc_base),
                 _ptr(rms_weight), float(rms_eps), _ptr(mixes), _ptr(pre), _ptr(post), _ptr(comb),
                 _ptr(y), _ptr(workspace), wbytes, _stream(dev, stream)), "hc_mixes_pre_norm")
    return y, pre, post, comb, mixes


def hc_post_mixes_pre(out, residual, post, comb, w_mix, hc_scale, hc_base,
                      sinkhorn_iters: int = 20, eps: float = 1e-6, norm_eps: float = 1e-20,
                      x_next=None, want_mixes: bool = False, mixes=None, pre=None,
                      post_next=None, comb_next=None, y=None, workspace=None, stream=None):
    """hc_post of one sublayer and hc_mixes_pre of the next in one call:
    x_next = hc_post(out, residual, post, comb) (x_next may be residual), then
    the next sublayer's (y, pre, post, comb[, mixes]) from x_next with its
    parameters w_mix, hc_scale, hc_base.
    Returns (x_next, y, pre, post, comb, mixes-or-None)."""
    _need(residual, "residual", torch.bfloat16)
    dev = residual.device
    lead, n, hc, d = _stream_dims(residual)
    _need(out, "out", torch.bfloat16, dev)
    if out.numel() != n * d:
        raise ValueError("out must hold n*d values")
    _need(post, "post", torch.float32, dev)
    _need(comb, "comb", torch.float32, dev)
    if post.numel() != n * hc or comb.numel() != n * hc * hc:
        raise ValueError("post/comb sizes do not match residual")
    mix = (2 + hc) * hc
    _need(w_mix, "w_mix", torch.float32, dev)
    _need(hc_scale, "hc_scale", torch.float32, dev)
    _need(hc_base, "hc_base", torch.float32, dev)
    x_next = _out(x_next, "x_next", lead + (hc, d), torch.bfloat16, dev)
    if want_mixes or mixes is not None:
        mixes = _out(mixes, "mixes", lead + (mix,), torch.float32, dev)
    pre = _out(pre, "pre", lead + (hc,), torch.float32, dev)
    post_next = _out(post_next, "post_next", lead + (hc,), torch.float32, dev)
    comb_next = _out(comb_next, "comb_next", lead + (hc, hc), torch.float32, dev)
    y = _out(y, "y", lead + (d,), torch.bfloat16, dev)
    wbytes = 0
    if mixes is None or hc == 8:
        wbytes = hc_workspace_bytes(n, hc, d)
        if workspace is None and wbytes:
            workspace = torch.empty(wbytes, dtype=torch.uint8, device=dev)
    if workspace is not None:
        _need(workspace, "workspace", torch.uint8, dev)
        wbytes = workspace.numel()
    _check(_call(dev, lib().hc_post_mixes_pre, n, hc, d, _ptr(out), _ptr(residual), _ptr(post),
                 _ptr(comb), _ptr(x_next), int(sinkhorn_iters), float(eps), float(norm_eps),
                 _ptr(w_mix), _ptr(hc_scale), _ptr(hc_base), _ptr(mixes), _ptr(pre),
                 _ptr(post_next), _ptr(comb_next), _ptr(y), _ptr(workspace), wbytes,
                 _stream(dev, stream)), "hc_post_mixes_pre")
    return x_next, y, pre, post_next, comb_next, mixes


def hc_launch_count() -> int:
    """Kernels the library has enqueued in this process since it was loaded."""
    return int(lib().hc_launch_count())


def hc_device_error(clear: bool = True) -> int:
    """The current device's error word (bit 0: a bounded wait timed out)."""
    v = ctypes.c_uint(0)
    _check(lib().hc_device_error(ctypes.byref(v), 1 if clear else 0), "hc_device_error")
    return int(v.value)


def hc_selftest_wait_timeout(limit_ns: int = 1000000, device=None, stream=None) -> None:
    """Enqueues the library's bounded-wait self-test: a wait that can only
    time out, after which hc_device_error() reports bit 0."""
    dev = torch.device("cuda", torch.cuda.current_device() if device is None else device)
    _check(_call(dev, lib().hc_selftest_wait_timeout, int(limit_ns), _stream(dev, stream)),
           "hc_selftest_wait_timeout")
