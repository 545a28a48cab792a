"""Float64 CPU oracle for hyper-connection residual mixing (test infrastructure).

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package.  The GPU
library never imports, links or calls it, and it imports nothing from the GPU
library.  The arithmetic lives in ``hc_oracle.c`` (plain loops in double);
this module only marshals numpy arrays through ctypes.

Functions follow the "DeepSeek V4.1" model-atlas pages:
  * ``hc_mixes``           -- "Mix projection" page, formula for m, Block.hc_mixes
  * ``hc_split_sinkhorn``  -- "Reading weights" page, pre formula and the
                              hc_split_sinkhorn kernel
  * ``hc_pre``/``hc_post`` -- "Mix projection" page, Block.hc_pre / Block.hc_post
Every function is pinned by tests in ``tests/test_oracle_pins.py``.
"""
import ctypes
import os

import numpy as np

from . import build as _build

_lib = None


def _load():
    global _lib
    if _lib is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        P = ctypes.c_void_p
        i64, i32, f64 = ctypes.c_int64, ctypes.c_int, ctypes.c_double
        lib.orc_bf16_to_double.argtypes = [ctypes.c_uint16]
        lib.orc_bf16_to_double.restype = f64
        lib.orc_double_to_bf16.argtypes = [f64]
        lib.orc_double_to_bf16.restype = ctypes.c_uint16
        lib.orc_round_bf16_array.argtypes = [i64, P, P]
        lib.orc_round_bf16_array.restype = None
        lib.orc_hc_mixes.argtypes = [i64, i32, i64, f64, P, P, P, P]
        lib.orc_hc_split_sinkhorn.argtypes = [i64, i32, i32, f64, P, P, P, P, P, P]
        lib.orc_hc_pre.argtypes = [i64, i32, i64, P, P, P, P, P]
        lib.orc_hc_post.argtypes = [i64, i32, i64, P, P, P, P, P, P, P]
        lib.orc_hc_rmsnorm.argtypes = [i64, i64, P, P, f64, P, P]
        lib.orc_num_threads.restype = i32
        lib.orc_set_num_threads.argtypes = [i32]
        for f in ("orc_hc_mixes", "orc_hc_split_sinkhorn", "orc_hc_pre",
                  "orc_hc_post", "orc_hc_rmsnorm", "orc_set_num_threads"):
            getattr(lib, f).restype = None
        _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def num_threads() -> int:
    return _load().orc_num_threads()


def set_num_threads(k: int) -> None:
    _load().orc_set_num_threads(int(k))


def bf16_bits_to_f64(bits) -> np.ndarray:
    """Exact decode of bf16 bit patterns (uint16) to float64."""
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def f64_to_bf16_bits(v) -> np.ndarray:
    """Round float64 values to bf16 bit patterns, nearest-even, in one step."""
    v = np.ascontiguousarray(v, dtype=np.float64)
    out = np.empty(v.shape, dtype=np.uint16)
    _load().orc_round_bf16_array(v.size, _ptr(v), _ptr(out))
    return out


def hc_mixes(x_bits, w, norm_eps=1e-20, return_rms_inv=False):
    """x_bits: uint16 [n, hc, d]; w: float32 [(2+hc)*hc, hc*d] -> float64 [n, mix_hc]."""
    x = _c(x_bits, np.uint16)
    n, hc, d = x.shape
    mix_hc = (2 + hc) * hc
    w = _c(w, np.float32)
    assert w.shape == (mix_hc, hc * d), w.shape
    mixes = np.empty((n, mix_hc), dtype=np.float64)
    r = np.empty((n,), dtype=np.float64)
    _load().orc_hc_mixes(n, hc, d, float(norm_eps), _ptr(x), _ptr(w), _ptr(mixes), _ptr(r))
    return (mixes, r) if return_rms_inv else mixes


def hc_split_sinkhorn(mixes, hc_scale, hc_base, hc=4, iters=20, eps=1e-6):
    """mixes: [n, (2+hc)*hc] (any float dtype, converted exactly to float64)
    -> pre [n, hc], post [n, hc], comb [n, hc, hc], all float64."""
    m = _c(mixes, np.float64)
    n = m.shape[0]
    mix_hc = (2 + hc) * hc
    assert m.shape == (n, mix_hc), m.shape
    assert 1 <= hc <= 16 and iters >= 1
    s = _c(hc_scale, np.float32)
    b = _c(hc_base, np.float32)
    assert s.shape == (3,) and b.shape == (mix_hc,)
    pre = np.empty((n, hc))
    post = np.empty((n, hc))
    comb = np.empty((n, hc, hc))
    _load().orc_hc_split_sinkhorn(n, hc, int(iters), float(eps), _ptr(m), _ptr(s),
                                  _ptr(b), _ptr(pre), _ptr(post), _ptr(comb))
    return pre, post, comb


def hc_pre(x_bits, pre):
    """x_bits: uint16 [n, hc, d]; pre: [n, hc] -> (y float64 [n, d],
    y bf16 bits [n, d], term magnitude sum float64 [n, d])."""
    x = _c(x_bits, np.uint16)
    n, hc, d = x.shape
    p = _c(pre, np.float64)
    assert p.shape == (n, hc)
    y = np.empty((n, d))
    yb = np.empty((n, d), dtype=np.uint16)
    mag = np.empty((n, d))
    _load().orc_hc_pre(n, hc, d, _ptr(x), _ptr(p), _ptr(y), _ptr(yb), _ptr(mag))
    return y, yb, mag


def hc_rmsnorm(y_bits, weight, eps=1e-20):
    """RMSNorm of the bf16 collapse output (standard form; not on the pages):
    y_bits uint16 [n, d], weight float32 [d] -> (out float64 [n, d], out bf16
    bits [n, d])."""
    y = _c(y_bits, np.uint16)
    n, d = y.shape
    g = _c(weight, np.float32)
    assert g.shape == (d,)
    out = np.empty((n, d))
    ob = np.empty((n, d), dtype=np.uint16)
    _load().orc_hc_rmsnorm(n, d, _ptr(y), _ptr(g), float(eps), _ptr(out), _ptr(ob))
    return out, ob


def hc_post(out_bits, res_bits, post, comb):
    """out_bits: uint16 [n, d]; res_bits: uint16 [n, hc, d]; post [n, hc];
    comb [n, hc, hc] -> (y float64 [n, hc, d], y bf16 bits, magnitude sum)."""
    o = _c(out_bits, np.uint16)
    r = _c(res_bits, np.uint16)
    n, hc, d = r.shape
    assert o.shape == (n, d)
    p = _c(post, np.float64)
    cb = _c(comb, np.float64)
    assert p.shape == (n, hc) and cb.shape == (n, hc, hc)
    y = np.empty((n, hc, d))
    yb = np.empty((n, hc, d), dtype=np.uint16)
    mag = np.empty((n, hc, d))
    _load().orc_hc_post(n, hc, d, _ptr(o), _ptr(r), _ptr(p), _ptr(cb), _ptr(y),
                        _ptr(yb), _ptr(mag))
    return y, yb, mag


def chain(x_bits, w, hc_scale, hc_base, out_bits, res_bits=None, iters=20,
          eps=1e-6, norm_eps=1e-20):
    """The whole path in float64: mixes -> split/Sinkhorn -> pre collapse ->
    post expansion (res defaults to the stream x itself, as in a block)."""
    x = _c(x_bits, np.uint16)
    hc = x.shape[1]
    mixes = hc_mixes(x, w, norm_eps)
    pre, post, comb = hc_split_sinkhorn(mixes, hc_scale, hc_base, hc, iters, eps)
    y_pre, y_pre_bits, _ = hc_pre(x, pre)
    res = x if res_bits is None else res_bits
    y_post, y_post_bits, _ = hc_post(out_bits, res, post, comb)
    return dict(mixes=mixes, pre=pre, post=post, comb=comb, y_pre=y_pre,
                y_pre_bits=y_pre_bits, y_post=y_post, y_post_bits=y_post_bits)
