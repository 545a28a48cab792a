"""Full-size parity helpers for the GPU tests: the float64 oracle is run over
token chunks (bounded host memory) and compared with the GPU's results on
every token, with the statistics of every chunk summed.

Tolerances are those of ``oracle/compare.py``.  For bf16 outputs the number
of elements accepted only through the binary32 cancellation band (beyond 1 ulp
of the correctly rounded value, inside the evaluation's own error bound) is
counted and bounded: at most ``MAX_CANCEL_FRAC`` of the elements (a random
model of the binary32 evaluation gives ~2e-6 on these workloads).
"""
import numpy as np

import oracle
from oracle import compare

MAX_CANCEL_FRAC = 1e-4
CHUNK = 4096

# oracle mix numbers per (workload name, parameter set, seed offset, n):
# the projection dominates the oracle's time and several tests share it
_MIXES = {}


def bits(t):
    """uint16 bit patterns of a bf16 tensor (host numpy)."""
    import torch
    assert t.dtype == torch.bfloat16
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view("uint16")


def np64(t):
    return t.detach().cpu().double().numpy()


def oracle_mixes(key, x_bits, w, norm_eps):
    """Float64 mix numbers of every token, cached under `key`."""
    if key is not None and key in _MIXES:
        return _MIXES[key]
    n = x_bits.shape[0]
    out = np.empty((n, w.shape[0]))
    for t0 in range(0, n, CHUNK):
        t1 = min(n, t0 + CHUNK)
        out[t0:t1] = oracle.hc_mixes(x_bits[t0:t1], w, norm_eps)
    if key is not None:
        _MIXES[key] = out
    return out


class Bf16Stats:
    """Sums compare.check_bf16 statistics over chunks."""

    def __init__(self, what):
        self.what = what
        self.count = self.exact = self.within = self.cancel = 0
        self.max_ulp = 0

    def add(self, st):
        self.count += st["count"]
        self.exact += st["exact"]
        self.within += st["within_1ulp"]
        self.cancel += st["cancellation"]
        self.max_ulp = max(self.max_ulp, st["max_ulp"])

    def finish(self):
        frac = self.cancel / max(1, self.count)
        print("PARITY %s: %d elements, %d exact, %d within 1 ulp, %d in the cancellation "
              "band (%.2e), max %d ulp" % (self.what, self.count, self.exact, self.within,
                                           self.cancel, frac, self.max_ulp))
        assert frac <= MAX_CANCEL_FRAC, "%s: %d of %d elements needed the cancellation band" % (
            self.what, self.cancel, self.count)
        return self


def check_mixes_all(m_gpu, want):
    st = compare.check_mixes(m_gpu, want)
    print("PARITY mixes: %d tokens, max scaled error %.3e" % (want.shape[0], st["max_scaled"]))
    return st


def check_split_all(m_gpu, pre, post, comb, scale, base, hc, iters, eps):
    """pre/post/comb against the oracle's split + Sinkhorn of the GPU's own
    mix numbers (stage parity), every token."""
    n = m_gpu.shape[0]
    worst = dict(pre=0.0, post=0.0, comb=0.0)
    for t0 in range(0, n, 8 * CHUNK):
        t1 = min(n, t0 + 8 * CHUNK)
        o_pre, o_post, o_comb = oracle.hc_split_sinkhorn(m_gpu[t0:t1], scale, base, hc, iters,
                                                         eps)
        for name, got, want in (("pre", pre[t0:t1], o_pre), ("post", post[t0:t1], o_post),
                                ("comb", comb[t0:t1], o_comb)):
            st = compare.check_abs(got, want, 1e-5, name)
            worst[name] = max(worst[name], st["max_abs"])
    print("PARITY split (iters %d): %d tokens, max abs error pre %.2e post %.2e comb %.2e"
          % (iters, n, worst["pre"], worst["post"], worst["comb"]))
    return worst


def check_pre_all(y_bits, x_bits, pre, hc, what="hc_pre y"):
    """The collapse y against the oracle's collapse with the given pre
    (float64), every token; returns the summed statistics."""
    n = x_bits.shape[0]
    acc = Bf16Stats(what)
    for t0 in range(0, n, CHUNK):
        t1 = min(n, t0 + CHUNK)
        want, _, mag = oracle.hc_pre(x_bits[t0:t1], pre[t0:t1])
        acc.add(compare.check_bf16(y_bits[t0:t1], want, mag, hc, what))
    return acc.finish()


def check_post_all(y_bits, out_bits, res_bits, post, comb, hc, what="hc_post y"):
    n = res_bits.shape[0]
    acc = Bf16Stats(what)
    for t0 in range(0, n, CHUNK):
        t1 = min(n, t0 + CHUNK)
        want, _, mag = oracle.hc_post(out_bits[t0:t1], res_bits[t0:t1], post[t0:t1],
                                      comb[t0:t1])
        acc.add(compare.check_bf16(y_bits[t0:t1], want, mag, hc + 1, what))
    return acc.finish()


def check_norm_all(y_bits, x_bits, pre, rms_w, hc, rms_eps=1e-20, what="normalised y"):
    """The normalised collapse against the oracle's RMSNorm of the oracle's
    collapse with the GPU's pre, every token.  The GPU's row may differ from
    it by one bf16 step of the collapse (or, where the hc terms cancel, by hc
    binary32 roundings of their magnitude), scaled by the norm factor, plus
    one step of the output; away from cancellation more than 99.9% of the
    elements are within one step."""
    n = x_bits.shape[0]
    g = np.abs(np.asarray(rms_w, dtype=np.float64))
    count = near = 0
    worst = 0.0
    for t0 in range(0, n, CHUNK):
        t1 = min(n, t0 + CHUNK)
        _, yc_bits, mag = oracle.hc_pre(x_bits[t0:t1], pre[t0:t1])
        out_want, want_bits = oracle.hc_rmsnorm(yc_bits, rms_w, rms_eps)
        yc = oracle.bf16_bits_to_f64(yc_bits)
        inv = 1.0 / np.sqrt((yc ** 2).mean(axis=1, keepdims=True) + rms_eps)
        got = oracle.bf16_bits_to_f64(y_bits[t0:t1])
        allowed = (g * inv * (compare.bf16_ulp(yc) + hc * 2.0 ** -24 * mag) +
                   compare.bf16_ulp(out_want) + 1e-5 * np.abs(out_want))
        err = np.abs(got - out_want)
        assert np.all(err <= allowed), (t0, float((err / allowed).max()))
        worst = max(worst, float((err / allowed).max()))
        count += err.size
        near += int(np.sum(np.abs(compare.bf16_key(y_bits[t0:t1]) -
                                  compare.bf16_key(want_bits)) <= 1))
    print("PARITY %s: %d elements, %d within one bf16 step (%.6f), worst error %.3f of the "
          "allowance" % (what, count, near, near / count, worst))
    assert near / count > 0.999
    return near / count
