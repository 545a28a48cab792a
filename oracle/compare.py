"""Tolerance checks between GPU results and the float64 oracle (test
infrastructure, used by tests/, the smoke check and the benchmark).

Tolerances:
  * mix numbers:      |g - o| <= 1e-4 * max(|o|, 1)
  * pre, post, comb:  |g - o| <= 1e-5 (absolute), with o computed by the
                      oracle from the GPU's own mix numbers (stage parity)
  * bf16 outputs:     g within 1 bf16 ulp of the correctly rounded oracle
                      value.  Where the terms of the sum cancel, the binary32
                      evaluation itself carries an error up to
                      k * 2^-24 * sum|terms| (k = number of roundings), which
                      can exceed 1 ulp of a small result; such elements are
                      accepted when |g - o| <= 1 ulp(o) + k * 2^-24 * sum|terms|,
                      and counted separately.
"""
import numpy as np

from . import bf16_bits_to_f64, f64_to_bf16_bits

U32 = 2.0 ** -24


def bf16_key(bits):
    """Monotone integer key of bf16 bit patterns (adjacent values differ by 1)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.int64)
    mag = b & 0x7FFF
    return np.where(b & 0x8000, -mag, mag)


def bf16_ulp(v):
    a = np.abs(np.asarray(v, dtype=np.float64))
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, -126.0)
    return np.where(a > 0, 2.0 ** (e - 7), 2.0 ** -133)


def check_bf16(got_bits, want, mag, n_round, what="bf16"):
    """got_bits: uint16 GPU result; want: float64 exact oracle value; mag:
    float64 sum of |terms|; n_round: binary32 roundings on the GPU side."""
    got_bits = np.asarray(got_bits, dtype=np.uint16)
    want = np.asarray(want, dtype=np.float64)
    ref_bits = f64_to_bf16_bits(want)
    dk = np.abs(bf16_key(got_bits) - bf16_key(ref_bits))
    primary = dk <= 1
    g = bf16_bits_to_f64(got_bits)
    band = bf16_ulp(want) + n_round * U32 * np.asarray(mag, dtype=np.float64)
    secondary = np.abs(g - want) <= band
    ok = primary | secondary
    stats = dict(what=what, count=int(want.size), exact=int(np.sum(dk == 0)),
                 within_1ulp=int(np.sum(primary)), cancellation=int(np.sum(~primary & secondary)),
                 max_ulp=int(dk.max()) if dk.size else 0)
    if not np.all(ok):
        i = np.flatnonzero(~ok.ravel())[:5]
        raise AssertionError("%s: %d of %d outside tolerance; first %s: got %s want %s mag %s"
                             % (what, int(np.sum(~ok)), want.size, i.tolist(),
                                g.ravel()[i].tolist(), want.ravel()[i].tolist(),
                                np.asarray(mag).ravel()[i].tolist()))
    return stats


def check_abs(got, want, atol, what="value"):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    err = np.abs(got - want)
    if not np.all(err <= atol):
        i = int(np.argmax(err))
        raise AssertionError("%s: max abs err %.3e > %.1e at %d (got %r want %r)"
                             % (what, err.ravel()[i], atol, i, got.ravel()[i], want.ravel()[i]))
    return dict(what=what, max_abs=float(err.max()) if err.size else 0.0)


def check_mixes(got, want, rtol=1e-4, what="mixes"):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    err = np.abs(got - want) / np.maximum(np.abs(want), 1.0)
    if not np.all(err <= rtol):
        i = int(np.argmax(err))
        raise AssertionError("%s: max scaled err %.3e > %.1e at %d (got %r want %r)"
                             % (what, err.ravel()[i], rtol, i, got.ravel()[i], want.ravel()[i]))
    return dict(what=what, max_scaled=float(err.max()) if err.size else 0.0)
