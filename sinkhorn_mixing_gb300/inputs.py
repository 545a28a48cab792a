"""Seeded synthetic inputs for the hyper-connection mixing path.

This module holds the workload recipes and the random draws only -- none of
the method's arithmetic -- so that the CUDA path and the float64 oracle can be
fed identical inputs without sharing any other code.

Recipes (distributions written N(mean, variance)):
  * streams x (and the residual, when separate): N(0, 1) in fp32, optionally
    times a per-token scale exp(U(ln lo, ln hi)) applied to all hc copies,
    then rounded to bf16 (nearest-even);
  * W_mix: fp32 [(2+hc)*hc, hc*d] ~ N(0, 1/(hc*d));
  * hc_scale: fp32 [3] ~ U(lo, hi);  hc_base: fp32 [(2+hc)*hc] ~ N(0, var);
  * sublayer output ``out``: bf16 [n, d] from N(0, 1).
The shapes and constants are those of the "DeepSeek V4.1" model config
(dim 5120, hc_mult 4, hc_sinkhorn_iters 20, hc_eps 1e-6, norm_eps 1e-20).
"""
from dataclasses import dataclass, field
from typing import Optional, Tuple

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    config_id: int
    B: int
    T: int
    hc: int
    d: int
    token_scale: Optional[Tuple[float, float]] = None  # log-uniform range
    base_var: float = 1.0
    scale_range: Tuple[float, float] = (0.5, 2.0)
    iters: Tuple[int, ...] = (20,)
    separate_residual: bool = False
    eps: float = 1e-6
    norm_eps: float = 1e-20

    @property
    def n(self) -> int:
        return self.B * self.T

    @property
    def mix_hc(self) -> int:
        return (2 + self.hc) * self.hc

    @property
    def F(self) -> int:
        return self.hc * self.d

    @property
    def seed(self) -> int:
        return 1000 + self.config_id


WORKLOADS = {
    "tiny": Workload("tiny", 0, 1, 8, 4, 64, separate_residual=True),
    "decode": Workload("decode", 1, 64, 1, 4, 5120, token_scale=(0.1, 10.0)),
    "prefill": Workload("prefill", 2, 1, 4096, 4, 5120, token_scale=(0.1, 10.0)),
    "large": Workload("large", 3, 8, 8192, 4, 5120, token_scale=(1e-3, 1e3)),
    "stress": Workload("stress", 4, 4, 16384, 8, 5120, base_var=5.0,
                       scale_range=(2.0, 8.0), iters=(1, 20, 50)),
}


def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def make_streams(wl: Workload, n: Optional[int] = None, device="cpu",
                 seed_offset: int = 0, chunk: int = 4096):
    """x (and residual) bf16 [n, hc, d] and out bf16 [n, d].

    Drawn in token chunks so that the fp32 intermediate stays small.  Tokens
    are a pure function of (seed, chunk index), so a prefix of a longer draw
    equals the shorter draw.
    """
    n = wl.n if n is None else n
    dev = torch.device(device)
    x = torch.empty((n, wl.hc, wl.d), dtype=torch.bfloat16, device=dev)
    res = (torch.empty_like(x) if wl.separate_residual else None)
    out = torch.empty((n, wl.d), dtype=torch.bfloat16, device=dev)
    for ci, t0 in enumerate(range(0, n, chunk)):
        t1 = min(n, t0 + chunk)
        g = _gen(dev, wl.seed * 1_000_003 + seed_offset * 7919 + ci)
        v = torch.randn((t1 - t0, wl.hc, wl.d), generator=g, device=dev)
        if wl.token_scale is not None:
            lo, hi = wl.token_scale
            u = torch.rand((t1 - t0, 1, 1), generator=g, device=dev)
            lnlo = torch.log(torch.tensor(lo, device=dev))
            lnhi = torch.log(torch.tensor(hi, device=dev))
            v = v * torch.exp(lnlo + (lnhi - lnlo) * u)
        x[t0:t1] = v.to(torch.bfloat16)
        if res is not None:
            res[t0:t1] = torch.randn((t1 - t0, wl.hc, wl.d), generator=g,
                                     device=dev).to(torch.bfloat16)
        out[t0:t1] = torch.randn((t1 - t0, wl.d), generator=g,
                                 device=dev).to(torch.bfloat16)
    return dict(x=x, residual=(res if res is not None else x), out=out)


def make_params(wl: Workload, param_set: int = 0, device="cpu"):
    """W_mix fp32 [mix_hc, F], hc_scale fp32 [3], hc_base fp32 [mix_hc]."""
    g = _gen(torch.device("cpu"), wl.seed * 31 + 17 + param_set)
    w = torch.randn((wl.mix_hc, wl.F), generator=g) * (1.0 / wl.F) ** 0.5
    lo, hi = wl.scale_range
    scale = lo + (hi - lo) * torch.rand((3,), generator=g)
    base = torch.randn((wl.mix_hc,), generator=g) * wl.base_var ** 0.5
    return dict(w=w.to(device), hc_scale=scale.to(device),
                hc_base=base.to(device))


def bf16_bits(t: torch.Tensor):
    """The uint16 bit patterns of a bf16 tensor, as a numpy array (host)."""
    assert t.dtype == torch.bfloat16
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view("uint16")
