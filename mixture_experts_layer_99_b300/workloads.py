"""Seeded synthetic workloads for the top-k routed MoE FFN layer.

This module only draws inputs. It holds none of the layer's arithmetic, so the
CUDA path and the CPU oracle can both take their inputs from here without
sharing any of the computation they are compared on.

The five workloads follow the shapes the MoE pages use:

* ``ref_fp32``    - small fp32 case (T=256, d=64, E=4, k=2, GELU 64->256->64,
  zero expert biases, capacity factor 1.25).
* ``switch_top1`` - Switch-style top-1 routing ("Switch Gating" in the
  intelliparadigm tutorial, section 2.2), bf16, T=8192, d=1024, E=8, GELU
  1024->4096->1024, c=1.0.
* ``mixtral``     - 8 experts top-2, SwiGLU 4096->14336->4096 (the
  4096->14336 expert of the lpnh.cn guide, section 3.2), bf16, T=16384, no drops
  (c = E/k).
* ``longtail``    - 64 experts top-2, SwiGLU 2048->1408->2048, bf16, T=32768,
  c=2.0, a fixed Zipf-like router bias b_i = 2*log(1/(i+1)) and Gumbel noise
  -log(-log(u)) supplied as an input tensor (lpnh.cn guide, sections 2.2/3.3).
* ``decode``      - decode-like step, T=64, d=4096, E=64, k=2, SwiGLU
  4096->1408->4096, no drops.
* ``sweep_e16_k4`` - the 16-expert, top-4 point of the expert-count x
  active-count sweep of the intelliparadigm tutorial (section 2.1), with the
  switch layer's total hidden width split over 16 experts (GELU
  1024->2048->1024), c=1.25, and Gaussian router noise of standard deviation
  0.05 added to the logits (the ``noise_std`` of the kwkr.cn MoE article,
  section 3.3, whose typical range is 0.01 to 0.1).
* ``sweep_std_noise`` - the same layer with the refined noise of that
  section: standard normal noise whose strength is 0.1 times each token's
  standard deviation of its logits (the router applies the scaling; the
  drawn tensor is N(0, 1)).

Draw order (one ``torch.Generator('cpu')`` per workload, seeded): x, W_g, W1,
W3 (SwiGLU only), W2, then the router noise (u for Gumbel noise, a
standard normal draw scaled by ``noise_std``, or an unscaled standard normal
draw for std-scaled noise). All normal draws are fp32
``randn``; weights are scaled by 1/sqrt(fan_in) and then cast to the workload
dtype. Weights use the ``nn.Linear`` storage convention [out, in]:
W_g [E, d], W1 and W3 [E, H, d], W2 [E, d, H].
"""
from __future__ import annotations

import dataclasses
import math
from fractions import Fraction
from typing import Optional

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    T: int
    d: int
    E: int
    k: int
    H: int
    act: str                 # "gelu" or "swiglu"
    dtype: str               # "f32" or "bf16"
    c: Fraction              # capacity factor, exact
    expert_bias: bool = False    # b1 [E,H], b2 [E,d] present (zeros)
    router_bias: Optional[str] = None   # None or "zipf"
    noise: Optional[str] = None         # None, "gumbel", "gaussian" or "gaussian_std"
    noise_std: float = 0.0              # std of "gaussian" noise; the scale of "gaussian_std"
    tau: float = 1.0
    seed: int = 0
    shared_H: int = 0                   # > 0: a shared expert of this hidden size

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    @property
    def elem_bytes(self):
        return 4 if self.dtype == "f32" else 2

    @property
    def nmat(self):
        return 3 if self.act == "swiglu" else 2

    @property
    def noise_scale(self) -> float:
        """The router's noise_scale: > 0 for noise whose strength follows each
        token's logit standard deviation ("gaussian_std"), else 0 (the noise
        tensor is added as drawn)."""
        return self.noise_std if self.noise == "gaussian_std" else 0.0

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    "ref_fp32": Workload("ref_fp32", T=256, d=64, E=4, k=2, H=256, act="gelu",
                         dtype="f32", c=Fraction(5, 4), expert_bias=True),
    "switch_top1": Workload("switch_top1", T=8192, d=1024, E=8, k=1, H=4096,
                            act="gelu", dtype="bf16", c=Fraction(1)),
    "mixtral": Workload("mixtral", T=16384, d=4096, E=8, k=2, H=14336,
                        act="swiglu", dtype="bf16", c=Fraction(4)),
    "longtail": Workload("longtail", T=32768, d=2048, E=64, k=2, H=1408,
                         act="swiglu", dtype="bf16", c=Fraction(2),
                         router_bias="zipf", noise="gumbel", tau=1.0),
    "decode": Workload("decode", T=64, d=4096, E=64, k=2, H=1408,
                       act="swiglu", dtype="bf16", c=Fraction(32)),
    "sweep_e16_k4": Workload("sweep_e16_k4", T=8192, d=1024, E=16, k=4, H=2048,
                             act="gelu", dtype="bf16", c=Fraction(5, 4),
                             noise="gaussian", noise_std=0.05),
    # the same sweep point with std-scaled router noise (strength 0.1 times
    # each token's logit standard deviation)
    "sweep_std_noise": Workload("sweep_std_noise", T=8192, d=1024, E=16, k=4, H=2048,
                                act="gelu", dtype="bf16", c=Fraction(5, 4),
                                noise="gaussian_std", noise_std=0.1),
    # the long-tail layer plus one always-on shared expert of the same width
    "longtail_shared": Workload("longtail_shared", T=32768, d=2048, E=64, k=2, H=1408,
                                act="swiglu", dtype="bf16", c=Fraction(2),
                                router_bias="zipf", noise="gumbel", tau=1.0, shared_H=1408),
}


def _randn(gen, shape, std, dtype):
    """fp32 N(0,1) draw scaled by std, then cast to ``dtype``."""
    a = torch.randn(*shape, generator=gen, dtype=torch.float32)
    if std != 1.0:
        a.mul_(std)
    return a.to(dtype)


def _randn_stacked(gen, E, rows, cols, std, dtype):
    """[E, rows, cols] drawn one expert after another (bounded host memory)."""
    out = torch.empty(E, rows, cols, dtype=dtype)
    for e in range(E):
        out[e] = _randn(gen, (rows, cols), std, dtype)
    return out


def make_inputs(w: Workload, seed: Optional[int] = None) -> dict:
    """Draw every input of one layer call on the host (CPU tensors).

    Returns a dict with x [T,d], Wg [E,d], W1 [E,H,d], W3 [E,H,d] or None,
    W2 [E,d,H], b1 [E,H] or None, b2 [E,d] or None, bias [E] fp32 or None,
    noise [T,E] fp32 or None.
    """
    seed = w.seed if seed is None else seed
    gen = torch.Generator(device="cpu").manual_seed(seed)
    dt = w.torch_dtype
    x = _randn(gen, (w.T, w.d), 1.0, dt)
    Wg = _randn(gen, (w.E, w.d), 1.0 / math.sqrt(w.d), dt)
    W1 = _randn_stacked(gen, w.E, w.H, w.d, 1.0 / math.sqrt(w.d), dt)
    W3 = (_randn_stacked(gen, w.E, w.H, w.d, 1.0 / math.sqrt(w.d), dt)
          if w.act == "swiglu" else None)
    W2 = _randn_stacked(gen, w.E, w.d, w.H, 1.0 / math.sqrt(w.H), dt)
    b1 = torch.zeros(w.E, w.H, dtype=dt) if w.expert_bias else None
    b2 = torch.zeros(w.E, w.d, dtype=dt) if w.expert_bias else None
    bias = None
    if w.router_bias == "zipf":
        i = torch.arange(w.E, dtype=torch.float64)
        bias = (2.0 * torch.log(1.0 / (i + 1.0))).to(torch.float32)
    noise = None
    if w.noise == "gumbel":
        u = torch.rand(w.T, w.E, generator=gen, dtype=torch.float64)
        u = u.clamp_(1e-12, 1.0 - 1e-12)
        noise = (-torch.log(-torch.log(u))).to(torch.float32)
    elif w.noise == "gaussian":
        noise = _randn(gen, (w.T, w.E), w.noise_std, torch.float32)
    elif w.noise == "gaussian_std":   # N(0, 1); the router scales it per token
        noise = _randn(gen, (w.T, w.E), 1.0, torch.float32)
    out = dict(x=x, Wg=Wg, W1=W1, W3=W3, W2=W2, b1=b1, b2=b2, bias=bias, noise=noise)
    if w.shared_H > 0:   # drawn last, so the routed inputs do not change
        Hs = w.shared_H
        out["shared"] = dict(
            W1=_randn(gen, (Hs, w.d), 1.0 / math.sqrt(w.d), dt),
            W3=(_randn(gen, (Hs, w.d), 1.0 / math.sqrt(w.d), dt)
                if w.act == "swiglu" else None),
            W2=_randn(gen, (w.d, Hs), 1.0 / math.sqrt(Hs), dt),
            b1=torch.zeros(Hs, dtype=dt) if w.expert_bias else None,
            b2=torch.zeros(w.d, dtype=dt) if w.expert_bias else None)
    return out


def small(w: Workload, T: int, d: int, H: int, E: Optional[int] = None,
          k: Optional[int] = None, c: Optional[Fraction] = None) -> Workload:
    """A reduced-size variant of a workload with the same structure."""
    return w.with_(T=T, d=d, H=H, E=E if E is not None else w.E,
                   k=k if k is not None else w.k, c=c if c is not None else w.c,
                   name=f"{w.name}[T{T},d{d},H{H}]")


def make_routing(T: int, E: int, k: int, seed: int = 0, skew: float = 0.0):
    """Random top-k expert ids [T, k] int32 (distinct per token) for tests of
    the stages after the router. ``skew`` > 0 tilts the choice towards low
    expert ids (ids are the k largest of u + skew * (E - i) / E, u uniform)."""
    gen = torch.Generator(device="cpu").manual_seed(seed)
    keys = torch.rand(T, E, generator=gen, dtype=torch.float64)
    if skew:
        keys = keys + skew * (E - torch.arange(E, dtype=torch.float64)) / E
    ids = torch.argsort(keys, dim=1, descending=True, stable=True)[:, :k]
    return ids.to(torch.int32).contiguous()


def make_gates(T: int, k: int, seed: int = 0):
    """Random positive gates [T, k] fp32 (rows need not sum to 1)."""
    gen = torch.Generator(device="cpu").manual_seed(seed)
    return torch.rand(T, k, generator=gen, dtype=torch.float32).add_(0.05)


def make_rows(R: int, d: int, dtype, seed: int = 0):
    """Random rows [R, d] of ``dtype`` (N(0,1))."""
    gen = torch.Generator(device="cpu").manual_seed(seed)
    return torch.randn(R, d, generator=gen, dtype=torch.float32).to(dtype)


def to_device(inp: dict, device) -> dict:
    def mv(v):
        if v is None:
            return None
        if isinstance(v, dict):
            return to_device(v, device)
        return v.to(device).contiguous()
    return {k: mv(v) for k, v in inp.items()}
