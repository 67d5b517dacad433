"""Seeded synthetic inputs for the routed MoE FFN layer.

This module is shared by the oracle's tests and the CUDA library's tests and
benchmark, and it holds none of the layer's arithmetic: it only draws inputs.

Recipe (the pages print no tensors, so these stand in for the real model's):
  * x       bf16 [T, H]     ~ N(0, 1)
  * W_gate  bf16 [E, I, H]  ~ N(0, 0.02^2)  (fp32 normal, rounded to bf16)
  * W_up    bf16 [E, I, H]  ~ N(0, 0.02^2)
  * W_down  bf16 [E, H, I]  ~ N(0, 0.02^2)
  * logits  fp32 [T, E]     ~ N(0, 1) + b_e
    with an optional Zipf-skewed expert bias b_e = -s * ln(rank_e), rank a
    seeded random permutation of 1..E (s = 1.1 for the skewed workloads), so
    expert popularity falls off like rank^-s.
Seeds: x uses ``seed``; each expert matrix has its own generator derived
from (seed, layer, expert, matrix) so single experts can be drawn alone; logits
``seed + 2000 + layer + 7919 * rep`` (``rep`` rotates independent logit sets
so repeated timing runs do not hit the same experts in L2), the Zipf ranks
``seed + 3000 + layer``.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Shape:
    T: int
    E: int
    k: int
    H: int
    I: int

    @property
    def P(self) -> int:
        return self.T * self.k


# The workloads the pages describe, as (name, shape, zipf exponent, layers).
TINY = Shape(T=64, E=16, k=2, H=512, I=256)
DECODE_B1 = Shape(T=1, E=384, k=8, H=4096, I=2048)
DECODE_B4 = Shape(T=4, E=384, k=8, H=4096, I=2048)
PREFILL = Shape(T=16384, E=384, k=8, H=4096, I=2048)
OFFLOAD = Shape(T=16384, E=384, k=8, H=2048, I=1024)
DECODE_SWEEP_BATCHES = (1, 2, 4, 8, 16, 24)
ZIPF_S = 1.1


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def make_x(T: int, H: int, seed: int = 0, device="cpu") -> torch.Tensor:
    g = _gen(seed, device)
    return torch.randn((T, H), generator=g, device=device,
                       dtype=torch.float32).to(torch.bfloat16)


def _expert_seed(seed: int, layer: int, e: int, which: int) -> int:
    # One generator per (layer, expert, matrix), so any single expert can be
    # drawn on its own.
    return ((seed + 1000 + layer) * 1_000_003 + e) * 4 + which


def make_expert(e: int, H: int, I: int, seed: int = 0, layer: int = 0, device="cpu",
                std: float = 0.02):
    """Expert e's (Wg [I, H], Wu [I, H], Wd [H, I]) in bf16."""
    out = []
    for which, shp in enumerate(((I, H), (I, H), (H, I))):
        g = _gen(_expert_seed(seed, layer, e, which), device)
        out.append((torch.randn(shp, generator=g, device=device, dtype=torch.float32)
                    * std).to(torch.bfloat16))
    return tuple(out)


def make_weights(E: int, H: int, I: int, seed: int = 0, layer: int = 0,
                 device="cpu", std: float = 0.02):
    """Returns (Wg [E, I, H], Wu [E, I, H], Wd [E, H, I]) in bf16; expert e
    equals make_expert(e, ...) drawn on the same device."""
    Wg = torch.empty((E, I, H), dtype=torch.bfloat16, device=device)
    Wu = torch.empty((E, I, H), dtype=torch.bfloat16, device=device)
    Wd = torch.empty((E, H, I), dtype=torch.bfloat16, device=device)
    for e in range(E):
        Wg[e], Wu[e], Wd[e] = make_expert(e, H, I, seed, layer, device, std)
    return Wg, Wu, Wd


def zipf_bias(E: int, s: float, seed: int = 0, layer: int = 0) -> torch.Tensor:
    """b_e = -s * ln(rank_e), rank a seeded permutation of 1..E (fp32)."""
    g = _gen(seed + 3000 + layer, "cpu")
    rank = torch.randperm(E, generator=g).to(torch.float64) + 1.0
    return (-s * torch.log(rank)).to(torch.float32)


def make_logits(T: int, E: int, seed: int = 0, layer: int = 0, rep: int = 0,
                zipf_s: float | None = None, device="cpu") -> torch.Tensor:
    g = _gen(seed + 2000 + layer + 7919 * rep, device)
    lg = torch.randn((T, E), generator=g, device=device, dtype=torch.float32)
    if zipf_s:
        lg = lg + zipf_bias(E, zipf_s, seed, layer).to(device)
    return lg


def make_layer(shape: Shape, seed: int = 0, layer: int = 0, rep: int = 0,
               zipf_s: float | None = None, device="cpu"):
    """All inputs of one layer: dict with x, logits, Wg, Wu, Wd."""
    Wg, Wu, Wd = make_weights(shape.E, shape.H, shape.I, seed, layer, device)
    return dict(
        x=make_x(shape.T, shape.H, seed, device),
        logits=make_logits(shape.T, shape.E, seed, layer, rep, zipf_s, device),
        Wg=Wg, Wu=Wu, Wd=Wd,
    )


def bf16_bits(t: torch.Tensor):
    """Raw bf16 bit patterns of a tensor as a numpy uint16 array (CPU)."""
    import numpy as np
    return t.detach().to("cpu").contiguous().view(torch.int16).numpy().view(np.uint16)


def tied_logits(T: int, E: int, seed: int = 0, levels: int = 3) -> torch.Tensor:
    """Logits drawn from a handful of integer levels, so ties are frequent
    (exercises the lower-index tie-break)."""
    g = _gen(seed + 4000, "cpu")
    return torch.randint(0, levels, (T, E), generator=g).to(torch.float32)
