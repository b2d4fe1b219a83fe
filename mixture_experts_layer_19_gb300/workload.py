"""Seeded synthetic inputs for the fused MoE layer.

This module is shared by the CUDA path's tests and benchmark and by the CPU
oracle's tests.  It holds only the input recipe (random draws and the load-skew
bias), none of the layer's arithmetic.

Recipe (one ``torch.Generator`` seeded with ``seed``; draws in this order):

* ``X``      [T, d]    N(0, 1), stored bf16.
* ``logits`` [T, E]    N(0, 1) fp32, plus a per-expert bias ``ln p_e`` with
  ``p_e`` proportional to ``rank_e ** -alpha``; ``rank`` is a seeded permutation
  of 1..E drawn right after the logits.  ``alpha = 0`` gives a uniform bias
  (no skew).  This stands in for the frontier MoE models' real routing skew.
* ``Wg``, ``Wu`` [E, F, d]  N(0, std=1/sqrt(d)), bf16, drawn expert by expert.
* ``Wd``     [E, d, F]  N(0, std=1/sqrt(F)), bf16, drawn expert by expert.
* ``dY``     [T, d]    N(0, 1), bf16 (the upstream gradient).
* ``Wr``     [E, d]    N(0, std=1/sqrt(d)), bf16, the router weight, drawn
  last and only when asked for (``router=True``), so the draws above do not
  depend on it.

The layer shape used by the pages' benchmark models is hidden 7168 and expert
width 2048 (Mixture-of-Kittens coverage, kucoin page, section 02); the weights
are random because no trained checkpoint is available.
"""
from __future__ import annotations

import math
from dataclasses import dataclass
from typing import Optional

import torch


@dataclass
class LayerShape:
    T: int
    d: int
    F: int
    E: int
    k: int

    @property
    def R(self) -> int:
        return self.T * self.k


@dataclass
class LayerInputs:
    X: torch.Tensor
    logits: torch.Tensor
    Wg: Optional[torch.Tensor]
    Wu: Optional[torch.Tensor]
    Wd: Optional[torch.Tensor]
    dY: torch.Tensor
    Wr: Optional[torch.Tensor] = None


def zipf_bias(E: int, alpha: float, gen: torch.Generator, device) -> torch.Tensor:
    """Per-expert additive logit bias ln p_e, p_e ~ rank_e^-alpha (normalised)."""
    rank = torch.randperm(E, generator=gen, device=device).to(torch.float64) + 1.0
    p = rank.pow(-float(alpha))
    p = p / p.sum()
    return p.log().to(torch.float32)


def make_inputs(shape: LayerShape, seed: int = 0, alpha: float = 0.0,
                device="cpu", weights: bool = True, router: bool = False) -> LayerInputs:
    """Draw the layer inputs on ``device`` following the recipe above."""
    T, d, F, E = shape.T, shape.d, shape.F, shape.E
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    X = torch.randn((T, d), generator=gen, device=device).to(torch.bfloat16)
    logits = torch.randn((T, E), generator=gen, device=device)
    logits = logits + zipf_bias(E, alpha, gen, device)[None, :]
    Wg = Wu = Wd = None
    if weights:
        Wg = torch.empty((E, F, d), dtype=torch.bfloat16, device=device)
        Wu = torch.empty((E, F, d), dtype=torch.bfloat16, device=device)
        Wd = torch.empty((E, d, F), dtype=torch.bfloat16, device=device)
        sg, sd = 1.0 / math.sqrt(d), 1.0 / math.sqrt(F)
        for W, s in ((Wg, sg), (Wu, sg), (Wd, sd)):
            for e in range(E):
                W[e].copy_(torch.randn(W.shape[1:], generator=gen, device=device) * s)
    dY = torch.randn((T, d), generator=gen, device=device).to(torch.bfloat16)
    Wr = None
    if router:
        Wr = (torch.randn((E, d), generator=gen, device=device) / math.sqrt(d)).to(torch.bfloat16)
    return LayerInputs(X=X, logits=logits.contiguous(), Wg=Wg, Wu=Wu, Wd=Wd, dY=dY, Wr=Wr)


def to_f64(t: torch.Tensor):
    """Exact widening of a bf16/fp32 tensor to a float64 numpy array."""
    return t.detach().to("cpu", torch.float64).numpy()
