"""Seeded synthetic inputs for the capacity-limited top-k MoE layer forward.

This module only draws random tensors; it holds none of the layer's arithmetic.
Both the CPU oracle (through the tests and the benchmark) and the CUDA library
consume the exact bytes produced here, so a parity comparison never depends on
two generators agreeing.

Recipe (one ``torch.Generator`` on the device that will hold the tensors,
seeded with the workload's seed, draws taken in this order):

1. ``x  [T, d]``      ~ N(0, 1)
2. ``Wg [E, d]``      ~ N(0, 1/d)
3. ``W1 [E, f, d]``   ~ N(0, 1/d)          (gate projection, nn.Linear out x in)
4. ``W3 [E, f, d]``   ~ N(0, 1/d)          (up projection; SwiGLU only)
5. ``W2 [E, d, f]``   ~ N(0, 1/f)          (down projection)
   (each expert weight tensor is drawn one expert at a time, expert 0 first)
6. skewed router only: a permutation ``perm`` of the E experts; expert
   ``perm[j]`` gets Zipf rank ``j + 1`` and logit bias ``-s * ln(rank)``
   (the log of a Zipf(s) pmf up to a constant, which softmax and top-k ignore).

Draws are fp32 and, for bf16 workloads, rounded to bf16 (round to nearest
even, ``Tensor.to(torch.bfloat16)``).  The router bias stays fp32.

The workloads are the synthetic stand-ins for the shapes the expert
parallelism pages talk about (Mixtral-style 8-expert top-2 layers, Switch-style
top-1 with many experts, fine-grained 64-expert layers with hot experts); the
pages name no dataset.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace
from typing import Optional

import torch

BF16 = "bf16"
F32 = "f32"
SWIGLU = "swiglu"
GELU = "gelu"


@dataclass(frozen=True)
class Workload:
    """Shape and recipe of one synthetic MoE layer."""

    name: str
    T: int
    d: int
    E: int
    D: int
    k: int
    ffn: int
    capacity_factor: float
    dtype: str = BF16
    act: str = SWIGLU
    seed: int = 0
    zipf_s: Optional[float] = None  # skewed router bias; None = no bias
    renorm: bool = False            # renormalise the k gates of a token to sum to one
    ffn_shared: int = 0             # width of a shared expert every token goes through; 0 = none
    expert_choice: bool = False     # experts take their tokens (instead of tokens their experts)
    reroute: bool = False           # a choice over capacity moves to the token's next-best expert

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


# The five workloads the layer is measured and checked on.
WORKLOADS = {
    "tiny_fp32": Workload("tiny_fp32", T=64, d=32, E=8, D=4, k=2, ffn=64,
                          capacity_factor=1.0, dtype=F32, act=GELU, seed=0),
    "mixtral_scaled": Workload("mixtral_scaled", T=4096, d=1024, E=8, D=8, k=2,
                               ffn=3584, capacity_factor=1.25, seed=1),
    "skewed_64e": Workload("skewed_64e", T=8192, d=2048, E=64, D=8, k=2,
                           ffn=1024, capacity_factor=1.0, seed=2, zipf_s=1.2),
    "switch_top1_c1.0": Workload("switch_top1_c1.0", T=16384, d=1024, E=128, D=8,
                                 k=1, ffn=4096, capacity_factor=1.0, seed=3),
    "switch_top1_c1.25": Workload("switch_top1_c1.25", T=16384, d=1024, E=128, D=8,
                                  k=1, ffn=4096, capacity_factor=1.25, seed=3),
    "switch_top1_c2.0": Workload("switch_top1_c2.0", T=16384, d=1024, E=128, D=8,
                                 k=1, ffn=4096, capacity_factor=2.0, seed=3),
    "mixtral_8x7b": Workload("mixtral_8x7b", T=32768, d=4096, E=8, D=8, k=2,
                             ffn=14336, capacity_factor=math.inf, seed=4),
}


@dataclass
class LayerInputs:
    """Tensors of one layer instance (all on one device).

    bf16 tensors have dtype ``torch.bfloat16``; fp32 ones ``torch.float32``.
    ``W3`` is None for the GeLU FFN, ``bias`` None without a router bias.
    """

    wl: Workload
    x: torch.Tensor
    Wg: torch.Tensor
    W1: torch.Tensor
    W3: Optional[torch.Tensor]
    W2: torch.Tensor
    bias: Optional[torch.Tensor]
    Ws1: Optional[torch.Tensor] = None  # shared expert [ffn_shared, d]
    Ws3: Optional[torch.Tensor] = None  # [ffn_shared, d] (SwiGLU only)
    Ws2: Optional[torch.Tensor] = None  # [d, ffn_shared]

    def to(self, device) -> "LayerInputs":
        mv = lambda t: None if t is None else t.to(device)
        return LayerInputs(self.wl, mv(self.x), mv(self.Wg), mv(self.W1),
                           mv(self.W3), mv(self.W2), mv(self.bias), mv(self.Ws1), mv(self.Ws3),
                           mv(self.Ws2))


def torch_dtype(dtype: str) -> torch.dtype:
    return {BF16: torch.bfloat16, F32: torch.float32}[dtype]


def _normal(gen, shape, std, dtype, device, per_expert=False):
    """N(0, std^2) fp32 draw, rounded to the storage dtype.

    Expert weights are drawn one expert (leading index) at a time, which
    bounds the fp32 temporary for the multi-GB weight sets.
    """
    out_dtype = torch_dtype(dtype)
    if not per_expert:
        t = torch.randn(shape, generator=gen, dtype=torch.float32, device=device)
        t.mul_(std)
        return t.to(out_dtype)
    out = torch.empty(shape, dtype=out_dtype, device=device)
    for e in range(shape[0]):
        t = torch.randn(shape[1:], generator=gen, dtype=torch.float32, device=device)
        t.mul_(std)
        out[e].copy_(t)
    return out


def make_inputs(wl: Workload, device="cpu") -> LayerInputs:
    """Draw one layer instance following the module recipe."""
    device = torch.device(device)
    gen = torch.Generator(device=device)
    gen.manual_seed(wl.seed)
    T, d, E, f = wl.T, wl.d, wl.E, wl.ffn
    x = _normal(gen, (T, d), 1.0, wl.dtype, device)
    Wg = _normal(gen, (E, d), 1.0 / math.sqrt(d), wl.dtype, device)
    W1 = _normal(gen, (E, f, d), 1.0 / math.sqrt(d), wl.dtype, device, True)
    W3 = (_normal(gen, (E, f, d), 1.0 / math.sqrt(d), wl.dtype, device, True)
          if wl.act == SWIGLU else None)
    W2 = _normal(gen, (E, d, f), 1.0 / math.sqrt(f), wl.dtype, device, True)
    bias = None
    if wl.zipf_s is not None:
        perm = torch.randperm(E, generator=gen, device=device)
        rank = torch.empty(E, dtype=torch.float64, device=device)
        rank[perm] = torch.arange(1, E + 1, dtype=torch.float64, device=device)
        bias = (-wl.zipf_s * torch.log(rank)).to(torch.float32)
    Ws1 = Ws3 = Ws2 = None
    if wl.ffn_shared:
        # drawn last, so the other tensors are the same with or without it
        fs = wl.ffn_shared
        Ws1 = _normal(gen, (fs, d), 1.0 / math.sqrt(d), wl.dtype, device)
        Ws3 = _normal(gen, (fs, d), 1.0 / math.sqrt(d), wl.dtype, device) if wl.act == SWIGLU else None
        Ws2 = _normal(gen, (d, fs), 1.0 / math.sqrt(fs), wl.dtype, device)
    return LayerInputs(wl, x, Wg, W1, W3, W2, bias, Ws1, Ws3, Ws2)
