"""Seeded synthetic inputs for the MoE FFN hot path.

This module only draws random tensors with the shapes and distributions of
the workloads; it holds none of the method's arithmetic.  Both the CUDA path
(bench, GPU tests) and the CPU oracle's tests take their inputs from here.

Workloads (all seeded with 0; tensors are drawn in the fixed order
logits, x, W_gate, W_up, W_down, dY from one generator on the target device):

  tiny          T=64    H=128  F=256   E=8   k=2
  fine_grained  T=4096  H=2048 F=1408  E=64  k=6
  mixtral       T=8192  H=4096 F=14336 E=8   k=2   (forward + backward)
  skewed        T=16384 H=4096 F=2048  E=128 k=8   (Zipf-like expert bias)
  dsv3_mxfp8    T=8192  H=7168 F=2048  E=256 k=8   (MXFP8 forward)

x ~ N(0,1) bf16, weights ~ N(0, 0.02) bf16, router logits ~ N(0,1) fp32,
dY ~ N(0,1) bf16.  The skewed workload adds a per-expert bias
b_e = 3*ln(1/rank_e^1.2) with rank = randperm(E, seed 0) + 1 drawn on the CPU,
and sets b_e = -inf for the 16 experts with e % 8 == 7 (zero-token experts).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, asdict

import torch

__all__ = ["MoeShape", "CONFIGS", "make_inputs", "skew_bias", "small_shape"]


@dataclass(frozen=True)
class MoeShape:
    name: str
    T: int
    H: int
    F: int
    E: int
    k: int
    skew: bool = False
    backward: bool = False
    mxfp8: bool = False
    router: str = "softmax"   # or "sigmoid" (sigmoid scores + expert routing bias)
    weight_at: str = "combine"   # where the router weight is applied: combine, fc1 or fc2

    @property
    def R(self) -> int:
        return self.T * self.k

    def asdict(self) -> dict:
        return asdict(self)


CONFIGS: dict[str, MoeShape] = {
    "tiny": MoeShape("tiny", T=64, H=128, F=256, E=8, k=2),
    "fine_grained": MoeShape("fine_grained", T=4096, H=2048, F=1408, E=64, k=6),
    "mixtral": MoeShape("mixtral", T=8192, H=4096, F=14336, E=8, k=2, backward=True),
    "skewed": MoeShape("skewed", T=16384, H=4096, F=2048, E=128, k=8, skew=True),
    "dsv3_mxfp8": MoeShape("dsv3_mxfp8", T=8192, H=7168, F=2048, E=256, k=8, mxfp8=True),
}


def small_shape(name: str, T: int, H: int, F: int, E: int, k: int, **kw) -> MoeShape:
    """A custom (usually small) shape with the same distributions."""
    return MoeShape(name, T=T, H=H, F=F, E=E, k=k, **kw)


def skew_bias(E: int, seed: int = 0) -> torch.Tensor:
    """Per-expert logit bias of the skewed workload, fp32 [E] on the CPU.

    b_e = 3 * ln(1 / rank_e**1.2), rank = randperm(E) + 1 (seeded CPU draw);
    experts with e % 8 == 7 get -inf so that they receive no tokens.
    """
    g = torch.Generator(device="cpu").manual_seed(seed)
    rank = torch.randperm(E, generator=g).to(torch.float64) + 1.0
    b = 3.0 * torch.log(1.0 / rank.pow(1.2))
    b[torch.arange(E) % 8 == 7] = -math.inf
    return b.to(torch.float32)


def make_inputs(shape: MoeShape, device="cpu", seed: int = 0, with_dy: bool | None = None,
                weights: bool = True, with_expert_bias: bool = False) -> dict[str, torch.Tensor]:
    """Draw the inputs of one workload on `device`.

    Returns a dict with logits fp32 [T,E], x bf16 [T,H], W_gate/W_up bf16
    [E,H,F], W_down bf16 [E,F,H] and (if requested) dY bf16 [T,H] and an
    expert routing bias fp32 [E] ~ N(0, 0.05^2) for the sigmoid router, drawn
    last so that the other tensors do not depend on it.  Weights are
    drawn one expert at a time so that large workloads never hold an fp32
    copy of the whole weight set.
    """
    device = torch.device(device)
    if with_dy is None:
        with_dy = shape.backward
    g = torch.Generator(device=device).manual_seed(seed)
    T, H, F, E = shape.T, shape.H, shape.F, shape.E
    out: dict[str, torch.Tensor] = {}
    logits = torch.randn(T, E, generator=g, device=device, dtype=torch.float32)
    if shape.skew:
        logits += skew_bias(E, seed).to(device)
    out["logits"] = logits
    out["x"] = torch.randn(T, H, generator=g, device=device, dtype=torch.bfloat16)
    if weights:
        for name, (a, b) in (("W_gate", (H, F)), ("W_up", (H, F)), ("W_down", (F, H))):
            w = torch.empty(E, a, b, device=device, dtype=torch.bfloat16)
            for e in range(E):
                w[e] = torch.randn(a, b, generator=g, device=device, dtype=torch.bfloat16) * 0.02
            out[name] = w
    if with_dy:
        out["dY"] = torch.randn(T, H, generator=g, device=device, dtype=torch.bfloat16)
    if with_expert_bias:
        out["expert_bias"] = torch.randn(E, generator=g, device=device, dtype=torch.float32) * 0.05
    return out
