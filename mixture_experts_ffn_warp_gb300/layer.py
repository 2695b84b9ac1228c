"""The whole forward hot path (A1 route -> A2 permute -> A3/A4 FFN -> A5 combine)
with every buffer allocated once, so a step enqueues kernels only.

Follows the MoE block dataflow of "[Draft][JAX] MoE block optimization"
(diagram: route tokens, dispatch, fused grouped GEMM + SwiGLU, down
projection, combine), on one GPU with the dispatch/combine done by the
permute and combine kernels.
"""
from __future__ import annotations

import torch

from ._binding import (Permutation, Workspace, moe_grouped_fc1_swiglu, moe_grouped_fc2, moe_permute,
                       moe_route_topk, moe_unpermute_combine, rows_capacity)


class MoeForward:
    """Pre-allocated forward pass for fixed (T, H, F, E, k)."""

    def __init__(self, T: int, H: int, F: int, E: int, k: int, device="cuda", align: int = 1,
                 keep_fc1_c: bool = False):
        self.T, self.H, self.F, self.E, self.k, self.align = T, H, F, E, k, align
        dev = torch.device(device)
        self.device = dev
        self.ws = Workspace(T, E, k, dev)
        cap = rows_capacity(T, k, E, align)
        self.rows_cap = cap
        self.topk_idx = torch.empty(T, k, dtype=torch.int32, device=dev)
        self.topk_w = torch.empty(T, k, dtype=torch.float32, device=dev)
        self.perm = Permutation(
            x_perm=torch.empty(cap, H, dtype=torch.bfloat16, device=dev),
            dst_of_route=torch.empty(T, k, dtype=torch.int32, device=dev),
            src_of_row=torch.empty(cap, dtype=torch.int32, device=dev),
            group_sizes=torch.empty(E, dtype=torch.int32, device=dev),
            group_offsets=torch.empty(E + 1, dtype=torch.int32, device=dev),
            rows_cap=cap, align=align)
        self.h = torch.empty(cap, F, dtype=torch.bfloat16, device=dev)
        self.y_perm = torch.empty(cap, H, dtype=torch.float32, device=dev)
        self.fc1_c = torch.empty(cap, 2 * F, dtype=torch.bfloat16, device=dev) if keep_fc1_c else None
        self.out = torch.empty(T, H, dtype=torch.bfloat16, device=dev)

    # the steps, each one launch group on the current stream
    def route(self, logits, stream=None):
        moe_route_topk(logits, self.k, self.topk_idx, self.topk_w, stream=stream)

    def permute(self, x, stream=None):
        moe_permute(x, self.topk_idx, self.E, self.ws, self.align, out=self.perm, stream=stream)

    def fc1(self, W_gate, W_up, stream=None):
        moe_grouped_fc1_swiglu(self.perm.x_perm, W_gate, W_up, self.perm.group_offsets, self.ws, self.h,
                               self.fc1_c, stream=stream)

    def fc2(self, W_down, stream=None):
        moe_grouped_fc2(self.h, W_down, self.perm.group_offsets, self.ws, self.y_perm, stream=stream)

    def ffn(self, W_gate, W_up, W_down, stream=None):
        self.fc1(W_gate, W_up, stream)
        self.fc2(W_down, stream)

    def combine(self, stream=None):
        moe_unpermute_combine(self.y_perm, self.perm.dst_of_route, self.topk_w, out=self.out, stream=stream)

    def __call__(self, x, logits, W_gate, W_up, W_down, stream=None) -> torch.Tensor:
        self.route(logits, stream)
        self.permute(x, stream)
        self.ffn(W_gate, W_up, W_down, stream)
        self.combine(stream)
        return self.out


def moe_forward(x, logits, W_gate, W_up, W_down, k: int, align: int = 1, keep_fc1_c: bool = False):
    """One-shot forward (allocates its buffers); returns (out, MoeForward)."""
    T, H = x.shape
    E, _, F = W_gate.shape
    m = MoeForward(T, H, F, E, k, x.device, align, keep_fc1_c)
    return m(x, logits, W_gate, W_up, W_down), m
