"""The whole forward hot path (A1 route -> A2 permute -> A3/A4 FFN -> A5 combine)
with every buffer allocated once, so a step enqueues kernels only.

Follows the MoE block dataflow of "[Draft][JAX] MoE block optimization"
(diagram: route tokens, dispatch, fused grouped GEMM + SwiGLU, down
projection, combine), on one GPU with the dispatch/combine done by the
permute and combine kernels.
"""
from __future__ import annotations

import torch

from ._binding import (SCORE_SIGMOID, SCORE_SOFTMAX, Permutation, PermutationMX, Workspace, moe_combine_bwd,
                       moe_grouped_dgrad_fc1, moe_route_topk_bwd, moe_route_topk_sigmoid,
                       moe_grouped_fc1_swiglu_mxfp8, moe_grouped_fc2_mxfp8, moe_permute_mxfp8,
                       moe_dequantize_rows_mxfp8, moe_dequantize_weights_mxfp8, moe_unpermute_combine_mxfp8,
                       moe_unpermute_combine_nvfp4,
                       moe_quantize_weights_mxfp8, mx_tile_scale_bytes,
                       moe_grouped_dgrad_fc2_dswiglu, moe_grouped_fc1_swiglu, moe_grouped_fc2,
                       moe_grouped_wgrad, moe_permute, moe_route_topk, moe_unpermute_combine,
                       moe_unpermute_sum, rows_capacity)


class MoeForward:
    """Pre-allocated forward pass for fixed (T, H, F, E, k).

    router: "softmax" (softmax over the k selected logits) or "sigmoid" (sigmoid
    scores; `expert_bias` [E] fp32 takes part in the selection only; weights
    normalised by their sum + 1e-20 when `normalize`).
    weight_at: where the router weight is applied: "combine" (default), "fc1"
    (h scaled before its bf16 rounding) or "fc2" (y scaled); the early placements
    are forward only.
    out_format: "bf16" (out [T, H]), "mxfp8" (out_q E4M3 [T, H] + out_sf UE8M0
    [T, H/32]) or "nvfp4" (out_q two E2M1 codes per byte [T, H/2] + out_sf E4M3
    [T, H/16]): block-scaled encodings of the same fp32 combine sum.
    swiglu_clamp: None or (gate_lo, gate_hi, up_lo, up_hi): the SwiGLU inputs clamped to
    those inclusive bounds (the optional DeepSeek-style clamp; a MoeBackward of this layer
    uses the same bounds)."""

    def __init__(self, T: int, H: int, F: int, E: int, k: int, device="cuda", align: int = 1,
                 keep_fc1_c: bool = False, router: str = "softmax", expert_bias=None, normalize: bool = True,
                 weight_at: str = "combine", out_format: str = "bf16", swiglu_clamp=None):
        if router not in ("softmax", "sigmoid"):
            raise ValueError("router must be 'softmax' or 'sigmoid'")
        if weight_at not in ("combine", "fc1", "fc2"):
            raise ValueError("weight_at must be 'combine', 'fc1' or 'fc2'")
        self.weight_at = weight_at
        self.swiglu_clamp = None if swiglu_clamp is None else tuple(float(v) for v in swiglu_clamp)
        if self.swiglu_clamp is not None and len(self.swiglu_clamp) != 4:
            raise ValueError("swiglu_clamp is (gate_lo, gate_hi, up_lo, up_hi)")
        self.T, self.H, self.F, self.E, self.k, self.align = T, H, F, E, k, align
        self.router, self.expert_bias, self.normalize = router, expert_bias, normalize
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
        self.y_perm = torch.empty(cap, H, dtype=torch.bfloat16, device=dev)
        self.fc1_c = torch.empty(cap, 2 * F, dtype=torch.bfloat16, device=dev) if keep_fc1_c else None
        _output_buffers(self, out_format, T, H, dev)

    # the steps, each one launch group on the current stream
    def route(self, logits, stream=None):
        if self.router == "sigmoid":
            moe_route_topk_sigmoid(logits, self.k, self.expert_bias, self.normalize, self.topk_idx, self.topk_w,
                                   stream=stream)
        else:
            moe_route_topk(logits, self.k, self.topk_idx, self.topk_w, stream=stream)

    def permute(self, x, stream=None):
        moe_permute(x, self.topk_idx, self.E, self.ws, self.align, out=self.perm, stream=stream)

    def _route_weights(self, at):
        return (self.perm.src_of_row, self.topk_w) if self.weight_at == at else None

    def fc1(self, W_gate, W_up, stream=None):
        moe_grouped_fc1_swiglu(self.perm.x_perm, W_gate, W_up, self.perm.group_offsets, self.ws, self.h,
                               self.fc1_c, stream=stream, route_weights=self._route_weights("fc1"),
                               clamp=self.swiglu_clamp)

    def fc2(self, W_down, stream=None):
        moe_grouped_fc2(self.h, W_down, self.perm.group_offsets, self.ws, self.y_perm, stream=stream,
                        route_weights=self._route_weights("fc2"))

    def ffn(self, W_gate, W_up, W_down, stream=None):
        self.fc1(W_gate, W_up, stream)
        self.fc2(W_down, stream)

    def combine(self, stream=None):
        _combine(self, self.topk_w if self.weight_at == "combine" else None, stream)

    def __call__(self, x, logits, W_gate, W_up, W_down, stream=None):
        """Returns out (bf16) or, with a block-scaled out_format, (out_q, out_sf)."""
        self.route(logits, stream)
        self.permute(x, stream)
        self.ffn(W_gate, W_up, W_down, stream)
        self.combine(stream)
        return self.out if self.out_format == "bf16" else (self.out_q, self.out_sf)


def _output_buffers(m, out_format: str, T: int, H: int, dev):
    if out_format not in ("bf16", "mxfp8", "nvfp4"):
        raise ValueError("out_format must be 'bf16', 'mxfp8' or 'nvfp4'")
    m.out_format = out_format
    m.out = m.out_q = m.out_sf = None
    if out_format == "bf16":
        m.out = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
    elif out_format == "mxfp8":
        if H % 32:
            raise ValueError("an MXFP8 output needs H % 32 == 0")
        m.out_q = torch.empty(T, H, dtype=torch.uint8, device=dev)
        m.out_sf = torch.empty(T, H // 32, dtype=torch.uint8, device=dev)
    else:
        if H % 16:
            raise ValueError("an NVFP4 output needs H % 16 == 0")
        m.out_q = torch.empty(T, H // 2, dtype=torch.uint8, device=dev)
        m.out_sf = torch.empty(T, H // 16, dtype=torch.uint8, device=dev)


def _combine(m, w, stream):
    if m.out_format == "bf16":
        moe_unpermute_combine(m.y_perm, m.perm.dst_of_route, w, out=m.out, stream=stream)
    elif m.out_format == "mxfp8":
        moe_unpermute_combine_mxfp8(m.y_perm, m.perm.dst_of_route, w, out_q=m.out_q, out_sf=m.out_sf, stream=stream)
    else:
        moe_unpermute_combine_nvfp4(m.y_perm, m.perm.dst_of_route, w, out_q=m.out_q, out_sf=m.out_sf, stream=stream)


def moe_forward(x, logits, W_gate, W_up, W_down, k: int, align: int = 1, keep_fc1_c: bool = False):
    """One-shot forward (allocates its buffers); returns (out, MoeForward)."""
    T, H = x.shape
    E, _, F = W_gate.shape
    m = MoeForward(T, H, F, E, k, x.device, align, keep_fc1_c)
    return m(x, logits, W_gate, W_up, W_down), m


class MoeBackward:
    """Pre-allocated backward for a MoeForward built with keep_fc1_c=True.

    Produces dx (bf16), fp32 dW_gate / dW_up / dW_down and fp32 d_topk_w,
    following the backward contract of "Add MoE + expert-parallel Python API
    surface, PyTorch reference, and tests" (FP32 weight and route gradients);
    with want_d_logits also the fp32 router-logits gradient ("[JAX] Expert
    Parallelism: JAX primitives + VJPs", commit log: the router backward).
    dw_dtype=torch.bfloat16 stores the weight gradients as bf16 instead (the
    same fp32 accumulators, rounded once)."""

    def __init__(self, fwd: MoeForward, want_d_topk_w: bool = True, want_d_logits: bool = False,
                 dw_dtype=torch.float32):
        if dw_dtype not in (torch.float32, torch.bfloat16):
            raise ValueError("dw_dtype: torch.float32 or torch.bfloat16")
        if want_d_logits and not want_d_topk_w:
            raise ValueError("the logits gradient needs d_topk_w")
        if fwd.fc1_c is None:
            raise ValueError("the forward must keep the fc1_c stash (keep_fc1_c=True)")
        if fwd.weight_at != "combine":
            raise ValueError("the backward needs the router weight applied in the combine")
        self.fwd = fwd
        T, H, F, E, k, dev, cap = fwd.T, fwd.H, fwd.F, fwd.E, fwd.k, fwd.device, fwd.rows_cap
        self.dy_perm = torch.empty(cap, H, dtype=torch.bfloat16, device=dev)
        self.dgu = torch.empty(cap, 2 * F, dtype=torch.bfloat16, device=dev)
        self.dx_perm = torch.empty(cap, H, dtype=torch.float32, device=dev)
        self.dx = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
        self.dW_gate = torch.empty(E, H, F, dtype=dw_dtype, device=dev)
        self.dW_up = torch.empty(E, H, F, dtype=dw_dtype, device=dev)
        self.dW_down = torch.empty(E, F, H, dtype=dw_dtype, device=dev)
        self.d_topk_w = torch.empty(T, k, dtype=torch.float32, device=dev) if want_d_topk_w else None
        self.d_logits = torch.empty(T, E, dtype=torch.float32, device=dev) if want_d_logits else None

    def combine_bwd(self, dY, stream=None):
        f = self.fwd
        moe_combine_bwd(dY, f.y_perm, f.perm, f.topk_w, self.dy_perm, self.d_topk_w, stream=stream)

    def dgrad_fc2(self, W_down, stream=None):
        f = self.fwd
        moe_grouped_dgrad_fc2_dswiglu(self.dy_perm, W_down, f.fc1_c, f.perm.group_offsets, f.ws, self.dgu,
                                      stream=stream, clamp=getattr(f, "swiglu_clamp", None))

    def dgrad_fc1(self, W_gate, W_up, stream=None):
        f = self.fwd
        moe_grouped_dgrad_fc1(self.dgu, W_gate, W_up, f.perm.group_offsets, f.ws, self.dx_perm, stream=stream)

    def wgrad(self, stream=None):
        f = self.fwd
        moe_grouped_wgrad(f.perm.x_perm, f.h, self.dy_perm, self.dgu, f.perm.group_offsets, f.ws, self.dW_gate,
                          self.dW_up, self.dW_down, stream=stream)

    def unpermute_sum(self, stream=None):
        moe_unpermute_sum(self.dx_perm, self.fwd.perm.dst_of_route, self.dx, stream=stream)

    def router_bwd(self, logits, stream=None):
        f = self.fwd
        moe_route_topk_bwd(logits, f.topk_idx, self.d_topk_w, SCORE_SIGMOID if f.router == "sigmoid" else SCORE_SOFTMAX,
                           f.normalize, self.d_logits, stream=stream)

    def __call__(self, dY, W_gate, W_up, W_down, stream=None, logits=None):
        """logits: the forward's router logits, needed for d_logits."""
        if self.d_logits is not None and logits is None:
            raise ValueError("the logits gradient needs the forward's logits")
        self.combine_bwd(dY, stream)
        if self.d_logits is not None:
            self.router_bwd(logits, stream)
        self.dgrad_fc2(W_down, stream)
        self.dgrad_fc1(W_gate, W_up, stream)
        self.wgrad(stream)
        self.unpermute_sum(stream)
        return self.dx


class MxWeights:
    """Expert weights quantised once to MXFP8 (K-major codes + tile-layout scales)."""

    def __init__(self, W_gate, W_up, W_down, stream=None):
        self.E, self.H, self.F = W_gate.shape
        self.Wg_q, self.Wg_sf = moe_quantize_weights_mxfp8(W_gate, stream)   # K = H, N = F
        self.Wu_q, self.Wu_sf = moe_quantize_weights_mxfp8(W_up, stream)
        self.Wd_q, self.Wd_sf = moe_quantize_weights_mxfp8(W_down, stream)   # K = F, N = H
        self._deq = None

    def dequantized(self, stream=None):
        """(W_gate, W_up, W_down) as the bf16 values of their MXFP8 codes, in the
        original layouts [E, H, F] / [E, F, H]; computed once."""
        if self._deq is None:
            E, H, F = self.E, self.H, self.F
            self._deq = (moe_dequantize_weights_mxfp8(self.Wg_q, self.Wg_sf, E, H, F, stream=stream),
                         moe_dequantize_weights_mxfp8(self.Wu_q, self.Wu_sf, E, H, F, stream=stream),
                         moe_dequantize_weights_mxfp8(self.Wd_q, self.Wd_sf, E, F, H, stream=stream))
        return self._deq


class MoeForwardMX:
    """Pre-allocated MXFP8 forward: route -> quantising permute -> block-scaled
    FC1 + SwiGLU (h to MXFP8) -> block-scaled FC2 -> combine (bf16 out).
    router / expert_bias / normalize as for MoeForward.  y_perm (the expert outputs)
    is bf16, as on the bf16 path."""

    def __init__(self, T: int, H: int, F: int, E: int, k: int, device="cuda", router: str = "softmax",
                 expert_bias=None, normalize: bool = True, keep_fc1_c: bool = False, out_format: str = "bf16",
                 swiglu_clamp=None):
        if router not in ("softmax", "sigmoid"):
            raise ValueError("router must be 'softmax' or 'sigmoid'")
        self.weight_at = "combine"
        self.swiglu_clamp = None if swiglu_clamp is None else tuple(float(v) for v in swiglu_clamp)
        self.T, self.H, self.F, self.E, self.k = T, H, F, E, k
        self.router, self.expert_bias, self.normalize = router, expert_bias, normalize
        dev = torch.device(device)
        self.device = dev
        self.ws = Workspace(T, E, k, dev)
        cap = T * k
        self.rows_cap = cap
        self.topk_idx = torch.empty(T, k, dtype=torch.int32, device=dev)
        self.topk_w = torch.empty(T, k, dtype=torch.float32, device=dev)
        self.perm = PermutationMX(
            x_q=torch.empty(cap, H, dtype=torch.uint8, device=dev),
            x_sf=torch.zeros(mx_tile_scale_bytes(cap, E, H), dtype=torch.uint8, device=dev),
            dst_of_route=torch.empty(T, k, dtype=torch.int32, device=dev),
            src_of_row=torch.empty(cap, dtype=torch.int32, device=dev),
            group_sizes=torch.empty(E, dtype=torch.int32, device=dev),
            group_offsets=torch.empty(E + 1, dtype=torch.int32, device=dev), rows_cap=cap)
        self.h_q = torch.empty(cap, F, dtype=torch.uint8, device=dev)
        self.h_sf = torch.zeros(mx_tile_scale_bytes(cap, E, F), dtype=torch.uint8, device=dev)
        self.y_perm = torch.empty(cap, H, dtype=torch.bfloat16, device=dev)
        _output_buffers(self, out_format, T, H, dev)
        self.fc1_c = torch.empty(cap, 2 * F, dtype=torch.bfloat16, device=dev) if keep_fc1_c else None

    route = MoeForward.route

    def permute(self, x, stream=None):
        moe_permute_mxfp8(x, self.topk_idx, self.E, self.ws, out=self.perm, stream=stream)

    def fc1(self, w: MxWeights, stream=None):
        p = self.perm
        moe_grouped_fc1_swiglu_mxfp8(p.x_q, p.x_sf, w.Wg_q, w.Wg_sf, w.Wu_q, w.Wu_sf, p.group_offsets, self.ws,
                                     self.h_q, self.h_sf, fc1_c=self.fc1_c, stream=stream, clamp=self.swiglu_clamp)

    def fc2(self, w: MxWeights, stream=None):
        moe_grouped_fc2_mxfp8(self.h_q, self.h_sf, w.Wd_q, w.Wd_sf, self.perm.group_offsets, self.ws, self.y_perm,
                              stream=stream)

    def combine(self, stream=None):
        _combine(self, self.topk_w, stream)

    def __call__(self, x, logits, w: MxWeights, stream=None):
        """Returns out (bf16) or, with a block-scaled out_format, (out_q, out_sf)."""
        self.route(logits, stream)
        self.permute(x, stream)
        self.fc1(w, stream)
        self.fc2(w, stream)
        self.combine(stream)
        return self.out if self.out_format == "bf16" else (self.out_q, self.out_sf)


class MoeBackwardMX(MoeBackward):
    """Straight-through backward of a MoeForwardMX built with keep_fc1_c=True
    ("Add MoE + expert-parallel Python API surface, PyTorch reference, and tests",
    Summary: quantization round-trips are straight-through): the bf16 backward
    kernels run on the values the forward's block-scaled MMAs consumed -- x and h
    dequantised from their MXFP8 rows, the weights from their MXFP8 codes
    (MxWeights.dequantized) -- with the g | u stash of the MXFP8 FC1.  Outputs as
    MoeBackward (gradients with respect to the unquantised x and weights)."""

    def __init__(self, fwd: MoeForwardMX, want_d_topk_w: bool = True, want_d_logits: bool = False,
                 dw_dtype=torch.float32):
        super().__init__(fwd, want_d_topk_w, want_d_logits, dw_dtype)
        cap, dev = fwd.rows_cap, fwd.device
        self.x_deq = torch.empty(cap, fwd.H, dtype=torch.bfloat16, device=dev)
        self.h_deq = torch.empty(cap, fwd.F, dtype=torch.bfloat16, device=dev)

    def dequantize(self, stream=None):
        f = self.fwd
        moe_dequantize_rows_mxfp8(f.perm.x_q, f.perm.x_sf, f.perm.group_offsets, f.ws, out=self.x_deq, stream=stream)
        moe_dequantize_rows_mxfp8(f.h_q, f.h_sf, f.perm.group_offsets, f.ws, out=self.h_deq, stream=stream)

    def wgrad(self, stream=None):
        f = self.fwd
        moe_grouped_wgrad(self.x_deq, self.h_deq, self.dy_perm, self.dgu, f.perm.group_offsets, f.ws, self.dW_gate,
                          self.dW_up, self.dW_down, stream=stream)

    def __call__(self, dY, w: MxWeights, stream=None, logits=None):
        """logits: the forward's router logits, needed for d_logits."""
        if self.d_logits is not None and logits is None:
            raise ValueError("the logits gradient needs the forward's logits")
        Wg, Wu, Wd = w.dequantized(stream)
        self.dequantize(stream)
        self.combine_bwd(dY, stream)
        if self.d_logits is not None:
            self.router_bwd(logits, stream)
        self.dgrad_fc2(Wd, stream)
        self.dgrad_fc1(Wg, Wu, stream)
        self.wgrad(stream)
        self.unpermute_sum(stream)
        return self.dx


class HostPipeline:
    """Batches that live in pinned host memory, run through per-slot layers with the
    host <-> device copies of neighbouring batches overlapped with compute.

    Three streams: uploads (host -> device inputs), compute, downloads (device ->
    host results), ordered by CUDA events per slot.  With two slots, batch i+1's
    inputs are copied in while batch i computes and batch i-1's results are copied
    out; nothing synchronises with the host.  Per slot b:
      upload    waits until compute has consumed the slot's previous inputs
      compute   waits for its inputs and until the slot's previous results left
      download  waits for the compute
    slots[b]   dict: input name -> device tensor of slot b (the copy targets)
    run(b, s)  enqueues slot b's compute on stream s
    outputs(b) the device tensors of slot b whose values go back to the host"""

    def __init__(self, slots, run, outputs, device=None):
        dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
        self.slots, self.run, self.outputs = slots, run, outputs
        self.up, self.comp, self.down = (torch.cuda.Stream(device=dev) for _ in range(3))
        n = len(slots)
        self.ev_in = [torch.cuda.Event() for _ in range(n)]
        self.ev_comp = [torch.cuda.Event() for _ in range(n)]
        self.ev_out = [torch.cuda.Event() for _ in range(n)]
        self.recorded = [False] * n
        self.i = 0

    def submit(self, host_inputs: dict, host_outputs: list):
        """Enqueue one batch: host_inputs name -> pinned host tensor (copied into the
        slot's device tensor of that name), host_outputs pinned host tensors that
        receive outputs(b) in order.  Returns without waiting."""
        b = self.i % len(self.slots)
        self.i += 1
        if self.recorded[b]:
            self.up.wait_event(self.ev_comp[b])
        with torch.cuda.stream(self.up):
            for name, h in host_inputs.items():
                self.slots[b][name].copy_(h, non_blocking=True)
            self.ev_in[b].record(self.up)
        self.comp.wait_event(self.ev_in[b])
        if self.recorded[b]:
            self.comp.wait_event(self.ev_out[b])
        with torch.cuda.stream(self.comp):
            self.run(b, self.comp)
            self.ev_comp[b].record(self.comp)
        self.down.wait_event(self.ev_comp[b])
        with torch.cuda.stream(self.down):
            for h, d in zip(host_outputs, self.outputs(b)):
                h.copy_(d, non_blocking=True)
            self.ev_out[b].record(self.down)
        self.recorded[b] = True
