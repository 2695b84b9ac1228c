"""The GEMMs' bounded device waits, exercised on the GPU without faulting it.

Every pipeline wait of the grouped GEMM kernels gives up after a limit kept in
the workspace header (moe_workspace_set_wait_limit; 2 s by default): it sets
MOE_DEVERR_TIMEOUT, lets the copies and MMAs already issued finish, frees its
tensor memory and exits.  With the limit at 1 ns every wait that has to spin
gives up, so the call must report the timeout; the same call at the default
limit must then give the oracle's result on the same context (no trap, no
hang, nothing left allocated).  Both kernels: the CTA-pair GEMM (FC1 + SwiGLU)
and the one-CTA GEMM (FC2 at H % 256 != 0)."""
import numpy as np
import pytest
import torch

import oracle
from mixture_experts_ffn_warp_gb300 import (Workspace, moe_grouped_fc1_swiglu, moe_grouped_fc2, moe_permute,
                                            moe_route_topk)
from mixture_experts_ffn_warp_gb300._binding import DEVERR_TIMEOUT
from mixture_experts_ffn_warp_gb300.synthetic import small_shape
from helpers import assert_close_ulp, bits, gpu_inputs, to_f64

pytestmark = pytest.mark.gpu


def _setup(H):
    shape = small_shape("tmo", T=256, H=H, F=512, E=4, k=2)
    inp = gpu_inputs(shape, with_dy=False)
    ws = Workspace(shape.T, shape.E, shape.k)
    idx, w = moe_route_topk(inp["logits"], shape.k)
    p = moe_permute(inp["x"], idx, shape.E, ws)
    torch.cuda.synchronize()
    assert ws.read_error() == 0
    return shape, inp, ws, idx, w, p


def test_pair_gemm_wait_timeout_then_recovery():
    shape, inp, ws, idx, w, p = _setup(256)
    h = torch.zeros(p.rows_cap, shape.F, dtype=torch.bfloat16, device="cuda")
    ws.set_wait_limit(1)
    moe_grouped_fc1_swiglu(p.x_perm, inp["W_gate"], inp["W_up"], p.group_offsets, ws, h)
    torch.cuda.synchronize()
    assert ws.read_error() & DEVERR_TIMEOUT
    ws.reset()                               # error word cleared, default limit again
    moe_grouped_fc1_swiglu(p.x_perm, inp["W_gate"], inp["W_up"], p.group_offsets, ws, h)
    torch.cuda.synchronize()
    assert ws.read_error() == 0
    ref_p = oracle.permute(idx.cpu().numpy(), shape.E)
    used = int(ref_p["group_offsets"][-1])
    ref = oracle.moe_fwd(bits(inp["x"]), bits(inp["W_gate"]), bits(inp["W_up"]), bits(inp["W_down"]),
                         idx.cpu().numpy(), w.cpu().numpy(), want_h=True)
    assert_close_ulp(to_f64(h[:used]), ref["h"][ref_p["src_of_row"][:used]], what="h after recovery")


def test_one_cta_gemm_wait_timeout_then_recovery():
    shape, inp, ws, idx, w, p = _setup(384)          # H % 256 != 0: FC2 on the one-CTA kernel
    h = torch.empty(p.rows_cap, shape.F, dtype=torch.bfloat16, device="cuda")
    moe_grouped_fc1_swiglu(p.x_perm, inp["W_gate"], inp["W_up"], p.group_offsets, ws, h)
    y = torch.zeros(p.rows_cap, shape.H, dtype=torch.bfloat16, device="cuda")
    ws.set_wait_limit(1)
    moe_grouped_fc2(h, inp["W_down"], p.group_offsets, ws, y)
    torch.cuda.synchronize()
    assert ws.read_error() & DEVERR_TIMEOUT
    ws.set_wait_limit(0)                     # the default limit; the error word stays set
    ws.reset()
    moe_grouped_fc2(h, inp["W_down"], p.group_offsets, ws, y)
    torch.cuda.synchronize()
    assert ws.read_error() == 0
    ref_p = oracle.permute(idx.cpu().numpy(), shape.E)
    used = int(ref_p["group_offsets"][-1])
    ref = oracle.moe_fwd(bits(inp["x"]), bits(inp["W_gate"]), bits(inp["W_up"]), bits(inp["W_down"]),
                         idx.cpu().numpy(), w.cpu().numpy(), want_y=True)
    assert_close_ulp(to_f64(y[:used]), ref["y"][ref_p["src_of_row"][:used]], what="y after recovery")
