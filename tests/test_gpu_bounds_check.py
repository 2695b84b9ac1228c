"""The bounds-check build (-DMOE_BOUNDS_CHECK), the stand-in for a memory sanitizer: the
GEMMs check the group offsets they read from device memory (the one data-dependent
extent their loads, MMAs and stores trust) before any access.

Through the C ABI of that build (compiled on the GPU machine into _build_bounds/): with valid
offsets its outputs equal the normal build's bit for bit; with offsets that leave the
rows' buffer it reports MOE_DEVERR_BOUNDS, computes nothing and faults nothing.  Such
offsets are only ever given to the bounds-check build."""
import ctypes as C
import os

import pytest
import torch

from mixture_experts_ffn_warp_gb300 import Workspace, moe_grouped_fc1_swiglu, moe_permute, moe_route_topk
from mixture_experts_ffn_warp_gb300 import build as B
from mixture_experts_ffn_warp_gb300.synthetic import small_shape
from helpers import gpu_inputs

pytestmark = pytest.mark.gpu

DEVERR_BOUNDS = 0x8


@pytest.fixture(scope="module")
def bounds_lib():
    path = B.build(extra_flags=["-DMOE_BOUNDS_CHECK"], out_dir=os.path.join(B.HERE, "_build_bounds"))
    L = C.CDLL(path)
    for name in ("moe_grouped_fc1_swiglu", "moe_grouped_wgrad"):
        getattr(L, name).restype = C.c_int
    return L


def _p(t):
    return C.c_void_p(t.data_ptr())


def _error_word(ws):
    torch.cuda.synchronize()
    return int(ws.buf[:4].view(torch.int32).item())


def test_bounds_build_matches_and_refuses_bad_offsets(bounds_lib):
    shape = small_shape("bounds", T=400, H=256, F=512, E=6, k=2)
    inp = gpu_inputs(shape, with_dy=False)
    ws = Workspace(shape.T, shape.E, shape.k)
    idx, _ = moe_route_topk(inp["logits"], shape.k)
    p = moe_permute(inp["x"], idx, shape.E, ws)
    cap, H, F, E = p.rows_cap, shape.H, shape.F, shape.E
    h_ref = torch.zeros(cap, F, dtype=torch.bfloat16, device="cuda")
    moe_grouped_fc1_swiglu(p.x_perm, inp["W_gate"], inp["W_up"], p.group_offsets, ws, h_ref)
    torch.cuda.synchronize()
    assert ws.read_error() == 0

    def fc1(offsets, h):
        st = bounds_lib.moe_grouped_fc1_swiglu(_p(p.x_perm), _p(inp["W_gate"]), _p(inp["W_up"]), _p(offsets), E, H,
                                               F, C.c_int64(cap), _p(h), None, _p(ws.buf), C.c_size_t(ws.nbytes),
                                               None)
        assert st == 0
        return _error_word(ws)

    h = torch.zeros_like(h_ref)
    assert fc1(p.group_offsets, h) == 0
    used = int(p.group_offsets[-1].item())
    assert torch.equal(h[:used], h_ref[:used])
    # offsets past the rows' buffer: reported, nothing computed
    bad = p.group_offsets.clone()
    bad[-1] = cap + 4096
    ws.reset()
    h_bad = torch.full_like(h_ref, 7.0)
    assert fc1(bad, h_bad) & DEVERR_BOUNDS
    assert bool((h_bad == 7.0).all())
    # decreasing offsets, through the K-grouped weight-gradient GEMM
    bad2 = p.group_offsets.clone()
    bad2[2] = bad2[3] + 1
    ws.reset()
    dW = [torch.full((E, H, F), 7.0, device="cuda"), torch.full((E, H, F), 7.0, device="cuda"),
          torch.full((E, F, H), 7.0, device="cuda")]
    dy = torch.zeros(cap, H, dtype=torch.bfloat16, device="cuda")
    dgu = torch.zeros(cap, 2 * F, dtype=torch.bfloat16, device="cuda")
    st = bounds_lib.moe_grouped_wgrad(_p(p.x_perm), _p(h_ref), _p(dy), _p(dgu), _p(bad2), E, H, F, C.c_int64(cap),
                                      _p(dW[0]), _p(dW[1]), _p(dW[2]), _p(ws.buf), C.c_size_t(ws.nbytes), None)
    assert st == 0
    assert _error_word(ws) & DEVERR_BOUNDS
    assert all(bool((t == 7.0).all()) for t in dW)
