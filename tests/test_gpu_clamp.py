"""GPU parity of the optional SwiGLU clamp (the pages' DeepSeek-style clamp with
inclusive bounds, bounds chosen by the caller) against the CPU oracle, through the
C ABI: forward h and output, and the backward (dSwiGLU at the clamped values, zero
derivative outside the bounds), within the same tolerances as the unclamped path."""
import numpy as np
import pytest
import torch

import oracle
from mixture_experts_ffn_warp_gb300 import MoeBackward, MoeForward
from mixture_experts_ffn_warp_gb300.synthetic import small_shape
from helpers import assert_close_rms, assert_close_ulp, bits, gpu_inputs, to_f64

pytestmark = pytest.mark.gpu

# g, u of these shapes are ~N(0, 0.02^2 H): the bounds clip a good share of both
SHAPES = {
    "ragged": (small_shape("ragged", T=300, H=256, F=384, E=5, k=2, backward=True), (-0.3, 0.2, -0.25, 0.25)),
    "many": (small_shape("many", T=512, H=128, F=128, E=64, k=4, skew=True, backward=True), (-np.inf, 0.1, -0.1, 0.15)),
    # H a multiple of 256: the FC1 dgrad runs on CTA pairs, the 256-wide dSwiGLU dgrad tiles;
    # ~450 rows per expert, two token blocks each
    "pairs": (small_shape("pairs", T=900, H=256, F=512, E=4, k=2, backward=True), (-0.3, 0.2, -0.25, 0.25)),
}


@pytest.mark.parametrize("name", list(SHAPES))
def test_clamped_forward_and_backward(name):
    shape, clamp = SHAPES[name]
    inp = gpu_inputs(shape, with_dy=True)
    m = MoeForward(shape.T, shape.H, shape.F, shape.E, shape.k, keep_fc1_c=True, swiglu_clamp=clamp)
    out = m(inp["x"], inp["logits"], inp["W_gate"], inp["W_up"], inp["W_down"])
    b = MoeBackward(m)
    b(inp["dY"], inp["W_gate"], inp["W_up"], inp["W_down"])
    torch.cuda.synchronize()
    assert m.ws.read_error() == 0
    idx, w = m.topk_idx.cpu().numpy(), m.topk_w.cpu().numpy()
    hb = {n: bits(inp[n]) for n in ("x", "W_gate", "W_up", "W_down", "dY")}
    with oracle.swiglu_clamp(*clamp):
        fwd = oracle.moe_fwd(hb["x"], hb["W_gate"], hb["W_up"], hb["W_down"], idx, w, round_mode=1,
                             want_h=True, want_fc1=True)
        fwd2 = oracle.moe_fwd(hb["x"], hb["W_gate"], hb["W_up"], hb["W_down"], idx, w, round_mode=2)
        bwd = oracle.moe_bwd(hb["x"], hb["W_gate"], hb["W_up"], hb["W_down"], idx, w, hb["dY"], round_mode=2)
    dst = m.perm.dst_of_route.cpu().numpy().reshape(-1)
    g = fwd["fc1"][:, :shape.F]
    clipped = np.mean((g < clamp[0]) | (g > clamp[1]))
    assert clipped > 0.05, clipped                      # the clamp is active
    assert_close_ulp(to_f64(m.h)[dst], fwd["h"], what="clamped h")
    assert_close_ulp(to_f64(m.fc1_c)[dst], oracle.round_bf16(fwd["fc1"]), what="unclamped stash")
    assert_close_rms(to_f64(out), fwd2["out"], what="clamped out", bf16_out=True)
    assert_close_rms(to_f64(b.dx), bwd["dx"], what="dx", bf16_out=True)
    for n in ("dW_gate", "dW_up", "dW_down"):
        assert_close_rms(getattr(b, n).double().cpu().numpy(), bwd[n], what=n)
    assert_close_rms(b.d_topk_w.double().cpu().numpy(), bwd["d_topk_w"], what="d_topk_w")


def test_clamp_with_weight_in_fc1():
    shape, clamp = SHAPES["ragged"]
    inp = gpu_inputs(shape, with_dy=False)
    m = MoeForward(shape.T, shape.H, shape.F, shape.E, shape.k, weight_at="fc1", swiglu_clamp=clamp)
    out = m(inp["x"], inp["logits"], inp["W_gate"], inp["W_up"], inp["W_down"])
    torch.cuda.synchronize()
    idx, w = m.topk_idx.cpu().numpy(), m.topk_w.cpu().numpy()
    hb = {n: bits(inp[n]) for n in ("x", "W_gate", "W_up", "W_down")}
    with oracle.swiglu_clamp(*clamp):
        ref = oracle.moe_fwd(hb["x"], hb["W_gate"], hb["W_up"], hb["W_down"], idx, w, round_mode=2,
                             weight_at=oracle.WEIGHT_IN_FC1)["out"]
    assert_close_rms(to_f64(out), ref, what="clamped, weight in FC1", bf16_out=True)


def test_clamped_mxfp8_forward_and_straight_through_backward():
    from mixture_experts_ffn_warp_gb300 import MoeBackwardMX, MoeForwardMX, MxWeights
    from helpers import TOL_MXFP8
    shape = small_shape("mxclamp", T=300, H=256, F=384, E=5, k=2, backward=True, mxfp8=True)
    clamp = (-0.3, 0.2, -0.25, 0.25)
    inp = gpu_inputs(shape, with_dy=True)
    mw = MxWeights(inp["W_gate"], inp["W_up"], inp["W_down"])
    m = MoeForwardMX(shape.T, shape.H, shape.F, shape.E, shape.k, keep_fc1_c=True, swiglu_clamp=clamp)
    out = m(inp["x"], inp["logits"], mw)
    b = MoeBackwardMX(m)
    b(inp["dY"], mw)
    torch.cuda.synchronize()
    assert m.ws.read_error() == 0
    idx, w = m.topk_idx.cpu().numpy(), m.topk_w.cpu().numpy()
    hb = {n: bits(inp[n]) for n in ("x", "W_gate", "W_up", "W_down", "dY")}
    xq = oracle.mx_roundtrip_rows(hb["x"])
    wg, wu, wd = oracle.mx_roundtrip_weights(hb["W_gate"], hb["W_up"], hb["W_down"])
    with oracle.swiglu_clamp(*clamp):
        ref_out = oracle.moe_fwd(xq, wg, wu, wd, idx, w, round_mode=2, h_mx=True)["out"]
        ref = oracle.moe_bwd_mxfp8(hb["x"], hb["W_gate"], hb["W_up"], hb["W_down"], idx, w, hb["dY"], round_mode=2)
    assert_close_rms(to_f64(out), ref_out, tol=TOL_MXFP8, what="clamped MXFP8 out", bf16_out=True)
    assert_close_rms(to_f64(b.dx), ref["dx"], tol=TOL_MXFP8, what="dx", bf16_out=True)
    for n in ("dW_gate", "dW_up", "dW_down"):
        assert_close_rms(getattr(b, n).double().cpu().numpy(), ref[n], tol=TOL_MXFP8, what=n)


def test_clamped_mxfp8_forward_on_cta_pairs():
    """Without the stash the MXFP8 FC1 runs on CTA pairs: the clamped forward there matches the
    clamped oracle, and its expert outputs are the ones of the one-CTA kernel (which runs when
    the stash is kept), bit for bit."""
    from mixture_experts_ffn_warp_gb300 import MoeForwardMX, MxWeights
    from helpers import TOL_MXFP8
    shape = small_shape("mxclamp_pairs", T=700, H=256, F=384, E=5, k=2, mxfp8=True)
    clamp = (-0.3, 0.2, -0.25, 0.25)
    inp = gpu_inputs(shape, with_dy=False)
    mw = MxWeights(inp["W_gate"], inp["W_up"], inp["W_down"])
    m0 = MoeForwardMX(shape.T, shape.H, shape.F, shape.E, shape.k, swiglu_clamp=clamp)
    m1 = MoeForwardMX(shape.T, shape.H, shape.F, shape.E, shape.k, keep_fc1_c=True, swiglu_clamp=clamp)
    out0 = m0(inp["x"], inp["logits"], mw)
    m1(inp["x"], inp["logits"], mw)
    torch.cuda.synchronize()
    assert m0.ws.read_error() == 0 and m1.ws.read_error() == 0
    rows = int(m0.perm.group_offsets[-1].item())
    assert torch.equal(m0.h_q[:rows], m1.h_q[:rows])
    assert torch.equal(m0.h_sf, m1.h_sf)
    assert torch.equal(m0.y_perm[:rows], m1.y_perm[:rows])
    idx, w = m0.topk_idx.cpu().numpy(), m0.topk_w.cpu().numpy()
    hb = {n: bits(inp[n]) for n in ("x", "W_gate", "W_up", "W_down")}
    xq = oracle.mx_roundtrip_rows(hb["x"])
    wg, wu, wd = oracle.mx_roundtrip_weights(hb["W_gate"], hb["W_up"], hb["W_down"])
    with oracle.swiglu_clamp(*clamp):
        ref_out = oracle.moe_fwd(xq, wg, wu, wd, idx, w, round_mode=2, h_mx=True)["out"]
    assert_close_rms(to_f64(out0), ref_out, tol=TOL_MXFP8, what="clamped MXFP8 out (CTA pairs)", bf16_out=True)
