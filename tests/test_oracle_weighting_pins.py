"""Pins of the oracle's router-weight placement (CPU only): the weight applied in
the combine, in the FC1 epilogue (to h, before its bf16 rounding) or in the FC2
epilogue (to y).  In exact arithmetic the three are one function; the pins check
that, that each route is scaled by its own weight, and where the rounding falls."""
import numpy as np
import torch

import oracle
from mixture_experts_ffn_warp_gb300.synthetic import make_inputs, small_shape

SHAPE = small_shape("wpin", T=24, H=64, F=96, E=5, k=3)


def _case():
    inp = make_inputs(SHAPE, device="cpu")
    idx, w = oracle.route_topk(inp["logits"].numpy(), SHAPE.k)
    b = {n: oracle.bf16_bits(inp[n]) for n in ("x", "W_gate", "W_up", "W_down")}
    return b, idx, w


def _fwd(b, idx, w, **kw):
    return oracle.moe_fwd(b["x"], b["W_gate"], b["W_up"], b["W_down"], idx, w, **kw)


def test_weight_placement_is_the_same_function_in_exact_arithmetic():
    b, idx, w = _case()
    ref = _fwd(b, idx, w, round_mode=0)["out"]
    for at in (oracle.WEIGHT_IN_FC1, oracle.WEIGHT_IN_FC2):
        got = _fwd(b, idx, w, round_mode=0, weight_at=at)["out"]
        np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-14)


def test_each_route_is_scaled_by_its_own_weight():
    """h (FC1 placement) and y (FC2 placement) of route (t, j) equal w[t, j] times the
    unweighted h and y of that route."""
    b, idx, w = _case()
    base = _fwd(b, idx, w, round_mode=0, want_h=True, want_y=True)
    f1 = _fwd(b, idx, w, round_mode=0, want_h=True, want_y=True, weight_at=oracle.WEIGHT_IN_FC1)
    f2 = _fwd(b, idx, w, round_mode=0, want_h=True, want_y=True, weight_at=oracle.WEIGHT_IN_FC2)
    wr = w.reshape(-1, 1).astype(np.float64)
    np.testing.assert_allclose(f1["h"], wr * base["h"], rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(f1["y"], wr * base["y"], rtol=1e-11, atol=1e-14)
    np.testing.assert_allclose(f2["h"], base["h"], rtol=0, atol=0)
    np.testing.assert_allclose(f2["y"], wr * base["y"], rtol=1e-13, atol=1e-15)


def test_fc1_placement_rounds_the_weighted_h():
    """round_mode 1: h = bf16(w * silu(g) u), rounded by torch's own bf16 conversion
    of the exact weighted value."""
    b, idx, w = _case()
    exact = _fwd(b, idx, w, round_mode=0, want_h=True, weight_at=oracle.WEIGHT_IN_FC1)["h"]
    got = _fwd(b, idx, w, round_mode=1, want_h=True, weight_at=oracle.WEIGHT_IN_FC1)["h"]
    ref = torch.from_numpy(exact).to(torch.bfloat16).double().numpy()
    assert np.array_equal(got, ref)


def test_fc2_placement_rounds_the_weighted_y():
    """round_mode 1: y = bf16(w * (h Wd)) on the (rounded, unweighted) h, rounded by
    torch's own bf16 conversion of the product, not w times a rounded y."""
    b, idx, w = _case()
    base = _fwd(b, idx, w, round_mode=1, want_h=True, want_y=True)
    got = _fwd(b, idx, w, round_mode=1, want_h=True, want_y=True, weight_at=oracle.WEIGHT_IN_FC2)
    assert np.array_equal(got["h"], base["h"])
    hr = torch.from_numpy(base["h"])
    wd = torch.from_numpy(oracle.bits_to_float(b["W_down"]))
    y_exact = torch.stack([hr[r] @ wd[int(idx.flat[r])] for r in range(idx.size)])
    wr = torch.from_numpy(w.reshape(-1, 1).astype(np.float64))
    ref = (wr * y_exact).to(torch.bfloat16).double().numpy()
    assert np.array_equal(got["y"], ref)
    assert not np.array_equal(got["y"], (wr.numpy() * base["y"]))


def test_unit_weights_make_the_placements_identical():
    """k = 1: the softmax over one logit is exactly 1, so every placement gives the same
    bits even with bf16 rounding."""
    inp = make_inputs(small_shape("wpin1", T=16, H=64, F=96, E=4, k=1), device="cpu")
    idx, w = oracle.route_topk(inp["logits"].numpy(), 1)
    assert (w == 1.0).all()
    b = {n: oracle.bf16_bits(inp[n]) for n in ("x", "W_gate", "W_up", "W_down")}
    outs = [_fwd(b, idx, w, round_mode=1, weight_at=at)["out"] for at in (0, 1, 2)]
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])
