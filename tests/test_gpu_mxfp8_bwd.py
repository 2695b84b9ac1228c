"""GPU parity of the MXFP8 path's straight-through backward against the CPU
oracle, through the C ABI.

The backward of the MXFP8 forward treats every quantisation round trip as the
identity ("Add MoE + expert-parallel Python API surface, PyTorch reference, and
tests", Summary).  The dequantised operands must equal the oracle's round trips
bit for bit; the g | u stash of the MXFP8 FC1 is a stored bf16 intermediate
(within one bf16 ulp of the oracle's); dx, the fp32 weight gradients and the
route-weight gradients must satisfy max|err| <= 6e-2 * RMS (the bar for the
MXFP8 path) against the oracle's straight-through backward, which applies the
same quantisation."""
import numpy as np
import pytest
import torch

import oracle
from mixture_experts_ffn_warp_gb300 import MoeBackwardMX, MoeForwardMX, MxWeights
from mixture_experts_ffn_warp_gb300.synthetic import small_shape
from helpers import TOL_MXFP8, assert_close_rms, assert_close_ulp, bits, gpu_inputs, host_experts, to_f64

pytestmark = pytest.mark.gpu

SHAPES = {
    # ragged groups over several M tiles, 256-wide tiles
    "ragged": small_shape("ragged", T=300, H=256, F=512, E=5, k=2, backward=True, mxfp8=True),
    # 128-wide tiles in dgrad and wgrad (H, F not multiples of 256)
    "h384": small_shape("h384", T=257, H=384, F=384, E=7, k=3, backward=True, mxfp8=True),
    # many experts, several with no routes
    "many": small_shape("many", T=512, H=128, F=128, E=64, k=4, skew=True, backward=True, mxfp8=True),
}


def _run(shape, seed=0):
    inp = gpu_inputs(shape, seed=seed, with_dy=True)
    mw = MxWeights(inp["W_gate"], inp["W_up"], inp["W_down"])
    m = MoeForwardMX(shape.T, shape.H, shape.F, shape.E, shape.k, keep_fc1_c=True)
    m(inp["x"], inp["logits"], mw)
    b = MoeBackwardMX(m)
    b(inp["dY"], mw)
    torch.cuda.synchronize()
    assert m.ws.read_error() == 0
    return inp, mw, m, b


def test_dequantized_operands_bit_exact():
    shape = SHAPES["ragged"]
    inp, mw, m, b = _run(shape)
    # x rows: the round trip of the token each row holds
    src = m.perm.src_of_row.cpu().numpy()
    used = int(m.perm.group_offsets[-1])
    xq = oracle.mx_roundtrip_rows(bits(inp["x"]))
    assert np.array_equal(bits(b.x_deq[:used]), xq[src[:used] // shape.k])
    # weights: the round trips along H (W_gate, W_up) and along F (W_down)
    Wg, Wu, Wd = mw.dequantized()
    for e in range(shape.E):
        assert np.array_equal(bits(Wg[e]), oracle.mx_roundtrip_cols(bits(inp["W_gate"][e]))), e
        assert np.array_equal(bits(Wu[e]), oracle.mx_roundtrip_cols(bits(inp["W_up"][e]))), e
        assert np.array_equal(bits(Wd[e]), oracle.mx_roundtrip_cols(bits(inp["W_down"][e]))), e
    # h rows: the MXFP8 h of the forward, dequantised -- the values of its codes
    hq_vals = oracle.bits_to_float(bits(b.h_deq[:used]))
    codes = m.h_q[:used].cpu().numpy()
    from test_gpu_mxfp8 import tiles_to_rowmajor
    sc = tiles_to_rowmajor(m.h_sf.cpu().numpy(), m.perm.group_offsets.cpu().numpy(), used, shape.F)
    assert np.array_equal(hq_vals, oracle.mx_dequantize(codes, sc))


def test_fc1_mx_stash_matches_oracle():
    shape = SHAPES["h384"]
    inp, mw, m, b = _run(shape)
    idx, w = m.topk_idx.cpu().numpy(), m.topk_w.cpu().numpy()
    xq = oracle.mx_roundtrip_rows(bits(inp["x"]))
    wg, wu, wd = oracle.mx_roundtrip_weights(bits(inp["W_gate"]), bits(inp["W_up"]), bits(inp["W_down"]))
    ref = oracle.moe_fwd(xq, wg, wu, wd, idx, w, round_mode=1, want_fc1=True, h_mx=True)
    dst = m.perm.dst_of_route.cpu().numpy().reshape(-1)
    got = to_f64(m.fc1_c)[dst]
    assert_close_ulp(got, oracle.round_bf16(ref["fc1"]), what="fc1_c (MXFP8 FC1)")


@pytest.mark.parametrize("name", list(SHAPES))
def test_mx_backward_parity_small(name):
    shape = SHAPES[name]
    inp, mw, m, b = _run(shape)
    idx, w = m.topk_idx.cpu().numpy(), m.topk_w.cpu().numpy()
    hb = {n: bits(inp[n]) for n in ("x", "W_gate", "W_up", "W_down", "dY")}
    ref = oracle.moe_bwd_mxfp8(hb["x"], hb["W_gate"], hb["W_up"], hb["W_down"], idx, w, hb["dY"], round_mode=2)
    assert_close_rms(to_f64(b.dx), ref["dx"], tol=TOL_MXFP8, what="dx", bf16_out=True)
    for n in ("dW_gate", "dW_up", "dW_down"):
        assert_close_rms(getattr(b, n).double().cpu().numpy(), ref[n], tol=TOL_MXFP8, what=n)
    assert_close_rms(b.d_topk_w.double().cpu().numpy(), ref["d_topk_w"], tol=TOL_MXFP8, what="d_topk_w")
    empty = (m.perm.group_sizes == 0).nonzero().flatten().tolist()
    if name == "many":
        assert len(empty) >= 8
    for e in empty:
        for t in (b.dW_gate, b.dW_up, b.dW_down):
            assert torch.count_nonzero(t[e]) == 0


def test_mx_backward_deepseek_shaped_sampled():
    """DeepSeek-V3 expert shapes (H=7168, F=2048, top-8) on 16 experts and 512 tokens
    (256 rows per expert, as in the full workload): dx and d_topk_w of sampled
    tokens and sampled weight-gradient entries against the oracle."""
    shape = small_shape("dsv3_e16", T=512, H=7168, F=2048, E=16, k=8, backward=True, mxfp8=True)
    inp, mw, m, b = _run(shape)
    idx, w = m.topk_idx.cpu().numpy(), m.topk_w.cpu().numpy()
    E, H, F = shape.E, shape.H, shape.F
    Wg, Wu, Wd = (host_experts(inp[n], range(E)) for n in ("W_gate", "W_up", "W_down"))
    wg, wu, wd = oracle.mx_roundtrip_weights([Wg[e] for e in range(E)], [Wu[e] for e in range(E)],
                                             [Wd[e] for e in range(E)])
    xq = oracle.mx_roundtrip_rows(bits(inp["x"]))
    dyb = bits(inp["dY"])
    rng = np.random.default_rng(5)
    toks = np.sort(rng.choice(shape.T, size=4, replace=False))
    ref = oracle.moe_bwd_dx_tokens(xq, wg, wu, wd, idx, w, dyb, toks, round_mode=2, h_mx=True)
    sel = torch.from_numpy(toks).cuda()
    assert_close_rms(to_f64(b.dx[sel]), ref["dx"], tol=TOL_MXFP8, what="dx", bf16_out=True)
    assert_close_rms(b.d_topk_w[sel].double().cpu().numpy(), ref["d_topk_w"], tol=TOL_MXFP8, what="d_topk_w")
    ents = []
    for which, (a_dim, b_dim) in ((0, (H, F)), (1, (H, F)), (2, (F, H))):
        for _ in range(6):
            ents.append((which, int(rng.integers(E)), int(rng.integers(a_dim)), int(rng.integers(b_dim))))
    vals = oracle.moe_bwd_dw_entries(ents, xq, wg, wu, wd, idx, w, dyb, round_mode=2, h_mx=True)
    for which in range(3):
        t = (b.dW_gate, b.dW_up, b.dW_down)[which]
        rms = float(t.double().pow(2).mean().sqrt())
        err = max(abs(float(t[e, a, c]) - vals[i]) for i, (q, e, a, c) in enumerate(ents) if q == which)
        assert err <= TOL_MXFP8 * rms, f"dW[{which}] max|err| {err:.3e} > {TOL_MXFP8} * RMS {rms:.3e}"
