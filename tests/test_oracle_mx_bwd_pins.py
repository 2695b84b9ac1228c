"""Pins of the oracle's straight-through backward of the MXFP8 forward (CPU only).

The pages fix the convention: the reference MoE backward treats every
quantisation round trip as straight-through ("Add MoE + expert-parallel Python
API surface, PyTorch reference, and tests", Summary).  The oracle realises it as
the bf16 backward formulas on the MXFP8 round trips of x and the weights, with
the MXFP8 forward's h.  It is pinned here against
  * the MXFP8 forward oracle (pinned separately): the forward behind the
    backward must be that forward, value for value, which fixes the
    quantisation axes (x along H, W_gate / W_up along H, W_down along F, h along F);
  * an independent fp64 torch-autograd implementation of the straight-through
    function, in which each quantisation enters as v + (Q(v) - v).detach() and
    the Q values come from the oracle's pinned quantisers;
  * invariants: round trips are idempotent and exact in bf16; zero-token experts
    get exactly zero weight gradients.
"""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.filterwarnings("ignore::UserWarning")


def _problem(T=6, H=64, F=64, E=3, k=2, seed=0, zero_expert=None):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(T, H, generator=g).to(torch.bfloat16)
    Wg = (torch.randn(E, H, F, generator=g) * 0.1).to(torch.bfloat16)
    Wu = (torch.randn(E, H, F, generator=g) * 0.1).to(torch.bfloat16)
    Wd = (torch.randn(E, F, H, generator=g) * 0.1).to(torch.bfloat16)
    logits = torch.randn(T, E, generator=g)
    if zero_expert is not None:
        logits[:, zero_expert] = -1e30
    dY = torch.randn(T, H, generator=g).to(torch.bfloat16)
    idx, w = oracle.route_topk(logits.numpy(), k)
    return dict(x=oracle.bf16_bits(x), Wg=oracle.bf16_bits(Wg), Wu=oracle.bf16_bits(Wu),
                Wd=oracle.bf16_bits(Wd), idx=idx, w=w, dY=oracle.bf16_bits(dY), E=E)


def test_roundtrip_is_idempotent_and_exact():
    p = _problem()
    xq = oracle.mx_roundtrip_rows(p["x"])
    assert np.array_equal(oracle.mx_roundtrip_rows(xq), xq)
    wq = oracle.mx_roundtrip_cols(p["Wg"][0])
    assert np.array_equal(oracle.mx_roundtrip_cols(wq), wq)
    # the values are the dequantised codes of the pinned quantiser, along the stated axis
    q, s = oracle.quantize_rows_mxfp8(p["x"])
    assert np.array_equal(oracle.bits_to_float(xq), oracle.mx_dequantize(q, s))
    qc, sc = oracle.quantize_cols_mxfp8(p["Wg"][0])          # columns of [H, F] along H
    assert np.array_equal(oracle.bits_to_float(wq), oracle.mx_dequantize(qc, sc).T)
    # round trips change values but stay within half an E4M3 step: 2^-4 |v| for normal
    # codes (3 mantissa bits), half the subnormal step 2^(X-10) near zero (X = block scale)
    xv, xqv = oracle.bits_to_float(p["x"]), oracle.bits_to_float(xq)
    assert not np.array_equal(xv, xqv)
    X = np.repeat(s.astype(np.int64) - 127, 32, axis=1)
    assert np.all(np.abs(xqv - xv) <= np.maximum(2.0 ** -4 * np.abs(xv), np.ldexp(1.0, X - 10)))


def test_forward_behind_the_backward_is_the_mxfp8_forward():
    p = _problem(T=8, H=96, F=64, E=3, k=2)
    xq = oracle.mx_roundtrip_rows(p["x"])
    wg, wu, wd = oracle.mx_roundtrip_weights(p["Wg"], p["Wu"], p["Wd"])
    st = oracle.moe_fwd(xq, wg, wu, wd, p["idx"], p["w"], round_mode=1, h_mx=True)["out"]
    codes = [oracle.quantize_cols_mxfp8(p[n][e]) for n in ("Wg", "Wu", "Wd") for e in range(p["E"])]
    E = p["E"]
    gq, gs = [c[0] for c in codes[:E]], [c[1] for c in codes[:E]]
    uq, us = [c[0] for c in codes[E:2 * E]], [c[1] for c in codes[E:2 * E]]
    dq, ds = [c[0] for c in codes[2 * E:]], [c[1] for c in codes[2 * E:]]
    ref = oracle.moe_fwd_mxfp8(p["x"], gq, gs, uq, us, dq, ds, p["idx"], p["w"], round_mode=1)["out"]
    assert np.array_equal(st, ref)
    # and it differs from the bf16 forward (h quantised to MXFP8, not rounded to bf16)
    plain = oracle.moe_fwd(xq, wg, wu, wd, p["idx"], p["w"], round_mode=1)["out"]
    assert not np.array_equal(st, plain)


def _autograd_straight_through(p):
    """fp64 torch autograd of out = sum_j w_j Q(h_j) Q(Wd), h = silu(Q(x) Q(Wg)) * (Q(x) Q(Wu)),
    with d Q(v)/dv = identity; loss = <dY, out>."""
    f = lambda b: torch.tensor(oracle.bits_to_float(b), dtype=torch.float64)  # noqa: E731
    E = p["E"]
    x = f(p["x"]).requires_grad_(True)
    Wg = f(p["Wg"]).requires_grad_(True)
    Wu = f(p["Wu"]).requires_grad_(True)
    Wd = f(p["Wd"]).requires_grad_(True)
    w = torch.tensor(p["w"], dtype=torch.float64, requires_grad=True)
    dY = f(p["dY"])
    st = lambda v, q: v + (q - v).detach()  # noqa: E731
    xq = st(x, f(oracle.mx_roundtrip_rows(p["x"])))
    Wgq = st(Wg, torch.stack([f(oracle.mx_roundtrip_cols(p["Wg"][e])) for e in range(E)]))
    Wuq = st(Wu, torch.stack([f(oracle.mx_roundtrip_cols(p["Wu"][e])) for e in range(E)]))
    Wdq = st(Wd, torch.stack([f(oracle.mx_roundtrip_cols(p["Wd"][e])) for e in range(E)]))
    T, k = p["idx"].shape
    outs = []
    for t in range(T):
        acc = torch.zeros(x.shape[1], dtype=torch.float64)
        for j in range(k):
            e = int(p["idx"][t, j])
            g = xq[t] @ Wgq[e]
            u = xq[t] @ Wuq[e]
            h = torch.nn.functional.silu(g) * u
            hq = st(h, torch.tensor(oracle.mx_fake_quant(h.detach().numpy()[None])[0]))
            acc = acc + w[t, j] * (hq @ Wdq[e])
        outs.append(acc)
    out = torch.stack(outs)
    (out * dY).sum().backward()
    return {"dx": x.grad.numpy(), "dW_gate": Wg.grad.numpy(), "dW_up": Wu.grad.numpy(),
            "dW_down": Wd.grad.numpy(), "d_topk_w": w.grad.numpy()}


@pytest.mark.parametrize("seed", [0, 1])
def test_straight_through_backward_matches_autograd(seed):
    p = _problem(seed=seed)
    ref = _autograd_straight_through(p)
    got = oracle.moe_bwd_mxfp8(p["x"], p["Wg"], p["Wu"], p["Wd"], p["idx"], p["w"], p["dY"], round_mode=0)
    for name in ("dx", "dW_gate", "dW_up", "dW_down", "d_topk_w"):
        a, b = got[name], ref[name]
        scale = max(np.abs(b).max(), 1e-300)
        assert np.abs(a - b).max() <= 1e-11 * scale, name
    # the quantisation matters: the bf16 backward on the unquantised operands differs
    plain = oracle.moe_bwd(p["x"], p["Wg"], p["Wu"], p["Wd"], p["idx"], p["w"], p["dY"], round_mode=0)
    assert np.abs(plain["dW_down"] - got["dW_down"]).max() > 1e-6 * np.abs(got["dW_down"]).max()


def test_zero_token_expert_gets_zero_gradients():
    p = _problem(E=4, zero_expert=2)
    assert not np.any(p["idx"] == 2)
    got = oracle.moe_bwd_mxfp8(p["x"], p["Wg"], p["Wu"], p["Wd"], p["idx"], p["w"], p["dY"])
    for name in ("dW_gate", "dW_up", "dW_down"):
        assert np.all(got[name][2] == 0.0)


def test_sampled_entry_and_token_functions_match_the_full_backward():
    p = _problem(T=8, H=64, F=64, E=3, k=2, seed=3)
    full = oracle.moe_bwd_mxfp8(p["x"], p["Wg"], p["Wu"], p["Wd"], p["idx"], p["w"], p["dY"])
    xq = oracle.mx_roundtrip_rows(p["x"])
    wg, wu, wd = oracle.mx_roundtrip_weights(p["Wg"], p["Wu"], p["Wd"])
    toks = np.array([0, 5, 7])
    tk = oracle.moe_bwd_dx_tokens(xq, wg, wu, wd, p["idx"], p["w"], p["dY"], toks, h_mx=True)
    assert np.array_equal(tk["dx"], full["dx"][toks])
    assert np.array_equal(tk["d_topk_w"], full["d_topk_w"][toks])
    e = int(p["idx"][0, 0])
    ents = [(0, e, 3, 17), (1, e, 60, 5), (2, e, 33, 40), (2, e, 0, 63)]
    val = oracle.moe_bwd_dw_entries(ents, xq, wg, wu, wd, p["idx"], p["w"], p["dY"], h_mx=True)
    ref = [full["dW_gate"][e, 3, 17], full["dW_up"][e, 60, 5], full["dW_down"][e, 33, 40], full["dW_down"][e, 0, 63]]
    assert np.allclose(val, ref, rtol=1e-12, atol=1e-300)
