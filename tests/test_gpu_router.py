"""GPU parity of the router variants against the CPU oracle, through the C ABI:
the sigmoid router with an expert routing bias, and the router backward for
both score functions.

Selections must match the oracle bit for bit, except where two fp32 keys are
within rounding of each other (the oracle ranks in double): there the GPU's
choice is checked to be a valid top-k.  Weights: |err| <= 2e-6.  d_logits:
|err| <= 2e-5 * max|d_logits| + 1e-6 * max|d_topk_w| and exact zeros off the
selection."""
import numpy as np
import pytest
import torch

import oracle
from mixture_experts_ffn_warp_gb300 import (SCORE_SIGMOID, SCORE_SOFTMAX, moe_route_topk, moe_route_topk_bwd,
                                            moe_route_topk_sigmoid)

pytestmark = pytest.mark.gpu

SHAPES = {"fine_grained": (4096, 64, 6), "dsv3": (8192, 256, 8), "ragged_e": (777, 40, 3), "k1": (300, 16, 1)}


def _inputs(T, E, k, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    logits = torch.randn(T, E, generator=g, device="cuda", dtype=torch.float32)
    bias = torch.randn(E, generator=g, device="cuda", dtype=torch.float32) * 0.05
    dw = torch.randn(T, k, generator=g, device="cuda", dtype=torch.float32)
    return logits, bias, dw


def _check_selection(idx_gpu, idx_ref, keys, k, tol=1e-6):
    """Equal rows must dominate.  A row that differs (two keys within fp32 rounding of each
    other: the GPU ranks fp32 keys, the oracle double ones) must still be a valid ranked
    top-k of the double keys up to `tol`: k distinct ids; every unselected key at most the
    smallest selected one (+ tol); slots in descending key order (up to tol); and where two
    keys are exactly equal in double, the lower id first, an unselected id never below a
    selected one of the same key."""
    diff = np.nonzero((idx_gpu != idx_ref).any(1))[0]
    assert len(diff) <= max(2, len(idx_ref) // 500), f"{len(diff)} rows differ"
    E = keys.shape[1]
    for t in diff:
        sel = idx_gpu[t]
        assert len(set(sel.tolist())) == k and (sel >= 0).all() and (sel < E).all(), (t, sel)
        ks = keys[t, sel]
        rest = np.setdiff1d(np.arange(E), sel)
        assert (keys[t, rest] <= ks.min() + tol).all(), (t, ks, keys[t, rest].max())
        for j in range(k - 1):
            assert ks[j] >= ks[j + 1] - tol, (t, j, ks)
            if ks[j] == ks[j + 1]:
                assert sel[j] < sel[j + 1], (t, j, sel)
        for e in rest:
            same = sel[ks == keys[t, e]]
            assert (same < e).all(), (t, e, same)
    return diff


def _sigmoid_weights_of(idx, lg, normalize):
    """Weights of a given selection in double: the selected unbiased sigmoid scores,
    divided by (their sum + 1e-20) when normalising."""
    s = 1.0 / (1.0 + np.exp(-np.take_along_axis(lg.astype(np.float64), idx.astype(np.int64), axis=1)))
    return s / (s.sum(1, keepdims=True) + 1e-20) if normalize else s


@pytest.mark.parametrize("name", list(SHAPES))
@pytest.mark.parametrize("use_bias,normalize", [(False, True), (True, True), (True, False)])
def test_sigmoid_router_matches_oracle(name, use_bias, normalize):
    T, E, k = SHAPES[name]
    logits, bias, _ = _inputs(T, E, k, 11)
    b = bias if use_bias else None
    idx, w = moe_route_topk_sigmoid(logits, k, b, normalize)
    torch.cuda.synchronize()
    lg = logits.cpu().numpy()
    bn = None if b is None else b.cpu().numpy()
    ref_idx, ref_w = oracle.route_topk_sigmoid(lg, k, bn, normalize)
    idx, w = idx.cpu().numpy(), w.cpu().numpy()
    keys = torch.sigmoid(torch.from_numpy(lg).double()).numpy() + (0 if bn is None else bn.astype(np.float64))
    diff = _check_selection(idx, ref_idx, keys, k)
    same = np.setdiff1d(np.arange(T), diff)
    assert np.abs(w[same] - ref_w[same]).max() <= 2e-6
    # every row's weights, those of differing rows included, from the GPU's own selection
    assert np.abs(w - _sigmoid_weights_of(idx, lg, normalize)).max() <= 2e-6


def test_sigmoid_router_special_rows():
    E, k = 40, 4
    lg = torch.randn(6, E, device="cuda")
    lg[0] = -torch.inf                  # all scores 0: ids 0..k-1, weights 0 (not NaN)
    lg[1] = 0.0                         # all tied: ids 0..k-1, weights 1/k
    lg[2, 5] = torch.nan                # a NaN logit ranks last
    lg[3, :] = -30.0
    lg[3, 7] = 5.0
    idx, w = moe_route_topk_sigmoid(lg, k)
    torch.cuda.synchronize()
    idx, w = idx.cpu().numpy(), w.cpu().numpy()
    assert (idx[0] == np.arange(k)).all() and (w[0] == 0).all()
    assert (idx[1] == np.arange(k)).all() and np.allclose(w[1], 0.25, atol=1e-7)
    assert 5 not in idx[2] and np.isfinite(w).all()
    assert idx[3, 0] == 7
    ref_idx, ref_w = oracle.route_topk_sigmoid(lg.cpu().numpy()[[0, 1, 3]], k)
    assert np.array_equal(idx[[0, 1, 3]], ref_idx)
    assert np.abs(w[[0, 1, 3]] - ref_w).max() <= 2e-6


@pytest.mark.parametrize("name", list(SHAPES))
@pytest.mark.parametrize("score_fn,normalize", [(SCORE_SOFTMAX, True), (SCORE_SIGMOID, True),
                                                (SCORE_SIGMOID, False)])
def test_router_bwd_matches_oracle(name, score_fn, normalize):
    T, E, k = SHAPES[name]
    logits, _, dw = _inputs(T, E, k, 12)
    lg = logits.cpu().numpy()
    if score_fn == SCORE_SOFTMAX:
        sel, _ = oracle.route_topk(lg, k)
    else:
        sel, _ = oracle.route_topk_sigmoid(lg, k, None, normalize)
    sel = sel.copy()
    sel[::5, k - 1] = -1                # dropped routes: skipped
    idx = torch.from_numpy(sel).cuda()
    dl = moe_route_topk_bwd(logits, idx, dw, score_fn, normalize)
    torch.cuda.synchronize()
    ref = oracle.route_topk_bwd(lg, sel, dw.cpu().numpy(), score_fn, normalize)
    got = dl.cpu().numpy().astype(np.float64)
    # relative to the largest gradient, with an fp32 floor for rows whose exact
    # gradient is far below fp32 resolution (k = 1 with normalisation: ~1e-17)
    tol = 2e-5 * np.abs(ref).max() + 1e-6 * np.abs(dw.cpu().numpy()).max()
    assert np.abs(got - ref).max() <= tol
    assert (got[ref == 0] == 0).all()


def test_router_bwd_softmax_selection_from_the_gpu_router():
    """The softmax router's own output as the selection; k = 1 gives exact zeros."""
    T, E, k = 2048, 64, 6
    logits, _, dw = _inputs(T, E, k, 13)
    idx, _ = moe_route_topk(logits, k)
    dl = moe_route_topk_bwd(logits, idx, dw, SCORE_SOFTMAX)
    torch.cuda.synchronize()
    ref_idx, _ = oracle.route_topk(logits.cpu().numpy(), k)
    assert np.array_equal(idx.cpu().numpy(), ref_idx)
    ref = oracle.route_topk_bwd(logits.cpu().numpy(), ref_idx, dw.cpu().numpy(), SCORE_SOFTMAX)
    assert np.abs(dl.cpu().numpy() - ref).max() <= 2e-5 * np.abs(ref).max()
    idx1, _ = moe_route_topk(logits, 1)
    dl1 = moe_route_topk_bwd(logits, idx1, dw[:, :1].contiguous(), SCORE_SOFTMAX)
    torch.cuda.synchronize()
    assert (dl1 == 0).all()
