"""Pins of the oracle's router variants (CPU only): the sigmoid score function
with an expert routing bias, and the router backward for both score functions.

Each pin checks the oracle against something other than itself: the softmax
router, torch's fp64 sigmoid and autograd, numpy's stable sort, finite
differences, and special cases with a known answer."""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _logits(T, E, seed):
    return np.random.default_rng(seed).standard_normal((T, E)).astype(np.float32)


def _select_by_keys(keys: np.ndarray, k: int) -> np.ndarray:
    """Top-k by (key descending, expert id ascending) with numpy's stable sort."""
    T, E = keys.shape
    out = np.empty((T, k), np.int64)
    for t in range(T):
        out[t] = np.lexsort((np.arange(E), -keys[t]))[:k]
    return out


def test_sigmoid_without_bias_selects_like_the_softmax_router():
    """sigmoid is increasing, so with no bias the selection is the logits' top-k."""
    lg = _logits(400, 64, 1)
    i_sig, _ = oracle.route_topk_sigmoid(lg, 6)
    i_soft, _ = oracle.route_topk(lg, 6)
    assert np.array_equal(i_sig, i_soft)


@pytest.mark.parametrize("normalize", [True, False])
def test_sigmoid_router_matches_torch_fp64(normalize):
    T, E, k = 300, 48, 5
    lg = _logits(T, E, 2)
    bias = (np.random.default_rng(3).standard_normal(E) * 0.3).astype(np.float32)
    idx, w = oracle.route_topk_sigmoid(lg, k, bias, normalize)
    s = torch.sigmoid(torch.from_numpy(lg).double()).numpy()
    ref_idx = _select_by_keys(s + bias.astype(np.float64), k)
    assert np.array_equal(idx, ref_idx)
    sel = np.take_along_axis(s, ref_idx, axis=1)
    ref_w = sel / (sel.sum(1, keepdims=True) + 1e-20) if normalize else sel
    np.testing.assert_allclose(w, ref_w.astype(np.float32), rtol=0, atol=0)   # fp32 rounding of the same double


def test_sigmoid_bias_drives_the_selection_only():
    """A strong bias forces experts into the top-k; their weights stay the unbiased scores."""
    T, E, k = 50, 32, 4
    lg = _logits(T, E, 4)
    bias = np.zeros(E, np.float32)
    bias[[3, 11]] = 10.0
    idx, w = oracle.route_topk_sigmoid(lg, k, bias, normalize=False)
    assert all({3, 11} <= set(r.tolist()) for r in idx)
    s = torch.sigmoid(torch.from_numpy(lg).double()).numpy()
    np.testing.assert_allclose(w, np.take_along_axis(s, idx.astype(np.int64), 1).astype(np.float32), atol=0)


def test_sigmoid_ties_go_to_the_lowest_expert_id():
    lg = np.zeros((3, 10), np.float32)
    idx, w = oracle.route_topk_sigmoid(lg, 4)
    assert (idx == np.arange(4)).all()
    np.testing.assert_allclose(w, 0.25, atol=0)


def test_sigmoid_underflow_gives_zero_weights_not_nan():
    """All selected scores ~0: weights / (sum + 1e-20) stays finite (the case the
    normalisation's epsilon exists for)."""
    lg = np.full((2, 8), -np.inf, np.float32)
    lg[1] = -200.0                      # sigmoid = e^-200 in double
    idx, w = oracle.route_topk_sigmoid(lg, 3)
    assert np.isfinite(w).all() and (w == 0).all()
    assert (idx == np.arange(3)).all()


def _autograd_dlogits(lg, idx, g, score_fn, normalize):
    l = torch.from_numpy(lg).double().requires_grad_(True)
    ii = torch.from_numpy(np.where(idx < 0, 0, idx).astype(np.int64))
    valid = torch.from_numpy(idx >= 0)
    sel = torch.gather(l, 1, ii)
    if score_fn == oracle.SCORE_SOFTMAX:
        sel = torch.where(valid, sel, torch.full_like(sel, -torch.inf))
        w = torch.softmax(sel, dim=1)
    else:
        s = torch.where(valid, torch.sigmoid(sel), torch.zeros_like(sel))
        w = s / (s.sum(1, keepdim=True) + 1e-20) if normalize else s
    (w * torch.from_numpy(g).double() * valid).sum().backward()
    return l.grad.numpy()


@pytest.mark.parametrize("score_fn,normalize", [(oracle.SCORE_SOFTMAX, True), (oracle.SCORE_SIGMOID, True),
                                                (oracle.SCORE_SIGMOID, False)])
def test_router_bwd_matches_fp64_autograd(score_fn, normalize):
    T, E, k = 64, 32, 4
    lg = _logits(T, E, 5)
    if score_fn == oracle.SCORE_SOFTMAX:
        idx, _ = oracle.route_topk(lg, k)
    else:
        idx, _ = oracle.route_topk_sigmoid(lg, k, normalize=normalize)
    idx = idx.copy()
    idx[::7, 2] = -1                    # dropped routes get no gradient
    g = np.random.default_rng(6).standard_normal((T, k)).astype(np.float32)
    got = oracle.route_topk_bwd(lg, idx, g, score_fn, normalize)
    ref = _autograd_dlogits(lg, idx, g, score_fn, normalize)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-15)
    selected = np.zeros((T, E), bool)
    for t, j in zip(*np.nonzero(idx >= 0)):
        selected[t, idx[t, j]] = True
    assert (got[~selected] == 0).all()


def test_router_bwd_single_expert_softmax_is_zero():
    """k = 1 softmax: the weight is identically 1, so its logits get no gradient."""
    lg = _logits(20, 16, 7)
    idx, _ = oracle.route_topk(lg, 1)
    g = np.random.default_rng(8).standard_normal((20, 1)).astype(np.float32)
    assert (oracle.route_topk_bwd(lg, idx, g, oracle.SCORE_SOFTMAX) == 0).all()


def test_router_bwd_sigmoid_finite_differences():
    """Central differences of sum(g * w) through the oracle's own forward, at a
    selection that the step does not change."""
    T, E, k = 6, 12, 3
    lg = _logits(T, E, 9).astype(np.float64)
    idx, _ = oracle.route_topk_sigmoid(lg.astype(np.float32), k)
    g = np.random.default_rng(10).standard_normal((T, k)).astype(np.float32)
    got = oracle.route_topk_bwd(lg.astype(np.float32), idx, g, oracle.SCORE_SIGMOID)
    h = 2.0 ** -7
    for t in range(T):
        for j in range(k):
            e = idx[t, j]
            vals = []
            for sgn in (1, -1):
                p = lg.astype(np.float32).copy()
                p[t, e] += sgn * h
                i2, w2 = oracle.route_topk_sigmoid(p, k)
                assert np.array_equal(i2[t], idx[t])
                vals.append(float((g[t].astype(np.float64) * w2[t]).sum()))
            fd = (vals[0] - vals[1]) / (2 * h)
            assert abs(fd - got[t, e]) <= 2e-4 * max(1.0, abs(got[t, e])) + 2e-5, (t, e, fd, got[t, e])
