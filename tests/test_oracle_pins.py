"""Pins of the CPU oracle against things other than itself.

Each test checks the oracle against the pages' definitions, closed forms,
library routines (numpy / torch fp64 on the CPU), brute force on tiny inputs
or invariants, chosen so that a dropped term, a wrong sign, a wrong index or
a transposed operand in the oracle fails at least one of them.  No GPU.
"""
import itertools
import math
import os

import numpy as np
import pytest
import torch

import oracle
from mixture_experts_ffn_warp_gb300.synthetic import CONFIGS, make_inputs, small_shape, skew_bias

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _expand(field: str):
    out = []
    for tok in field.split(","):
        tok = tok.strip()
        if "*" in tok:
            v, n = tok.split("*")
            out += [v] * int(n)
        else:
            out.append(tok)
    return out


def _lines(name):
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                yield [p.strip() for p in line.split(";")]


def _bits_of(vals):
    return np.array([oracle.double_to_bf16_bits(np.array(float(v))) for v in vals], dtype=np.uint16)


# ------------------------------------------------------------ number formats

def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(1)
    vals = np.concatenate([rng.standard_normal(4000).astype(np.float32),
                           (rng.standard_normal(1000) * 1e-39).astype(np.float32),   # subnormals
                           np.array([3.3895314e38, -3.3895314e38, 0.0, -0.0, 1.0], np.float32)])
    want = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle.double_to_bf16_bits(vals.astype(np.float64))
    assert np.array_equal(got, want)
    # ties go to even: 1 + 2^-8 is halfway between 1 and 1 + 2^-7
    assert oracle.double_to_bf16_bits(np.array(1.0 + 2.0 ** -8)) == 0x3F80
    assert oracle.double_to_bf16_bits(np.array(1.0 + 3 * 2.0 ** -8)) == 0x3F82


def test_e4m3_decode_matches_torch_table():
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([oracle.e4m3_to_double(int(c)) for c in range(256)])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    # spec facts of E4M3
    assert oracle.e4m3_to_double(0x7E) == 448.0
    assert oracle.e4m3_to_double(0x08) == 2.0 ** -6
    assert oracle.e4m3_to_double(0x01) == 2.0 ** -9


def test_e4m3_encode_matches_torch_rne_in_range():
    rng = np.random.default_rng(2)
    vals = np.concatenate([rng.uniform(-447, 447, 3000), rng.standard_normal(3000) * 0.01,
                           rng.standard_normal(1000)]).astype(np.float32)
    ref = torch.from_numpy(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.double_to_e4m3(float(v)) for v in vals], dtype=np.uint8)
    assert np.array_equal(got, ref)
    # round trip of every finite code
    for c in range(256):
        v = oracle.e4m3_to_double(c)
        if math.isnan(v):
            continue
        back = oracle.double_to_e4m3(v)
        assert back == c or (v == 0.0 and (back & 0x7F) == 0)
    # saturation (the conversion is "satfinite")
    assert oracle.double_to_e4m3(1e6) == 0x7E and oracle.double_to_e4m3(-465.0) == 0xFE


@pytest.mark.parametrize("case", list(_lines("mx_blocks.txt")), ids=lambda c: c[0])
def test_mx_block_golden(case):
    name, vals, scale, codes = case
    vals = [float(v) for v in _expand(vals)]
    assert len(vals) == 32
    bits = _bits_of(vals)
    assert np.array_equal(oracle.bits_to_float(bits), np.array(vals)), "fixture values must be bf16-exact"
    data, sc = oracle.quantize_rows_mxfp8(bits.reshape(1, 32))
    assert sc[0, 0] == int(scale, 16)
    assert [int(c, 16) for c in _expand(codes)] == list(data[0])


def test_mx_quantize_layouts_and_error_bound():
    rng = np.random.default_rng(3)
    m = torch.from_numpy(rng.standard_normal((64, 96)).astype(np.float32)).to(torch.bfloat16)
    bits = oracle.bf16_bits(m)
    rq, rs = oracle.quantize_rows_mxfp8(bits)                  # along the 96-long rows
    cq, cs = oracle.quantize_cols_mxfp8(bits[:, :64].copy())   # along the 64-long columns
    assert rq.shape == (64, 96) and rs.shape == (64, 3)
    assert cq.shape == (64, 64) and cs.shape == (64, 2)
    # column quantisation of M equals row quantisation of M^T
    tq, ts = oracle.quantize_rows_mxfp8(np.ascontiguousarray(bits[:, :64].T))
    assert np.array_equal(cq, tq) and np.array_equal(cs, ts)
    # dequantised values are within half an E4M3 step (relative 2^-4) of the input, or below
    # the smallest subnormal step of the block; the rounded-up scale never saturates
    deq = np.vectorize(oracle.e4m3_to_double)(rq) * np.exp2(np.repeat(rs.astype(np.int64) - 127, 32, axis=1))
    x = oracle.bits_to_float(bits)
    X = np.repeat(rs.astype(np.int64) - 127, 32, axis=1)
    tol = np.maximum(np.abs(x) * 2.0 ** -4, np.exp2(X - 10.0))
    assert np.all(np.abs(x) <= 448.0 * np.exp2(X))
    assert np.all(np.abs(deq - x) <= tol)
    # the scale is the smallest power of two that avoids saturation
    amax = np.abs(x).reshape(64, 3, 32).max(2)
    Xb = rs.astype(np.int64) - 127
    assert np.all(amax <= 448.0 * np.exp2(Xb)) and np.all(amax > 448.0 * np.exp2(Xb - 1))


# ------------------------------------------------------------ A1 routing

def _brute_topk(row, k):
    """Enumerate all k-subsets; the selected set is the one whose worst member
    ranks before the best non-member, ordered by the ranking."""
    E = len(row)

    def key(e):
        v = row[e]
        return (1, 0.0, e) if math.isnan(v) else (0, -v, e)   # sort ascending

    best = None
    for S in itertools.combinations(range(E), k):
        rest = [e for e in range(E) if e not in S]
        if not rest or max(key(e) for e in S) < min(key(e) for e in rest):
            assert best is None
            best = sorted(S, key=key)
    return best


def test_topk_brute_force_tiny():
    inp = make_inputs(CONFIGS["tiny"])
    lg = inp["logits"].numpy()
    idx, w = oracle.route_topk(lg, 2)
    for t in range(lg.shape[0]):
        assert list(idx[t]) == _brute_topk(lg[t], 2)


def test_topk_ties_integer_logits_vs_stable_lexsort():
    rng = np.random.default_rng(4)
    lg = rng.integers(-3, 4, size=(500, 16)).astype(np.float32)
    idx, _ = oracle.route_topk(lg, 5)
    for t in range(lg.shape[0]):
        order = np.lexsort((np.arange(16), -lg[t]))      # by -logit, then by id
        assert list(idx[t]) == list(order[:5])
        assert list(idx[t]) == _brute_topk(lg[t], 5) if t < 40 else True


@pytest.mark.parametrize("case", list(_lines("topk_ties.txt")), ids=lambda c: c[0])
def test_topk_golden(case):
    row = np.array([float(v) for v in case[0].split(",")], np.float32)
    want = [int(v) for v in case[1].split(",")]
    idx, w = oracle.route_topk(row.reshape(1, 8), 3)
    assert list(idx[0]) == want


def test_topk_weights_softmax_of_selected():
    inp = make_inputs(CONFIGS["fine_grained"], weights=False)
    lg = inp["logits"][:256].numpy()
    idx, w = oracle.route_topk(lg, 6)
    sel = torch.from_numpy(np.take_along_axis(lg, idx, axis=1)).double()
    ref = torch.softmax(sel, dim=1).numpy()
    assert np.allclose(w, ref, rtol=2 ** -23, atol=0)
    # equals the softmax over all E renormalised over the top-k
    full = torch.softmax(torch.from_numpy(lg).double(), dim=1).numpy()
    ren = np.take_along_axis(full, idx, axis=1)
    ren = ren / ren.sum(1, keepdims=True)
    assert np.allclose(w, ren, rtol=1e-6)
    # closed forms of the golden rows: equal logits share equally; 5,5,2
    _, w1 = oracle.route_topk(np.array([[1, 3, 3, 2, 3, 0, 0, 1]], np.float32), 3)
    assert np.allclose(w1, 1.0 / 3.0, rtol=2 ** -23)
    _, w3 = oracle.route_topk(np.array([[-np.inf, 5, -np.inf, 5, 1, np.nan, 2, 2]], np.float32), 3)
    e3 = math.exp(-3.0)
    assert np.allclose(w3[0], [1 / (2 + e3), 1 / (2 + e3), e3 / (2 + e3)], rtol=2 ** -23)
    # every selected logit -inf -> every weight 0
    _, w4 = oracle.route_topk(np.array([[np.nan, np.nan] + [-np.inf] * 6], np.float32), 3)
    assert np.all(w4 == 0.0)


def test_skewed_workload_has_zero_token_experts():
    b = skew_bias(128)
    assert torch.isinf(b[7::8]).all() and torch.isfinite(b[0::8]).all()
    lg = torch.randn(2048, 128, generator=torch.Generator().manual_seed(0)) + b
    idx, _ = oracle.route_topk(lg.numpy(), 8)
    assert not np.isin(np.arange(7, 128, 8), idx).any()


# ------------------------------------------------------------ A2 permutation

def _check_perm(idx, E, align, p):
    T, k = idx.shape
    flat = idx.reshape(-1)
    valid = (flat >= 0) & (flat < E)
    order = np.argsort(np.where(valid, flat, E), kind="stable")[: valid.sum()]
    sizes = np.bincount(flat[valid], minlength=E)
    assert np.array_equal(p["group_sizes"], sizes)
    padded = (sizes + align - 1) // align * align
    assert np.array_equal(p["group_offsets"], np.concatenate([[0], np.cumsum(padded)]))
    src = p["src_of_row"]
    rows = [src[p["group_offsets"][e]: p["group_offsets"][e] + sizes[e]] for e in range(E)]
    assert np.array_equal(np.concatenate(rows), order)          # stable argsort of expert ids
    dst = p["dst_of_route"].reshape(-1)
    assert np.all(dst[~valid] == -1)
    assert np.array_equal(src[dst[valid]], np.nonzero(valid)[0])  # inverse maps
    assert len(set(dst[valid].tolist())) == valid.sum()            # injective
    pad_rows = np.ones(len(src), bool)
    pad_rows[dst[valid]] = False
    assert np.all(src[pad_rows] == -1)
    assert p["n_invalid"] == int(((flat != -1) & ~valid).sum())


@pytest.mark.parametrize("align", [1, 4, 128])
def test_permute_vs_stable_argsort(align):
    inp = make_inputs(CONFIGS["fine_grained"], weights=False)
    idx, _ = oracle.route_topk(inp["logits"].numpy(), 6)
    p = oracle.permute(idx, 64, align=align)
    _check_perm(idx, 64, align, p)
    if align == 1:
        assert p["group_sizes"].sum() == idx.size and p["group_offsets"][-1] == idx.size


def test_permute_dropped_and_invalid_routes():
    rng = np.random.default_rng(5)
    idx = rng.integers(-1, 9, size=(300, 4)).astype(np.int32)
    idx[5, 1] = 100
    idx[7, 0] = -7
    p = oracle.permute(idx, 8)
    _check_perm(idx, 8, 1, p)
    assert p["n_invalid"] == int(((idx >= 8) | (idx < -1)).sum())


def test_gather_rows_bitwise():
    inp = make_inputs(CONFIGS["tiny"])
    idx, _ = oracle.route_topk(inp["logits"].numpy(), 2)
    p = oracle.permute(idx, 8, align=8)
    xb = oracle.bf16_bits(inp["x"])
    rows = int(p["group_offsets"][-1])
    xp = oracle.gather_rows(xb, 2, p["src_of_row"], rows)
    dst = p["dst_of_route"]
    for t in range(64):
        for j in range(2):
            assert np.array_equal(xp[dst[t, j]], xb[t])
    assert np.all(xp[p["src_of_row"][:rows] < 0] == 0)


# ------------------------------------------------------------ A5 combine

def test_identity_experts_return_input():
    """Experts set to identity (y_perm = x_perm) with weights summing to 1
    give back x to within one bf16 rounding."""
    inp = make_inputs(CONFIGS["fine_grained"], weights=False)
    lg = inp["logits"][:512].numpy()
    idx, w = oracle.route_topk(lg, 6)
    p = oracle.permute(idx, 64)
    xb = oracle.bf16_bits(inp["x"][:512])
    xp = oracle.bits_to_float(oracle.gather_rows(xb, 6, p["src_of_row"], idx.size)).astype(np.float32)
    out = oracle.unpermute_combine(xp, p["dst_of_route"], w, round_mode=0)
    x = oracle.bits_to_float(xb)
    s = w.astype(np.float64).sum(1, keepdims=True)
    assert np.allclose(out, x * s, rtol=1e-15, atol=0)
    assert np.all(np.abs(s - 1) < 1e-6)
    out_r = oracle.unpermute_combine(xp, p["dst_of_route"], w, round_mode=1)
    assert np.all(np.abs(out_r - x) <= np.abs(x) * 2.0 ** -7)


def test_combine_slot_weights_and_drops():
    yb = np.array([[1.0, 2.0], [10.0, -4.0], [0.5, 0.25]], np.float32)
    dst = np.array([[1, 0], [-1, 2]], np.int32)
    w = np.array([[0.25, 0.75], [0.9, 2.0]], np.float32)
    out = oracle.unpermute_combine(yb, dst, w, round_mode=0)
    assert np.array_equal(out, [[0.25 * 10 + 0.75 * 1, 0.25 * -4 + 0.75 * 2], [1.0, 0.5]])


# ------------------------------------------------------------ A3/A4 experts

def _golden_values(name):
    return {k: float(v) for k, v in _lines(name)}


def test_swiglu_route_closed_form():
    g = _golden_values("swiglu_route.txt")
    x = oracle.double_to_bf16_bits(np.array([[1.0, 2.0]]))
    Wg = oracle.double_to_bf16_bits(np.array([[[0.5], [0.25]]]))
    Wu = oracle.double_to_bf16_bits(np.array([[[1.0], [0.5]]]))
    Wd = oracle.double_to_bf16_bits(np.array([[[0.5, -1.0]]]))
    idx = np.zeros((1, 1), np.int32)
    w = np.ones((1, 1), np.float32)
    r = oracle.moe_fwd(x, Wg, Wu, Wd, idx, w, round_mode=0, want_h=True, want_y=True, want_fc1=True)
    assert np.allclose(r["fc1"][0], [1.0, 2.0], rtol=0, atol=0)
    assert abs(r["h"][0, 0] - g["h"]) < 1e-15
    assert np.allclose(r["out"][0], [g["y0"], g["y1"]], rtol=1e-15, atol=0)
    dY = oracle.double_to_bf16_bits(np.array([[1.0, 1.0]]))
    b = oracle.moe_bwd(x, Wg, Wu, Wd, idx, w, dY, round_mode=0)
    assert np.allclose(b["dx"][0], [g["dx0"], g["dx1"]], rtol=1e-14, atol=0)
    assert np.allclose(b["dW_gate"][0, :, 0], [g["dg"], 2 * g["dg"]], rtol=1e-14, atol=0)
    assert np.allclose(b["dW_up"][0, :, 0], [g["du"], 2 * g["du"]], rtol=1e-14, atol=0)
    assert np.allclose(b["dW_down"][0, 0], [g["h"], g["h"]], rtol=1e-14, atol=0)
    assert abs(b["d_topk_w"][0, 0] - g["d_topk_w"]) < 1e-14


def _rand_problem(seed, T, H, F, E, k):
    shape = small_shape("pin", T=T, H=H, F=F, E=E, k=k, backward=True)
    inp = make_inputs(shape, seed=seed)
    idx, w = oracle.route_topk(inp["logits"].numpy(), k)
    bits = {n: oracle.bf16_bits(inp[n]) for n in ("x", "W_gate", "W_up", "W_down", "dY")}
    return inp, idx, w, bits


def _torch_moe(inp, idx, w):
    """Independent fp64 torch implementation (autograd-capable) of the
    per-token MoE forward: out[t] = sum_j w_j * (silu(x Wg) * (x Wu)) Wd."""
    x = inp["x"].double().requires_grad_(True)
    Wg = inp["W_gate"].double().requires_grad_(True)
    Wu = inp["W_up"].double().requires_grad_(True)
    Wd = inp["W_down"].double().requires_grad_(True)
    tw = torch.from_numpy(w).double().requires_grad_(True)
    T, k = idx.shape
    out = torch.zeros(T, x.shape[1], dtype=torch.float64)
    for e in range(Wg.shape[0]):
        t_sel, j_sel = np.nonzero(idx == e)
        if len(t_sel) == 0:
            continue
        ts = torch.from_numpy(t_sel)
        xe = x[ts]
        he = torch.nn.functional.silu(xe @ Wg[e]) * (xe @ Wu[e])
        ye = he @ Wd[e]
        out = out.index_add(0, ts, tw[ts, torch.from_numpy(j_sel)].unsqueeze(1) * ye)
    return out, (x, Wg, Wu, Wd, tw)


def test_dense_special_case_E1_k1_vs_torch_matmul():
    """E = 1, k = 1 reduces to a dense SwiGLU MLP."""
    inp, idx, w, b = _rand_problem(6, T=24, H=64, F=96, E=1, k=1)
    assert np.all(idx == 0) and np.all(w == 1.0)
    r = oracle.moe_fwd(b["x"], b["W_gate"], b["W_up"], b["W_down"], idx, w, round_mode=0)
    x = inp["x"].double()
    ref = (torch.nn.functional.silu(x @ inp["W_gate"][0].double()) * (x @ inp["W_up"][0].double())) \
        @ inp["W_down"][0].double()
    assert np.allclose(r["out"], ref.numpy(), rtol=1e-12, atol=1e-15)


def test_forward_vs_torch_fp64_multi_expert():
    inp, idx, w, b = _rand_problem(7, T=40, H=64, F=32, E=6, k=3)
    r = oracle.moe_fwd(b["x"], b["W_gate"], b["W_up"], b["W_down"], idx, w, round_mode=0)
    ref, _ = _torch_moe(inp, idx, w)
    assert np.allclose(r["out"], ref.detach().numpy(), rtol=1e-12, atol=1e-16)
    # round_mode 1 stays within the stated bf16 tolerance of the exact result
    r1 = oracle.moe_fwd(b["x"], b["W_gate"], b["W_up"], b["W_down"], idx, w, round_mode=1)
    rms = np.sqrt((r["out"] ** 2).mean())
    assert np.abs(r1["out"] - r["out"]).max() <= 2e-2 * rms


def test_forward_rounding_points_vs_torch_bf16_stores():
    """round_mode 1 stores h and the expert output y in bf16 and rounds the output: an
    independent torch implementation that casts to bf16 (torch's own RNE conversion) at
    exactly those three points gives the same values.  A rounding point left out or moved
    (y unrounded, h rounded after Wd, out rounded per slot) changes many elements."""
    inp, idx, w, b = _rand_problem(16, T=40, H=64, F=96, E=6, k=3)
    r = oracle.moe_fwd(b["x"], b["W_gate"], b["W_up"], b["W_down"], idx, w, round_mode=1,
                       want_h=True, want_y=True)
    x = inp["x"].double()
    T, k = idx.shape
    out = torch.zeros(T, x.shape[1], dtype=torch.float64)
    bf = lambda v: v.to(torch.bfloat16).double()  # noqa: E731
    for t in range(T):
        for j in range(k):
            e = int(idx[t, j])
            hr = bf(torch.nn.functional.silu(x[t] @ inp["W_gate"][e].double()) * (x[t] @ inp["W_up"][e].double()))
            yr = bf(hr @ inp["W_down"][e].double())
            assert np.array_equal(r["h"][t * k + j], hr.numpy())
            assert np.array_equal(r["y"][t * k + j], yr.numpy())
            out[t] += float(w[t, j]) * yr
    assert np.array_equal(r["out"], bf(out).numpy())
    # the unrounded y differs from the stored one: the rounding point is really there
    r0 = oracle.moe_fwd(b["x"], b["W_gate"], b["W_up"], b["W_down"], idx, w, round_mode=0, want_y=True)
    assert not np.array_equal(r0["y"], r["y"])


def test_zero_token_experts_contribute_nothing():
    inp, idx, w, b = _rand_problem(8, T=32, H=32, F=64, E=8, k=2)
    idx = np.where(idx >= 6, idx - 6, idx).astype(np.int32)      # experts 6, 7 get no tokens
    r = oracle.moe_fwd(b["x"], b["W_gate"], b["W_up"], b["W_down"], idx, w)
    Wg, Wu, Wd = (b[n].copy() for n in ("W_gate", "W_up", "W_down"))
    for W in (Wg, Wu, Wd):
        W[6:] = 0x7FC0                                            # NaN weights
    r2 = oracle.moe_fwd(b["x"], Wg, Wu, Wd, idx, w)
    assert np.array_equal(r["out"], r2["out"]) and np.isfinite(r2["out"]).all()
    bw = oracle.moe_bwd(b["x"], Wg, Wu, Wd, idx, w, b["dY"])
    assert np.all(bw["dW_gate"][6:] == 0) and np.all(bw["dW_up"][6:] == 0) and np.all(bw["dW_down"][6:] == 0)
    assert np.isfinite(bw["dx"]).all()


def test_dropped_routes_skip():
    inp, idx, w, b = _rand_problem(9, T=16, H=32, F=32, E=4, k=2)
    idx2 = idx.copy()
    idx2[:, 1] = -1
    r = oracle.moe_fwd(b["x"], b["W_gate"], b["W_up"], b["W_down"], idx2, w, round_mode=0)
    w1 = w.copy()
    w1[:, 1] = 0
    r1 = oracle.moe_fwd(b["x"], b["W_gate"], b["W_up"], b["W_down"], idx, w1, round_mode=0)
    assert np.allclose(r["out"], r1["out"], rtol=0, atol=0)


# ------------------------------------------------------------ A8 backward

def test_backward_vs_torch_autograd():
    inp, idx, w, b = _rand_problem(10, T=40, H=48, F=32, E=5, k=2)
    idx[3, 1] = -1                                               # one dropped route
    r = oracle.moe_bwd(b["x"], b["W_gate"], b["W_up"], b["W_down"], idx, w, b["dY"], round_mode=0)
    out, (x, Wg, Wu, Wd, tw) = _torch_moe(inp, idx, w)
    out.backward(inp["dY"].double())
    for name, ref in (("dx", x.grad), ("dW_gate", Wg.grad), ("dW_up", Wu.grad), ("dW_down", Wd.grad)):
        assert np.allclose(r[name], ref.numpy(), rtol=1e-10, atol=1e-14), name
    ref_dtw = tw.grad.numpy().copy()
    ref_dtw[idx < 0] = 0
    assert np.allclose(r["d_topk_w"], ref_dtw, rtol=1e-10, atol=1e-14)


def test_backward_central_differences():
    """Finite differences of the exact (round_mode 0) forward w.r.t. the
    router weights and one weight entry."""
    inp, idx, w, b = _rand_problem(11, T=6, H=16, F=16, E=3, k=2)
    dY = oracle.bits_to_float(b["dY"])
    r = oracle.moe_bwd(b["x"], b["W_gate"], b["W_up"], b["W_down"], idx, w, b["dY"], round_mode=0)
    # the forward is linear in each router weight: d/dw_(t,j) <dY, out> = <dY[t], y(t,j)>
    f0 = oracle.moe_fwd(b["x"], b["W_gate"], b["W_up"], b["W_down"], idx, w, round_mode=0, want_y=True)
    y = f0["y"].reshape(6, 2, 16)
    assert np.allclose(r["d_topk_w"], np.einsum("tn,tjn->tj", dY, y), rtol=1e-12)
    # d/dWg[e,h,f]: perturb one entry by a bf16-representable step in both directions
    e, hh, ff = int(idx[0, 0]), 3, 5
    base = oracle.bits_to_float(b["W_gate"][e, hh, ff])

    def loss(val):
        Wg = b["W_gate"].copy()
        Wg[e, hh, ff] = oracle.double_to_bf16_bits(np.array(val))
        return float((oracle.moe_fwd(b["x"], Wg, b["W_up"], b["W_down"], idx, w, round_mode=0)["out"] * dY).sum())

    step = 2.0 ** (math.floor(math.log2(abs(base))) - 6)
    fd = (loss(base + step) - loss(base - step)) / (2 * step)
    assert abs(fd - r["dW_gate"][e, hh, ff]) <= 1e-3 * abs(r["dW_gate"][e, hh, ff]) + 1e-9


def test_sampled_backward_functions_agree_with_full():
    inp, idx, w, b = _rand_problem(12, T=24, H=32, F=32, E=4, k=2)
    full = oracle.moe_bwd(b["x"], b["W_gate"], b["W_up"], b["W_down"], idx, w, b["dY"])
    toks = np.array([0, 5, 23])
    dx = oracle.moe_bwd_dx_tokens(b["x"], b["W_gate"], b["W_up"], b["W_down"], idx, w, b["dY"], toks)
    assert np.array_equal(dx["dx"], full["dx"][toks])
    assert np.array_equal(dx["d_topk_w"], full["d_topk_w"][toks])
    ents = [(0, 1, 3, 4), (1, 2, 0, 31), (2, 3, 7, 9), (2, 0, 31, 0)]
    vals = oracle.moe_bwd_dw_entries(ents, b["x"], b["W_gate"], b["W_up"], b["W_down"], idx, w, b["dY"])
    ref = [full["dW_gate"][1, 3, 4], full["dW_up"][2, 0, 31], full["dW_down"][3, 7, 9], full["dW_down"][0, 31, 0]]
    # same definition, summed in a different order
    assert np.allclose(vals, ref, rtol=1e-12, atol=0)


# ------------------------------------------------------------ A7 MXFP8 forward

def _quantize_experts(b, E):
    q = {}
    for e in range(E):
        q.setdefault("gq", []), q.setdefault("gs", []), q.setdefault("uq", []), q.setdefault("us", [])
        q.setdefault("dq", []), q.setdefault("ds", [])
        a, s = oracle.quantize_cols_mxfp8(b["W_gate"][e]); q["gq"].append(a); q["gs"].append(s)
        a, s = oracle.quantize_cols_mxfp8(b["W_up"][e]); q["uq"].append(a); q["us"].append(s)
        a, s = oracle.quantize_cols_mxfp8(b["W_down"][e]); q["dq"].append(a); q["ds"].append(s)
    return q


def test_mxfp8_forward_exact_operands_match_bf16_up_to_h():
    """With x and weights exactly representable in MXFP8, the MXFP8 forward
    differs from the exact forward only by the quantisation of h (relative
    2^-4 per element at most) -- and a transposed weight or a wrong scale
    index would break both bounds below."""
    rng = np.random.default_rng(13)
    T, H, F, E, k = 8, 64, 64, 3, 2
    grid = np.array([0.0, 0.25, 0.5, 0.75, 1.0, -0.25, -0.5, -1.0])
    x = oracle.double_to_bf16_bits(rng.choice(grid, size=(T, H)) * 2.0)
    Wg = oracle.double_to_bf16_bits(rng.choice(grid, size=(E, H, F)) * 0.03125)
    Wu = oracle.double_to_bf16_bits(rng.choice(grid, size=(E, H, F)) * 0.03125)
    Wd = oracle.double_to_bf16_bits(rng.choice(grid, size=(E, F, H)) * 0.0625)
    b = {"x": x, "W_gate": Wg, "W_up": Wu, "W_down": Wd}
    lg = rng.standard_normal((T, E)).astype(np.float32)
    idx, w = oracle.route_topk(lg, k)
    q = _quantize_experts(b, E)
    # exactly representable: dequantised codes reproduce the inputs
    deq = np.vectorize(oracle.e4m3_to_double)(q["gq"][0]) * np.exp2(np.repeat(q["gs"][0].astype(int) - 127, 32, axis=1))
    assert np.array_equal(deq, oracle.bits_to_float(Wg[0]).T)
    mx = oracle.moe_fwd_mxfp8(x, q["gq"], q["gs"], q["uq"], q["us"], q["dq"], q["ds"], idx, w, round_mode=0)
    ex = oracle.moe_fwd(x, Wg, Wu, Wd, idx, w, round_mode=0, want_h=True)
    # bound: |dy_n| <= sum_f |dh_f| |Wd[f,n]|, |dh_f| <= 2^-4 |h_f| (normal range) + subnormal step
    bound = np.zeros((T, H))
    for t in range(T):
        for j in range(k):
            e = idx[t, j]
            h = ex["h"][t * k + j]
            bound[t] += w[t, j] * (np.abs(h) * 2.0 ** -4 + 2.0 ** -20) @ np.abs(oracle.bits_to_float(Wd[e]))
    assert np.all(np.abs(mx["out"] - ex["out"]) <= bound + 1e-15)
    assert np.abs(mx["out"] - ex["out"]).max() > 0      # h quantisation is really applied


def test_mxfp8_forward_close_to_exact_on_random_inputs():
    inp, idx, w, b = _rand_problem(14, T=16, H=64, F=96, E=4, k=2)
    q = _quantize_experts(b, 4)
    mx = oracle.moe_fwd_mxfp8(b["x"], q["gq"], q["gs"], q["uq"], q["us"], q["dq"], q["ds"], idx, w)
    ex = oracle.moe_fwd(b["x"], b["W_gate"], b["W_up"], b["W_down"], idx, w, round_mode=0)
    # E4M3 keeps 3 mantissa bits (relative half-step 2^-4, ~3.6% RMS per element); with x, the
    # weights and h each quantised the output's relative RMS error is ~10%.  A transposed operand
    # or a wrong scale index gives errors of order 100%.
    rms = np.sqrt((ex["out"] ** 2).mean())
    rel = np.sqrt(((mx["out"] - ex["out"]) ** 2).mean()) / rms
    assert 1e-3 < rel < 0.15


def test_round_mode_2_is_mode_1_before_the_final_rounding():
    inp, idx, w, b = _rand_problem(15, T=20, H=32, F=64, E=4, k=2)
    f1 = oracle.moe_fwd(b["x"], b["W_gate"], b["W_up"], b["W_down"], idx, w, round_mode=1, want_y=True)
    f2 = oracle.moe_fwd(b["x"], b["W_gate"], b["W_up"], b["W_down"], idx, w, round_mode=2, want_y=True)
    assert np.array_equal(f1["y"], f2["y"])                      # same intermediates
    assert np.array_equal(oracle.round_bf16(f2["out"]), f1["out"])
    assert not np.array_equal(f2["out"], f1["out"])
    g1 = oracle.moe_bwd(b["x"], b["W_gate"], b["W_up"], b["W_down"], idx, w, b["dY"], round_mode=1)
    g2 = oracle.moe_bwd(b["x"], b["W_gate"], b["W_up"], b["W_down"], idx, w, b["dY"], round_mode=2)
    assert np.array_equal(oracle.round_bf16(g2["dx"]), g1["dx"])
    for n in ("dW_gate", "dW_up", "dW_down"):                   # fp32 on the path: never rounded
        assert np.array_equal(g2[n], g1[n]), n
