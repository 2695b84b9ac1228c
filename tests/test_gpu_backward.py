"""GPU parity of the backward (A8) against the CPU oracle, through the C ABI.

dx (bf16), the fp32 weight gradients and the fp32 route-weight gradients are
compared with the oracle's exact result of the same arithmetic (dy_perm and
dg/du rounded to bf16 where the path stores them; round_mode 2) at
max|err| <= 2e-2 * RMS.  Experts with no routes must get exactly zero weight
gradients."""
import numpy as np
import pytest
import torch

import oracle
from mixture_experts_ffn_warp_gb300 import MoeBackward, MoeForward, Workspace, moe_grouped_ffn_bwd, moe_grouped_wgrad
from mixture_experts_ffn_warp_gb300.synthetic import CONFIGS, small_shape
from helpers import assert_close_rms, assert_close_ulp, bits, gpu_inputs, host_experts, to_f64

pytestmark = pytest.mark.gpu

SHAPES = {
    "tiny": small_shape("tiny", T=64, H=128, F=256, E=8, k=2, backward=True),
    # ragged groups, several M tiles; 256-wide tiles everywhere
    "ragged": small_shape("ragged", T=300, H=256, F=512, E=5, k=2, backward=True),
    # 128-wide tiles (H % 256 and F % 256 != 0) in dgrad and wgrad
    "h384": small_shape("h384", T=257, H=384, F=384, E=7, k=3, backward=True),
    # wgrad tiles straddling the dW_gate | dW_up split (F % 256 != 0), long K per group
    "f1408": small_shape("f1408", T=1024, H=256, F=1408, E=4, k=2, backward=True),
    # many experts, several with no routes
    "many": small_shape("many", T=512, H=128, F=128, E=64, k=4, skew=True, backward=True),
    # >= 1024 rows per expert: the weight gradients on CTA pairs, with ragged K tails
    "pair_wgrad": small_shape("pair_wgrad", T=2200, H=256, F=256, E=4, k=2, backward=True),
    # the same with a Zipf-like load and one expert without routes
    "pair_wgrad_skew": small_shape("pair_wgrad_skew", T=4500, H=256, F=256, E=8, k=2, skew=True, backward=True),
}


def _run(shape, align=1):
    inp = gpu_inputs(shape, with_dy=True)
    m = MoeForward(shape.T, shape.H, shape.F, shape.E, shape.k, align=align, keep_fc1_c=True)
    m(inp["x"], inp["logits"], inp["W_gate"], inp["W_up"], inp["W_down"])
    b = MoeBackward(m)
    b(inp["dY"], inp["W_gate"], inp["W_up"], inp["W_down"])
    torch.cuda.synchronize()
    assert m.ws.read_error() == 0
    return inp, m, b


@pytest.mark.parametrize("name", list(SHAPES))
def test_backward_parity_small(name):
    shape = SHAPES[name]
    inp, m, b = _run(shape)
    idx, w = m.topk_idx.cpu().numpy(), m.topk_w.cpu().numpy()
    hb = {n: bits(inp[n]) for n in ("x", "W_gate", "W_up", "W_down", "dY")}
    ref = oracle.moe_bwd(hb["x"], hb["W_gate"], hb["W_up"], hb["W_down"], idx, w, hb["dY"], round_mode=2)
    assert_close_rms(to_f64(b.dx), ref["dx"], what="dx", bf16_out=True)
    for n in ("dW_gate", "dW_up", "dW_down"):
        assert_close_rms(getattr(b, n).double().cpu().numpy(), ref[n], what=n)
    assert_close_rms(b.d_topk_w.double().cpu().numpy(), ref["d_topk_w"], what="d_topk_w")
    # dy_perm = bf16(w * dY) on the forward rows
    dst = m.perm.dst_of_route.cpu().numpy()
    dY = oracle.bits_to_float(hb["dY"])
    used = int(m.perm.group_offsets[-1])
    want = np.zeros((used, shape.H))
    for t in range(shape.T):
        for j in range(shape.k):
            want[dst[t, j]] = oracle.round_bf16(np.float64(w[t, j]) * dY[t])
    assert_close_ulp(to_f64(b.dy_perm[:used]), want, what="dy_perm", slack=0.0)
    # experts without routes: exact zeros
    empty = (m.perm.group_sizes == 0).nonzero().flatten().tolist()
    if name == "many":
        assert len(empty) >= 8
    for e in empty:
        assert torch.count_nonzero(b.dW_gate[e]) == 0 and torch.count_nonzero(b.dW_up[e]) == 0
        assert torch.count_nonzero(b.dW_down[e]) == 0


def test_backward_aligned_groups_and_one_call_api():
    """Padded groups (align 8): padding rows get zero gradient rows, so the
    weight gradients are unchanged; the single-call ABI matches the steps."""
    shape = SHAPES["many"]
    inp, m, b = _run(shape, align=8)
    idx, w = m.topk_idx.cpu().numpy(), m.topk_w.cpu().numpy()
    hb = {n: bits(inp[n]) for n in ("x", "W_gate", "W_up", "W_down", "dY")}
    ref = oracle.moe_bwd(hb["x"], hb["W_gate"], hb["W_up"], hb["W_down"], idx, w, hb["dY"], round_mode=2)
    for n in ("dW_gate", "dW_up", "dW_down"):
        assert_close_rms(getattr(b, n).double().cpu().numpy(), ref[n], what=n)
    assert_close_rms(to_f64(b.dx), ref["dx"], what="dx", bf16_out=True)
    one = moe_grouped_ffn_bwd(inp["dY"], m.perm.x_perm, inp["W_gate"], inp["W_up"], inp["W_down"], m.fc1_c, m.h,
                              m.y_perm, m.perm, m.topk_w, m.ws)
    torch.cuda.synchronize()
    assert torch.equal(one["dx"], b.dx)
    for n in ("dW_gate", "dW_up", "dW_down", "d_topk_w"):
        assert torch.equal(one[n], getattr(b, n)), n


def test_backward_is_deterministic():
    shape = SHAPES["ragged"]
    inp, m, b = _run(shape)
    first = {n: getattr(b, n).clone() for n in ("dx", "dW_gate", "dW_up", "dW_down", "d_topk_w")}
    b(inp["dY"], inp["W_gate"], inp["W_up"], inp["W_down"])
    torch.cuda.synchronize()
    for n, v in first.items():
        assert torch.equal(v, getattr(b, n)), n


def _edge_or_random(rng, n):
    """A coordinate on a 128 / 256 tile edge (the last of a tile, the first of the next, the
    first or last overall) or a random one."""
    edges = [0, 127, 128, 255, 256, n - 257, n - 256, n - 1]
    return int(rng.choice(edges)) if rng.random() < 0.6 else int(rng.integers(n))


def test_backward_parity_mixtral_full_size_sampled():
    """Mixtral-like fwd+bwd at full size (T=8192, H=4096, F=14336, E=8, top-2),
    in the bench's launch configuration (expert groups padded to 16 rows): dx and d_topk_w of
    64 sampled tokens, and entries of every weight gradient of every expert -- most on the
    edges of the 256 x 256 gradient tiles (each entry sums over all of its expert's rows and
    its zero padding rows) -- against the oracle.  The tolerance scale is the RMS of the
    oracle's own values.  (The K tail of unpadded groups: test_wgrad_group_sizes_on_cta_pairs.)"""
    shape = CONFIGS["mixtral"]
    inp, m, b = _run(shape, align=16)
    idx, w = m.topk_idx.cpu().numpy(), m.topk_w.cpu().numpy()
    E, H, F = shape.E, shape.H, shape.F
    Wg, Wu, Wd = (host_experts(inp[n], range(E)) for n in ("W_gate", "W_up", "W_down"))
    xb, dyb = bits(inp["x"]), bits(inp["dY"])
    rng = np.random.default_rng(1)
    toks = np.sort(rng.choice(shape.T, size=64, replace=False))
    ref = oracle.moe_bwd_dx_tokens(xb, Wg, Wu, Wd, idx, w, dyb, toks, round_mode=2)
    sel = torch.from_numpy(toks).cuda()
    assert_close_rms(to_f64(b.dx[sel]), ref["dx"], what="mixtral dx", bf16_out=True)
    assert_close_rms(b.d_topk_w[sel].double().cpu().numpy(), ref["d_topk_w"], what="mixtral d_topk_w")
    ents = []
    for which, (a_dim, b_dim) in ((0, (H, F)), (1, (H, F)), (2, (F, H))):
        for e in range(E):
            for _ in range(5):
                ents.append((which, e, _edge_or_random(rng, a_dim), _edge_or_random(rng, b_dim)))
    vals = np.asarray(oracle.moe_bwd_dw_entries(ents, xb, Wg, Wu, Wd, idx, w, dyb, round_mode=2))
    grads = (b.dW_gate, b.dW_up, b.dW_down)
    got = np.array([float(grads[which][e, a, c]) for which, e, a, c in ents])
    for which in range(3):
        sel_w = np.array([i for i, q in enumerate(ents) if q[0] == which])
        rms = float(np.sqrt(np.mean(vals[sel_w] ** 2)))
        err = float(np.abs(got[sel_w] - vals[sel_w]).max())
        assert err <= 2e-2 * rms, f"dW[{which}] max|err| {err:.3e} > 2e-2 * RMS {rms:.3e}"


def test_wgrad_group_sizes_on_cta_pairs():
    """moe_grouped_wgrad on chosen group sizes (0 rows, fewer than 16, whole 16-row slices,
    ragged tails; >= 1024 rows per expert on average, so the CTA-pair kernel runs): each
    expert's gradients against the fp64 products of its rows."""
    H, F = 256, 512
    sizes = [0, 5, 16, 1100, 4077, 1000, 37, 2000]
    E, R = len(sizes), sum(sizes)
    assert R >= 1024 * E
    g = torch.Generator(device="cuda").manual_seed(11)
    x = torch.randn(R, H, generator=g, device="cuda").to(torch.bfloat16)
    h = torch.randn(R, F, generator=g, device="cuda").to(torch.bfloat16)
    dy = torch.randn(R, H, generator=g, device="cuda").to(torch.bfloat16)
    dgu = torch.randn(R, 2 * F, generator=g, device="cuda").to(torch.bfloat16)
    offs = torch.tensor(np.concatenate([[0], np.cumsum(sizes)]), dtype=torch.int32, device="cuda")
    dWg = torch.full((E, H, F), float("nan"), device="cuda")
    dWu = torch.full((E, H, F), float("nan"), device="cuda")
    dWd = torch.full((E, F, H), float("nan"), device="cuda")
    ws = Workspace(R, E, 1)
    moe_grouped_wgrad(x, h, dy, dgu, offs, ws, dWg, dWu, dWd)
    torch.cuda.synchronize()
    assert ws.read_error() == 0
    xd, hd, dyd, dgud = (t.double().cpu() for t in (x, h, dy, dgu))
    o = offs.cpu().tolist()
    for e in range(E):
        r0, r1 = o[e], o[e + 1]
        want = {"dW_down": hd[r0:r1].T @ dyd[r0:r1], "dW_gate": xd[r0:r1].T @ dgud[r0:r1, :F],
                "dW_up": xd[r0:r1].T @ dgud[r0:r1, F:]}
        for n, got in (("dW_down", dWd[e]), ("dW_gate", dWg[e]), ("dW_up", dWu[e])):
            got = got.double().cpu()
            if sizes[e] == 0:
                assert torch.count_nonzero(got) == 0, (e, n)
                continue
            err = (got - want[n]).abs().max().item()
            assert err <= 1e-4 * want[n].abs().max().item(), (e, n, err)   # fp32 accumulation


@pytest.mark.parametrize("sizes", [[0, 5, 16, 1100, 4077, 1000, 37, 2000],   # CTA pairs (>= 1024 rows on average)
                                   [0, 5, 16, 300, 77, 129, 37, 200]])       # the one-CTA kernels
def test_wgrad_bf16_is_the_rounded_fp32(sizes):
    """moe_grouped_wgrad_bf16 stores the same fp32 accumulators as moe_grouped_wgrad, each rounded
    to the nearest bf16 (ties to even) once: bit for bit, on both weight-gradient kernels, with
    experts of no rows (exact zeros), of fewer than 16 rows and of ragged tails."""
    H, F = 256, 512
    E, R = len(sizes), sum(sizes)
    g = torch.Generator(device="cuda").manual_seed(12)
    x = torch.randn(R, H, generator=g, device="cuda").to(torch.bfloat16)
    h = torch.randn(R, F, generator=g, device="cuda").to(torch.bfloat16)
    dy = torch.randn(R, H, generator=g, device="cuda").to(torch.bfloat16)
    dgu = torch.randn(R, 2 * F, generator=g, device="cuda").to(torch.bfloat16)
    offs = torch.tensor(np.concatenate([[0], np.cumsum(sizes)]), dtype=torch.int32, device="cuda")
    ws = Workspace(R, E, 1)
    out = {}
    for dt in (torch.float32, torch.bfloat16):
        dWg = torch.full((E, H, F), float("nan"), device="cuda", dtype=dt)
        dWu = torch.full((E, H, F), float("nan"), device="cuda", dtype=dt)
        dWd = torch.full((E, F, H), float("nan"), device="cuda", dtype=dt)
        moe_grouped_wgrad(x, h, dy, dgu, offs, ws, dWg, dWu, dWd)
        out[dt] = (dWg, dWu, dWd)
    torch.cuda.synchronize()
    assert ws.read_error() == 0
    for f32, b16 in zip(out[torch.float32], out[torch.bfloat16]):
        assert torch.equal(f32.to(torch.bfloat16), b16)
    assert torch.count_nonzero(out[torch.bfloat16][0][0]) == 0   # the expert without rows


def test_one_call_backward_with_bf16_weight_gradients():
    """moe_grouped_ffn_bwd_bf16: dx and d_topk_w as moe_grouped_ffn_bwd, the weight gradients its
    fp32 ones rounded to bf16."""
    shape = SHAPES["ragged"]
    inp, m, b = _run(shape)
    res = {}
    for dt in (torch.float32, torch.bfloat16):
        res[dt] = moe_grouped_ffn_bwd(inp["dY"], m.perm.x_perm, inp["W_gate"], inp["W_up"], inp["W_down"], m.fc1_c,
                                      m.h, m.y_perm, m.perm, m.topk_w, m.ws, dw_dtype=dt)
    torch.cuda.synchronize()
    assert m.ws.read_error() == 0
    f, q = res[torch.float32], res[torch.bfloat16]
    assert torch.equal(f["dx"], q["dx"]) and torch.equal(f["d_topk_w"], q["d_topk_w"])
    for n in ("dW_gate", "dW_up", "dW_down"):
        assert q[n].dtype == torch.bfloat16
        assert torch.equal(f[n].to(torch.bfloat16), q[n])
