"""Pins of the oracle's optional SwiGLU clamp (CPU only).

The pages name an optional DeepSeek-style clamp of the SwiGLU experts with
inclusive bounds ("Add MoE + expert-parallel Python API surface, PyTorch
reference, and tests", Summary) but no form or values.  The oracle's reading:
h = silu(clamp(g, gate_lo, gate_hi)) * clamp(u, up_lo, up_hi), a value equal to a
bound being inside (its derivative passes).  Pinned against an independent fp64
torch implementation (torch.clamp's derivative passes exactly where lo <= x <= hi),
a constructed on-the-bound case, and the no-op case."""
import numpy as np
import torch

import oracle

BOUNDS = (-1.0, 0.75, -0.5, 0.5)     # gate_lo, gate_hi, up_lo, up_hi: clip a good share of values


def _problem(T=6, H=64, F=64, E=3, k=2, seed=0):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(T, H, generator=g).to(torch.bfloat16)
    Wg = (torch.randn(E, H, F, generator=g) * 0.2).to(torch.bfloat16)
    Wu = (torch.randn(E, H, F, generator=g) * 0.2).to(torch.bfloat16)
    Wd = (torch.randn(E, F, H, generator=g) * 0.2).to(torch.bfloat16)
    logits = torch.randn(T, E, generator=g)
    dY = torch.randn(T, H, generator=g).to(torch.bfloat16)
    idx, w = oracle.route_topk(logits.numpy(), k)
    return dict(x=oracle.bf16_bits(x), Wg=oracle.bf16_bits(Wg), Wu=oracle.bf16_bits(Wu), Wd=oracle.bf16_bits(Wd),
                idx=idx, w=w, dY=oracle.bf16_bits(dY))


def _torch(p, bounds):
    f = lambda b: torch.tensor(oracle.bits_to_float(b), dtype=torch.float64)  # noqa: E731
    x, Wg, Wu, Wd = (f(p[n]).requires_grad_(True) for n in ("x", "Wg", "Wu", "Wd"))
    w = torch.tensor(p["w"], dtype=torch.float64, requires_grad=True)
    gl, gh, ul, uh = bounds
    T, k = p["idx"].shape
    outs = []
    for t in range(T):
        acc = torch.zeros(x.shape[1], dtype=torch.float64)
        for j in range(k):
            e = int(p["idx"][t, j])
            g = torch.clamp(x[t] @ Wg[e], gl, gh)
            u = torch.clamp(x[t] @ Wu[e], ul, uh)
            acc = acc + w[t, j] * ((torch.nn.functional.silu(g) * u) @ Wd[e])
        outs.append(acc)
    out = torch.stack(outs)
    (out * f(p["dY"])).sum().backward()
    return out.detach().numpy(), {"dx": x.grad.numpy(), "dW_gate": Wg.grad.numpy(), "dW_up": Wu.grad.numpy(),
                                  "dW_down": Wd.grad.numpy(), "d_topk_w": w.grad.numpy()}


def test_clamped_forward_and_backward_match_torch():
    p = _problem()
    ref_out, ref = _torch(p, BOUNDS)
    with oracle.swiglu_clamp(*BOUNDS):
        out = oracle.moe_fwd(p["x"], p["Wg"], p["Wu"], p["Wd"], p["idx"], p["w"], round_mode=0)["out"]
        got = oracle.moe_bwd(p["x"], p["Wg"], p["Wu"], p["Wd"], p["idx"], p["w"], p["dY"], round_mode=0)
    assert np.abs(out - ref_out).max() <= 1e-12 * np.abs(ref_out).max()
    for n in ("dx", "dW_gate", "dW_up", "dW_down", "d_topk_w"):
        assert np.abs(got[n] - ref[n]).max() <= 1e-11 * np.abs(ref[n]).max(), n
    # the clamp changed the result
    plain = oracle.moe_fwd(p["x"], p["Wg"], p["Wu"], p["Wd"], p["idx"], p["w"], round_mode=0)["out"]
    assert np.abs(plain - out).max() > 1e-3 * np.abs(out).max()


def test_bounds_enclosing_every_value_change_nothing():
    p = _problem(seed=1)
    plain_f = oracle.moe_fwd(p["x"], p["Wg"], p["Wu"], p["Wd"], p["idx"], p["w"])["out"]
    plain_b = oracle.moe_bwd(p["x"], p["Wg"], p["Wu"], p["Wd"], p["idx"], p["w"], p["dY"])
    with oracle.swiglu_clamp(-1e6, 1e6, -1e6, 1e6):
        f = oracle.moe_fwd(p["x"], p["Wg"], p["Wu"], p["Wd"], p["idx"], p["w"])["out"]
        b = oracle.moe_bwd(p["x"], p["Wg"], p["Wu"], p["Wd"], p["idx"], p["w"], p["dY"])
    assert np.array_equal(f, plain_f)
    for n in plain_b:
        assert np.array_equal(b[n], plain_b[n]), n


def test_bounds_are_inclusive():
    """One token, one expert, H = F = 32 with integer data: g and u of column 0 are exact
    integers.  A bound equal to the value keeps the derivative; a bound just below it
    zeroes the derivative (the value is clamped)."""
    H = F = 32
    x = np.zeros((1, H), np.float32)
    x[0, :3] = [1.0, 2.0, 1.0]
    Wg = np.zeros((1, H, F), np.float32)
    Wu = np.zeros((1, H, F), np.float32)
    Wd = np.zeros((1, F, H), np.float32)
    Wg[0, :3, 0] = [1.0, 0.0, 1.0]       # g[0] = 2
    Wu[0, :3, 0] = [0.0, 1.0, 1.0]       # u[0] = 3
    Wd[0, 0, 0] = 1.0
    dY = np.zeros((1, H), np.float32)
    dY[0, 0] = 1.0
    b = lambda a: oracle.double_to_bf16_bits(a.astype(np.float64))  # noqa: E731
    idx, w = np.zeros((1, 1), np.int32), np.ones((1, 1), np.float32)
    args = (b(x), b(Wg), b(Wu), b(Wd), idx, w, b(dY))

    def dg_du(bounds):
        with oracle.swiglu_clamp(*bounds):
            g = oracle.moe_bwd(*args, round_mode=0)
        # dW_gate[0, 0, 0] = x0 * dg ; dW_up[0, 0, 0] = x0 * du  (x0 = 1)
        return g["dW_gate"][0, 0, 0], g["dW_up"][0, 0, 0]

    s = 1.0 / (1.0 + np.exp(-2.0))
    dg_free = 3.0 * s * (1.0 + 2.0 * (1.0 - s))
    du_free = 2.0 * s
    dg, du = dg_du((-np.inf, 2.0, -np.inf, 3.0))          # both exactly on their upper bound
    assert np.isclose(dg, dg_free, rtol=1e-14) and np.isclose(du, du_free, rtol=1e-14)
    dg, du = dg_du((2.0, np.inf, 3.0, np.inf))            # both exactly on their lower bound
    assert np.isclose(dg, dg_free, rtol=1e-14) and np.isclose(du, du_free, rtol=1e-14)
    dg, du = dg_du((-np.inf, 1.5, -np.inf, 2.5))          # both clamped: derivatives zero
    assert dg == 0.0 and du == 0.0
    # and the clamped forward uses the bound: h = silu(1.5) * 2.5
    with oracle.swiglu_clamp(-np.inf, 1.5, -np.inf, 2.5):
        h = oracle.moe_fwd(args[0], args[1], args[2], args[3], idx, w, round_mode=0, want_h=True)["h"]
    assert np.isclose(h[0, 0], 1.5 / (1.0 + np.exp(-1.5)) * 2.5, rtol=1e-14)
