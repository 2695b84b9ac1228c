"""GPU parity of the forward hot path (A1 route, A2 permute, A3/A4 grouped
FFN, A5 combine) against the CPU oracle, called through the C ABI.

Integer outputs (expert ids, permutation maps, group sizes/offsets, copied
rows) must match bit for bit; floating-point outputs must satisfy
max|err| <= 2e-2 * RMS(oracle) (fp32 weights: 2e-6 absolute), for the bf16 layer
output counting the error beyond its own bf16 rounding of the exact value."""
import numpy as np
import pytest
import torch

import oracle
from mixture_experts_ffn_warp_gb300 import (MoeForward, Workspace, moe_grouped_ffn_fwd, moe_permute,
                                            moe_route_topk, moe_unpermute_combine)
from mixture_experts_ffn_warp_gb300.synthetic import CONFIGS, small_shape
from helpers import TOL_BF16, assert_close_rms, assert_close_ulp, bits, gpu_inputs, host_experts, to_f64

pytestmark = pytest.mark.gpu

SMALL = {
    "tiny": CONFIGS["tiny"],
    # several M tiles with ragged tails, 3 FC1 N tiles, one 256-wide FC2 tile
    "ragged": small_shape("ragged", T=300, H=256, F=384, E=5, k=2),
    # FC2 with 128-wide tiles (H % 256 != 0), odd T, larger k
    "h384": small_shape("h384", T=257, H=384, F=256, E=7, k=3),
    # dense special case
    "dense": small_shape("dense", T=200, H=128, F=128, E=1, k=1),
    # many experts, several empty
    "many": small_shape("many", T=512, H=128, F=128, E=64, k=4, skew=True),
    # ~1000 rows per expert: several 256-token blocks per expert and a ragged last block
    "blocks": small_shape("blocks", T=1500, H=256, F=256, E=3, k=2),
    # the largest expert count: most of the 1024 experts get 0-3 rows (tiles of 16-token MMAs)
    "e1024": small_shape("e1024", T=600, H=256, F=256, E=1024, k=4),
    # ~4700 rows per expert: more than 16 token blocks, so two bands of the pair GEMM's tile order
    "bands": small_shape("bands", T=7000, H=256, F=256, E=3, k=2),
}


def _route_and_check(inp, k):
    idx, w = moe_route_topk(inp["logits"], k)
    ref_idx, ref_w = oracle.route_topk(inp["logits"].cpu().numpy(), k)
    assert np.array_equal(idx.cpu().numpy(), ref_idx)
    assert np.abs(w.cpu().numpy() - ref_w).max() <= 2e-6
    return idx, w, ref_idx, ref_w


def _check_perm(p, ref, R):
    used = int(ref["group_offsets"][-1])
    assert np.array_equal(p.group_sizes.cpu().numpy(), ref["group_sizes"])
    assert np.array_equal(p.group_offsets.cpu().numpy(), ref["group_offsets"])
    assert np.array_equal(p.dst_of_route.cpu().numpy(), ref["dst_of_route"])
    assert np.array_equal(p.src_of_row[:used].cpu().numpy(), ref["src_of_row"][:used])


@pytest.mark.parametrize("name", list(SMALL))
def test_forward_parity_small(name):
    shape = SMALL[name]
    inp = gpu_inputs(shape)
    T, H, F, E, k = shape.T, shape.H, shape.F, shape.E, shape.k
    ws = Workspace(T, E, k)
    idx, w, ref_idx, ref_w = _route_and_check(inp, k)

    p = moe_permute(inp["x"], idx, E, ws)
    ref_p = oracle.permute(ref_idx, E)
    _check_perm(p, ref_p, T * k)
    xb = bits(inp["x"])
    used = int(ref_p["group_offsets"][-1])
    ref_xp = oracle.gather_rows(xb, k, ref_p["src_of_row"], used)
    assert np.array_equal(bits(p.x_perm[:used]), ref_xp)

    h, y_perm, fc1_c = moe_grouped_ffn_fwd(p.x_perm, inp["W_gate"], inp["W_up"], inp["W_down"],
                                           p.group_offsets, ws, want_fc1_c=True)
    out = moe_unpermute_combine(y_perm, p.dst_of_route, w)
    torch.cuda.synchronize()
    assert ws.read_error() == 0

    Wg, Wu, Wd = bits(inp["W_gate"]), bits(inp["W_up"]), bits(inp["W_down"])
    ref = oracle.moe_fwd(xb, Wg, Wu, Wd, ref_idx, ref_w, want_fc1=True, want_h=True, want_y=True)
    # stored intermediates, per route, against the oracle rounding at the same points
    route_of_row = ref_p["src_of_row"][:used]
    assert_close_ulp(to_f64(h[:used]), ref["h"][route_of_row], what="h")
    assert_close_ulp(to_f64(fc1_c[:used]), oracle.round_bf16(ref["fc1"][route_of_row]), what="fc1_c")
    # y_perm within the bar of the oracle's y (the GPU's h may round one ulp away from the
    # oracle's, which can move y by more than one of its own ulps) ...
    assert_close_rms(to_f64(y_perm[:used]), ref["y"][route_of_row], what="y_perm")
    # ... and within one bf16 ulp of bf16(h W_down) taken in fp64 on the GPU's own h
    offs = ref_p["group_offsets"]
    hd = h[:used].double().cpu()
    y_own = torch.cat([hd[offs[e]:offs[e + 1]] @ inp["W_down"][e].double().cpu() for e in range(E)])
    assert_close_ulp(to_f64(y_perm[:used]), y_own.to(torch.bfloat16).double().numpy(), what="y_perm (own h)")
    # the layer output against the exact value of the same arithmetic (h and y rounded to
    # bf16 where the path stores them, the output sum unrounded): max|err| <= 2e-2 * RMS
    exact = oracle.moe_fwd(xb, Wg, Wu, Wd, ref_idx, ref_w, round_mode=2)
    assert_close_rms(to_f64(out), exact["out"], what="out", bf16_out=True)
    # combine on the GPU's own y_perm: fp32 slot-order sum vs the oracle's double sum
    ref_c = oracle.unpermute_combine(y_perm.float().cpu().numpy(), p.dst_of_route.cpu().numpy(), w.cpu().numpy(),
                                     round_mode=2)
    assert np.abs(to_f64(out) - ref_c).max() <= 2.0 ** -7 * np.abs(ref_c).max()


def test_layer_object_matches_steps():
    shape = SMALL["ragged"]
    inp = gpu_inputs(shape)
    m = MoeForward(shape.T, shape.H, shape.F, shape.E, shape.k)
    out1 = m(inp["x"], inp["logits"], inp["W_gate"], inp["W_up"], inp["W_down"]).clone()
    out2 = m(inp["x"], inp["logits"], inp["W_gate"], inp["W_up"], inp["W_down"]).clone()
    torch.cuda.synchronize()
    assert torch.equal(out1, out2)     # deterministic
    assert m.ws.read_error() == 0


def test_identity_experts_permute_combine_returns_x():
    """Experts set to identity (y_perm = x_perm) with weights summing to 1."""
    shape = CONFIGS["fine_grained"]
    inp = gpu_inputs(shape)
    idx, w = moe_route_topk(inp["logits"], shape.k)
    ws = Workspace(shape.T, shape.E, shape.k)
    p = moe_permute(inp["x"], idx, shape.E, ws)
    out = moe_unpermute_combine(p.x_perm, p.dst_of_route, w)
    x = to_f64(inp["x"])
    assert np.all(np.abs(to_f64(out) - x) <= np.abs(x) * 2.0 ** -7)


@pytest.mark.parametrize("align", [8, 128])
def test_permute_aligned_groups(align):
    shape = SMALL["many"]
    inp = gpu_inputs(shape)
    idx, w = moe_route_topk(inp["logits"], shape.k)
    ws = Workspace(shape.T, shape.E, shape.k)
    p = moe_permute(inp["x"], idx, shape.E, ws, align=align)
    ref = oracle.permute(idx.cpu().numpy(), shape.E, align=align)
    _check_perm(p, ref, shape.T * shape.k)
    used = int(ref["group_offsets"][-1])
    ref_xp = oracle.gather_rows(bits(inp["x"]), shape.k, ref["src_of_row"], used)
    assert np.array_equal(bits(p.x_perm[:used]), ref_xp)     # padding rows are zero
    # the FFN runs on the padded layout and the combine ignores the padding
    h, y_perm, _ = moe_grouped_ffn_fwd(p.x_perm, inp["W_gate"], inp["W_up"], inp["W_down"],
                                       p.group_offsets, ws)
    out = moe_unpermute_combine(y_perm, p.dst_of_route, w)
    refo = oracle.moe_fwd(bits(inp["x"]), bits(inp["W_gate"]), bits(inp["W_up"]), bits(inp["W_down"]),
                          idx.cpu().numpy(), w.cpu().numpy(), round_mode=2)
    assert_close_rms(to_f64(out), refo["out"], what="out", bf16_out=True)


@pytest.mark.parametrize("T,k,E,align", [
    (2000, 8, 40, 1),      # 16000 routes: one cluster of 8 CTAs exchanging counts on chip
    (4096, 8, 256, 128),   # 32768 routes, 16 warps a CTA: the cluster pass's largest problem
    (1000, 32, 1024, 1),   # 32000 routes, a [16][1024] count table a CTA, in one cluster
    (4097, 8, 256, 16),    # 32776 routes: chunk counts and the last block's scan
    (3000, 32, 1024, 8),   # 96000 routes over 1024 experts: chunk counts
])
def test_permute_counting_paths(T, k, E, align):
    """Both counting passes (one cluster while the routes fit it, chunk counts otherwise)
    give the oracle's maps, group sizes and offsets and copy the rows bit for bit, with a
    skewed load, dropped routes and padded groups."""
    H = 64
    g = torch.Generator(device="cuda").manual_seed(T + k + E)
    x = torch.randn(T, H, generator=g, device="cuda", dtype=torch.bfloat16)
    # a Zipf-like load: expert e drawn with weight 1 / (e + 1)
    wts = 1.0 / torch.arange(1, E + 1, device="cuda", dtype=torch.float32)
    idx = torch.multinomial(wts.expand(T, E), k, replacement=False, generator=g).to(torch.int32)
    idx[::97, 0] = -1                     # dropped routes
    ws = Workspace(T, E, k)
    p = moe_permute(x, idx, E, ws, align=align)
    torch.cuda.synchronize()
    assert ws.read_error() == 0
    ref = oracle.permute(idx.cpu().numpy(), E, align=align)
    _check_perm(p, ref, T * k)
    used = int(ref["group_offsets"][-1])
    assert np.array_equal(bits(p.x_perm[:used]), oracle.gather_rows(bits(x), k, ref["src_of_row"], used))


def test_permute_dropped_and_invalid_ids():
    T, H, E, k = 700, 64, 6, 3
    g = torch.Generator(device="cuda").manual_seed(3)
    x = torch.randn(T, H, generator=g, device="cuda", dtype=torch.bfloat16)
    idx = torch.randint(-1, E, (T, k), generator=g, device="cuda", dtype=torch.int32)
    idx[5, 1] = 99
    idx[17, 0] = -5
    ws = Workspace(T, E, k)
    p = moe_permute(x, idx, E, ws)
    ref = oracle.permute(idx.cpu().numpy(), E)
    _check_perm(p, ref, T * k)
    assert ws.read_error() == 1          # MOE_DEVERR_BAD_EXPERT_ID
    ws.reset()
    assert ws.read_error() == 0


def test_zero_token_experts_ignore_their_weights():
    shape = SMALL["many"]
    inp = gpu_inputs(shape)
    m = MoeForward(shape.T, shape.H, shape.F, shape.E, shape.k)
    out = m(inp["x"], inp["logits"], inp["W_gate"], inp["W_up"], inp["W_down"]).clone()
    sizes = m.perm.group_sizes.cpu()
    empty = torch.nonzero(sizes == 0).flatten().tolist()
    assert len(empty) >= 8
    for name in ("W_gate", "W_up", "W_down"):
        inp[name][empty] = float("nan")
    out2 = m(inp["x"], inp["logits"], inp["W_gate"], inp["W_up"], inp["W_down"]).clone()
    torch.cuda.synchronize()
    assert torch.equal(out, out2) and torch.isfinite(out2.float()).all()


def test_empty_and_degenerate_sizes():
    ws = Workspace(0, 4, 2)
    x = torch.empty(0, 64, dtype=torch.bfloat16, device="cuda")
    lg = torch.empty(0, 4, dtype=torch.float32, device="cuda")
    idx, w = moe_route_topk(lg, 2)
    p = moe_permute(x, idx, 4, ws)
    assert p.group_offsets.cpu().tolist() == [0, 0, 0, 0, 0]
    # all routes dropped: the FFN has no tiles, the combine gives zeros
    T, H, F, E = 40, 128, 128, 3
    xx = torch.randn(T, H, device="cuda", dtype=torch.bfloat16)
    dropped = torch.full((T, 2), -1, dtype=torch.int32, device="cuda")
    ws2 = Workspace(T, E, 2)
    p2 = moe_permute(xx, dropped, E, ws2)
    W = torch.randn(E, H, F, device="cuda", dtype=torch.bfloat16)
    Wd = torch.randn(E, F, H, device="cuda", dtype=torch.bfloat16)
    h, y, _ = moe_grouped_ffn_fwd(p2.x_perm, W, W, Wd, p2.group_offsets, ws2)
    out = moe_unpermute_combine(y, p2.dst_of_route, torch.ones(T, 2, device="cuda"))
    torch.cuda.synchronize()
    assert p2.group_offsets.cpu().tolist() == [0] * (E + 1)
    assert torch.count_nonzero(out) == 0
    assert ws2.read_error() == 0


@pytest.mark.parametrize("name", ["fine_grained", "mixtral", "skewed"])
def test_forward_parity_full_size_sampled(name):
    """Full-size workload in the bench's launch configuration: routing and
    permutation checked on every token, outputs on sampled tokens."""
    shape = CONFIGS[name]
    inp = gpu_inputs(shape, with_dy=False)
    T, E, k = shape.T, shape.E, shape.k
    m = MoeForward(shape.T, shape.H, shape.F, E, k)
    out = m(inp["x"], inp["logits"], inp["W_gate"], inp["W_up"], inp["W_down"])
    torch.cuda.synchronize()
    assert m.ws.read_error() == 0
    ref_idx, ref_w = oracle.route_topk(inp["logits"].cpu().numpy(), k)
    assert np.array_equal(m.topk_idx.cpu().numpy(), ref_idx)
    assert np.abs(m.topk_w.cpu().numpy() - ref_w).max() <= 2e-6
    ref_p = oracle.permute(ref_idx, E)
    _check_perm(m.perm, ref_p, T * k)
    # every permuted row equals its source token, bit for bit
    src = m.perm.src_of_row[: T * k].long()
    assert torch.equal(m.perm.x_perm[: T * k], inp["x"][src // k])
    # sampled tokens through the oracle
    rng = np.random.default_rng(0)
    toks = np.sort(rng.choice(T, size=12, replace=False))
    experts = np.unique(ref_idx[toks])
    Wg, Wu, Wd = (host_experts(inp[n], experts) for n in ("W_gate", "W_up", "W_down"))
    ref = oracle.moe_fwd(bits(inp["x"]), Wg, Wu, Wd, ref_idx, ref_w, tokens=toks, round_mode=2,
                         want_y=True)
    assert_close_rms(to_f64(out[torch.from_numpy(toks).cuda()]), ref["out"], what=f"{name} out", bf16_out=True)
    # the bf16 expert outputs of the sampled routes, within one bf16 ulp of bf16(h W_down)
    # taken in fp64 on the GPU's own h (the GPU's h may round one ulp away from the
    # oracle's, and that moves y by up to a few of its own ulps)
    rows = torch.from_numpy(ref_p["dst_of_route"][toks].reshape(-1).astype(np.int64)).cuda()
    hr = to_f64(m.h[rows])
    y_own = np.stack([hr[i] @ oracle.bits_to_float(Wd[int(e)]) for i, e in enumerate(ref_idx[toks].reshape(-1))])
    assert_close_ulp(to_f64(m.y_perm[rows]), oracle.round_bf16(y_own), what=f"{name} y_perm (own h)")


def test_route_and_permute_at_the_largest_sizes():
    """E = 1024 experts and k = 32 (the ABI's limits): selection, weights and maps
    against the oracle (the route kernel's widest per-lane slice, 32 values per lane)."""
    T, E, k, H = 300, 1024, 32, 64
    g = torch.Generator(device="cuda").manual_seed(7)
    logits = torch.randn(T, E, generator=g, device="cuda")
    logits[0, :40] = 0.5                     # a tied block: lowest ids first
    x = torch.randn(T, H, generator=g, device="cuda").to(torch.bfloat16)
    idx, w, ref_idx, _ = _route_and_check({"logits": logits}, k)
    ws = Workspace(T, E, k)
    p = moe_permute(x, idx, E, ws)
    torch.cuda.synchronize()
    assert ws.read_error() == 0
    _check_perm(p, oracle.permute(ref_idx, E), T * k)
    src = p.src_of_row[: T * k].long()
    assert torch.equal(p.x_perm[: T * k], x[src // k])


def test_every_token_to_every_expert():
    """k = E: each expert receives every token; the forward against the oracle."""
    shape = small_shape("kE", T=200, H=128, F=256, E=4, k=4)
    inp = gpu_inputs(shape, with_dy=False)
    m = MoeForward(shape.T, shape.H, shape.F, shape.E, shape.k)
    out = m(inp["x"], inp["logits"], inp["W_gate"], inp["W_up"], inp["W_down"])
    torch.cuda.synchronize()
    assert m.ws.read_error() == 0
    assert m.perm.group_sizes.cpu().tolist() == [shape.T] * shape.E
    idx, w = m.topk_idx.cpu().numpy(), m.topk_w.cpu().numpy()
    hb = {n: bits(inp[n]) for n in ("x", "W_gate", "W_up", "W_down")}
    ref = oracle.moe_fwd(hb["x"], hb["W_gate"], hb["W_up"], hb["W_down"], idx, w, round_mode=2)
    assert_close_rms(to_f64(out), ref["out"], what="k = E out", bf16_out=True)


def test_misaligned_row_pointers_are_refused_before_launch():
    """Entry points whose kernels move 16-byte vectors return MOE_ERR_UNSUPPORTED for a
    row pointer off a 16-byte boundary, without launching (the error word stays 0)."""
    import ctypes as C
    from mixture_experts_ffn_warp_gb300 import Workspace, _binding
    L = _binding.load_library()
    T, H, E, k = 64, 128, 8, 2
    dev = torch.device("cuda")
    x = torch.zeros(T * H + 8, dtype=torch.bfloat16, device=dev)
    xp = torch.zeros(T * k * H + 8, dtype=torch.bfloat16, device=dev)
    idx = torch.zeros(T, k, dtype=torch.int32, device=dev)
    maps = [torch.zeros(n, dtype=torch.int32, device=dev) for n in (T * k, T * k, E, E + 1)]
    ws = Workspace(T, E, k)
    off = lambda t, b: C.c_void_p(t.data_ptr() + b)   # noqa: E731
    unsupported = 2
    st = L.moe_permute(off(x, 2), C.c_void_p(idx.data_ptr()), T, H, E, k, 1, C.c_void_p(xp.data_ptr()), T * k,
                       *[C.c_void_p(m.data_ptr()) for m in maps], C.c_void_p(ws.buf.data_ptr()), ws.nbytes, None)
    assert st == unsupported
    out = torch.zeros(T * H + 8, dtype=torch.bfloat16, device=dev)
    st = L.moe_unpermute_combine(off(xp, 4), C.c_void_p(maps[0].data_ptr()), None, T, H, k,
                                 C.c_void_p(out.data_ptr()), None)
    assert st == unsupported
    st = L.moe_unpermute_combine(C.c_void_p(xp.data_ptr()), C.c_void_p(maps[0].data_ptr()), None, T, H, k,
                                 off(out, 8), None)
    assert st == unsupported
    torch.cuda.synchronize()
    assert ws.read_error() == 0
