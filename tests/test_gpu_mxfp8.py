"""GPU parity of the MXFP8 path (A6 quantisers, the quantising permute, A7
block-scaled grouped FFN) against the CPU oracle, through the C ABI.

Quantised codes and scales must match the oracle's quantiser bit for bit;
the FFN outputs must satisfy max|err| <= 6e-2 * RMS against the oracle that
applies the same quantisation (x, weights and h in MXFP8)."""
import numpy as np
import pytest
import torch

import oracle
from mixture_experts_ffn_warp_gb300 import (MoeForwardMX, MxWeights, Workspace, moe_grouped_quantize_mxfp8,
                                            moe_permute, moe_permute_mxfp8, moe_quantize_weights_mxfp8,
                                            moe_route_topk, moe_unpermute_combine)
from mixture_experts_ffn_warp_gb300.synthetic import CONFIGS, small_shape
from helpers import TOL_MXFP8, assert_close_rms, assert_close_rms_mx, bits, gpu_inputs, to_f64

pytestmark = pytest.mark.gpu


def tiles_to_rowmajor(sf_tiles: np.ndarray, group_offsets: np.ndarray, rows: int, K: int) -> np.ndarray:
    """Scales of every grouped row read back from the MMA tile layout."""
    out = np.zeros((rows, K // 32), np.uint8)
    go = group_offsets.astype(np.int64)
    G = len(go) - 1
    sizes = np.maximum(go[1:] - go[:-1], 0)
    mts = np.concatenate([[0], np.cumsum((sizes + 127) // 128)])
    kb = np.arange(K // 32)
    for g in range(G):
        for i in range(int(sizes[g])):
            tile, m = mts[g] + i // 128, i % 128
            off = (tile * (K // 128) + kb // 4) * 512 + (m % 32) * 16 + (m // 32) * 4 + kb % 4
            out[go[g] + i] = sf_tiles[off]
    return out


def weight_scales_rowmajor(sf: np.ndarray, E: int, K: int, N: int) -> np.ndarray:
    """[E, N, K/32] from the weights' [E][K/128][N/128] atom layout."""
    e, n, kb = np.meshgrid(np.arange(E), np.arange(N), np.arange(K // 32), indexing="ij")
    atom = (e * (K // 128) + kb // 4) * (N // 128) + n // 128
    off = atom * 512 + (n % 32) * 16 + ((n % 128) // 32) * 4 + kb % 4
    return sf[off]


def weight_codes_nk(data: torch.Tensor, e: int, K: int, N: int) -> np.ndarray:
    """Codes of expert e as [N, K] from the tiled layout: 16 KB blocks ordered
    [K/128][N/128], row r of a block holding its 16-byte chunk j at j ^ (r % 8)."""
    blk = data[e * K * N:(e + 1) * K * N].cpu().numpy().reshape(K // 128, N // 128, 128, 8, 16)
    r = np.arange(128)[:, None]
    phys = np.arange(8)[None, :] ^ (r % 8)                      # [r, logical chunk] -> stored chunk
    logical = blk[:, :, r, phys, :]                             # [KB, NB, 128, 8, 16]
    return np.ascontiguousarray(logical.transpose(1, 2, 0, 3, 4)).reshape(N, K)


def _special_rows(g, rows, K):
    x = torch.randn(rows, K, generator=g, device="cuda", dtype=torch.float32)
    x[0] = 0.0                                    # amax = 0 blocks
    x[1, :32] = 448.0                             # exact largest finite
    x[1, 32:64] = 500.0                           # significand > 1.75: scale rounds up
    x[2] *= 1e-30                                 # tiny blocks
    x[3] *= 1e30                                  # huge blocks
    x[4, :32] = torch.tensor([2.0 ** i for i in range(-16, 16)], device="cuda")
    return x.to(torch.bfloat16)


def test_quantize_rows_bit_exact():
    g = torch.Generator(device="cuda").manual_seed(21)
    x = _special_rows(g, 777, 384)
    data, srm, _ = moe_grouped_quantize_mxfp8(x)
    torch.cuda.synchronize()
    rd, rs = oracle.quantize_rows_mxfp8(bits(x))
    assert np.array_equal(data.cpu().numpy(), rd)
    assert np.array_equal(srm.cpu().numpy(), rs)


def test_quantize_tile_layout_matches_rowmajor():
    shape = small_shape("many", T=700, H=256, F=128, E=24, k=3, skew=True)
    inp = gpu_inputs(shape, with_dy=False)
    idx, _ = moe_route_topk(inp["logits"], shape.k)
    ws = Workspace(shape.T, shape.E, shape.k)
    p = moe_permute(inp["x"], idx, shape.E, ws)
    used = int(p.group_offsets[-1])
    data, srm, stl = moe_grouped_quantize_mxfp8(p.x_perm[:used], p.group_offsets, ws, rowmajor=True, tiles=True)
    torch.cuda.synchronize()
    back = tiles_to_rowmajor(stl.cpu().numpy(), p.group_offsets.cpu().numpy(), used, shape.H)
    assert np.array_equal(back, srm.cpu().numpy())
    rd, rs = oracle.quantize_rows_mxfp8(bits(p.x_perm[:used]))
    assert np.array_equal(data.cpu().numpy(), rd) and np.array_equal(srm.cpu().numpy(), rs)


def test_quantize_weights_bit_exact():
    g = torch.Generator(device="cuda").manual_seed(22)
    E, K, N = 3, 256, 384
    W = (torch.randn(E, K, N, generator=g, device="cuda") * 0.02).to(torch.bfloat16)
    W[1, :32, 5] = 0.0
    data, sf = moe_quantize_weights_mxfp8(W)
    torch.cuda.synchronize()
    rs_all = weight_scales_rowmajor(sf.cpu().numpy(), E, K, N)
    wb = bits(W)
    for e in range(E):
        rd, rs = oracle.quantize_cols_mxfp8(wb[e])
        assert np.array_equal(weight_codes_nk(data, e, K, N), rd)
        assert np.array_equal(rs_all[e], rs)


@pytest.mark.parametrize("T,H,E,k", [(1500, 384, 16, 4),    # counted in one cluster
                                     (8500, 128, 16, 8)])   # 68000 routes: chunk counts
def test_permute_mxfp8_bit_exact(T, H, E, k):
    shape = small_shape("perm", T=T, H=H, F=128, E=E, k=k)
    inp = gpu_inputs(shape, with_dy=False)
    idx, _ = moe_route_topk(inp["logits"], shape.k)
    ws = Workspace(shape.T, shape.E, shape.k)
    p = moe_permute_mxfp8(inp["x"], idx, shape.E, ws)
    torch.cuda.synchronize()
    assert ws.read_error() == 0
    ref = oracle.permute(idx.cpu().numpy(), shape.E)
    assert np.array_equal(p.group_offsets.cpu().numpy(), ref["group_offsets"])
    assert np.array_equal(p.dst_of_route.cpu().numpy(), ref["dst_of_route"])
    R = shape.T * shape.k
    src = ref["src_of_row"][:R]
    xq, xs = oracle.quantize_rows_mxfp8(bits(inp["x"]))
    assert np.array_equal(p.x_q.cpu().numpy(), xq[src // shape.k])
    back = tiles_to_rowmajor(p.x_sf.cpu().numpy(), ref["group_offsets"], R, shape.H)
    assert np.array_equal(back, xs[src // shape.k])


def _oracle_mx_weights(inp, experts):
    q = {n: {} for n in ("gq", "gs", "uq", "us", "dq", "ds")}
    for e in experts:
        e = int(e)
        q["gq"][e], q["gs"][e] = oracle.quantize_cols_mxfp8(bits(inp["W_gate"][e]))
        q["uq"][e], q["us"][e] = oracle.quantize_cols_mxfp8(bits(inp["W_up"][e]))
        q["dq"][e], q["ds"][e] = oracle.quantize_cols_mxfp8(bits(inp["W_down"][e]))
    return q


SMALL = {
    "tiny": small_shape("tiny", T=64, H=128, F=256, E=8, k=2),
    "ragged": small_shape("ragged", T=300, H=256, F=384, E=5, k=2),
    "h384": small_shape("h384", T=257, H=384, F=256, E=7, k=3),   # FC2 with 128-wide tiles
    "many": small_shape("many", T=512, H=256, F=128, E=64, k=4, skew=True),
    # experts of 1011, 25, 317, 1400, 1367 and 80 rows: several 256-token blocks, last blocks
    # of every kind (one CTA's half of at most 32 tokens, or more)
    "blocks": small_shape("blocks", T=1400, H=256, F=384, E=6, k=3, skew=True),
}


@pytest.mark.parametrize("name", list(SMALL))
def test_mxfp8_forward_parity_small(name):
    shape = SMALL[name]
    inp = gpu_inputs(shape, with_dy=False)
    w = MxWeights(inp["W_gate"], inp["W_up"], inp["W_down"])
    m = MoeForwardMX(shape.T, shape.H, shape.F, shape.E, shape.k)
    out = m(inp["x"], inp["logits"], w)
    torch.cuda.synchronize()
    assert m.ws.read_error() == 0
    idx, tw = m.topk_idx.cpu().numpy(), m.topk_w.cpu().numpy()
    q = _oracle_mx_weights(inp, range(shape.E))
    ref = oracle.moe_fwd_mxfp8(bits(inp["x"]), q["gq"], q["gs"], q["uq"], q["us"], q["dq"], q["ds"], idx, tw,
                               round_mode=2, want_y=True)
    assert_close_rms(to_f64(out), ref["out"], tol=TOL_MXFP8, what="out", bf16_out=True)
    dst = torch.from_numpy(m.perm.dst_of_route.cpu().numpy().reshape(-1).astype(np.int64)).cuda()
    assert_close_rms(to_f64(m.y_perm[dst]), ref["y"], tol=TOL_MXFP8, what="y_perm")


def test_mxfp8_forward_dsv3_full_size_sampled():
    """DeepSeek-V3-shaped MXFP8 forward at full size (T=8192, H=7168, F=2048,
    E=256, top-8) in the bench's launch configuration: weight quantisation
    bit-exact on sampled experts, outputs of sampled tokens vs the oracle."""
    shape = CONFIGS["dsv3_mxfp8"]
    inp = gpu_inputs(shape, with_dy=False)
    w = MxWeights(inp["W_gate"], inp["W_up"], inp["W_down"])
    m = MoeForwardMX(shape.T, shape.H, shape.F, shape.E, shape.k)
    out = m(inp["x"], inp["logits"], w)
    torch.cuda.synchronize()
    assert m.ws.read_error() == 0
    idx, tw = m.topk_idx.cpu().numpy(), m.topk_w.cpu().numpy()
    ref_idx, _ = oracle.route_topk(inp["logits"].cpu().numpy(), shape.k)
    assert np.array_equal(idx, ref_idx)
    rng = np.random.default_rng(3)
    toks = np.sort(rng.choice(shape.T, size=4, replace=False))
    experts = np.unique(idx[toks])
    q = _oracle_mx_weights(inp, experts)
    # the GPU's weight codes for two of those experts, bit for bit
    for e in experts[:2]:
        e = int(e)
        assert np.array_equal(weight_codes_nk(w.Wg_q, e, shape.H, shape.F), q["gq"][e])
        assert np.array_equal(weight_codes_nk(w.Wd_q, e, shape.F, shape.H), q["dq"][e])
    ref = oracle.moe_fwd_mxfp8(bits(inp["x"]), q["gq"], q["gs"], q["uq"], q["us"], q["dq"], q["ds"], idx, tw,
                               tokens=toks, round_mode=2)
    assert_close_rms(to_f64(out[torch.from_numpy(toks).cuda()]), ref["out"], tol=TOL_MXFP8, what="dsv3 out", bf16_out=True)


def test_mxfp8_stash_leaves_the_forward_unchanged():
    """Keeping the bf16 g | u stash for the straight-through backward changes nothing in
    the forward: y_perm and the output are bit-identical with and without it, and the
    combine over the bf16 rows is the plain combine of the same rows."""
    shape = small_shape("ystash", T=600, H=256, F=384, E=6, k=3, mxfp8=True)
    inp = gpu_inputs(shape, with_dy=False)
    w = MxWeights(inp["W_gate"], inp["W_up"], inp["W_down"])
    m0 = MoeForwardMX(shape.T, shape.H, shape.F, shape.E, shape.k)
    m1 = MoeForwardMX(shape.T, shape.H, shape.F, shape.E, shape.k, keep_fc1_c=True)
    assert m0.y_perm.dtype == torch.bfloat16 and m1.y_perm.dtype == torch.bfloat16
    out0 = m0(inp["x"], inp["logits"], w)
    out1 = m1(inp["x"], inp["logits"], w)
    torch.cuda.synchronize()
    assert m0.ws.read_error() == 0 and m1.ws.read_error() == 0
    rows = int(m0.perm.group_offsets[-1].item())
    assert rows == shape.T * shape.k
    assert torch.equal(m0.y_perm[:rows], m1.y_perm[:rows])
    assert torch.equal(out0, out1)
    ref = moe_unpermute_combine(m0.y_perm, m0.perm.dst_of_route, m0.topk_w)
    assert torch.equal(out0, ref)


def _e4m3_values() -> np.ndarray:
    return np.array([oracle.e4m3_to_double(c) for c in range(256)])


def test_mxfp8_h_codes_over_token_blocks():
    """The FC1 epilogue's h codes and scales on experts cut into several 256-token blocks:
    decoded, they are the exact h of the MXFP8 operands within the encoding's own rounding
    (oracle, fp64), and every 32-feature block's scale is the smallest power of two that
    keeps the block within E4M3's 448 (its largest code is at least 224 in magnitude)."""
    shape = SMALL["blocks"]
    inp = gpu_inputs(shape, with_dy=False)
    w = MxWeights(inp["W_gate"], inp["W_up"], inp["W_down"])
    m = MoeForwardMX(shape.T, shape.H, shape.F, shape.E, shape.k)
    m(inp["x"], inp["logits"], w)
    torch.cuda.synchronize()
    assert m.ws.read_error() == 0
    sizes = m.perm.group_sizes.cpu().numpy()
    tail = sizes % 256
    assert (sizes > 512).any() and ((tail > 0) & (tail <= 64)).any() and (tail > 64).any(), sizes
    go = m.perm.group_offsets.cpu().numpy()
    used = int(go[-1])
    codes = m.h_q[:used].cpu().numpy()
    sc = tiles_to_rowmajor(m.h_sf.cpu().numpy(), go, used, shape.F)
    vals = _e4m3_values()
    mag = np.abs(vals[codes]).reshape(used, shape.F // 32, 32).max(axis=2)
    assert np.all((mag >= 224) | (sc == 0)), "a block scale is not the smallest that fits"
    got = oracle.mx_dequantize(codes, sc)
    idx, tw = m.topk_idx.cpu().numpy(), m.topk_w.cpu().numpy()
    xq = oracle.mx_roundtrip_rows(bits(inp["x"]))
    wg, wu, wd = oracle.mx_roundtrip_weights(bits(inp["W_gate"]), bits(inp["W_up"]), bits(inp["W_down"]))
    ref = oracle.moe_fwd(xq, wg, wu, wd, idx, tw, round_mode=0, want_h=True)
    dst = m.perm.dst_of_route.cpu().numpy().reshape(-1)
    assert_close_rms_mx(got[dst], ref["h"], sc[dst], what="h (MXFP8) over token blocks")
