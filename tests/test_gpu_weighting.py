"""GPU parity of the early router-weight placements (the weight applied in the FC1
or the FC2 epilogue, the combine summing unweighted) against the oracle's same
placement, through the C ABI: outputs max|err| <= 2e-2 * RMS beyond their own bf16
rounding, the weighted h
within one bf16 ulp, the weighted fp32 y within 2e-2 * RMS."""
import numpy as np
import pytest
import torch

import oracle
from mixture_experts_ffn_warp_gb300 import MoeBackward, MoeForward
from mixture_experts_ffn_warp_gb300.synthetic import CONFIGS, small_shape
from helpers import assert_close_rms, assert_close_ulp, bits, gpu_inputs, host_experts, to_f64

pytestmark = pytest.mark.gpu

AT = {"fc1": oracle.WEIGHT_IN_FC1, "fc2": oracle.WEIGHT_IN_FC2}
SMALL = {
    "ragged": (small_shape("ragged", T=300, H=256, F=384, E=5, k=2), 1),
    "many": (small_shape("many", T=512, H=256, F=128, E=64, k=4, skew=True), 1),
    "align128": (small_shape("al", T=200, H=128, F=256, E=6, k=3), 128),   # padding rows: weight 0
}


@pytest.mark.parametrize("name", list(SMALL))
@pytest.mark.parametrize("at", ["fc1", "fc2"])
def test_early_weighting_matches_oracle(name, at):
    shape, align = SMALL[name]
    inp = gpu_inputs(shape, with_dy=False)
    m = MoeForward(shape.T, shape.H, shape.F, shape.E, shape.k, align=align, weight_at=at)
    out = m(inp["x"], inp["logits"], inp["W_gate"], inp["W_up"], inp["W_down"])
    torch.cuda.synchronize()
    assert m.ws.read_error() == 0
    idx, w = oracle.route_topk(inp["logits"].cpu().numpy(), shape.k)
    assert np.array_equal(m.topk_idx.cpu().numpy(), idx)
    xb, Wg, Wu, Wd = (bits(inp[n]) for n in ("x", "W_gate", "W_up", "W_down"))
    # the oracle's per-route outputs use its own weights (the GPU's differ by <= 2e-6)
    ref = oracle.moe_fwd(xb, Wg, Wu, Wd, idx, w, round_mode=1, want_h=True, want_y=True, weight_at=AT[at])
    exact = oracle.moe_fwd(xb, Wg, Wu, Wd, idx, w, round_mode=2, weight_at=AT[at])
    assert_close_rms(to_f64(out), exact["out"], what=f"{at} out", bf16_out=True)
    used = int(m.perm.group_offsets[-1])
    src = m.perm.src_of_row[:used].cpu().numpy()   # rows past the groups are never written
    rows = np.nonzero(src >= 0)[0]
    routes = src[rows]
    if at == "fc1":
        assert_close_ulp(to_f64(m.h[torch.from_numpy(rows).cuda()]), ref["h"][routes], what="weighted h", slack=4e-3)
    else:
        # y = bf16(w * (h W_down)) within one bf16 ulp, taken in fp64 on the GPU's own h and
        # weights (a one-ulp difference of h moves y by more than one of its own ulps)
        hr = to_f64(m.h[torch.from_numpy(rows).cuda()])
        wr = m.topk_w.reshape(-1).cpu().numpy().astype(np.float64)[routes]
        er = idx.reshape(-1)[routes]
        y_own = np.stack([wr[i] * (hr[i] @ oracle.bits_to_float(Wd[int(e)])) for i, e in enumerate(er)])
        assert_close_ulp(to_f64(m.y_perm[torch.from_numpy(rows).cuda()]), oracle.round_bf16(y_own),
                         what="weighted y (own h)")
    pad = np.nonzero(src < 0)[0]
    if len(pad):   # padding rows inside the groups carry weight 0
        t = m.h if at == "fc1" else m.y_perm
        assert (t[torch.from_numpy(pad).cuda()] == 0).all()


def test_early_weighting_agrees_with_late_weighting():
    """The three placements are one function; on the GPU they agree to the bf16
    roundings of the weighted h (FC1) or the weighted y (FC2) against the unweighted ones."""
    shape = small_shape("agree", T=400, H=256, F=256, E=8, k=3)
    inp = gpu_inputs(shape, with_dy=False)
    outs = {}
    for at in ("combine", "fc1", "fc2"):
        m = MoeForward(shape.T, shape.H, shape.F, shape.E, shape.k, weight_at=at)
        outs[at] = to_f64(m(inp["x"], inp["logits"], inp["W_gate"], inp["W_up"], inp["W_down"]).clone())
    torch.cuda.synchronize()
    rms = np.sqrt((outs["combine"] ** 2).mean())
    assert np.abs(outs["fc2"] - outs["combine"]).max() <= 2.0 ** -7 * np.abs(outs["combine"]).max() + 2e-2 * rms
    assert np.abs(outs["fc1"] - outs["combine"]).max() <= 2.0 ** -7 * np.abs(outs["combine"]).max() + 2e-2 * rms


def test_backward_refuses_early_weighting():
    shape = small_shape("bw", T=64, H=128, F=128, E=4, k=2)
    m = MoeForward(shape.T, shape.H, shape.F, shape.E, shape.k, keep_fc1_c=True, weight_at="fc2")
    with pytest.raises(ValueError):
        MoeBackward(m)


@pytest.mark.parametrize("at", ["fc1", "fc2"])
def test_early_weighting_full_size_sampled(at):
    """fine_grained (T=4096, H=2048, F=1408, E=64, top-6) with the weight in FC1 / FC2,
    sampled tokens against the oracle."""
    shape = CONFIGS["fine_grained"]
    inp = gpu_inputs(shape, with_dy=False)
    m = MoeForward(shape.T, shape.H, shape.F, shape.E, shape.k, weight_at=at)
    out = m(inp["x"], inp["logits"], inp["W_gate"], inp["W_up"], inp["W_down"])
    torch.cuda.synchronize()
    assert m.ws.read_error() == 0
    idx, w = oracle.route_topk(inp["logits"].cpu().numpy(), shape.k)
    toks = np.sort(np.random.default_rng(5).choice(shape.T, size=10, replace=False))
    experts = np.unique(idx[toks])
    Wg, Wu, Wd = (host_experts(inp[n], experts) for n in ("W_gate", "W_up", "W_down"))
    ref = oracle.moe_fwd(bits(inp["x"]), Wg, Wu, Wd, idx, w, tokens=toks, round_mode=2, weight_at=AT[at])
    assert_close_rms(to_f64(out[torch.from_numpy(toks).cuda()]), ref["out"], what=f"{at} out", bf16_out=True)
