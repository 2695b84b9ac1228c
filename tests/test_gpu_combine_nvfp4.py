"""GPU parity of the combine with an NVFP4 output encoding against the CPU oracle,
through the C ABI.

Given the same bf16 expert outputs, the kernel's codes and scales must equal the
oracle's bit for bit: both sum in fp32 in slot order with one rounding per
multiply-add and take every encoding decision on that fp32 value (the decisions
compare exact fp32 quantities).  Through the whole forward the decoded output must
be within the path's bar (2e-2 * RMS bf16, 6e-2 * RMS MXFP8) of the oracle's exact
forward beyond the encoding's own rounding (half a step of the E2M1 grid at the
block's scale, up to a sixth of the block maximum)."""
import numpy as np
import pytest
import torch

import oracle
from mixture_experts_ffn_warp_gb300 import MoeForward, MoeForwardMX, MxWeights, moe_unpermute_combine_nvfp4
from mixture_experts_ffn_warp_gb300.synthetic import small_shape
from helpers import TOL_BF16, TOL_MXFP8, assert_close_rms_nvfp4, bits, gpu_inputs

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("T,H,k,drop,plain", [(300, 256, 1, False, False), (257, 400, 2, True, False),
                                               (513, 2048, 6, True, False), (129, 7168, 8, False, False),
                                               (64, 16, 4, True, True), (40, 48, 32, False, False)])
def test_combine_nvfp4_bit_exact(T, H, k, drop, plain):
    g = torch.Generator(device="cuda").manual_seed(T + H + k)
    rows = T * k
    y = (torch.randn(rows, H, generator=g, device="cuda") * 3.0).to(torch.bfloat16)
    y[5] *= 1e-6                                             # a row of tiny values
    y[6] *= 3000.0                                           # a row whose blocks saturate
    dst = torch.randperm(rows, generator=g, device="cuda").to(torch.int32).reshape(T, k)
    if drop:
        dst[3] = -1                                          # all routes of a token dropped
        dst[7, 0] = -1
    w = None if plain else torch.rand(T, k, generator=g, device="cuda")
    q, sf = moe_unpermute_combine_nvfp4(y, dst, w)
    torch.cuda.synchronize()
    wn = np.ones((T, k), np.float32) if plain else w.cpu().numpy()
    rq, rs = oracle.unpermute_combine_nvfp4(y.float().cpu().numpy(), dst.cpu().numpy(), wn)
    assert np.array_equal(sf.cpu().numpy(), rs)
    assert np.array_equal(q.cpu().numpy(), rq)


@pytest.mark.parametrize("mx_path", [False, True])
def test_forward_with_nvfp4_output(mx_path):
    shape = small_shape("outnv", T=300, H=256, F=384, E=6, k=3, mxfp8=mx_path)
    inp = gpu_inputs(shape, with_dy=False)
    if mx_path:
        mw = MxWeights(inp["W_gate"], inp["W_up"], inp["W_down"])
        m = MoeForwardMX(shape.T, shape.H, shape.F, shape.E, shape.k, out_format="nvfp4")
        q, sf = m(inp["x"], inp["logits"], mw)
    else:
        m = MoeForward(shape.T, shape.H, shape.F, shape.E, shape.k, out_format="nvfp4")
        q, sf = m(inp["x"], inp["logits"], inp["W_gate"], inp["W_up"], inp["W_down"])
    torch.cuda.synchronize()
    assert m.ws.read_error() == 0
    assert q.shape == (shape.T, shape.H // 2) and sf.shape == (shape.T, shape.H // 16)
    # codes and scales: the oracle's encoding of this layer's own expert outputs
    rq, rs = oracle.unpermute_combine_nvfp4(m.y_perm.float().cpu().numpy(), m.perm.dst_of_route.cpu().numpy(),
                                            m.topk_w.cpu().numpy())
    assert np.array_equal(q.cpu().numpy(), rq) and np.array_equal(sf.cpu().numpy(), rs)
    vals = oracle.nvfp4_decode(q.cpu().numpy(), sf.cpu().numpy())
    # against the exact forward that applies the same operand quantisation
    idx, w = m.topk_idx.cpu().numpy(), m.topk_w.cpu().numpy()
    hb = {n: bits(inp[n]) for n in ("x", "W_gate", "W_up", "W_down")}
    if mx_path:
        xq = oracle.mx_roundtrip_rows(hb["x"])
        wg, wu, wd = oracle.mx_roundtrip_weights(hb["W_gate"], hb["W_up"], hb["W_down"])
        ref = oracle.moe_fwd(xq, wg, wu, wd, idx, w, round_mode=2, h_mx=True)["out"]
    else:
        ref = oracle.moe_fwd(hb["x"], hb["W_gate"], hb["W_up"], hb["W_down"], idx, w, round_mode=2)["out"]
    assert_close_rms_nvfp4(vals, ref, sf.cpu().numpy(), tol=TOL_MXFP8 if mx_path else TOL_BF16,
                           what="NVFP4 output")
