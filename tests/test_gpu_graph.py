"""The hot path captured in a CUDA graph (every call enqueues device work only and
reads routing-dependent sizes on the device, so a whole step can be captured):
replays on new inputs must equal, bit for bit, the same layer called directly on
those inputs.  Covers the programmatic launches, the CTA-pair GEMMs' cluster
launches and the device-side tile schedules inside a graph."""
import pytest
import torch

from mixture_experts_ffn_warp_gb300 import MoeBackward, MoeForward, MoeForwardMX, MxWeights
from mixture_experts_ffn_warp_gb300.synthetic import make_inputs, small_shape

pytestmark = pytest.mark.gpu


def _outputs(m, b):
    outs = [m.out]
    if b is not None:
        outs += [b.dx, b.dW_gate, b.dW_up, b.dW_down, b.d_topk_w, b.d_logits]
    return [t.clone() for t in outs]


@pytest.mark.parametrize("backward", [False, True])
def test_bf16_step_in_a_cuda_graph(backward):
    # H, F multiples of 256: FC1, FC2 and the FC1 dgrad on CTA pairs
    shape = small_shape("graph", T=700, H=256, F=512, E=6, k=2, backward=backward)
    inputs = [make_inputs(shape, device="cuda", seed=40 + i, with_dy=backward) for i in range(3)]
    W = inputs[0]
    names = ["x", "logits"] + (["dY"] if backward else [])
    m = MoeForward(shape.T, shape.H, shape.F, shape.E, shape.k, keep_fc1_c=backward)
    b = MoeBackward(m, want_d_logits=True) if backward else None
    static = {n: torch.empty_like(inputs[0][n]) for n in names}

    def step():
        m(static["x"], static["logits"], W["W_gate"], W["W_up"], W["W_down"])
        if b is not None:
            b(static["dY"], W["W_gate"], W["W_up"], W["W_down"], logits=static["logits"])

    # eager results for every input set (also the first call of every launcher, outside capture)
    ref = []
    for inp in inputs:
        for n in names:
            static[n].copy_(inp[n])
        step()
        ref.append(_outputs(m, b))
    torch.cuda.synchronize()

    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            step()
    torch.cuda.current_stream().wait_stream(s)
    for i in (2, 0, 1):
        for n in names:
            static[n].copy_(inputs[i][n])
        g.replay()
        got = _outputs(m, b)
        torch.cuda.synchronize()
        for a, r in zip(got, ref[i]):
            assert torch.equal(a, r)
    assert m.ws.read_error() == 0


def test_mxfp8_forward_in_a_cuda_graph():
    shape = small_shape("graph_mx", T=500, H=256, F=256, E=8, k=2)
    inputs = [make_inputs(shape, device="cuda", seed=60 + i) for i in range(2)]
    W = inputs[0]
    mw = MxWeights(W["W_gate"], W["W_up"], W["W_down"])
    m = MoeForwardMX(shape.T, shape.H, shape.F, shape.E, shape.k)
    static = {n: torch.empty_like(inputs[0][n]) for n in ("x", "logits")}
    ref = []
    for inp in inputs:
        for n in static:
            static[n].copy_(inp[n])
        ref.append(m(static["x"], static["logits"], mw).clone())
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            m(static["x"], static["logits"], mw)
    torch.cuda.current_stream().wait_stream(s)
    for i in (1, 0):
        for n in static:
            static[n].copy_(inputs[i][n])
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(m.out, ref[i])
    assert m.ws.read_error() == 0
