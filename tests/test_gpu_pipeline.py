"""The HostPipeline public API on the GPU: batches in pinned host memory, copies of
neighbouring batches overlapped with compute on separate streams.  Every batch's
result must equal, bit for bit, the same layer run directly on that batch (the
kernels are deterministic), which fails if a slot's buffers were reused before the
previous batch had left them or a stream ran ahead of its inputs."""
import pytest
import torch

from mixture_experts_ffn_warp_gb300 import HostPipeline, MoeBackward, MoeForward
from mixture_experts_ffn_warp_gb300.synthetic import make_inputs, small_shape

pytestmark = pytest.mark.gpu


def _batches(shape, n):
    return [make_inputs(shape, device="cuda", seed=100 + i, with_dy=shape.backward) for i in range(n)]


@pytest.mark.parametrize("backward", [False, True])
def test_pipeline_matches_direct_calls(backward):
    shape = small_shape("pipe", T=384, H=256, F=512, E=8, k=2, backward=backward)
    batches = _batches(shape, 5)
    W = batches[0]
    names = ["x", "logits"] + (["dY"] if backward else [])

    # direct: one layer, batch after batch
    ref = []
    m = MoeForward(shape.T, shape.H, shape.F, shape.E, shape.k, keep_fc1_c=backward)
    bw = MoeBackward(m) if backward else None
    for bt in batches:
        out = m(bt["x"], bt["logits"], W["W_gate"], W["W_up"], W["W_down"]).clone()
        dx = bw(bt["dY"], W["W_gate"], W["W_up"], W["W_down"]).clone() if backward else None
        ref.append((out, dx))
    torch.cuda.synchronize()

    layers = [MoeForward(shape.T, shape.H, shape.F, shape.E, shape.k, keep_fc1_c=backward) for _ in range(2)]
    bwds = [MoeBackward(l) for l in layers] if backward else None
    slots = [{n: torch.empty_like(batches[0][n]) for n in names} for _ in layers]

    def run(b, s):
        d = slots[b]
        layers[b](d["x"], d["logits"], W["W_gate"], W["W_up"], W["W_down"], s)
        if backward:
            bwds[b](d["dY"], W["W_gate"], W["W_up"], W["W_down"], s)

    def outputs(b):
        return [layers[b].out] + ([bwds[b].dx] if backward else [])

    pipe = HostPipeline(slots, run, outputs)
    host_in = [{n: bt[n].cpu().pin_memory() for n in names} for bt in batches]
    host_out = [[torch.empty(shape.T, shape.H, dtype=torch.bfloat16).pin_memory() for _ in outputs(0)]
                for _ in batches]
    for hi, ho in zip(host_in, host_out):
        pipe.submit(hi, ho)
    torch.cuda.synchronize()
    for (out, dx), ho in zip(ref, host_out):
        assert torch.equal(ho[0], out.cpu())
        if backward:
            assert torch.equal(ho[1], dx.cpu())
    for l in layers:
        assert l.ws.read_error() == 0
