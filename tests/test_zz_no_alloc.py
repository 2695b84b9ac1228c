"""moe_permute_static_scratch: the permutation entry point for callers that
cannot allocate device memory (its scratch is a fixed array inside the
library instead of a caller-provided workspace).

Called through the C ABI and compared with moe_permute on the same inputs,
on two calls in a row (the second with different routing, so that state kept
in the shared array from the first call would show).  The permutation's
outputs are integers and copied rows, so the comparison is bit for bit.  This
file is collected last so that a run stopping at its first failure has
already run every other test.
"""
import ctypes as C

import numpy as np
import pytest
import torch

import oracle
from mixture_experts_ffn_warp_gb300 import Workspace, load_library, moe_permute, moe_route_topk

pytestmark = pytest.mark.gpu


def _p(t):
    return C.c_void_p(t.data_ptr())


def _outputs(T, H, E, k, align, dev):
    cap = T * k + E * (align - 1)
    return {
        "x_perm": torch.zeros(cap, H, dtype=torch.bfloat16, device=dev),
        "dst_of_route": torch.empty(T, k, dtype=torch.int32, device=dev),
        "src_of_row": torch.full((cap,), -7, dtype=torch.int32, device=dev),
        "group_sizes": torch.empty(E, dtype=torch.int32, device=dev),
        "group_offsets": torch.empty(E + 1, dtype=torch.int32, device=dev),
        "err": torch.full((1,), 0xFF, dtype=torch.int32, device=dev),
    }


def _static_permute(x, idx, E, align=1, out=None):
    L = load_library()
    T, H = x.shape
    k = idx.shape[1]
    cap = T * k + E * (align - 1)
    if out is None:
        out = _outputs(T, H, E, k, align, x.device)
    st = L.moe_permute_static_scratch(
        _p(x), _p(idx), T, H, E, k, align, _p(out["x_perm"]), cap, _p(out["dst_of_route"]),
        _p(out["src_of_row"]), _p(out["group_sizes"]), _p(out["group_offsets"]), _p(out["err"]),
        C.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, f"moe_permute_static_scratch returned {st}"
    return out


def _compare(x, idx, E, align=1):
    ws = Workspace(x.shape[0], E, idx.shape[1])
    ref = moe_permute(x, idx, E, ws, align=align)
    got = _static_permute(x, idx, E, align)
    torch.cuda.synchronize()
    used = int(ref.group_offsets[-1])
    assert torch.equal(got["group_sizes"], ref.group_sizes)
    assert torch.equal(got["group_offsets"], ref.group_offsets)
    assert torch.equal(got["dst_of_route"], ref.dst_of_route)
    assert torch.equal(got["src_of_row"][:used], ref.src_of_row[:used])
    assert torch.equal(got["x_perm"][:used], ref.x_perm[:used])
    assert int(got["err"].item()) == ws.read_error()
    # and the maps against the CPU oracle's stable counting sort
    want = oracle.permute(idx.cpu().numpy(), E, align=align)
    assert np.array_equal(got["group_sizes"].cpu().numpy(), want["group_sizes"])
    assert np.array_equal(got["group_offsets"].cpu().numpy(), want["group_offsets"])
    assert np.array_equal(got["dst_of_route"].cpu().numpy(), want["dst_of_route"])
    assert np.array_equal(got["src_of_row"][:used].cpu().numpy(), want["src_of_row"][:used])
    return got


def test_static_scratch_matches_workspace_permute_twice():
    g = torch.Generator(device="cuda").manual_seed(11)
    # call 1: fine-grained-like routing
    T, H, E, k = 3000, 256, 64, 6
    x = torch.randn(T, H, generator=g, device="cuda", dtype=torch.bfloat16)
    lg = torch.randn(T, E, generator=g, device="cuda")
    idx, _ = moe_route_topk(lg, k)
    got1 = _compare(x, idx, E)
    assert int(got1["err"].item()) == 0
    # call 2, right after: different sizes, skewed routing and padding
    T2, H2, E2, k2 = 20000, 128, 16, 4
    x2 = torch.randn(T2, H2, generator=g, device="cuda", dtype=torch.bfloat16)
    lg2 = torch.randn(T2, E2, generator=g, device="cuda")
    lg2[:, :3] += 2.0
    idx2, _ = moe_route_topk(lg2, k2)
    got2 = _compare(x2, idx2, E2, align=8)
    assert int(got2["err"].item()) == 0


def test_static_scratch_reports_bad_ids_and_clears_them():
    g = torch.Generator(device="cuda").manual_seed(12)
    T, H, E, k = 500, 64, 8, 2
    x = torch.randn(T, H, generator=g, device="cuda", dtype=torch.bfloat16)
    idx = torch.randint(-1, E, (T, k), generator=g, device="cuda", dtype=torch.int32)
    idx[3, 0] = 50
    got = _compare(x, idx, E)
    assert int(got["err"].item()) == 1          # MOE_DEVERR_BAD_EXPERT_ID
    idx[3, 0] = 2
    got = _compare(x, idx, E)
    assert int(got["err"].item()) == 0          # the shared error word restarts at zero


def test_static_scratch_allocates_nothing():
    """After a first call (the address lookup, and the lazy loading of the kernels it
    launches), a second call of the same shape leaves the device's free memory unchanged:
    no allocation by the library, torch's caching allocator idle in between."""
    g = torch.Generator(device="cuda").manual_seed(13)
    T, H, E, k = 4000, 256, 32, 4
    x = torch.randn(T, H, generator=g, device="cuda", dtype=torch.bfloat16)
    idx, _ = moe_route_topk(torch.randn(T, E, generator=g, device="cuda"), k)
    out = _outputs(T, H, E, k, 1, x.device)
    _static_permute(x, idx, E, out=out)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    _static_permute(x, idx, E, out=out)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0
    assert int(out["err"].item()) == 0


def test_static_scratch_rejects_problems_beyond_the_array():
    """ceil(T*k / 2048) * E > 65472 -> MOE_ERR_UNSUPPORTED.  Every pointer is a real
    device buffer of the rejected problem's size, so that a refusal that regressed would
    still launch on valid memory."""
    L = load_library()
    T, H, E, k = 130000, 8, 1024, 1          # 64 chunks x 1024 experts = 65536 counts
    assert -(-T * k // 2048) * E > 65472
    dev = torch.device("cuda")
    x = torch.zeros(T, H, dtype=torch.bfloat16, device=dev)
    idx = torch.zeros(T, k, dtype=torch.int32, device=dev)
    out = _outputs(T, H, E, k, 1, dev)
    st = L.moe_permute_static_scratch(
        _p(x), _p(idx), T, H, E, k, 1, _p(out["x_perm"]), T * k, _p(out["dst_of_route"]), _p(out["src_of_row"]),
        _p(out["group_sizes"]), _p(out["group_offsets"]), _p(out["err"]),
        C.c_void_p(torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    assert st == 2
    assert int(out["err"].item()) == 0xFF     # nothing was launched or copied
