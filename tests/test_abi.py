"""The C-ABI library builds, loads and exports every symbol include/moe.h
declares; host-side validation answers without touching a GPU."""
import ctypes as C
import os
import re

import pytest

import __graft_entry__
from mixture_experts_ffn_warp_gb300 import _binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", text))
    return names


@pytest.fixture(scope="module")
def lib():
    __graft_entry__.build()
    return _binding.load_library()


def test_header_declares_the_path(lib):
    names = _declared()
    for n in ("moe_route_topk", "moe_permute", "moe_grouped_ffn_fwd", "moe_unpermute_combine"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in _declared() if not hasattr(lib, n)]
    assert not missing, missing
    # and the binding mirrors every declaration
    assert _declared() <= set(_binding.SIGNATURES)


def test_status_strings_and_version(lib):
    assert lib.moe_status_string(0) == b"MOE_OK"
    assert lib.moe_status_string(2) == b"MOE_ERR_UNSUPPORTED"
    assert lib.moe_abi_version() >= 1


def test_workspace_bytes(lib):
    # header + per-chunk counts (24576 routes -> 12 chunks of 2048) + M-tile prefix, 16-byte rounded
    assert lib.moe_workspace_bytes(4096, 64, 6) == 256 + 12 * 64 * 4 + 272
    assert lib.moe_workspace_bytes(0, 8, 2) == 256 + 0 + 48
    assert lib.moe_workspace_bytes(10, 0, 2) == 0
    assert lib.moe_workspace_bytes(10, 8, 33) == 0


def test_host_validation_before_launch(lib):
    nul = None
    # E, k out of range
    assert lib.moe_route_topk(nul, 10, 0, 1, nul, nul, nul) == 2
    assert lib.moe_route_topk(nul, 10, 8, 9, nul, nul, nul) == 2
    assert lib.moe_route_topk(nul, -1, 8, 2, nul, nul, nul) == 1
    assert lib.moe_route_topk(nul, 0, 8, 2, nul, nul, nul) == 0          # empty: no-op
    assert lib.moe_route_topk(nul, 5, 8, 2, nul, nul, nul) == 1          # null pointers
    # sigmoid router and router backward
    assert lib.moe_route_topk_sigmoid(nul, nul, 10, 8, 9, 1, nul, nul, nul) == 2
    assert lib.moe_route_topk_sigmoid(nul, nul, 0, 8, 2, 1, nul, nul, nul) == 0
    assert lib.moe_route_topk_sigmoid(nul, nul, 5, 8, 2, 1, nul, nul, nul) == 1
    fk = C.c_void_p(16)
    assert lib.moe_route_topk_bwd(fk, fk, fk, 5, 8, 2, 7, 1, fk, nul) == 1       # unknown score function
    assert lib.moe_route_topk_bwd(fk, fk, fk, 5, 2000, 2, 0, 1, fk, nul) == 2    # E > 1024
    assert lib.moe_route_topk_bwd(fk, nul, fk, 5, 8, 2, 1, 1, fk, nul) == 1      # null pointer
    # weighted FC1 / FC2: route maps required
    assert lib.moe_grouped_fc1_swiglu_weighted(fk, fk, fk, fk, nul, nul, 4, 128, 128, 8, fk, nul, fk, 4096, nul) == 1
    assert lib.moe_grouped_fc2_weighted(fk, fk, fk, fk, nul, 4, 128, 128, 8, fk, fk, 4096, nul) == 1
    # SwiGLU clamp: empty interval or NaN bound rejected before anything else
    inf, nan = float("inf"), float("nan")
    assert lib.moe_grouped_fc1_swiglu_clamped(fk, fk, fk, fk, nul, nul, 4, 128, 128, 8, 1.0, 0.5, -inf, inf, fk, nul,
                                              fk, 4096, nul) == 1
    assert lib.moe_grouped_fc1_swiglu_clamped(fk, fk, fk, fk, nul, nul, 4, 128, 128, 8, -inf, inf, nan, 1.0, fk, nul,
                                              fk, 4096, nul) == 1
    assert lib.moe_grouped_fc1_swiglu_clamped(fk, fk, fk, fk, fk, nul, 4, 128, 128, 8, -1.0, 1.0, -1.0, 1.0, fk, nul,
                                              fk, 4096, nul) == 1                 # half of the route maps
    assert lib.moe_grouped_dgrad_fc2_dswiglu_clamped(fk, fk, fk, fk, 4, 128, 128, 8, 0.0, -1.0, -1.0, 1.0, fk, fk,
                                                     4096, nul) == 1
    assert lib.moe_grouped_fc1_swiglu_mxfp8_clamped(fk, fk, fk, fk, fk, fk, fk, 4, 128, 128, 8, 1.0, 0.0, -1.0, 1.0,
                                                    fk, fk, nul, fk, 4096, nul) == 1
    # permute: H % 8, capacity, workspace
    assert lib.moe_permute(nul, nul, 4, 12, 4, 2, 1, nul, 8, nul, nul, nul, nul, nul, 0, nul) == 2
    assert lib.moe_permute(nul, nul, 4, 16, 4, 2, 1, nul, 7, nul, nul, nul, nul, nul, 0, nul) == 1
    fake = C.c_void_p(16)
    assert lib.moe_permute(fake, fake, 4, 16, 4, 2, 1, fake, 8, fake, fake, fake, fake, nul, 0, nul) == 5
    # ffn: H, F multiples of 128
    assert lib.moe_grouped_ffn_fwd(fake, fake, fake, fake, fake, 4, 100, 128, 8, fake, fake, nul, fake, 256, nul) == 2
    assert lib.moe_grouped_ffn_fwd(fake, fake, fake, fake, fake, 4, 128, 128, 8, fake, fake, nul, nul, 0, nul) == 5
    # combine
    assert lib.moe_unpermute_combine(nul, nul, nul, 3, 12, 2, nul, nul) == 2
    assert lib.moe_unpermute_combine(nul, nul, nul, 3, 16, 2, nul, nul) == 1
    # row pointers off a 16-byte boundary (the kernels move 16-byte vectors): refused
    # before the workspace check and before any launch
    mis = C.c_void_p(24)
    assert lib.moe_permute(mis, fake, 4, 16, 4, 2, 1, fake, 8, fake, fake, fake, fake, nul, 0, nul) == 2
    assert lib.moe_permute(fake, fake, 4, 16, 4, 2, 1, mis, 8, fake, fake, fake, fake, nul, 0, nul) == 2
    assert lib.moe_unpermute_combine(mis, fake, nul, 3, 16, 2, fake, nul) == 2
    assert lib.moe_unpermute_combine(fake, fake, nul, 3, 16, 2, mis, nul) == 2
    assert lib.moe_unpermute_sum(mis, fake, 3, 16, 2, fake, nul) == 2
    # weight gradients, fp32 and bf16: null outputs, sizes, workspace -- refused before a launch
    for wg in (lib.moe_grouped_wgrad, lib.moe_grouped_wgrad_bf16):
        assert wg(fake, fake, fake, fake, fake, 4, 128, 128, 64, nul, fake, fake, fake, 256, nul) == 1
        assert wg(fake, fake, fake, fake, fake, 4, 100, 128, 64, fake, fake, fake, fake, 256, nul) == 2
        assert wg(fake, fake, fake, fake, fake, 4, 128, 128, 64, fake, fake, fake, nul, 0, nul) == 5
    assert lib.moe_grouped_ffn_bwd_bf16(*([fake] * 12), 4, 100, 128, 4, 2, 8, *([fake] * 8), fake, 256, nul) == 2


def test_product_path_has_no_oracle_dependency():
    pkg_dir = os.path.join(ROOT, "mixture_experts_ffn_warp_gb300")
    for dirpath, _, files in os.walk(pkg_dir):
        for fn in files:
            if fn.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, fn)).read()
                assert "import oracle" not in text and "from oracle" not in text, fn
                assert "moe_oracle" not in text, fn
