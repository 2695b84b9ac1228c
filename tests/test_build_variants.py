"""The bounds-check build variant (-DMOE_BOUNDS_CHECK) compiles for sm_103a (no GPU: nvcc
cross-compiles one GEMM translation unit with the flag)."""
import os
import shutil
import subprocess

import pytest

from mixture_experts_ffn_warp_gb300 import build as B


@pytest.mark.skipif(shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"),
                    reason="nvcc not available")
def test_bounds_check_build_compiles(tmp_path):
    src = os.path.join(B.CSRC, "ffn_fwd.cu")
    cmd = [B._nvcc(), *B.ARCH, *B.NVCC_FLAGS, "-DMOE_BOUNDS_CHECK", "-c", src, "-o", str(tmp_path / "ffn_fwd.o")]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr[-2000:]
