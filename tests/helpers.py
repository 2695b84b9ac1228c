"""Shared helpers for the GPU parity tests: seeded inputs on the device, host
copies for the oracle, and the tolerance checks."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from mixture_experts_ffn_warp_gb300.synthetic import MoeShape, make_inputs

# Floating-point bar: max |err| <= 2e-2 * RMS(reference) for bf16 outputs with
# fp32 accumulation; 6e-2 * RMS for MXFP8 against an oracle that applies the
# same quantisation.
TOL_BF16 = 2e-2
TOL_MXFP8 = 6e-2


def bits(t: torch.Tensor) -> np.ndarray:
    return oracle.bf16_bits(t)


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().double().numpy()


def bf16_half_ulp(ref) -> np.ndarray:
    """Half the spacing of the bf16 grid at each value (8 significant bits): the
    largest error of a correctly rounded bf16 representation of `ref`."""
    ref = np.abs(np.asarray(ref, dtype=np.float64))
    _, e = np.frexp(ref)                 # ref = m * 2^e, m in [0.5, 1)
    return np.ldexp(1.0, np.maximum(e, -125) - 9)


def assert_close_rms(got, ref, tol=TOL_BF16, what="", bf16_out=False):
    """max |got - ref| <= tol * RMS(ref).  bf16_out: `got` is a bf16 output compared with
    the exact value, and the bar applies to the error beyond the output format's own
    rounding of that value (half a bf16 ulp), which alone reaches 2^-9 * max|ref|: more
    than 2e-2 * RMS once the largest element exceeds about 5 * RMS."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.isfinite(got).all(), f"{what}: non-finite values"
    rms = float(np.sqrt(np.mean(ref ** 2)))
    dev = np.abs(got - ref)
    if bf16_out:
        dev = np.maximum(dev - bf16_half_ulp(ref), 0.0)
    err = float(dev.max()) if got.size else 0.0
    assert err <= tol * rms, f"{what}: max|err| {err:.3e} > {tol} * RMS {rms:.3e}"
    return err / rms if rms > 0 else 0.0


def e4m3_half_step(ref, scale_bytes) -> np.ndarray:
    """Half the spacing of the MXFP8 grid at each value of `ref` [rows, K] given the
    blocks' UE8M0 scale bytes [rows, K/32]: 2^(floor(log2 |v|) - 4) for normal E4M3
    codes (3 mantissa bits), at least half the subnormal step 2^(X - 10)."""
    ref = np.abs(np.asarray(ref, dtype=np.float64))
    X = np.repeat(np.asarray(scale_bytes).astype(np.int64) - 127, 32, axis=-1)
    _, e = np.frexp(ref)                 # ref = m * 2^e, m in [0.5, 1)
    return np.maximum(np.ldexp(1.0, e - 5), np.ldexp(1.0, X - 10))


def assert_close_rms_mx(got, ref, scale_bytes, tol=TOL_MXFP8, what=""):
    """max |got - ref| <= tol * RMS(ref) for an MXFP8-encoded output compared with the
    exact value, the bar applied to the error beyond the encoding's own rounding of that
    value (half an E4M3 step at the block's scale), as for bf16 outputs."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.isfinite(got).all(), f"{what}: non-finite values"
    rms = float(np.sqrt(np.mean(ref ** 2)))
    dev = np.maximum(np.abs(got - ref) - e4m3_half_step(ref, scale_bytes), 0.0)
    err = float(dev.max()) if got.size else 0.0
    assert err <= tol * rms, f"{what}: max|err| beyond the encoding {err:.3e} > {tol} * RMS {rms:.3e}"
    return err / rms if rms > 0 else 0.0


def e2m1_half_step(values, scale_bytes) -> np.ndarray:
    """Half the spacing of the NVFP4 grid around each value [rows, K] given the blocks'
    E4M3 scale bytes [rows, K/16]: the E2M1 magnitudes are 0.5 apart below 2, 1 apart
    from 2 to 4 and 2 apart from 4 to 6 (times the block scale s)."""
    s = np.repeat(np.vectorize(oracle.e4m3_to_double)(np.asarray(scale_bytes, np.uint8)), 16, axis=-1)
    q = np.abs(np.asarray(values, np.float64)) / np.where(s > 0, s, 1.0)
    return np.where(q < 2, 0.25, np.where(q < 4, 0.5, 1.0)) * s


def assert_close_rms_nvfp4(got, ref, scale_bytes, tol, what=""):
    """max |got - ref| <= tol * RMS(ref) for an NVFP4-encoded output compared with the
    exact value, the bar applied to the error beyond the encoding's own rounding (half a
    step of the E2M1 grid at the block's scale, taken at the larger of |got| and |ref|)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.isfinite(got).all(), f"{what}: non-finite values"
    rms = float(np.sqrt(np.mean(ref ** 2)))
    hs = np.maximum(e2m1_half_step(got, scale_bytes), e2m1_half_step(ref, scale_bytes))
    dev = np.maximum(np.abs(got - ref) - hs, 0.0)
    err = float(dev.max()) if got.size else 0.0
    assert err <= tol * rms, f"{what}: max|err| beyond the encoding {err:.3e} > {tol} * RMS {rms:.3e}"
    return err / rms if rms > 0 else 0.0


def assert_close_ulp(got, ref, what="", slack=2e-3):
    """Element-wise check of a stored bf16 intermediate against the oracle that
    rounds at the same point: the two may round a value on either side of a
    bf16 rounding boundary (fp32 vs fp64 accumulation), so each element may
    differ by one bf16 ulp (2^-7 relative, at most) plus a small absolute
    slack of `slack` * RMS for the accumulation-order difference."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.isfinite(got).all(), f"{what}: non-finite values"
    rms = float(np.sqrt(np.mean(ref ** 2)))
    bound = 2.0 ** -7 * np.abs(ref) + slack * rms
    bad = np.abs(got - ref) > bound
    assert not bad.any(), f"{what}: {int(bad.sum())} elements beyond 1 ulp + {slack}*RMS; " \
                          f"worst {float(np.abs(got - ref).max()):.3e} (RMS {rms:.3e})"


def gpu_inputs(shape: MoeShape, seed: int = 0, with_dy=None):
    return make_inputs(shape, device="cuda", seed=seed, with_dy=with_dy)


def host_experts(W: torch.Tensor, experts) -> dict:
    """Copy selected experts of a [E, a, b] bf16 device tensor to host bits."""
    return {int(e): bits(W[int(e)]) for e in experts}
