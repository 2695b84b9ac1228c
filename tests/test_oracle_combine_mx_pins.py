"""Pins of the oracle's combine with an MXFP8 output encoding (CPU only).

The output of the MoE layer may be a block-scaled tensor ("Add MoE +
expert-parallel Python API surface, PyTorch reference, and tests", Summary:
bf16, mxfp8 and nvfp4 public outputs, logical unswizzled layout).  The oracle
sums in fp32 in slot order (the combine's stated accumulation) and applies the MX
rule to that fp32 value.  Pinned against the separately pinned MX quantiser, the
fp32 slot-order semantics, the exact fp64 combine within E4M3's error, and
special cases (dropped routes, all-zero rows)."""
import numpy as np

import oracle


def _case(T=5, H=64, k=3, rows=12, seed=0):
    rng = np.random.default_rng(seed)
    y = rng.standard_normal((rows, H)).astype(np.float32)
    dst = rng.permutation(rows)[:T * k].reshape(T, k).astype(np.int32)
    w = rng.random((T, k)).astype(np.float32)
    return y, dst, w


def test_matches_the_quantiser_when_sums_are_bf16_values():
    # small integers times powers of two: every fp32 sum is exact and bf16-representable
    rng = np.random.default_rng(1)
    T, H, k, rows = 4, 96, 2, 8
    y = (rng.integers(-8, 9, size=(rows, H)) * 0.25).astype(np.float32)
    dst = rng.permutation(rows).reshape(T, k).astype(np.int32)
    w = np.array([[0.5, 0.25]] * T, np.float32)
    codes, scales = oracle.unpermute_combine_mxfp8(y, dst, w)
    exact = oracle.unpermute_combine(y, dst, w, round_mode=0)
    qb, qs = oracle.quantize_rows_mxfp8(oracle.double_to_bf16_bits(exact))
    assert np.array_equal(codes, qb)
    assert np.array_equal(scales, qs)


def test_fp32_slot_order():
    # 1e8 + 1 rounds to 1e8 in fp32, so the slot-order sum 1e8 + 1 - 1e8 is 0, not 1
    H = 32
    y = np.zeros((3, H), np.float32)
    y[0, 0], y[1, 0], y[2, 0] = 1e8, 1.0, -1e8
    y[0, 1], y[1, 1], y[2, 1] = 1.0, 1e8, -1e8
    dst = np.array([[0, 1, 2]], np.int32)
    w = np.ones((1, 3), np.float32)
    codes, scales = oracle.unpermute_combine_mxfp8(y, dst, w)
    vals = oracle.mx_dequantize(codes, scales)
    assert vals[0, 0] == 0.0
    # second column: (0 + 1) + 1e8 = 1e8 (fp32), then - 1e8 = 0 as well
    assert vals[0, 1] == 0.0
    # reversed slots: (-1e8 + 1e8) + 1 = 1
    codes2, scales2 = oracle.unpermute_combine_mxfp8(y, np.array([[2, 0, 1]], np.int32), w)
    assert oracle.mx_dequantize(codes2, scales2)[0, 0] == 1.0


def test_within_e4m3_error_of_the_exact_combine():
    y, dst, w = _case(T=16, H=128, k=4, rows=64, seed=2)
    codes, scales = oracle.unpermute_combine_mxfp8(y, dst, w)
    vals = oracle.mx_dequantize(codes, scales)
    exact = oracle.unpermute_combine(y, dst, w, round_mode=0)
    X = np.repeat(scales.astype(np.int64) - 127, 32, axis=1)
    # half an E4M3 step (2^-4 relative for normal codes, 2^(X-10) near zero) plus the
    # fp32 accumulation's own rounding
    bound = np.maximum(2.0 ** -4 * np.abs(exact), np.ldexp(1.0, X - 10)) + 1e-6 * np.abs(exact).max()
    assert np.all(np.abs(vals - exact) <= bound)


def test_dropped_routes_and_zero_rows():
    y, dst, w = _case(T=4, H=64, k=3, rows=12, seed=3)
    dst[1] = -1                      # token 1: all routes dropped -> zero row
    dst[2, 1] = -1                   # token 2: one route dropped
    codes, scales = oracle.unpermute_combine_mxfp8(y, dst, w)
    assert np.all(codes[1] == 0) and np.all(scales[1] == 0)
    keep = dst[2] >= 0
    c2, s2 = oracle.unpermute_combine_mxfp8(y, dst[2:3, keep], w[2:3, keep])
    assert np.array_equal(codes[2], c2[0]) and np.array_equal(scales[2], s2[0])
