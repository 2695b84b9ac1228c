"""Pins of the oracle's NVFP4 output encoding (CPU only).

The layer's output may be an NVFP4 block-scaled tensor ("Add MoE + expert-parallel
Python API surface, PyTorch reference, and tests", Summary: bf16, mxfp8 and nvfp4
public outputs; BlockScaledTensor: data plus scale, block_size 16 for nvfp4).  The
oracle encodes the combine's fp32 slot-order sum with E2M1 elements and one E4M3
scale per 16 elements (the reading stated in moe_oracle.c).  Pinned against
hand-worked blocks, an independent implementation (round-to-nearest-even by
threshold counting, the E4M3 grid taken from torch's float8_e4m3fn decoding), the
format's error bound, the minimality of the scale, and the combine's fp32 sum."""
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
E2M1 = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def _expand(field):
    out = []
    for tok in field.split(","):
        tok = tok.strip()
        if "*" in tok:
            v, n = tok.split("*")
            out += [v] * int(n)
        else:
            out.append(tok)
    return out


def _golden():
    with open(os.path.join(GOLDEN, "nvfp4_blocks.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                yield [p.strip() for p in line.split(";")]


def _unpack(codes):
    c = np.asarray(codes, np.uint8)
    return np.stack([c & 0xF, c >> 4], axis=-1).reshape(c.shape[:-1] + (2 * c.shape[-1],))


@pytest.mark.parametrize("case", list(_golden()), ids=lambda c: c[0])
def test_nvfp4_block_golden(case):
    name, vals, scale, codes = case
    v = np.array([float(x) for x in _expand(vals)])
    assert v.size == 16
    assert np.array_equal(v.astype(np.float32).astype(np.float64), v), "fixture values must be fp32-exact"
    got_c, got_s = oracle.nvfp4_encode(v.astype(np.float32).reshape(1, 16))
    assert got_s[0, 0] == int(scale, 16)
    assert list(_unpack(got_c)[0]) == [int(c, 16) for c in _expand(codes)]


def _e4m3_positive_table():
    """(codes 1..0x7E, their values) from torch's own float8_e4m3fn decoding."""
    codes = torch.arange(1, 0x7F, dtype=torch.uint8)
    return codes.numpy(), codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def _independent_encode(v):
    """Scale: the first E4M3 value of torch's table with 6 s >= amax; codes: count the
    rounding thresholds (midpoints of the E2M1 magnitudes) that |v| / s passes, a value
    exactly on a midpoint rounding to the even code."""
    tc, tv = _e4m3_positive_table()
    mids = (E2M1[1:] + E2M1[:-1]) / 2                   # 0.25, 0.75, ..., 5
    up_is_even = (np.arange(1, 8) % 2) == 0             # code above each midpoint even?
    v = np.asarray(v, np.float64).reshape(-1, 16)
    codes = np.zeros(v.shape, np.uint8)
    scales = np.zeros(v.shape[0], np.uint8)
    for b in range(v.shape[0]):
        amax = np.abs(v[b]).max()
        if amax == 0:
            continue
        ok = np.nonzero(6.0 * tv >= amax)[0]
        i = ok[0] if ok.size else len(tv) - 1
        scales[b], s = tc[i], tv[i]
        for e in range(16):
            a = abs(v[b, e])
            thr = s * mids                               # exact: <= 7 significant bits
            c = int(np.sum((a > thr) | ((a == thr) & up_is_even)))
            codes[b, e] = c | (8 if v[b, e] < 0 else 0)
    return codes, scales


def test_matches_an_independent_encoder_on_random_blocks():
    rng = np.random.default_rng(7)
    blocks = []
    for mag in (1e-4, 3e-3, 0.05, 0.7, 1.0, 3.0, 40.0, 500.0, 5000.0):
        blocks.append(rng.standard_normal((40, 16)) * mag)
    # values exactly on rounding midpoints of a power-of-two scale
    grid = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0])
    blocks.append(rng.choice(grid, size=(40, 16)) * rng.choice([1, -1], size=(40, 16)))
    v = np.concatenate(blocks).astype(np.float32)
    codes, scales = oracle.nvfp4_encode(v)
    ic, isc = _independent_encode(v)
    assert np.array_equal(scales.reshape(-1), isc)
    assert np.array_equal(_unpack(codes).reshape(-1, 16), ic)


def test_error_bound_no_clipping_and_minimal_scale():
    rng = np.random.default_rng(8)
    v = (rng.standard_normal((200, 16)) * np.exp(rng.uniform(-6, 6, size=(200, 1)))).astype(np.float32)
    codes, scales = oracle.nvfp4_encode(v)
    vals = oracle.nvfp4_decode(codes, scales)
    s = np.repeat(np.vectorize(oracle.e4m3_to_double)(scales), 16, axis=1)
    q = np.abs(v.astype(np.float64)) / s
    half_step = np.where(q <= 2, 0.25, np.where(q <= 4, 0.5, 1.0)) * s
    assert np.all(np.abs(vals - v) <= half_step)
    amax = np.abs(v.astype(np.float64)).max(axis=1)
    sb = np.vectorize(oracle.e4m3_to_double)(scales[:, 0])
    assert np.all(6.0 * sb >= amax)                              # no element clips
    prev = np.vectorize(oracle.e4m3_to_double)((scales[:, 0] - 1).astype(np.uint8))
    assert np.all((scales[:, 0] == 1) | (6.0 * prev < amax))       # the smallest such scale


def test_combine_encodes_the_fp32_slot_order_sum():
    # small integers times powers of two: every product and fp32 sum is exact
    rng = np.random.default_rng(9)
    T, H, k, rows = 6, 64, 3, 18
    y = (rng.integers(-16, 17, size=(rows, H)) * 0.125).astype(np.float32)
    dst = rng.permutation(rows).reshape(T, k).astype(np.int32)
    dst[2, 1] = -1                                      # a dropped route
    dst[4] = -1                                         # a token with every route dropped
    w = np.array([[0.5, 0.25, 0.125]] * T, np.float32)
    codes, scales = oracle.unpermute_combine_nvfp4(y, dst, w)
    exact = oracle.unpermute_combine(y, dst, w, round_mode=0)
    ec, es = oracle.nvfp4_encode(exact.astype(np.float32))
    assert np.array_equal(codes, ec) and np.array_equal(scales, es)
    assert np.all(codes[4] == 0) and np.all(scales[4] == 0)
    # fp32 slot order: 1e8 + 1 - 1e8 is 0 in fp32
    y2 = np.zeros((3, 16), np.float32)
    y2[0, 0], y2[1, 0], y2[2, 0] = 1e8, 1.0, -1e8
    y2[:, 1] = 0.5
    c2, s2 = oracle.unpermute_combine_nvfp4(y2, np.array([[0, 1, 2]], np.int32), np.ones((1, 3), np.float32))
    assert oracle.nvfp4_decode(c2, s2)[0, 0] == 0.0
    assert oracle.nvfp4_decode(c2, s2)[0, 1] == 1.5
