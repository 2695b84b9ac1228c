"""CPU oracle for the MoE FFN hot path -- TEST INFRASTRUCTURE ONLY.

A plain fp64 C implementation (moe_oracle.c) of what the path computes,
loaded with ctypes.  Only tests/, __graft_entry__.smoke() and bench.py's
CPU-baseline / reference leg may import this package; the CUDA product path
never does, and the two share no code.

bf16 tensors cross this boundary as uint16 bit patterns (numpy), fp32 as
float32, indices as int32.  Every function cites the passage it follows in
moe_oracle.c.
"""
from __future__ import annotations

import ctypes as C
import os
from typing import Sequence

import numpy as np

from . import build as _build

_lib = None

_u16p = C.POINTER(C.c_uint16)
_u8p = C.POINTER(C.c_uint8)
_i32p = C.POINTER(C.c_int32)
_i64p = C.POINTER(C.c_int64)
_f32p = C.POINTER(C.c_float)
_f64p = C.POINTER(C.c_double)
_i64 = C.c_int64
_int = C.c_int


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = C.CDLL(path)
        L.oracle_bf16_to_double.restype = C.c_double
        L.oracle_bf16_to_double.argtypes = [C.c_uint16]
        L.oracle_double_to_bf16.restype = C.c_uint16
        L.oracle_double_to_bf16.argtypes = [C.c_double]
        L.oracle_e4m3_to_double.restype = C.c_double
        L.oracle_e4m3_to_double.argtypes = [C.c_uint8]
        L.oracle_double_to_e4m3.restype = C.c_uint8
        L.oracle_double_to_e4m3.argtypes = [C.c_double]
        L.oracle_quantize_mxfp8.restype = None
        L.oracle_quantize_mxfp8.argtypes = [_u16p, _i64, _i64, _i64, _i64, _u8p, _u8p]
        L.oracle_route_topk.restype = None
        L.oracle_route_topk.argtypes = [_f32p, _i64, _int, _int, _i32p, _f32p]
        L.oracle_route_topk_sigmoid.restype = None
        L.oracle_route_topk_sigmoid.argtypes = [_f32p, _f32p, _i64, _int, _int, _int, _i32p, _f32p]
        L.oracle_route_topk_bwd.restype = None
        L.oracle_route_topk_bwd.argtypes = [_f32p, _i32p, _f32p, _i64, _int, _int, _int, _int, _f64p]
        L.oracle_permute.restype = _i64
        L.oracle_permute.argtypes = [_i32p, _i64, _int, _int, _int, _i32p, _i32p, _i64, _i32p, _i32p]
        L.oracle_gather_rows.restype = None
        L.oracle_gather_rows.argtypes = [_u16p, _int, _int, _i32p, _i64, _u16p]
        pp16 = C.POINTER(_u16p)
        pp8 = C.POINTER(_u8p)
        L.oracle_moe_fwd_w.restype = None
        L.oracle_moe_fwd_w.argtypes = [_i64, _i64p, _int, _int, _int, _int, _u16p, pp16, pp16, pp16,
                                       _i32p, _f32p, _int, _int, _int, _f64p, _f64p, _f64p, _f64p]
        L.oracle_set_swiglu_clamp.restype = None
        L.oracle_set_swiglu_clamp.argtypes = [C.c_double] * 4
        L.oracle_mx_fake_quant.restype = None
        L.oracle_mx_fake_quant.argtypes = [_f64p, _i64, _i64, _f64p]
        L.oracle_moe_fwd.restype = None
        L.oracle_moe_fwd.argtypes = [_i64, _i64p, _int, _int, _int, _int, _u16p, pp16, pp16, pp16,
                                     _i32p, _f32p, _int, _f64p, _f64p, _f64p, _f64p]
        L.oracle_moe_fwd_mxfp8.restype = None
        L.oracle_moe_fwd_mxfp8.argtypes = [_i64, _i64p, _int, _int, _int, _int, _u16p,
                                           pp8, pp8, pp8, pp8, pp8, pp8, _i32p, _f32p, _int,
                                           _f64p, _f64p]
        L.oracle_moe_bwd.restype = None
        L.oracle_moe_bwd.argtypes = [_i64, _int, _int, _int, _int, _u16p, pp16, pp16, pp16,
                                     _i32p, _f32p, _u16p, _int, _int, _f64p, _f64p, _f64p, _f64p, _f64p]
        L.oracle_moe_bwd_dx_tokens.restype = None
        L.oracle_moe_bwd_dx_tokens.argtypes = [_i64, _i64p, _int, _int, _int, _int, _u16p, pp16, pp16,
                                               pp16, _i32p, _f32p, _u16p, _int, _int, _f64p, _f64p]
        L.oracle_moe_bwd_dw_entries.restype = None
        L.oracle_moe_bwd_dw_entries.argtypes = [_i64, _i32p, _i32p, _i32p, _i32p, _i64, _int, _int,
                                                _int, _int, _u16p, pp16, pp16, pp16, _i32p, _f32p,
                                                _u16p, _int, _int, _f64p]
        L.oracle_unpermute_combine.restype = None
        L.oracle_unpermute_combine.argtypes = [_f32p, _i32p, _f32p, _i64, _int, _int, _int, _f64p]
        L.oracle_unpermute_combine_mxfp8.restype = None
        L.oracle_unpermute_combine_mxfp8.argtypes = [_f32p, _i32p, _f32p, _i64, _int, _int, _u8p, _u8p]
        L.oracle_nvfp4_encode.restype = None
        L.oracle_nvfp4_encode.argtypes = [_f32p, _i64, _u8p, _u8p]
        L.oracle_nvfp4_value.restype = C.c_double
        L.oracle_nvfp4_value.argtypes = [C.c_uint8, C.c_uint8]
        L.oracle_unpermute_combine_nvfp4.restype = None
        L.oracle_unpermute_combine_nvfp4.argtypes = [_f32p, _i32p, _f32p, _i64, _int, _int, _u8p, _u8p]
        L.oracle_round_bf16_array.restype = None
        L.oracle_round_bf16_array.argtypes = [_f64p, _i64, _f64p]
        L.oracle_num_threads.restype = _int
        L.oracle_num_threads.argtypes = []
        _lib = L
    return _lib


# ---------------------------------------------------------------- helpers

def _c(a: np.ndarray, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


def _p(a: np.ndarray | None, ptype):
    if a is None:
        return None
    return a.ctypes.data_as(ptype)


def bf16_bits(t) -> np.ndarray:
    """uint16 bit patterns of a bf16 torch tensor (copied to the host)."""
    import torch
    return t.detach().to("cpu").contiguous().view(torch.int16).numpy().view(np.uint16)


def bits_to_float(b: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> float64 values (exact)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def double_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    L = lib()
    flat = np.asarray(a, dtype=np.float64).ravel()
    out = np.fromiter((L.oracle_double_to_bf16(float(v)) for v in flat), dtype=np.uint16, count=flat.size)
    return out.reshape(np.shape(a))


def round_bf16(a: np.ndarray) -> np.ndarray:
    """Round a float64 array to bf16 values (RNE), returned as float64."""
    src = _c(a, np.float64)
    out = np.empty_like(src)
    lib().oracle_round_bf16_array(_p(src, _f64p), src.size, _p(out, _f64p))
    return out


def e4m3_to_double(code: int) -> float:
    return lib().oracle_e4m3_to_double(code)


def double_to_e4m3(v: float) -> int:
    return lib().oracle_double_to_e4m3(v)


def num_threads() -> int:
    return lib().oracle_num_threads()


class _PtrArray:
    """Per-expert pointer array (None entries become NULL)."""

    def __init__(self, arrays: Sequence[np.ndarray | None], ptype, dtype):
        self.keep = [None if a is None else _c(a, dtype) for a in arrays]
        self.arr = (ptype * len(self.keep))(*[(_p(a, ptype) if a is not None else ptype()) for a in self.keep])


def _experts(W, E):
    """Accept an [E,...] array or a sequence/dict of per-expert arrays."""
    if isinstance(W, dict):
        if E is None:
            E = max(W.keys()) + 1
        return [W.get(e) for e in range(E)]
    if isinstance(W, np.ndarray):
        return [W[e] for e in range(E)]
    return list(W)


# ---------------------------------------------------------------- A1, A2

def route_topk(logits: np.ndarray, k: int):
    """Top-k routing, softmax over the selected k (moe_oracle.c, A1)."""
    lg = _c(logits, np.float32)
    T, E = lg.shape
    idx = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float32)
    lib().oracle_route_topk(_p(lg, _f32p), T, E, k, _p(idx, _i32p), _p(w, _f32p))
    return idx, w


def route_topk_sigmoid(logits: np.ndarray, k: int, bias: np.ndarray | None = None, normalize: bool = True):
    """Top-k routing on sigmoid scores with an optional expert routing bias
    (selection only); weights = selected scores / (sum + 1e-20) when normalize."""
    lg = _c(logits, np.float32)
    T, E = lg.shape
    b = None if bias is None else _c(bias, np.float32)
    idx = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float32)
    lib().oracle_route_topk_sigmoid(_p(lg, _f32p), None if b is None else _p(b, _f32p), T, E, k, int(normalize),
                                    _p(idx, _i32p), _p(w, _f32p))
    return idx, w


SCORE_SOFTMAX, SCORE_SIGMOID = 0, 1


def route_topk_bwd(logits: np.ndarray, topk_idx: np.ndarray, d_topk_w: np.ndarray, score_fn: int,
                   normalize: bool = True) -> np.ndarray:
    """d_logits [T, E] (float64) of the router for the given selection."""
    lg = _c(logits, np.float32)
    T, E = lg.shape
    ti = _c(topk_idx, np.int32)
    k = ti.shape[1]
    g = _c(d_topk_w, np.float32)
    out = np.empty((T, E), np.float64)
    lib().oracle_route_topk_bwd(_p(lg, _f32p), _p(ti, _i32p), _p(g, _f32p), T, E, k, int(score_fn), int(normalize),
                                _p(out, _f64p))
    return out


def permute(topk_idx: np.ndarray, E: int, align: int = 1, rows_cap: int | None = None):
    """Stable counting sort of routes by expert (moe_oracle.c, A2)."""
    ti = _c(topk_idx, np.int32)
    T, k = ti.shape
    R = T * k
    if rows_cap is None:
        rows_cap = R + E * (align - 1)
    dst = np.empty(R, np.int32)
    src = np.empty(rows_cap, np.int32)
    gs = np.empty(E, np.int32)
    go = np.empty(E + 1, np.int32)
    bad = lib().oracle_permute(_p(ti, _i32p), T, k, E, align, _p(dst, _i32p), _p(src, _i32p),
                               rows_cap, _p(gs, _i32p), _p(go, _i32p))
    return {"dst_of_route": dst.reshape(T, k), "src_of_row": src, "group_sizes": gs,
            "group_offsets": go, "n_invalid": int(bad)}


def gather_rows(x_bits: np.ndarray, k: int, src_of_row: np.ndarray, rows: int) -> np.ndarray:
    xb = _c(x_bits, np.uint16)
    H = xb.shape[1]
    src = _c(src_of_row, np.int32)
    out = np.empty((rows, H), np.uint16)
    lib().oracle_gather_rows(_p(xb, _u16p), H, k, _p(src, _i32p), rows, _p(out, _u16p))
    return out


def unpermute_combine(y_perm: np.ndarray, dst_of_route: np.ndarray, topk_w: np.ndarray,
                      round_mode: int = 1) -> np.ndarray:
    """Weighted combine in slot order of fp32 expert outputs (moe_oracle.c, A5)."""
    yb = _c(y_perm, np.float32)
    H = yb.shape[1]
    dst = _c(dst_of_route, np.int32)
    tw = _c(topk_w, np.float32)
    T, k = dst.shape
    out = np.empty((T, H))
    lib().oracle_unpermute_combine(_p(yb, _f32p), _p(dst, _i32p), _p(tw, _f32p), T, H, k,
                                   round_mode, _p(out, _f64p))
    return out


def unpermute_combine_mxfp8(y_perm: np.ndarray, dst_of_route: np.ndarray, topk_w: np.ndarray):
    """The combine with an MXFP8 output (moe_oracle.c, oracle_unpermute_combine_mxfp8):
    fp32 slot-order sum, then the MX rule along H.  Returns (codes uint8 [T, H],
    scales uint8 [T, H/32])."""
    yb = _c(y_perm, np.float32)
    H = yb.shape[1]
    dst = _c(dst_of_route, np.int32)
    tw = _c(topk_w, np.float32)
    T, k = dst.shape
    codes = np.empty((T, H), np.uint8)
    scales = np.empty((T, H // 32), np.uint8)
    lib().oracle_unpermute_combine_mxfp8(_p(yb, _f32p), _p(dst, _i32p), _p(tw, _f32p), T, H, k,
                                         _p(codes, _u8p), _p(scales, _u8p))
    return codes, scales


def nvfp4_encode(v: np.ndarray):
    """NVFP4 encoding of an fp32 array [..., K] (K % 16 == 0) along its last axis
    (moe_oracle.c, oracle_nvfp4_encode): returns (codes uint8 [..., K/2], two E2M1
    codes per byte with the even element in the low nibble; scales uint8 [..., K/16],
    E4M3 bytes)."""
    a = _c(v, np.float32)
    K = a.shape[-1]
    nb = a.size // 16
    codes = np.empty(a.shape[:-1] + (K // 2,), np.uint8)
    scales = np.empty(a.shape[:-1] + (K // 16,), np.uint8)
    lib().oracle_nvfp4_encode(_p(a, _f32p), nb, _p(codes, _u8p), _p(scales, _u8p))
    return codes, scales


def nvfp4_decode(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """Values of NVFP4 codes [..., K/2] with their block scales [..., K/16] (float64 [..., K])."""
    c = np.asarray(codes, np.uint8)
    nib = np.stack([c & 0xF, c >> 4], axis=-1).reshape(c.shape[:-1] + (c.shape[-1] * 2,))
    sc = np.repeat(np.asarray(scales, np.uint8), 16, axis=-1)
    f = lib().oracle_nvfp4_value
    return np.vectorize(lambda q, s: f(int(q), int(s)))(nib, sc).astype(np.float64)


def unpermute_combine_nvfp4(y_perm: np.ndarray, dst_of_route: np.ndarray, topk_w: np.ndarray):
    """The combine with an NVFP4 output (moe_oracle.c, oracle_unpermute_combine_nvfp4):
    fp32 slot-order sum, then the NVFP4 encoding along H.  Returns (codes uint8
    [T, H/2], scales uint8 [T, H/16])."""
    yb = _c(y_perm, np.float32)
    H = yb.shape[1]
    dst = _c(dst_of_route, np.int32)
    tw = _c(topk_w, np.float32)
    T, k = dst.shape
    codes = np.empty((T, H // 2), np.uint8)
    scales = np.empty((T, H // 16), np.uint8)
    lib().oracle_unpermute_combine_nvfp4(_p(yb, _f32p), _p(dst, _i32p), _p(tw, _f32p), T, H, k,
                                         _p(codes, _u8p), _p(scales, _u8p))
    return codes, scales


# ---------------------------------------------------------------- A3..A5

WEIGHT_IN_COMBINE, WEIGHT_IN_FC1, WEIGHT_IN_FC2 = 0, 1, 2


def moe_fwd(x_bits, Wg, Wu, Wd, topk_idx, topk_w, tokens=None, round_mode: int = 1,
            want_fc1: bool = False, want_h: bool = False, want_y: bool = False, weight_at: int = 0,
            h_mx: bool = False):
    """Per-token forward: SwiGLU experts + weighted combine (moe_oracle.c).

    weight_at: where the router weight is applied (WEIGHT_IN_COMBINE, _FC1, _FC2).
    h_mx: h quantised to MXFP8 along F (the MXFP8 forward's h; operands are then
    passed as their MXFP8 round trips, see moe_bwd_mxfp8).
    Returns dict with out (float64 [n,H]) and optional per-route fc1 [n*k,2F],
    h [n*k,F], y [n*k,H] (NaN rows for dropped routes)."""
    xb = _c(x_bits, np.uint16)
    T, H = xb.shape
    ti = _c(topk_idx, np.int32)
    tw = _c(topk_w, np.float32)
    k = ti.shape[1]
    wg = _experts(Wg, None if not isinstance(Wg, np.ndarray) else Wg.shape[0])
    E = len(wg)
    wu = _experts(Wu, E)
    wd = _experts(Wd, E)
    F = next(a for a in wg if a is not None).shape[1]
    toks = None if tokens is None else _c(tokens, np.int64)
    n = T if toks is None else toks.size
    out = np.empty((n, H), np.float64)
    fc1 = np.full((n * k, 2 * F), np.nan) if want_fc1 else None
    h = np.full((n * k, F), np.nan) if want_h else None
    y = np.full((n * k, H), np.nan) if want_y else None
    pg, pu, pd = (_PtrArray(a, _u16p, np.uint16) for a in (wg, wu, wd))
    lib().oracle_moe_fwd_w(n, _p(toks, _i64p), H, F, E, k, _p(xb, _u16p), pg.arr, pu.arr, pd.arr,
                           _p(ti, _i32p), _p(tw, _f32p), round_mode, int(weight_at), int(h_mx), _p(out, _f64p),
                           _p(fc1, _f64p), _p(h, _f64p), _p(y, _f64p))
    return {"out": out, "fc1": fc1, "h": h, "y": y}


def quantize_mxfp8(in_bits: np.ndarray, n_vec: int, K: int, stride_vec: int, stride_k: int):
    """MXFP8 (E4M3 + UE8M0 per 1x32 block along K) of n_vec vectors
    (moe_oracle.c, oracle_quantize_mxfp8).  Returns (codes [n_vec,K],
    scales [n_vec,K/32])."""
    ib = _c(in_bits, np.uint16)
    data = np.empty((n_vec, K), np.uint8)
    scale = np.empty((n_vec, K // 32), np.uint8)
    lib().oracle_quantize_mxfp8(_p(ib, _u16p), n_vec, K, stride_vec, stride_k,
                                _p(data, _u8p), _p(scale, _u8p))
    return data, scale


def quantize_rows_mxfp8(rows_bits: np.ndarray):
    """Quantise each row of a [n,K] bf16 matrix along K."""
    n, K = rows_bits.shape
    return quantize_mxfp8(rows_bits, n, K, K, 1)


def quantize_cols_mxfp8(mat_bits: np.ndarray):
    """Quantise each column of a [K,N] bf16 matrix along K; codes are
    returned K-contiguous as [N,K] with scales [N,K/32]."""
    K, N = mat_bits.shape
    return quantize_mxfp8(mat_bits, N, K, 1, N)


def moe_fwd_mxfp8(x_bits, Wg_q, Wg_s, Wu_q, Wu_s, Wd_q, Wd_s, topk_idx, topk_w,
                  tokens=None, round_mode: int = 1, want_y: bool = False):
    """MXFP8 forward for a list of tokens (moe_oracle.c, A7).  Weight codes
    and scales are per expert (None for experts not needed): W_gate/W_up as
    [F,H] codes with [F,H/32] scales, W_down as [H,F] codes with [H,F/32]."""
    xb = _c(x_bits, np.uint16)
    T, H = xb.shape
    ti = _c(topk_idx, np.int32)
    tw = _c(topk_w, np.float32)
    k = ti.shape[1]
    lists = [list(a) if not isinstance(a, dict) else a for a in (Wg_q, Wg_s, Wu_q, Wu_s, Wd_q, Wd_s)]
    E = len(lists[0]) if not isinstance(lists[0], dict) else max(lists[0].keys()) + 1
    lists = [_experts(a, E) for a in lists]
    F = next(a for a in lists[0] if a is not None).shape[0]
    toks = None if tokens is None else _c(tokens, np.int64)
    n = T if toks is None else toks.size
    out = np.empty((n, H), np.float64)
    y = np.full((n * k, H), np.nan) if want_y else None
    ptrs = [_PtrArray(a, _u8p, np.uint8) for a in lists]
    lib().oracle_moe_fwd_mxfp8(n, _p(toks, _i64p), H, F, E, k, _p(xb, _u16p),
                               *[p.arr for p in ptrs], _p(ti, _i32p), _p(tw, _f32p), round_mode,
                               _p(out, _f64p), _p(y, _f64p))
    return {"out": out, "y": y}


# ---------------------------------------------------------------- A8

def moe_bwd(x_bits, Wg, Wu, Wd, topk_idx, topk_w, dY_bits, round_mode: int = 1, h_mx: bool = False):
    """Full backward on a small problem (moe_oracle.c, oracle_moe_bwd).  h_mx: the
    MXFP8 forward's h (use through moe_bwd_mxfp8)."""
    xb = _c(x_bits, np.uint16)
    T, H = xb.shape
    ti = _c(topk_idx, np.int32)
    tw = _c(topk_w, np.float32)
    db = _c(dY_bits, np.uint16)
    k = ti.shape[1]
    wg = _experts(Wg, Wg.shape[0] if isinstance(Wg, np.ndarray) else None)
    E = len(wg)
    wu, wd = _experts(Wu, E), _experts(Wd, E)
    F = next(a for a in wg if a is not None).shape[1]
    dx = np.empty((T, H))
    dWg = np.empty((E, H, F))
    dWu = np.empty((E, H, F))
    dWd = np.empty((E, F, H))
    dtw = np.empty((T, k))
    pg, pu, pd = (_PtrArray(a, _u16p, np.uint16) for a in (wg, wu, wd))
    lib().oracle_moe_bwd(T, H, F, E, k, _p(xb, _u16p), pg.arr, pu.arr, pd.arr, _p(ti, _i32p),
                         _p(tw, _f32p), _p(db, _u16p), round_mode, int(h_mx), _p(dx, _f64p), _p(dWg, _f64p),
                         _p(dWu, _f64p), _p(dWd, _f64p), _p(dtw, _f64p))
    return {"dx": dx, "dW_gate": dWg, "dW_up": dWu, "dW_down": dWd, "d_topk_w": dtw}


def moe_bwd_dx_tokens(x_bits, Wg, Wu, Wd, topk_idx, topk_w, dY_bits, tokens, round_mode: int = 1,
                      h_mx: bool = False):
    """dx and d_topk_w of selected tokens (moe_oracle.c)."""
    xb = _c(x_bits, np.uint16)
    T, H = xb.shape
    ti = _c(topk_idx, np.int32)
    tw = _c(topk_w, np.float32)
    db = _c(dY_bits, np.uint16)
    k = ti.shape[1]
    wg = _experts(Wg, Wg.shape[0] if isinstance(Wg, np.ndarray) else None)
    E = len(wg)
    wu, wd = _experts(Wu, E), _experts(Wd, E)
    F = next(a for a in wg if a is not None).shape[1]
    toks = _c(tokens, np.int64)
    n = toks.size
    dx = np.empty((n, H))
    dtw = np.empty((n, k))
    pg, pu, pd = (_PtrArray(a, _u16p, np.uint16) for a in (wg, wu, wd))
    lib().oracle_moe_bwd_dx_tokens(n, _p(toks, _i64p), H, F, E, k, _p(xb, _u16p), pg.arr, pu.arr,
                                   pd.arr, _p(ti, _i32p), _p(tw, _f32p), _p(db, _u16p), round_mode,
                                   int(h_mx), _p(dx, _f64p), _p(dtw, _f64p))
    return {"dx": dx, "d_topk_w": dtw}


def moe_bwd_dw_entries(entries, x_bits, Wg, Wu, Wd, topk_idx, topk_w, dY_bits, round_mode: int = 1,
                       h_mx: bool = False):
    """Selected weight-gradient entries; entries = [(which, e, a, b)] with
    which 0 = dW_gate[e,h,f], 1 = dW_up[e,h,f], 2 = dW_down[e,f,n]."""
    ent = np.asarray(entries, dtype=np.int32).reshape(-1, 4)
    which, ee, aa, bb = (np.ascontiguousarray(ent[:, i]) for i in range(4))
    xb = _c(x_bits, np.uint16)
    T, H = xb.shape
    ti = _c(topk_idx, np.int32)
    tw = _c(topk_w, np.float32)
    db = _c(dY_bits, np.uint16)
    k = ti.shape[1]
    wg = _experts(Wg, Wg.shape[0] if isinstance(Wg, np.ndarray) else None)
    E = len(wg)
    wu, wd = _experts(Wu, E), _experts(Wd, E)
    F = next(a for a in wg if a is not None).shape[1]
    val = np.empty(len(ent))
    pg, pu, pd = (_PtrArray(a, _u16p, np.uint16) for a in (wg, wu, wd))
    lib().oracle_moe_bwd_dw_entries(len(ent), _p(which, _i32p), _p(ee, _i32p), _p(aa, _i32p),
                                    _p(bb, _i32p), T, H, F, E, k, _p(xb, _u16p), pg.arr, pu.arr,
                                    pd.arr, _p(ti, _i32p), _p(tw, _f32p), _p(db, _u16p),
                                    round_mode, int(h_mx), _p(val, _f64p))
    return val


# ---------------------------------------------------------------- A8 on the MXFP8 path

_E4M3_TABLE = None


def mx_dequantize(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """Values of MXFP8 vectors: codes [n, K] (E4M3) times 2^(scale - 127) per 32
    elements along K (moe_oracle.c, oracle_e4m3_to_double)."""
    global _E4M3_TABLE
    if _E4M3_TABLE is None:
        _E4M3_TABLE = np.array([e4m3_to_double(c) for c in range(256)])
    vals = _E4M3_TABLE[codes.astype(np.int64)]
    exp = np.repeat(scales.astype(np.int64) - 127, 32, axis=-1)
    return np.ldexp(vals, exp)


def _exact_bf16_bits(v: np.ndarray) -> np.ndarray:
    """bf16 bit patterns of values that bf16 holds exactly (raises otherwise)."""
    f32 = np.asarray(v, dtype=np.float64).astype(np.float32)
    u = f32.view(np.uint32)
    if not np.array_equal(f32.astype(np.float64), v) or np.any(u & 0xFFFF):
        raise ValueError("an MXFP8 value is not exactly representable in bf16")
    return (u >> 16).astype(np.uint16)


def mx_roundtrip_rows(rows_bits: np.ndarray) -> np.ndarray:
    """bf16 bits of deq(Q(row)) for each row of [n, K], quantised along K."""
    q, sc = quantize_rows_mxfp8(rows_bits)
    return _exact_bf16_bits(mx_dequantize(q, sc)).reshape(rows_bits.shape)


def mx_roundtrip_cols(mat_bits: np.ndarray) -> np.ndarray:
    """bf16 bits of deq(Q(column)) for each column of [K, N], quantised along K."""
    q, sc = quantize_cols_mxfp8(mat_bits)          # [N, K] codes, [N, K/32] scales
    return np.ascontiguousarray(_exact_bf16_bits(mx_dequantize(q, sc)).T)


def mx_roundtrip_weights(Wg, Wu, Wd, experts=None):
    """MXFP8 round trips of the expert weights along their forward contraction
    axes: W_gate / W_up [H, F] along H, W_down [F, H] along F.  Returns three
    per-expert lists (None for experts not in `experts`)."""
    E = len(Wg)
    keep = set(range(E)) if experts is None else {int(e) for e in experts}
    f = lambda W: [mx_roundtrip_cols(np.asarray(W[e])) if e in keep else None for e in range(E)]  # noqa: E731
    return f(Wg), f(Wu), f(Wd)


def moe_bwd_mxfp8(x_bits, Wg, Wu, Wd, topk_idx, topk_w, dY_bits, round_mode: int = 1):
    """Straight-through backward of the MXFP8 forward on a small problem: the bf16
    backward (oracle_moe_bwd) on the MXFP8 round trips of x and the weights, with
    the forward's MXFP8 h ("Add MoE + expert-parallel Python API surface, PyTorch
    reference, and tests", Summary: quantization round-trips are straight-through).
    Gradients are with respect to the unquantised x and weights."""
    xq = mx_roundtrip_rows(np.asarray(x_bits))
    wg, wu, wd = mx_roundtrip_weights(Wg, Wu, Wd)
    return moe_bwd(xq, wg, wu, wd, topk_idx, topk_w, dY_bits, round_mode=round_mode, h_mx=True)


def mx_fake_quant(v: np.ndarray) -> np.ndarray:
    """Values of the MXFP8 round trip of each row of a float64 [n, K] array along K
    (moe_oracle.c, mx_fake_quant: the rule applied to h on the MXFP8 path)."""
    a = np.ascontiguousarray(v, dtype=np.float64)
    n, K = a.reshape(-1, a.shape[-1]).shape
    out = np.empty_like(a)
    lib().oracle_mx_fake_quant(_p(a, _f64p), n, K, _p(out, _f64p))
    return out


class swiglu_clamp:
    """Context manager: the oracle's SwiGLU inputs clamped, g to [gate_lo, gate_hi] and u
    to [up_lo, up_hi], inclusive bounds (moe_oracle.c, oracle_set_swiglu_clamp); the
    clamp is off again on exit."""

    def __init__(self, gate_lo=-np.inf, gate_hi=np.inf, up_lo=-np.inf, up_hi=np.inf):
        self.bounds = (float(gate_lo), float(gate_hi), float(up_lo), float(up_hi))

    def __enter__(self):
        lib().oracle_set_swiglu_clamp(*self.bounds)
        return self

    def __exit__(self, *exc):
        lib().oracle_set_swiglu_clamp(-np.inf, np.inf, -np.inf, np.inf)
        return False
