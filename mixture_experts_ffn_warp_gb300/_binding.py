"""ctypes binding of the C ABI declared in include/moe.h.

Argument marshalling only: every step runs in the CUDA library
(_build/libmoe_gb300.so).  There is no CPU fallback -- if the library is
missing or CUDA is unavailable, calls raise.  torch supplies device memory
and the current stream.
"""
from __future__ import annotations

import ctypes as C
import os
from dataclasses import dataclass

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libmoe_gb300.so")

MOE_OK = 0
STATUS = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED", 3: "MOE_ERR_CUDA",
          4: "MOE_ERR_DEVICE_DATA", 5: "MOE_ERR_WORKSPACE"}
DEVERR_BAD_EXPERT_ID = 0x1
DEVERR_TIMEOUT = 0x2
DEVERR_CAPACITY = 0x4

_vp = C.c_void_p
_i64 = C.c_int64
_int = C.c_int
_sz = C.c_size_t
_st = C.c_int

# name -> (restype, argtypes); mirrors include/moe.h
SIGNATURES = {
    "moe_status_string": (C.c_char_p, [_int]),
    "moe_abi_version": (_int, []),
    "moe_workspace_bytes": (_sz, [_i64, _int, _int]),
    "moe_workspace_init": (_st, [_vp, _sz, _vp]),
    "moe_workspace_set_wait_limit": (_st, [_vp, _sz, C.c_uint32, _vp]),
    "moe_read_device_error": (_st, [_vp, _vp, C.POINTER(C.c_uint32)]),
    "moe_route_topk": (_st, [_vp, _i64, _int, _int, _vp, _vp, _vp]),
    "moe_route_topk_sigmoid": (_st, [_vp, _vp, _i64, _int, _int, _int, _vp, _vp, _vp]),
    "moe_route_topk_bwd": (_st, [_vp, _vp, _vp, _i64, _int, _int, _int, _int, _vp, _vp]),
    "moe_permute": (_st, [_vp, _vp, _i64, _int, _int, _int, _int, _vp, _i64, _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "moe_permute_static_scratch": (_st, [_vp, _vp, _i64, _int, _int, _int, _int, _vp, _i64, _vp, _vp, _vp, _vp,
                                         _vp, _vp]),
    "moe_grouped_ffn_fwd": (_st, [_vp, _vp, _vp, _vp, _vp, _int, _int, _int, _i64, _vp, _vp, _vp, _vp, _sz, _vp]),
    "moe_grouped_fc1_swiglu": (_st, [_vp, _vp, _vp, _vp, _int, _int, _int, _i64, _vp, _vp, _vp, _sz, _vp]),
    "moe_grouped_fc2": (_st, [_vp, _vp, _vp, _int, _int, _int, _i64, _vp, _vp, _sz, _vp]),
    "moe_grouped_fc1_swiglu_weighted": (_st, [_vp, _vp, _vp, _vp, _vp, _vp, _int, _int, _int, _i64, _vp, _vp, _vp,
                                              _sz, _vp]),
    "moe_grouped_fc2_weighted": (_st, [_vp, _vp, _vp, _vp, _vp, _int, _int, _int, _i64, _vp, _vp, _sz, _vp]),
    "moe_unpermute_combine": (_st, [_vp, _vp, _vp, _i64, _int, _int, _vp, _vp]),
    "moe_grouped_ffn_bwd": (_st, [_vp] * 12 + [_i64, _int, _int, _int, _int, _i64] + [_vp] * 8 + [_vp, _sz, _vp]),
    "moe_grouped_ffn_bwd_bf16": (_st, [_vp] * 12 + [_i64, _int, _int, _int, _int, _i64] + [_vp] * 8 + [_vp, _sz, _vp]),
    "moe_combine_bwd": (_st, [_vp, _vp, _vp, _vp, _vp, _vp, _i64, _int, _int, _int, _i64, _vp, _vp, _vp]),
    "moe_grouped_dgrad_fc2_dswiglu": (_st, [_vp, _vp, _vp, _vp, _int, _int, _int, _i64, _vp, _vp, _sz, _vp]),
    "moe_grouped_dgrad_fc2_dswiglu_clamped": (_st, [_vp, _vp, _vp, _vp, _int, _int, _int, _i64] + [C.c_float] * 4
                                              + [_vp, _vp, _sz, _vp]),
    "moe_grouped_fc1_swiglu_clamped": (_st, [_vp] * 6 + [_int, _int, _int, _i64] + [C.c_float] * 4
                                       + [_vp, _vp, _vp, _sz, _vp]),
    "moe_grouped_dgrad_fc1": (_st, [_vp, _vp, _vp, _vp, _int, _int, _int, _i64, _vp, _vp, _sz, _vp]),
    "moe_grouped_wgrad": (_st, [_vp, _vp, _vp, _vp, _vp, _int, _int, _int, _i64, _vp, _vp, _vp, _vp, _sz, _vp]),
    "moe_grouped_wgrad_bf16": (_st, [_vp, _vp, _vp, _vp, _vp, _int, _int, _int, _i64, _vp, _vp, _vp, _vp, _sz, _vp]),
    "moe_unpermute_sum": (_st, [_vp, _vp, _i64, _int, _int, _vp, _vp]),
    "moe_mx_tile_scale_bytes": (_sz, [_i64, _int, _int]),
    "moe_grouped_quantize_mxfp8": (_st, [_vp, _i64, _int, _vp, _int, _vp, _vp, _vp, _vp, _sz, _vp]),
    "moe_quantize_weights_mxfp8": (_st, [_vp, _int, _int, _int, _vp, _vp, _vp]),
    "moe_permute_mxfp8": (_st, [_vp, _vp, _i64, _int, _int, _int, _vp, _vp, _i64, _vp, _vp, _vp, _vp, _vp, _sz,
                                _vp]),
    "moe_grouped_ffn_fwd_mxfp8": (_st, [_vp] * 9 + [_int, _int, _int, _i64, _vp, _vp, _vp, _vp, _sz, _vp]),
    "moe_grouped_fc1_swiglu_mxfp8": (_st, [_vp] * 7 + [_int, _int, _int, _i64, _vp, _vp, _vp, _vp, _sz, _vp]),
    "moe_dequantize_rows_mxfp8": (_st, [_vp, _vp, _vp, _int, _i64, _int, _vp, _vp, _sz, _vp]),
    "moe_grouped_fc1_swiglu_mxfp8_clamped": (_st, [_vp] * 7 + [_int, _int, _int, _i64] + [C.c_float] * 4
                                             + [_vp, _vp, _vp, _vp, _sz, _vp]),
    "moe_unpermute_combine_mxfp8": (_st, [_vp, _vp, _vp, _i64, _int, _int, _vp, _vp, _vp]),
    "moe_unpermute_combine_nvfp4": (_st, [_vp, _vp, _vp, _i64, _int, _int, _vp, _vp, _vp]),
    "moe_dequantize_weights_mxfp8": (_st, [_vp, _vp, _int, _int, _int, _vp, _vp]),
    "moe_grouped_fc2_mxfp8": (_st, [_vp] * 5 + [_int, _int, _int, _i64, _vp, _vp, _sz, _vp]),
}

_lib = None


class MoeError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} failed: {STATUS.get(status, status)}")
        self.status = status


def load_library(path: str | None = None):
    """Load (once) the CUDA library; raises if it has not been built."""
    global _lib
    if _lib is None:
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(f"CUDA library not built: {p} (run __graft_entry__.build())")
        L = C.CDLL(p)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _check(fn: str, status: int):
    if status != MOE_OK:
        raise MoeError(fn, status)


def _ptr(t: torch.Tensor | None):
    return None if t is None else C.c_void_p(t.data_ptr())


def _stream(stream) -> C.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return C.c_void_p(stream.cuda_stream)


def _need(t: torch.Tensor, name: str, dtype: torch.dtype, shape: tuple | None = None, device=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} shape must be {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if device is not None and t.device != device:
        raise ValueError(f"{name} must be on {device}, got {t.device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


# ------------------------------------------------------------------ workspace

class Workspace:
    """Device workspace (error word + permutation scratch) for T, E, k."""

    def __init__(self, T: int, E: int, k: int, device=None, stream=None):
        L = load_library()
        n = L.moe_workspace_bytes(T, E, k)
        if n == 0:
            raise ValueError(f"invalid sizes T={T} E={E} k={k}")
        self.nbytes = int(n)
        self.buf = torch.empty(self.nbytes, dtype=torch.uint8, device=device or "cuda")
        _check("moe_workspace_init", L.moe_workspace_init(_ptr(self.buf), self.nbytes, _stream(stream)))

    def reset(self, stream=None):
        _check("moe_workspace_init", load_library().moe_workspace_init(_ptr(self.buf), self.nbytes, _stream(stream)))

    def set_wait_limit(self, limit_ns: int, stream=None):
        """Limit of the GEMMs' device spin waits in ns (0: the default 2 s)."""
        _check("moe_workspace_set_wait_limit", load_library().moe_workspace_set_wait_limit(
            _ptr(self.buf), self.nbytes, int(limit_ns), _stream(stream)))

    def read_error(self, stream=None) -> int:
        """Device error word (synchronises the stream)."""
        v = C.c_uint32(0)
        st = load_library().moe_read_device_error(_ptr(self.buf), _stream(stream), C.byref(v))
        if st not in (MOE_OK, 4):
            raise MoeError("moe_read_device_error", st)
        return int(v.value)


# ------------------------------------------------------------------ A1

def moe_route_topk(logits: torch.Tensor, k: int, topk_idx=None, topk_w=None, stream=None):
    """Top-k routing with a softmax over the selected k logits (moe.h)."""
    _need(logits, "logits", torch.float32)
    if logits.dim() != 2:
        raise ValueError("logits must be [T, E]")
    T, E = logits.shape
    if topk_idx is None:
        topk_idx = torch.empty(T, k, dtype=torch.int32, device=logits.device)
    if topk_w is None:
        topk_w = torch.empty(T, k, dtype=torch.float32, device=logits.device)
    _need(topk_idx, "topk_idx", torch.int32, (T, k), logits.device)
    _need(topk_w, "topk_w", torch.float32, (T, k), logits.device)
    _check("moe_route_topk", load_library().moe_route_topk(
        _ptr(logits), T, E, k, _ptr(topk_idx), _ptr(topk_w), _stream(stream)))
    return topk_idx, topk_w


SCORE_SOFTMAX, SCORE_SIGMOID = 0, 1   # moe.h MOE_SCORE_*


def moe_route_topk_sigmoid(logits: torch.Tensor, k: int, expert_bias=None, normalize: bool = True, topk_idx=None,
                           topk_w=None, stream=None):
    """Top-k routing on sigmoid scores; the expert routing bias takes part in the
    selection only; weights / (sum + 1e-20) when normalize (moe.h)."""
    _need(logits, "logits", torch.float32)
    if logits.dim() != 2:
        raise ValueError("logits must be [T, E]")
    T, E = logits.shape
    if expert_bias is not None:
        _need(expert_bias, "expert_bias", torch.float32, (E,), logits.device)
    if topk_idx is None:
        topk_idx = torch.empty(T, k, dtype=torch.int32, device=logits.device)
    if topk_w is None:
        topk_w = torch.empty(T, k, dtype=torch.float32, device=logits.device)
    _need(topk_idx, "topk_idx", torch.int32, (T, k), logits.device)
    _need(topk_w, "topk_w", torch.float32, (T, k), logits.device)
    _check("moe_route_topk_sigmoid", load_library().moe_route_topk_sigmoid(
        _ptr(logits), _ptr(expert_bias), T, E, k, int(bool(normalize)), _ptr(topk_idx), _ptr(topk_w),
        _stream(stream)))
    return topk_idx, topk_w


def moe_route_topk_bwd(logits: torch.Tensor, topk_idx: torch.Tensor, d_topk_w: torch.Tensor, score_fn: int,
                       normalize: bool = True, d_logits=None, stream=None):
    """fp32 logits gradient of the router for the given selection (moe.h)."""
    _need(logits, "logits", torch.float32)
    if logits.dim() != 2:
        raise ValueError("logits must be [T, E]")
    T, E = logits.shape
    k = topk_idx.shape[1] if topk_idx.dim() == 2 else -1
    _need(topk_idx, "topk_idx", torch.int32, (T, k), logits.device)
    _need(d_topk_w, "d_topk_w", torch.float32, (T, k), logits.device)
    if d_logits is None:
        d_logits = torch.empty(T, E, dtype=torch.float32, device=logits.device)
    _need(d_logits, "d_logits", torch.float32, (T, E), logits.device)
    _check("moe_route_topk_bwd", load_library().moe_route_topk_bwd(
        _ptr(logits), _ptr(topk_idx), _ptr(d_topk_w), T, E, k, int(score_fn), int(bool(normalize)),
        _ptr(d_logits), _stream(stream)))
    return d_logits


# ------------------------------------------------------------------ A2

@dataclass
class Permutation:
    x_perm: torch.Tensor        # [rows_cap, H]
    dst_of_route: torch.Tensor  # [T, k] int32
    src_of_row: torch.Tensor    # [rows_cap] int32
    group_sizes: torch.Tensor   # [E] int32
    group_offsets: torch.Tensor # [E+1] int32
    rows_cap: int
    align: int


def rows_capacity(T: int, k: int, E: int, align: int = 1) -> int:
    return T * k + E * (align - 1)


def moe_permute(x: torch.Tensor, topk_idx: torch.Tensor, E: int, ws: Workspace, align: int = 1,
                out: Permutation | None = None, stream=None) -> Permutation:
    """Expert-contiguous permutation with device-side group sizes (moe.h)."""
    _need(x, "x", torch.bfloat16)
    T, H = x.shape
    _need(topk_idx, "topk_idx", torch.int32, None, x.device)
    if topk_idx.dim() != 2 or topk_idx.shape[0] != T:
        raise ValueError(f"topk_idx must be [{T}, k]")
    k = topk_idx.shape[1]
    cap = rows_capacity(T, k, E, align)
    if out is None:
        dev = x.device
        out = Permutation(
            x_perm=torch.empty(cap, H, dtype=torch.bfloat16, device=dev),
            dst_of_route=torch.empty(T, k, dtype=torch.int32, device=dev),
            src_of_row=torch.empty(cap, dtype=torch.int32, device=dev),
            group_sizes=torch.empty(E, dtype=torch.int32, device=dev),
            group_offsets=torch.empty(E + 1, dtype=torch.int32, device=dev),
            rows_cap=cap, align=align)
    _check("moe_permute", load_library().moe_permute(
        _ptr(x), _ptr(topk_idx), T, H, E, k, align, _ptr(out.x_perm), out.rows_cap,
        _ptr(out.dst_of_route), _ptr(out.src_of_row), _ptr(out.group_sizes), _ptr(out.group_offsets),
        _ptr(ws.buf), ws.nbytes, _stream(stream)))
    return out


# ------------------------------------------------------------------ A3 + A4

def moe_grouped_ffn_fwd(x_perm: torch.Tensor, W_gate: torch.Tensor, W_up: torch.Tensor,
                        W_down: torch.Tensor, group_offsets: torch.Tensor, ws: Workspace,
                        want_fc1_c: bool = False, h=None, y_perm=None, fc1_c=None, stream=None):
    """Grouped SwiGLU expert FFN on tcgen05 (moe.h).  Returns (h, y_perm, fc1_c)."""
    _need(x_perm, "x_perm", torch.bfloat16)
    rows_cap, H = x_perm.shape
    dev = x_perm.device
    E, H2, F = W_gate.shape
    if H2 != H:
        raise ValueError(f"W_gate must be [E, {H}, F]")
    _need(W_gate, "W_gate", torch.bfloat16, (E, H, F), dev)
    _need(W_up, "W_up", torch.bfloat16, (E, H, F), dev)
    _need(W_down, "W_down", torch.bfloat16, (E, F, H), dev)
    _need(group_offsets, "group_offsets", torch.int32, (E + 1,), dev)
    if h is None:
        h = torch.empty(rows_cap, F, dtype=torch.bfloat16, device=dev)
    if y_perm is None:
        y_perm = torch.empty(rows_cap, H, dtype=torch.bfloat16, device=dev)
    if want_fc1_c and fc1_c is None:
        fc1_c = torch.empty(rows_cap, 2 * F, dtype=torch.bfloat16, device=dev)
    _need(h, "h", torch.bfloat16, (rows_cap, F), dev)
    _need(y_perm, "y_perm", torch.bfloat16, (rows_cap, H), dev)
    if fc1_c is not None:
        _need(fc1_c, "fc1_c", torch.bfloat16, (rows_cap, 2 * F), dev)
    _check("moe_grouped_ffn_fwd", load_library().moe_grouped_ffn_fwd(
        _ptr(x_perm), _ptr(W_gate), _ptr(W_up), _ptr(W_down), _ptr(group_offsets), E, H, F, rows_cap,
        _ptr(h), _ptr(y_perm), _ptr(fc1_c), _ptr(ws.buf), ws.nbytes, _stream(stream)))
    return h, y_perm, fc1_c


def moe_grouped_fc1_swiglu(x_perm, W_gate, W_up, group_offsets, ws: Workspace, h, fc1_c=None, stream=None,
                           route_weights=None, clamp=None):
    """A3 alone: h = silu(x W_gate) * (x W_up) per group (moe.h).  route_weights =
    (src_of_row, topk_w): h of each row scaled by its route's router weight.  clamp =
    (gate_lo, gate_hi, up_lo, up_hi): the SwiGLU inputs clamped to those inclusive bounds."""
    rows_cap, H = x_perm.shape
    E, _, F = W_gate.shape
    if clamp is not None:
        src, tw = route_weights if route_weights is not None else (None, None)
        _check("moe_grouped_fc1_swiglu_clamped", load_library().moe_grouped_fc1_swiglu_clamped(
            _ptr(x_perm), _ptr(W_gate), _ptr(W_up), _ptr(group_offsets), _ptr(src), _ptr(tw), E, H, F, rows_cap,
            *[float(v) for v in clamp], _ptr(h), _ptr(fc1_c), _ptr(ws.buf), ws.nbytes, _stream(stream)))
    elif route_weights is None:
        _check("moe_grouped_fc1_swiglu", load_library().moe_grouped_fc1_swiglu(
            _ptr(x_perm), _ptr(W_gate), _ptr(W_up), _ptr(group_offsets), E, H, F, rows_cap, _ptr(h),
            _ptr(fc1_c), _ptr(ws.buf), ws.nbytes, _stream(stream)))
    else:
        src, tw = route_weights
        _check("moe_grouped_fc1_swiglu_weighted", load_library().moe_grouped_fc1_swiglu_weighted(
            _ptr(x_perm), _ptr(W_gate), _ptr(W_up), _ptr(group_offsets), _ptr(src), _ptr(tw), E, H, F, rows_cap,
            _ptr(h), _ptr(fc1_c), _ptr(ws.buf), ws.nbytes, _stream(stream)))
    return h


def moe_grouped_fc2(h, W_down, group_offsets, ws: Workspace, y_perm, stream=None, route_weights=None):
    """A4 alone: y_perm = bf16(h W_down) per group (moe.h).  route_weights = (src_of_row,
    topk_w): y of each row scaled by its route's router weight."""
    rows_cap, F = h.shape
    E, _, H = W_down.shape
    _need(y_perm, "y_perm", torch.bfloat16, (rows_cap, H), h.device)
    if route_weights is None:
        _check("moe_grouped_fc2", load_library().moe_grouped_fc2(
            _ptr(h), _ptr(W_down), _ptr(group_offsets), E, H, F, rows_cap, _ptr(y_perm),
            _ptr(ws.buf), ws.nbytes, _stream(stream)))
    else:
        src, tw = route_weights
        _check("moe_grouped_fc2_weighted", load_library().moe_grouped_fc2_weighted(
            _ptr(h), _ptr(W_down), _ptr(group_offsets), _ptr(src), _ptr(tw), E, H, F, rows_cap, _ptr(y_perm),
            _ptr(ws.buf), ws.nbytes, _stream(stream)))
    return y_perm


# ------------------------------------------------------------------ A5

def moe_unpermute_combine(y_perm: torch.Tensor, dst_of_route: torch.Tensor, topk_w,
                          out=None, stream=None) -> torch.Tensor:
    """out[t] = sum_j w[t,j] * y_perm[dst[t,j]] in fp32, slot order, over bf16 expert
    outputs (moe.h); topk_w None: the plain sum (weights already applied in FC1 or FC2)."""
    _need(y_perm, "y_perm", torch.bfloat16)
    H = y_perm.shape[1]
    dev = y_perm.device
    _need(dst_of_route, "dst_of_route", torch.int32, None, dev)
    T, k = dst_of_route.shape
    if topk_w is not None:
        _need(topk_w, "topk_w", torch.float32, (T, k), dev)
    if out is None:
        out = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
    _need(out, "out", torch.bfloat16, (T, H), dev)
    _check("moe_unpermute_combine", load_library().moe_unpermute_combine(
        _ptr(y_perm), _ptr(dst_of_route), _ptr(topk_w), T, H, k, _ptr(out), _stream(stream)))
    return out


# ------------------------------------------------------------------ A8 backward steps

def moe_combine_bwd(dY, y_perm, perm: "Permutation", topk_w, dy_perm, d_topk_w=None, stream=None):
    """dy_perm = w * dY scattered to the forward rows; d_topk_w = <dY, y> over the bf16
    expert outputs y_perm (moe.h)."""
    T, H = dY.shape
    if y_perm is not None:
        _need(y_perm, "y_perm", torch.bfloat16, None, dY.device)
    k = perm.dst_of_route.shape[1]
    E = perm.group_sizes.shape[0]
    _check("moe_combine_bwd", load_library().moe_combine_bwd(
        _ptr(dY), _ptr(y_perm), _ptr(perm.dst_of_route), _ptr(topk_w), _ptr(perm.group_sizes),
        _ptr(perm.group_offsets), T, H, E, k, perm.rows_cap, _ptr(dy_perm), _ptr(d_topk_w), _stream(stream)))


def moe_grouped_dgrad_fc2_dswiglu(dy_perm, W_down, fc1_c, group_offsets, ws: Workspace, dgu, stream=None, clamp=None):
    """dgu = dSwiGLU(dy_perm W_down^T) from the fc1_c stash (moe.h); clamp: the forward's
    SwiGLU input bounds (gate_lo, gate_hi, up_lo, up_hi)."""
    rows_cap, H = dy_perm.shape
    E, F, _ = W_down.shape
    if clamp is not None:
        _check("moe_grouped_dgrad_fc2_dswiglu_clamped", load_library().moe_grouped_dgrad_fc2_dswiglu_clamped(
            _ptr(dy_perm), _ptr(W_down), _ptr(fc1_c), _ptr(group_offsets), E, H, F, rows_cap,
            *[float(v) for v in clamp], _ptr(dgu), _ptr(ws.buf), ws.nbytes, _stream(stream)))
        return
    _check("moe_grouped_dgrad_fc2_dswiglu", load_library().moe_grouped_dgrad_fc2_dswiglu(
        _ptr(dy_perm), _ptr(W_down), _ptr(fc1_c), _ptr(group_offsets), E, H, F, rows_cap, _ptr(dgu),
        _ptr(ws.buf), ws.nbytes, _stream(stream)))


def moe_grouped_dgrad_fc1(dgu, W_gate, W_up, group_offsets, ws: Workspace, dx_perm, stream=None):
    """dx_perm = [dg|du] [W_gate; W_up]^T per group (moe.h)."""
    rows_cap = dgu.shape[0]
    E, H, F = W_gate.shape
    _check("moe_grouped_dgrad_fc1", load_library().moe_grouped_dgrad_fc1(
        _ptr(dgu), _ptr(W_gate), _ptr(W_up), _ptr(group_offsets), E, H, F, rows_cap, _ptr(dx_perm),
        _ptr(ws.buf), ws.nbytes, _stream(stream)))


def moe_grouped_wgrad(x_perm, h, dy_perm, dgu, group_offsets, ws: Workspace, dW_gate, dW_up, dW_down,
                      stream=None):
    """Weight gradients per expert, K = the group's rows (moe.h): fp32 accumulation, stored in
    the dtype of the dW tensors (fp32, or bf16 through moe_grouped_wgrad_bf16)."""
    rows_cap, H = x_perm.shape
    E, _, F = dW_gate.shape
    fn = "moe_grouped_wgrad_bf16" if dW_gate.dtype == torch.bfloat16 else "moe_grouped_wgrad"
    for name, t in (("dW_gate", dW_gate), ("dW_up", dW_up), ("dW_down", dW_down)):
        if t.dtype != dW_gate.dtype or t.dtype not in (torch.float32, torch.bfloat16):
            raise ValueError(f"{name}: fp32 or bf16, all three the same dtype")
    _check(fn, getattr(load_library(), fn)(
        _ptr(x_perm), _ptr(h), _ptr(dy_perm), _ptr(dgu), _ptr(group_offsets), E, H, F, rows_cap,
        _ptr(dW_gate), _ptr(dW_up), _ptr(dW_down), _ptr(ws.buf), ws.nbytes, _stream(stream)))


def moe_unpermute_sum(dx_perm, dst_of_route, dx, stream=None):
    """dx[t] = sum_j dx_perm[dst[t,j]] (moe.h)."""
    T, k = dst_of_route.shape
    H = dx_perm.shape[1]
    _check("moe_unpermute_sum", load_library().moe_unpermute_sum(
        _ptr(dx_perm), _ptr(dst_of_route), T, H, k, _ptr(dx), _stream(stream)))


def moe_grouped_ffn_bwd(dY, x_perm, W_gate, W_up, W_down, fc1_c, h, y_perm, perm: "Permutation", topk_w,
                        ws: Workspace, want_d_topk_w: bool = True, stream=None, dw_dtype=torch.float32):
    """The whole backward in one call (moe.h); allocates its outputs and scratch.  dw_dtype:
    fp32 weight gradients (moe_grouped_ffn_bwd) or bf16 (moe_grouped_ffn_bwd_bf16).
    Returns dict(dx, dW_gate, dW_up, dW_down, d_topk_w)."""
    if dw_dtype not in (torch.float32, torch.bfloat16):
        raise ValueError("dw_dtype: torch.float32 or torch.bfloat16")
    dev = dY.device
    T, H = dY.shape
    E, _, F = W_gate.shape
    k = perm.dst_of_route.shape[1]
    cap = perm.rows_cap
    for name, t, dt, shp in (("dY", dY, torch.bfloat16, (T, H)), ("x_perm", x_perm, torch.bfloat16, (cap, H)),
                             ("W_gate", W_gate, torch.bfloat16, (E, H, F)), ("W_up", W_up, torch.bfloat16, (E, H, F)),
                             ("W_down", W_down, torch.bfloat16, (E, F, H)),
                             ("fc1_c", fc1_c, torch.bfloat16, (cap, 2 * F)), ("h", h, torch.bfloat16, (cap, F)),
                             ("y_perm", y_perm, torch.bfloat16, (cap, H)), ("topk_w", topk_w, torch.float32, (T, k))):
        _need(t, name, dt, shp, dev)
    out = {
        "dx": torch.empty(T, H, dtype=torch.bfloat16, device=dev),
        "dW_gate": torch.empty(E, H, F, dtype=dw_dtype, device=dev),
        "dW_up": torch.empty(E, H, F, dtype=dw_dtype, device=dev),
        "dW_down": torch.empty(E, F, H, dtype=dw_dtype, device=dev),
        "d_topk_w": torch.empty(T, k, dtype=torch.float32, device=dev) if want_d_topk_w else None,
    }
    dy_perm = torch.empty(cap, H, dtype=torch.bfloat16, device=dev)
    dgu = torch.empty(cap, 2 * F, dtype=torch.bfloat16, device=dev)
    dx_perm = torch.empty(cap, H, dtype=torch.float32, device=dev)
    fn = "moe_grouped_ffn_bwd_bf16" if dw_dtype == torch.bfloat16 else "moe_grouped_ffn_bwd"
    _check(fn, getattr(load_library(), fn)(
        _ptr(dY), _ptr(x_perm), _ptr(W_gate), _ptr(W_up), _ptr(W_down), _ptr(fc1_c), _ptr(h), _ptr(y_perm),
        _ptr(perm.dst_of_route), _ptr(perm.group_sizes), _ptr(perm.group_offsets), _ptr(topk_w),
        T, H, F, E, k, cap, _ptr(dy_perm), _ptr(dgu), _ptr(dx_perm), _ptr(out["dx"]), _ptr(out["dW_gate"]),
        _ptr(out["dW_up"]), _ptr(out["dW_down"]), _ptr(out["d_topk_w"]), _ptr(ws.buf), ws.nbytes, _stream(stream)))
    return out


# ------------------------------------------------------------------ A6 + A7 MXFP8

def mx_tile_scale_bytes(rows_cap: int, E: int, K: int) -> int:
    return int(load_library().moe_mx_tile_scale_bytes(rows_cap, E, K))


def moe_grouped_quantize_mxfp8(x: torch.Tensor, group_offsets=None, ws: Workspace | None = None,
                               rowmajor: bool = True, tiles: bool = False, stream=None):
    """MXFP8 of each row of a bf16 [rows, K] matrix along K (moe.h).  Returns
    (data uint8 [rows, K], row-major scales [rows, K/32] or None, tile-layout
    scales or None)."""
    _need(x, "x", torch.bfloat16)
    rows, K = x.shape
    dev = x.device
    data = torch.empty(rows, K, dtype=torch.uint8, device=dev)
    srm = torch.empty(rows, K // 32, dtype=torch.uint8, device=dev) if rowmajor else None
    stl = None
    G = 0
    if tiles:
        G = group_offsets.shape[0] - 1
        stl = torch.zeros(mx_tile_scale_bytes(rows, G, K), dtype=torch.uint8, device=dev)
    _check("moe_grouped_quantize_mxfp8", load_library().moe_grouped_quantize_mxfp8(
        _ptr(x), rows, K, _ptr(group_offsets), G, _ptr(data), _ptr(srm), _ptr(stl),
        _ptr(ws.buf) if ws is not None else None, ws.nbytes if ws is not None else 0, _stream(stream)))
    return data, srm, stl


def moe_quantize_weights_mxfp8(W: torch.Tensor, stream=None):
    """MXFP8 of expert weights [E, K, N] along K -> (codes, scales), both uint8
    flat arrays in the MMA tile layout (moe.h): codes in 16 KB pre-swizzled
    blocks of 128 rows n x 128 K bytes, scales in 512-byte atoms, both ordered
    [E][K/128][N/128]."""
    _need(W, "W", torch.bfloat16)
    E, K, N = W.shape
    data = torch.empty(E * N * K, dtype=torch.uint8, device=W.device)
    scales = torch.empty(E * K * N // 32, dtype=torch.uint8, device=W.device)
    _check("moe_quantize_weights_mxfp8", load_library().moe_quantize_weights_mxfp8(
        _ptr(W), E, K, N, _ptr(data), _ptr(scales), _stream(stream)))
    return data, scales


@dataclass
class PermutationMX:
    x_q: torch.Tensor           # [rows_cap, H] uint8 (E4M3)
    x_sf: torch.Tensor          # tile-layout scales, uint8
    dst_of_route: torch.Tensor
    src_of_row: torch.Tensor
    group_sizes: torch.Tensor
    group_offsets: torch.Tensor
    rows_cap: int


def moe_permute_mxfp8(x: torch.Tensor, topk_idx: torch.Tensor, E: int, ws: Workspace,
                      out: PermutationMX | None = None, stream=None) -> PermutationMX:
    """Permutation with the rows quantised to MXFP8 on the way (moe.h)."""
    _need(x, "x", torch.bfloat16)
    T, H = x.shape
    k = topk_idx.shape[1]
    cap = T * k
    if out is None:
        dev = x.device
        out = PermutationMX(
            x_q=torch.empty(cap, H, dtype=torch.uint8, device=dev),
            x_sf=torch.zeros(mx_tile_scale_bytes(cap, E, H), dtype=torch.uint8, device=dev),
            dst_of_route=torch.empty(T, k, dtype=torch.int32, device=dev),
            src_of_row=torch.empty(cap, dtype=torch.int32, device=dev),
            group_sizes=torch.empty(E, dtype=torch.int32, device=dev),
            group_offsets=torch.empty(E + 1, dtype=torch.int32, device=dev), rows_cap=cap)
    _check("moe_permute_mxfp8", load_library().moe_permute_mxfp8(
        _ptr(x), _ptr(topk_idx), T, H, E, k, _ptr(out.x_q), _ptr(out.x_sf), out.rows_cap, _ptr(out.dst_of_route),
        _ptr(out.src_of_row), _ptr(out.group_sizes), _ptr(out.group_offsets), _ptr(ws.buf), ws.nbytes,
        _stream(stream)))
    return out


def moe_grouped_fc1_swiglu_mxfp8(x_q, x_sf, Wg_q, Wg_sf, Wu_q, Wu_sf, group_offsets, ws: Workspace, h_q, h_sf,
                                 fc1_c=None, stream=None, clamp=None):
    """A3 on MXFP8 operands; h quantised to MXFP8 along F (moe.h).  fc1_c (bf16
    [rows_cap, 2F], optional): the g | u stash for the backward.  clamp = (gate_lo,
    gate_hi, up_lo, up_hi): the SwiGLU inputs clamped to those inclusive bounds."""
    rows_cap, H = x_q.shape
    E = group_offsets.shape[0] - 1
    F = h_q.shape[1]
    if fc1_c is not None:
        _need(fc1_c, "fc1_c", torch.bfloat16, (rows_cap, 2 * F))
    if clamp is not None:
        _check("moe_grouped_fc1_swiglu_mxfp8_clamped", load_library().moe_grouped_fc1_swiglu_mxfp8_clamped(
            _ptr(x_q), _ptr(x_sf), _ptr(Wg_q), _ptr(Wg_sf), _ptr(Wu_q), _ptr(Wu_sf), _ptr(group_offsets), E, H, F,
            rows_cap, *[float(v) for v in clamp], _ptr(h_q), _ptr(h_sf), _ptr(fc1_c), _ptr(ws.buf), ws.nbytes,
            _stream(stream)))
        return
    _check("moe_grouped_fc1_swiglu_mxfp8", load_library().moe_grouped_fc1_swiglu_mxfp8(
        _ptr(x_q), _ptr(x_sf), _ptr(Wg_q), _ptr(Wg_sf), _ptr(Wu_q), _ptr(Wu_sf), _ptr(group_offsets), E, H, F,
        rows_cap, _ptr(h_q), _ptr(h_sf), _ptr(fc1_c), _ptr(ws.buf), ws.nbytes, _stream(stream)))


def moe_grouped_fc2_mxfp8(h_q, h_sf, Wd_q, Wd_sf, group_offsets, ws: Workspace, y_perm, stream=None):
    """A4 on MXFP8 operands, y_perm bf16 (moe.h)."""
    rows_cap, F = h_q.shape
    E = group_offsets.shape[0] - 1
    _need(y_perm, "y_perm", torch.bfloat16, None, h_q.device)
    H = y_perm.shape[1]
    _check("moe_grouped_fc2_mxfp8", load_library().moe_grouped_fc2_mxfp8(
        _ptr(h_q), _ptr(h_sf), _ptr(Wd_q), _ptr(Wd_sf), _ptr(group_offsets), E, H, F, rows_cap, _ptr(y_perm),
        _ptr(ws.buf), ws.nbytes, _stream(stream)))


# ------------------------------------------------------------------ A8 on the MXFP8 path

def moe_dequantize_rows_mxfp8(codes: torch.Tensor, tile_scales: torch.Tensor, group_offsets: torch.Tensor,
                              ws: Workspace, out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """MXFP8 rows (codes uint8 [rows, K], tile-layout scales of the groups in
    group_offsets) -> bf16 [rows, K], for the straight-through backward (moe.h)."""
    _need(codes, "codes", torch.uint8)
    _need(tile_scales, "tile_scales", torch.uint8)
    _need(group_offsets, "group_offsets", torch.int32)
    rows, K = codes.shape
    G = group_offsets.shape[0] - 1
    if out is None:
        out = torch.empty(rows, K, dtype=torch.bfloat16, device=codes.device)
    _need(out, "out", torch.bfloat16, (rows, K))
    _check("moe_dequantize_rows_mxfp8", load_library().moe_dequantize_rows_mxfp8(
        _ptr(codes), _ptr(tile_scales), _ptr(group_offsets), G, rows, K, _ptr(out), _ptr(ws.buf), ws.nbytes,
        _stream(stream)))
    return out


def moe_dequantize_weights_mxfp8(data: torch.Tensor, scales: torch.Tensor, E: int, K: int, N: int,
                                 out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Tiled MXFP8 expert weights (moe_quantize_weights_mxfp8) -> bf16 [E, K, N] (moe.h)."""
    _need(data, "data", torch.uint8)
    _need(scales, "scales", torch.uint8)
    if data.numel() != E * K * N or scales.numel() != E * K * N // 32:
        raise ValueError("data / scales do not match E, K, N")
    if out is None:
        out = torch.empty(E, K, N, dtype=torch.bfloat16, device=data.device)
    _need(out, "out", torch.bfloat16, (E, K, N))
    _check("moe_dequantize_weights_mxfp8", load_library().moe_dequantize_weights_mxfp8(
        _ptr(data), _ptr(scales), E, K, N, _ptr(out), _stream(stream)))
    return out


def moe_unpermute_combine_mxfp8(y_perm: torch.Tensor, dst_of_route: torch.Tensor, topk_w, out_q=None, out_sf=None,
                                stream=None):
    """The combine with an MXFP8 output (moe.h): (codes uint8 [T, H], scales uint8 [T, H/32])."""
    _need(y_perm, "y_perm", torch.bfloat16)
    _need(dst_of_route, "dst_of_route", torch.int32)
    T, k = dst_of_route.shape
    H = y_perm.shape[1]
    if topk_w is not None:
        _need(topk_w, "topk_w", torch.float32, (T, k))
    if out_q is None:
        out_q = torch.empty(T, H, dtype=torch.uint8, device=y_perm.device)
    if out_sf is None:
        out_sf = torch.empty(T, H // 32, dtype=torch.uint8, device=y_perm.device)
    _need(out_q, "out_q", torch.uint8, (T, H))
    _need(out_sf, "out_sf", torch.uint8, (T, H // 32))
    _check("moe_unpermute_combine_mxfp8", load_library().moe_unpermute_combine_mxfp8(
        _ptr(y_perm), _ptr(dst_of_route), _ptr(topk_w), T, H, k, _ptr(out_q), _ptr(out_sf), _stream(stream)))
    return out_q, out_sf


def moe_unpermute_combine_nvfp4(y_perm: torch.Tensor, dst_of_route: torch.Tensor, topk_w, out_q=None, out_sf=None,
                                stream=None):
    """The combine with an NVFP4 output (moe.h): (codes uint8 [T, H/2], two E2M1 codes per
    byte; scales uint8 [T, H/16], E4M3)."""
    _need(y_perm, "y_perm", torch.bfloat16)
    _need(dst_of_route, "dst_of_route", torch.int32)
    T, k = dst_of_route.shape
    H = y_perm.shape[1]
    if topk_w is not None:
        _need(topk_w, "topk_w", torch.float32, (T, k))
    if out_q is None:
        out_q = torch.empty(T, H // 2, dtype=torch.uint8, device=y_perm.device)
    if out_sf is None:
        out_sf = torch.empty(T, H // 16, dtype=torch.uint8, device=y_perm.device)
    _need(out_q, "out_q", torch.uint8, (T, H // 2))
    _need(out_sf, "out_sf", torch.uint8, (T, H // 16))
    _check("moe_unpermute_combine_nvfp4", load_library().moe_unpermute_combine_nvfp4(
        _ptr(y_perm), _ptr(dst_of_route), _ptr(topk_w), T, H, k, _ptr(out_q), _ptr(out_sf), _stream(stream)))
    return out_q, out_sf
