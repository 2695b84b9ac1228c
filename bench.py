"""Benchmark of the single-GPU MoE FFN hot path on GB300.

A step is one pass of the whole hot path over one batch of seeded synthetic
inputs resident in HBM:
  bf16 forward   route -> permute -> grouped FC1+SwiGLU -> grouped FC2 -> combine
  mixtral        the forward, then the backward (combine bwd, router bwd to the
                 logits, FC2 dgrad + dSwiGLU, FC1 dgrad, grouped wgrad, unpermute-sum)
  dsv3_mxfp8     route -> quantising permute -> block-scaled FC1 (h to MXFP8) ->
                 block-scaled FC2 -> combine; weights quantised once, untimed
Variants: --router sigmoid (sigmoid scores + a seeded expert routing bias);
--weight-at fc1|fc2 (the router weight applied in the FC1 / FC2 epilogue);
--backward (forward + backward; on dsv3_mxfp8 the straight-through backward:
MXFP8 rows dequantised, then the bf16 backward kernels on the values the
forward's MMAs consumed, weights dequantised once with the quantisation).
Default workload: mixtral forward + backward (T=8192, H=4096, F=14336, E=8, top-2), the
largest workload that fits one GPU and the one the tensor-core target is stated on.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME]
    python bench.py --impl reference ...   # the CPU oracle, timed on the host cores

Prints one JSON line (rank 0).  Under torchrun each rank runs an independent
replica of the workload on its own GPU (the path needs no collective); the
reported time is the max over ranks and `value` counts all ranks' tokens.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE layer tokens/s & grouped-GEMM TFLOP/s (% of GB300 peak); permute/combine GB/s"
UNIT = "tokens/s"
L2_FLUSH_BYTES = 256 << 20
FP8_OVER_BF16 = 2.0   # nominal dense fp8 / bf16 tensor rate (4.5 / 2.25 PFLOP/s)
# Dense MXFP8 (E4M3, UE8M0 per 32 along K) rate of the library block-scaled GEMM on this
# pool's GB300, measured by `python bench.py --measure-peaks` (torch._scaled_mm, 8192^3):
# 2847 TFLOP/s best single launch, 3254 TFLOP/s back to back for ~3 s (bf16 torch.matmul
# in the same run: 1913 / 1686).  The larger of the two is the denominator.
MEASURED_MXFP8_TFLOPS = 3254.0

# DRAM traffic (read + write bytes per launch) of a workload's dominant kernel from one
# ncu capture (profiles/), with a hash of the kernel sources it was taken on.  Reported as
# null once those sources change.
PROFILED_TRAFFIC = {
    ("fine_grained", "fc1_swiglu"): (904.0e6, "551f7a1898737b1d"),
    # captured at F = 2048 (both launches: 1200.0 MB) and scaled to F = 14336: reads by each
    # launch's measured/operand-byte ratio, writes = fp32 gradient bytes less the measured
    # L2-resident residue
    ("mixtral", "wgrad"): (7286.8e6, "551f7a1898737b1d"),
}
KERNEL_SOURCES = ["common.cuh", "sm100.cuh", "grouped_gemm.cuh", "grouped_gemm_pair.cuh", "gemm_launch.cuh", "tmap.cuh",
                  "ffn_fwd.cu", "ffn_bwd.cu"]


def kernel_source_hash() -> str:
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "mixture_experts_ffn_warp_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str, kernel: str):
    t = PROFILED_TRAFFIC.get((workload, kernel))
    if t is None or t[1] != kernel_source_hash():
        return None
    return t[0]


def measure_library_peaks(dev) -> dict:
    """Dense rates of the library GEMMs on this GPU, as timing comparators for the
    roofline's denominators: torch.matmul bf16 and torch._scaled_mm MXFP8 (E4M3 operands,
    UE8M0 scales per 32 elements along K), both 8192^3.  Burst = best of 10 single
    launches; sustained = back to back for about 3 s.  Only the timings are used."""
    import torch
    n = 8192
    flop = 2.0 * n ** 3

    def rate(fn):
        for _ in range(3):
            fn()
        torch.cuda.synchronize(dev)
        best = float("inf")
        for _ in range(10):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            torch.cuda.synchronize(dev)
            best = min(best, a.elapsed_time(b))
        reps = max(1, int(3000.0 / best))
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(reps):
            fn()
        b.record()
        torch.cuda.synchronize(dev)
        return flop / (best * 1e-3) / 1e12, flop * reps / (a.elapsed_time(b) * 1e-3) / 1e12

    out = {"how": "8192^3; burst: best of 10 launches; sustained: back to back for ~3 s; CUDA events"}
    x = torch.randn(n, n, device=dev, dtype=torch.bfloat16)
    y = torch.randn(n, n, device=dev, dtype=torch.bfloat16)
    out["bf16_tflops"], out["bf16_tflops_sustained"] = rate(lambda: torch.matmul(x, y))
    try:
        a8 = torch.randn(n, n, device=dev).to(torch.float8_e4m3fn)
        b8 = torch.randn(n, n, device=dev).to(torch.float8_e4m3fn).t()     # column-major [K, N]
        rows = (n + 127) // 128 * 128
        cols = ((n // 32) + 3) // 4 * 4
        sa = torch.ones(rows, cols, device=dev).to(torch.float8_e8m0fnu)
        sb = torch.ones(rows, cols, device=dev).to(torch.float8_e8m0fnu)
        fn = lambda: torch._scaled_mm(a8, b8, sa, sb, out_dtype=torch.bfloat16)  # noqa: E731
        out["mxfp8_tflops"], out["mxfp8_tflops_sustained"] = rate(fn)
        out["mxfp8_call"] = "torch._scaled_mm(E4M3 [M,K], E4M3 [K,N] column-major, UE8M0 scales, bf16 out)"
    except Exception as e:   # the library block-scaled GEMM is not available here
        out["mxfp8_unavailable"] = f"{type(e).__name__}: {e}"[:300]
    return out


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


# ------------------------------------------------------------------ distributed plumbing

def dist_env():
    return (int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")),
            int(os.environ.get("LOCAL_RANK", "0")))


def init_dist(backend: str):
    import torch.distributed as dist
    ws, rank, _ = dist_env()
    if ws > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend, rank=rank, world_size=ws)
    return ws, rank


def max_over_ranks(value: float, device=None) -> float:
    """Max of a float over all ranks (identity without a process group)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(device=None):
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        if device is not None and device.type == "cuda":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons, started before the
    warm-up and stopped after the timed steps."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")
    NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "20"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, FileNotFoundError):
            self.proc = None
        t0 = time.time()
        while self.proc is not None and not self.lines and time.time() - t0 < 3.0:
            time.sleep(0.01)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, mx, power, reasons = [], [], [], set()
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for n, v in zip(self.NAMES, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "power_w_max": max(power) if power else None, "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ workloads

class Group:
    """One timed kernel group of a step: its launches and its algorithmic work."""

    def __init__(self, name, run, flop=0.0, nbytes=0.0, launches=1, fp8=False):
        self.name, self.run, self.flop, self.nbytes, self.launches, self.fp8 = name, run, flop, nbytes, launches, fp8


def group_align(shape, requested=None) -> int:
    """Rows each expert's group is padded to (with zero rows) in the permutation.  The bf16
    forward + backward pads to 16, so that every expert's rows are whole 16-row K slices of
    the weight-gradient GEMM (no zero-padded tail slice to build per expert); the padding rows
    carry zeros through every GEMM and change no result."""
    if requested is not None:
        return requested
    return 16 if (shape.backward and not shape.mxfp8) else 1


def build_workload(shape, dev, stream, align=1, dw_bf16=False):
    """Inputs, pre-allocated layer objects and the step's kernel groups."""
    import torch
    from mixture_experts_ffn_warp_gb300 import MoeBackward, MoeBackwardMX, MoeForward, MoeForwardMX, MxWeights
    from mixture_experts_ffn_warp_gb300.synthetic import make_inputs

    T, H, F, E, k = shape.T, shape.H, shape.F, shape.E, shape.k
    R = T * k
    sigmoid = shape.router == "sigmoid"
    dw_dtype = torch.bfloat16 if dw_bf16 else torch.float32
    inp = make_inputs(shape, device=dev, with_dy=shape.backward, with_expert_bias=sigmoid)
    w = {"inp": inp, "shape": shape}
    if shape.mxfp8:
        mw = MxWeights(inp["W_gate"], inp["W_up"], inp["W_down"], stream)
        w["make_layer"] = lambda: MoeForwardMX(T, H, F, E, k, device=dev, router=shape.router,  # noqa: E731
                                               expert_bias=inp.get("expert_bias"), keep_fc1_c=shape.backward)
        w["make_bwd"] = lambda f: MoeBackwardMX(f, want_d_logits=True, dw_dtype=dw_dtype)  # noqa: E731
        m = w["make_layer"]()
        w.update(layer=m, mw=mw)
        m(inp["x"], inp["logits"], mw, stream)
        if shape.backward:
            # the backward's weights: the bf16 values of the MXFP8 codes, prepared once
            # with the quantisation (untimed)
            w["bwd"] = w["make_bwd"](m)
            w["bwd_weights"] = mw.dequantized(stream)
    else:
        w["make_layer"] = lambda: MoeForward(T, H, F, E, k, device=dev, align=align,  # noqa: E731
                                             keep_fc1_c=shape.backward,
                                             router="sigmoid" if sigmoid else "softmax",
                                             expert_bias=inp.get("expert_bias"), weight_at=shape.weight_at)
        w["make_bwd"] = lambda f: MoeBackward(f, want_d_logits=True, dw_dtype=dw_dtype)  # noqa: E731
        m = w["make_layer"]()
        w.update(layer=m)
        m(inp["x"], inp["logits"], inp["W_gate"], inp["W_up"], inp["W_down"], stream)
        if shape.backward:
            w["bwd"] = w["make_bwd"](m)
    torch.cuda.synchronize(dev)
    active = int((m.perm.group_sizes > 0).sum().item())     # experts whose weights are read
    w["active_experts"] = active
    wbytes = active * H * F * (1 if shape.mxfp8 else 2) * (1 + (1 / 32 if shape.mxfp8 else 0))
    ysz = m.y_perm.element_size()   # bf16 expert outputs

    g = [Group("route", lambda: m.route(inp["logits"], stream), nbytes=T * E * 4 + R * 8)]
    if shape.mxfp8:
        mw = w["mw"]
        g += [
            Group("permute_mxfp8", lambda: m.permute(inp["x"], stream),
                  nbytes=T * H * 2 + R * H * (1 + 1 / 32) + R * 8, launches=2),
            Group("fc1_swiglu_mxfp8", lambda: m.fc1(mw, stream), flop=4.0 * R * H * F,
                  nbytes=R * H * (1 + 1 / 32) + 2 * wbytes + R * F * (1 + 1 / 32)
                  + (R * 2 * F * 2 if shape.backward else 0), fp8=True),
            Group("fc2_mxfp8", lambda: m.fc2(mw, stream), flop=2.0 * R * H * F,
                  nbytes=R * F * (1 + 1 / 32) + wbytes + R * H * ysz, fp8=True),
        ]
    else:
        stash = R * 2 * F * 2 if shape.backward else 0
        g += [
            Group("permute", lambda: m.permute(inp["x"], stream), nbytes=T * H * 2 + R * H * 2 + R * 8,
                  launches=2),
            Group("fc1_swiglu", lambda: m.fc1(inp["W_gate"], inp["W_up"], stream), flop=4.0 * R * H * F,
                  nbytes=R * H * 2 + 2 * wbytes + R * F * 2 + stash),
            Group("fc2", lambda: m.fc2(inp["W_down"], stream), flop=2.0 * R * H * F,
                  nbytes=R * F * 2 + wbytes + R * H * ysz),
        ]
    g.append(Group("combine", lambda: m.combine(stream), nbytes=R * H * ysz + T * H * 2 + R * 8))
    if shape.backward:
        b = w["bwd"]
        # the backward's weights: bf16 (on the MXFP8 path the values of the MXFP8 codes)
        Wg_b, Wu_b, Wd_b = w.get("bwd_weights") or (inp["W_gate"], inp["W_up"], inp["W_down"])
        wb16 = active * H * F * 2
        if shape.mxfp8:
            g.append(Group("dequant_mx", lambda: b.dequantize(stream),
                           nbytes=R * (H + F) * (1 + 1 / 32) + R * (H + F) * 2, launches=4))
        g += [
            Group("combine_bwd", lambda: b.combine_bwd(inp["dY"], stream),
                  nbytes=T * H * 2 + R * H * ysz + R * H * 2 + R * 8),
            Group("route_bwd", lambda: b.router_bwd(inp["logits"], stream), nbytes=R * 4 + R * 8 + T * E * 4),
            Group("dgrad_fc2_dswiglu", lambda: b.dgrad_fc2(Wd_b, stream), flop=2.0 * R * H * F,
                  nbytes=R * H * 2 + wb16 + R * 2 * F * 2 * 2),
            Group("dgrad_fc1", lambda: b.dgrad_fc1(Wg_b, Wu_b, stream), flop=4.0 * R * H * F,
                  nbytes=R * 2 * F * 2 + 2 * wb16 + R * H * 4),
            Group("wgrad", lambda: b.wgrad(stream), flop=6.0 * R * H * F,
                  nbytes=R * (F + H + H + 2 * F) * 2 + 3 * E * H * F * (2 if dw_bf16 else 4), launches=2),
            Group("unpermute_sum", lambda: b.unpermute_sum(stream), nbytes=R * H * 4 + T * H * 2 + R * 8),
        ]
    w["groups"] = g
    return w


def e2e_pipeline(w, flush=None):
    """The public HostPipeline over two slots of the workload's layer (slot 0 is the
    layer the device-resident steps use): pinned host inputs are copied in, the
    step runs, and its result (and for a backward workload dx) is copied back, the
    copies of neighbouring steps overlapping compute.  flush (a device buffer) is
    rewritten inside every step's compute when the step's weights would fit in the
    L2.  Returns (pipeline, host inputs, host outputs, H2D bytes, D2H bytes)."""
    import torch
    from mixture_experts_ffn_warp_gb300 import HostPipeline
    inp, shape = w["inp"], w["shape"]
    layers = [w["layer"], w["make_layer"]()]
    bwds = [w["bwd"], w["make_bwd"](layers[1])] if shape.backward else None
    names = ["x", "logits"] + (["dY"] if shape.backward else [])
    slots = [{n: torch.empty_like(inp[n]) for n in names} for _ in layers]
    weights = w.get("mw")

    def run(bi, s):
        if flush is not None:
            flush.fill_(1.0)
        d, m = slots[bi], layers[bi]
        if shape.mxfp8:
            m(d["x"], d["logits"], weights, s)
        else:
            m(d["x"], d["logits"], inp["W_gate"], inp["W_up"], inp["W_down"], s)
        if shape.backward:
            if shape.mxfp8:
                bwds[bi](d["dY"], weights, s, logits=d["logits"])
            else:
                bwds[bi](d["dY"], inp["W_gate"], inp["W_up"], inp["W_down"], s, logits=d["logits"])

    def outputs(bi):
        return [layers[bi].out] + ([bwds[bi].dx] if shape.backward else [])

    pipe = HostPipeline(slots, run, outputs)
    host_in = {n: inp[n].cpu().pin_memory() for n in names}
    host_out = [torch.empty(shape.T, shape.H, dtype=torch.bfloat16).pin_memory() for _ in outputs(0)]
    h2d = sum(t.numel() * t.element_size() for t in host_in.values())
    d2h = sum(t.numel() * t.element_size() for t in host_out)
    return pipe, host_in, host_out, h2d, d2h


# ------------------------------------------------------------------ CPU oracle

def oracle_sample(shape, inp_dev, n_tokens: int, it: int = 0):
    """Run the oracle on a sample of n_tokens tokens of the workload (routing and
    permutation over all tokens; the expert FFN -- and for mixtral the backward,
    for dsv3_mxfp8 the MXFP8 arithmetic -- on the sampled tokens).  Weights of
    the experts the sample touches are copied to the host (and, for MXFP8,
    quantised by the oracle) before the clock starts.  Returns (seconds, tokens)."""
    import numpy as np
    import oracle
    T, k = shape.T, shape.k
    lg = inp_dev["logits"].cpu().numpy()
    bias = inp_dev["expert_bias"].cpu().numpy() if shape.router == "sigmoid" else None

    def route():
        return oracle.route_topk_sigmoid(lg, k, bias) if bias is not None else oracle.route_topk(lg, k)

    idx_all, w_all = route()
    toks = (np.arange(n_tokens) * max(1, T // n_tokens) + it) % T
    experts = np.unique(idx_all[toks])
    x_rows = oracle.bf16_bits(inp_dev["x"].index_select(0, _long(inp_dev, toks)))
    wts = {n: {int(e): oracle.bf16_bits(inp_dev[n][int(e)]) for e in experts} for n in ("W_gate", "W_up", "W_down")}
    idx_s, w_s = idx_all[toks], w_all[toks]
    if shape.mxfp8:
        q = {n: {} for n in ("gq", "gs", "uq", "us", "dq", "ds")}
        for e in experts:
            e = int(e)
            q["gq"][e], q["gs"][e] = oracle.quantize_cols_mxfp8(wts["W_gate"][e])
            q["uq"][e], q["us"][e] = oracle.quantize_cols_mxfp8(wts["W_up"][e])
            q["dq"][e], q["ds"][e] = oracle.quantize_cols_mxfp8(wts["W_down"][e])
        if shape.backward:   # the backward's operands: the weights' MXFP8 round trips
            rt = {n: {int(e): oracle.mx_roundtrip_cols(wts[n][int(e)]) for e in experts}
                  for n in ("W_gate", "W_up", "W_down")}
    dy_rows = oracle.bf16_bits(inp_dev["dY"].index_select(0, _long(inp_dev, toks))) if shape.backward else None
    t0 = time.perf_counter()
    idx, w = route()
    oracle.permute(idx, shape.E)
    if shape.mxfp8:
        oracle.moe_fwd_mxfp8(x_rows, q["gq"], q["gs"], q["uq"], q["us"], q["dq"], q["ds"], idx_s, w_s)
        if shape.backward:   # straight-through backward on the round-tripped operands
            g = oracle.moe_bwd(oracle.mx_roundtrip_rows(x_rows), _dense(rt["W_gate"], shape.E),
                               _dense(rt["W_up"], shape.E), _dense(rt["W_down"], shape.E), idx_s, w_s, dy_rows,
                               h_mx=True)
            oracle.route_topk_bwd(lg[toks], idx_s, g["d_topk_w"].astype("float32"),
                                  oracle.SCORE_SIGMOID if bias is not None else oracle.SCORE_SOFTMAX)
    else:
        oracle.moe_fwd(x_rows, wts["W_gate"], wts["W_up"], wts["W_down"], idx_s, w_s,
                       weight_at={"combine": 0, "fc1": 1, "fc2": 2}[shape.weight_at])
        if shape.backward:
            g = oracle.moe_bwd(x_rows, _dense(wts["W_gate"], shape.E), _dense(wts["W_up"], shape.E),
                               _dense(wts["W_down"], shape.E), idx_s, w_s, dy_rows)
            oracle.route_topk_bwd(lg[toks], idx_s, g["d_topk_w"].astype("float32"),
                                  oracle.SCORE_SIGMOID if bias is not None else oracle.SCORE_SOFTMAX)
    return time.perf_counter() - t0, n_tokens


def _long(inp_dev, toks):
    import torch
    return torch.from_numpy(toks.astype("int64")).to(inp_dev["x"].device)


def _dense(d: dict, E: int):
    """Per-expert dict -> list; experts the sample does not route to get a zero
    placeholder (never read by the oracle)."""
    import numpy as np
    zero = np.zeros_like(next(iter(d.values())))
    return [d[e] if e in d else zero for e in range(E)]


def cpu_baseline(shape, inp_dev, target_s: float):
    """The oracle as it stands on the host cores, on a bounded token sample."""
    import oracle
    n = 2 if (shape.backward or shape.mxfp8) else 8
    spent, done = 0.0, 0
    while spent < target_s and done < shape.T:
        n = min(n, shape.T - done)
        dt, m = oracle_sample(shape, inp_dev, n, it=done)
        spent += dt
        done += m
        if spent < target_s:
            n = max(1, min(4 * n, int(m * (target_s - spent) / max(dt, 1e-3))))
    return {"value": done / spent, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"{done} of {shape.T} tokens in {spent:.1f} s: routing + permutation over all tokens, "
                      f"the per-token fp64 oracle ({_pass_name(shape)}) on the sample"}


def _pass_name(shape) -> str:
    return ("MXFP8 " if shape.mxfp8 else "") + ("forward + backward" if shape.backward else "forward")


# ------------------------------------------------------------------ arms

def workload_shape(args):
    """The named workload, with sizes overridden by --shape (a smaller case of the
    same kernels, e.g. for profiling)."""
    import dataclasses
    from mixture_experts_ffn_warp_gb300.synthetic import CONFIGS
    shape = CONFIGS[args.config]
    if args.shape:
        kw = {kv.split("=")[0].strip(): int(kv.split("=")[1]) for kv in args.shape.split(",") if kv.strip()}
        shape = dataclasses.replace(shape, name=shape.name + "_" + "_".join(f"{a}{b}" for a, b in kw.items()), **kw)
    if args.router != "softmax":
        shape = dataclasses.replace(shape, name=shape.name + "_" + args.router, router=args.router)
    if args.weight_at != "combine":
        if shape.backward or shape.mxfp8:
            raise SystemExit("--weight-at fc1/fc2 applies to the bf16 forward workloads")
        shape = dataclasses.replace(shape, name=shape.name + "_w" + args.weight_at, weight_at=args.weight_at)
    if args.backward and not shape.backward:
        shape = dataclasses.replace(shape, name=shape.name + "_fwdbwd", backward=True)
    return shape


def workload_config(shape, active_experts: int) -> dict:
    """The `config` object of the JSON line, the same for both arms."""
    return {"workload": shape.name, "T": shape.T, "H": shape.H, "F": shape.F, "E": shape.E, "k": shape.k,
            "router": shape.router, "weight_at": shape.weight_at,
            "pass": ("MXFP8 " if shape.mxfp8 else "") + ("forward+backward" if shape.backward else "forward"),
            "active_experts": active_experts,
            "l2": "GPU arm: L2 flushed between timed steps (256 MiB write outside the timed events)"}


def run_reference(args):
    """The oracle as it stands, on the host cores, a bounded token sample per step."""
    import torch
    import oracle
    from mixture_experts_ffn_warp_gb300.synthetic import CONFIGS, make_inputs
    _, rank, _ = dist_env()
    if rank != 0:
        return 0
    shape = workload_shape(args)
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    inp = make_inputs(shape, device=dev, with_dy=shape.backward, with_expert_bias=shape.router == "sigmoid")
    sample = max(1, min(shape.T, args.ref_tokens if args.ref_tokens else (2 if shape.backward or shape.mxfp8 else 16)))
    lg = inp["logits"].cpu().numpy()
    if shape.router == "sigmoid":
        idx_all, _ = oracle.route_topk_sigmoid(lg, shape.k, inp["expert_bias"].cpu().numpy())
    else:
        idx_all, _ = oracle.route_topk(lg, shape.k)
    active = int(len(set(int(e) for e in idx_all.reshape(-1) if e >= 0)))
    times = []
    for it in range(args.warmup + args.steps):
        dt, _ = oracle_sample(shape, inp, sample, it=it)
        if it >= args.warmup:
            times.append(dt)
    ms = 1e3 * statistics.mean(times)
    value = sample / (ms / 1e3)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(shape, active),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
                         "sample": f"{sample} of {shape.T} tokens per step (routing and permutation over all tokens)"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_gpu(args):
    import torch
    from mixture_experts_ffn_warp_gb300.synthetic import CONFIGS

    if not torch.cuda.is_available():
        raise RuntimeError("bench.py needs a CUDA GPU (no CPU fallback)")
    world, rank = init_dist("nccl")
    _, _, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    shape = workload_shape(args)
    pk = peaks()
    stream = torch.cuda.Stream(device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731

    with torch.cuda.stream(stream):
        align = group_align(shape, args.align)
        w = build_workload(shape, dev, stream, align, args.wgrad_dtype == "bf16")
    groups = w["groups"]
    m = w["layer"]

    clocks = ClockSampler(local)
    clocks.start()
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            for g in groups:
                g.run()
        stream.synchronize()
        if m.ws.read_error(stream) != 0:
            raise RuntimeError("device error word set during warm-up")
        barrier(dev)
        torch.cuda.synchronize(dev)
        # the K timed steps: one event pair per step and nothing recorded between the
        # kernels, so each launch may overlap the tail of the one before it
        steps = []
        for it in range(args.steps):
            flush.fill_(float(it % 7))           # evict L2 between steps (outside the events)
            a, b = ev(), ev()
            a.record(stream)
            for g in groups:
                g.run()
            b.record(stream)
            steps.append((a, b))
        torch.cuda.synchronize(dev)
        barrier(dev)
        # breakdown (not the timed steps): the same steps with an event after each group
        marks = []
        for it in range(args.steps):
            flush.fill_(float(it % 7))
            e = [ev() for _ in range(len(groups) + 1)]
            e[0].record(stream)
            for i, g in enumerate(groups):
                g.run()
                e[i + 1].record(stream)
            marks.append(e)
        torch.cuda.synchronize(dev)
    clk = clocks.stop()
    if m.ws.read_error(stream) != 0:
        raise RuntimeError("device error word set during the timed steps")

    per = {g.name: statistics.mean(e[i].elapsed_time(e[i + 1]) for e in marks) for i, g in enumerate(groups)}
    step_ms = statistics.mean(a.elapsed_time(b) for a, b in steps)
    ms_step = max_over_ranks(step_ms, dev)

    # end to end through the public pipeline API: every step copies its inputs in from
    # pinned host memory and its result back; neighbouring steps overlap copies and compute
    weights_bytes = shape.E * 3 * shape.H * shape.F * (1 if shape.mxfp8 else 2)
    small = weights_bytes < 2 * L2_FLUSH_BYTES
    pipe, host_in, host_out, h2d, d2h = e2e_pipeline(w, flush if small else None)
    for _ in range(args.warmup):
        pipe.submit(host_in, host_out)
    torch.cuda.synchronize(dev)
    barrier(dev)
    t0, t1 = ev(), ev()
    t0.record(pipe.up)
    for _ in range(args.steps):
        pipe.submit(host_in, host_out)
    pipe.down.wait_event(pipe.ev_comp[(pipe.i - 1) % len(pipe.slots)])
    t1.record(pipe.down)
    torch.cuda.synchronize(dev)
    if m.ws.read_error(stream) != 0:
        raise RuntimeError("device error word set during the end-to-end steps")
    ms_e2e = max_over_ranks(t0.elapsed_time(t1) / args.steps, dev)

    # The library GEMM was measured twice: a burst at full clocks and a seconds-long loop
    # under the power cap.  A run whose own clocks sat under the power cap (sw_power_cap
    # active, median SM clock below 90 % of the maximum) is in the second regime.
    capped = ("sw_power_cap" in clk.get("reasons", []) and bool(clk.get("sm_mhz"))
              and clk["sm_mhz"] < 0.9 * (clk.get("sm_max_mhz") or float("inf")))
    use_sustained = capped and bool(pk.get("bf16_tflops_sustained"))

    def peak_flops(g, burst=False):
        if g.fp8:
            return MEASURED_MXFP8_TFLOPS if MEASURED_MXFP8_TFLOPS else pk["bf16_tflops"] * FP8_OVER_BF16
        return pk["bf16_tflops_sustained"] if use_sustained and not burst else pk["bf16_tflops"]

    rates = {}
    for g in groups:
        t = per[g.name] / 1e3
        r = {"ms": per[g.name], "gbs": g.nbytes / t / 1e9}
        if g.flop:
            r["tflops"] = g.flop / t / 1e12
            r["frac_tensor"] = r["tflops"] / peak_flops(g)
            if use_sustained and not g.fp8:
                r["frac_tensor_of_burst"] = r["tflops"] / peak_flops(g, burst=True)
        r["frac_hbm"] = r["gbs"] / pk["hbm_gbs"]
        rates[g.name] = r
    dom = max(groups, key=lambda g: per[g.name])
    t_dom = per[dom.name] / 1e3
    ridge = peak_flops(dom) * 1e12 / (pk["hbm_gbs"] * 1e9)
    tensor_bound = dom.flop > 0 and dom.flop / dom.nbytes >= ridge
    if tensor_bound:
        roof = {"bound": "tensor", "achieved": dom.flop / t_dom / 1e12, "peak": peak_flops(dom), "unit": "TFLOP/s",
                "peak_source": (("measured MXFP8 library GEMM rate (bench.py --measure-peaks)"
                                 if MEASURED_MXFP8_TFLOPS else f"{pk['source']} bf16 dense burst x 2 (nominal fp8/bf16)")
                                if dom.fp8 else f"{pk['source']} bf16 dense "
                                + ("sustained (this run was power-capped)" if use_sustained else "burst"))}
        if not dom.fp8:
            roof["frac_of_burst"] = roof["achieved"] / peak_flops(dom, burst=True)
    else:
        roof = {"bound": "hbm", "achieved": dom.nbytes / t_dom / 1e9, "peak": pk["hbm_gbs"], "unit": "GB/s",
                "peak_source": f"{pk['source']} HBM copy"}
    roof.update(kernel=dom.name, frac=roof["achieved"] / roof["peak"], traffic=profiled_traffic(shape.name + ("_dwbf16" if args.wgrad_dtype == "bf16" else ""), dom.name),
                algorithmic_bytes=dom.nbytes, algorithmic_flop=dom.flop)

    ffn = [g for g in groups if g.flop]
    ffn_flop = sum(g.flop for g in ffn)
    ffn_ms = sum(per[g.name] for g in ffn)
    tokens = shape.T * world
    line = {
        "metric": METRIC, "value": tokens / (ms_step / 1e3), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "mxfp8" if shape.mxfp8 else "bf16",
        "data": "synthetic (seeded; the workload's stated shapes and distributions)",
        "config": workload_config(shape, w["active_experts"]),
        "kernels": rates,
        "kernels_note": "per kernel group: a second pass of the same steps with an event after each group "
                        "(events between groups stop a launch from overlapping the previous group's tail, so "
                        "the groups sum to a little more than ms_per_step)",
        "ffn_tflops": ffn_flop / (ffn_ms / 1e3) / 1e12,
        "ffn_frac_of_peak": ffn_flop / (ffn_ms / 1e3) / 1e12 / peak_flops(ffn[0]),
        "roofline": roof,
        "clocks": clk,
        "gpu_launches": args.steps * sum(g.launches for g in groups),
        "group_align": align,
        "weight_grads": args.wgrad_dtype if shape.backward else None,
        "e2e": {"value": tokens / (ms_e2e / 1e3), "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": ms_e2e,
                "how": "HostPipeline (two slots; upload, compute and download streams): K steps from the first "
                       "upload to the last download, each step's inputs copied from pinned host memory and its "
                       "result copied back" + ("; L2 flushed inside every step" if small else
                                               "; no flush: each step streams more than the L2 in weights")},
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(shape, w["inp"], args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line), flush=True)
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--config", default="mixtral",
                    choices=["tiny", "fine_grained", "mixtral", "skewed", "dsv3_mxfp8"])
    ap.add_argument("--wgrad-dtype", default="fp32", choices=["fp32", "bf16"],
                    help="dtype the weight gradients are stored in (fp32 accumulation either way)")
    ap.add_argument("--align", type=int, default=None,
                    help="pad each expert's rows to a multiple of this (default: 16 for the bf16 "
                         "forward + backward, else 1)")
    ap.add_argument("--shape", default="",
                    help="override sizes of the workload, e.g. 'T=2048,F=4096' (same kind of pass)")
    ap.add_argument("--router", default="softmax", choices=["softmax", "sigmoid"],
                    help="score function of the routing step (sigmoid: + a seeded expert routing bias)")
    ap.add_argument("--weight-at", default="combine", choices=["combine", "fc1", "fc2"],
                    help="where the router weight is applied (bf16 forward workloads)")
    ap.add_argument("--backward", action="store_true",
                    help="time forward + backward (the MXFP8 workload: its straight-through backward)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--ref-tokens", type=int, default=0)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--measure-peaks", action="store_true",
                    help="print the library GEMMs' dense bf16 and MXFP8 rates on this GPU and exit")
    args = ap.parse_args(argv)
    if args.measure_peaks:
        import torch
        print(json.dumps(measure_library_peaks(torch.device("cuda", 0))), flush=True)
        return 0
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
