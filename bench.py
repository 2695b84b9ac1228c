"""Benchmark of the single-GPU MoE FFN forward hot path on GB300.

A step = route (A1) + permute (A2) + grouped FC1+SwiGLU (A3) + grouped FC2
(A4) + combine (A5) over one batch of seeded synthetic inputs resident in
HBM.  Default workload: fine_grained (T=4096, H=2048, F=1408, E=64, top-6).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME]
    python bench.py --impl reference ...     # the CPU oracle, timed on the host cores

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


# DRAM traffic (read + write bytes per launch) of the dominant kernel (grouped FC1 + SwiGLU),
# from one ncu capture per workload (profiles/<workload>_fwd_kernels.md), with a hash of the
# kernel sources the capture was taken on.  Reported as null once those sources change.
PROFILED_TRAFFIC = {"fine_grained": (900.8e6, "c26e88ae9aa42def")}
KERNEL_SOURCES = ["common.cuh", "sm100.cuh", "grouped_gemm.cuh", "gemm_launch.cuh", "tmap.cuh", "ffn_fwd.cu"]


def kernel_source_hash() -> str:
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "mixture_experts_ffn_warp_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str):
    t = PROFILED_TRAFFIC.get(workload)
    if t is None or t[1] != kernel_source_hash():
        return None
    return t[0]


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


# ------------------------------------------------------------------ distributed plumbing

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


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
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def wait_first(self, limit_s: float = 3.0):
        t0 = time.time()
        while self.proc is not None and not self.lines and time.time() - t0 < limit_s:
            time.sleep(0.01)

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ workload bookkeeping

def work(shape):
    """Algorithmic FLOPs and bytes of one forward step."""
    T, H, F, E, k = shape.T, shape.H, shape.F, shape.E, shape.k
    R = T * k
    return {
        "fc1_flop": 4.0 * R * H * F,
        # FC1 reads x_perm and W_gate/W_up of the experts that received routes, writes h
        "fc1_bytes": R * H * 2 + 2 * E * H * F * 2 + R * F * 2,
        "fc2_flop": 2.0 * R * H * F,
        "permute_bytes": T * H * 2 + R * H * 2 + R * 8 + E * 8,
        "combine_bytes": R * H * 4 + T * H * 2 + R * 8,   # fp32 expert outputs in, bf16 out
        "route_bytes": T * E * 4 + R * 8,
    }


# ------------------------------------------------------------------ CPU oracle baseline

def oracle_sample_rate(shape, inp_cpu, target_s: float, max_tokens: int = 4096):
    """Tokens/s of the oracle's per-token forward on a bounded sample of tokens,
    plus its routing + permutation over all tokens."""
    import numpy as np
    import oracle
    lg = inp_cpu["logits"].numpy()
    t0 = time.perf_counter()
    idx, w = oracle.route_topk(lg, shape.k)
    oracle.permute(idx, shape.E)
    t_route = time.perf_counter() - t0
    xb = oracle.bf16_bits(inp_cpu["x"])
    Wg, Wu, Wd = inp_cpu["Wg_bits"], inp_cpu["Wu_bits"], inp_cpu["Wd_bits"]
    n = 8
    spent, done = 0.0, 0
    while True:
        toks = np.arange(done, min(done + n, shape.T, max_tokens))
        if toks.size == 0:
            break
        t0 = time.perf_counter()
        oracle.moe_fwd(xb, Wg, Wu, Wd, idx, w, tokens=toks)
        spent += time.perf_counter() - t0
        done += toks.size
        if spent >= target_s or done >= min(shape.T, max_tokens):
            break
        n = min(4 * n, max(8, int(toks.size * (target_s - spent) / max(spent, 1e-3))))
    # tokens/s for the whole path: per-token FFN rate, plus routing amortised over T
    per_token = spent / done
    total = per_token * shape.T + t_route
    return shape.T / total, done, spent + t_route, oracle.num_threads()


def cpu_inputs(inp):
    import oracle
    c = {"logits": inp["logits"].cpu(), "x": inp["x"].cpu()}
    c["Wg_bits"] = oracle.bf16_bits(inp["W_gate"])
    c["Wu_bits"] = oracle.bf16_bits(inp["W_up"])
    c["Wd_bits"] = oracle.bf16_bits(inp["W_down"])
    return c


def run_reference(args):
    """The oracle as it stands, on the host cores, bounded sample per step."""
    import numpy as np
    import oracle
    from mixture_experts_ffn_warp_gb300.synthetic import CONFIGS, make_inputs
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    shape = CONFIGS[args.config]
    inp = make_inputs(shape, device="cpu")
    c = cpu_inputs(inp)
    lg = c["logits"].numpy()
    xb = oracle.bf16_bits(c["x"])
    sample = max(1, min(shape.T, args.ref_tokens))
    times = []
    for it in range(args.warmup + args.steps):
        toks = (np.arange(sample) * (shape.T // sample) + it) % shape.T
        t0 = time.perf_counter()
        idx, w = oracle.route_topk(lg, shape.k)
        oracle.permute(idx, shape.E)
        oracle.moe_fwd(xb, c["Wg_bits"], c["Wu_bits"], c["Wd_bits"], idx, w, tokens=toks)
        dt = time.perf_counter() - t0
        if it >= args.warmup:
            times.append(dt)
    ms = 1e3 * statistics.mean(times)
    value = sample / (ms / 1e3)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": shape.name, "T": shape.T, "H": shape.H, "F": shape.F, "E": shape.E,
                   "k": shape.k, "tokens_per_step": sample},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
                         "sample": f"{sample} of {shape.T} tokens per step (routing and permutation over all tokens)"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ GPU arm

def run_gpu(args):
    import torch
    from mixture_experts_ffn_warp_gb300 import MoeForward
    from mixture_experts_ffn_warp_gb300.synthetic import CONFIGS, make_inputs

    backend = "nccl" if torch.cuda.is_available() else "gloo"
    world, rank = init_dist(backend)
    _, _, local = dist_env()
    if not torch.cuda.is_available():
        raise RuntimeError("bench.py needs a CUDA GPU (no CPU fallback)")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    shape = CONFIGS[args.config]
    W = work(shape)
    peaks = _peaks()

    inp = make_inputs(shape, device=dev, with_dy=False)
    m = MoeForward(shape.T, shape.H, shape.F, shape.E, shape.k, device=dev)
    stream = torch.cuda.Stream(device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def step():
        m.route(inp["logits"], stream)
        m.permute(inp["x"], stream)
        m.fc1(inp["W_gate"], inp["W_up"], stream)
        m.fc2(inp["W_down"], stream)
        m.combine(stream)

    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    # clocks are sampled from the start of the warm-up to the end of the timed steps
    clocks = ClockSampler(local)
    clocks.start()
    clocks.wait_first()
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
        stream.synchronize()
        if m.ws.read_error(stream) != 0:
            raise RuntimeError("device error word set during warm-up")

        barrier(dev)
        torch.cuda.synchronize(dev)
        marks = []
        for it in range(args.steps):
            flush.fill_(float(it % 7))           # evict L2 between steps (outside the events)
            e = [ev() for _ in range(5)]
            e[0].record(stream)
            m.route(inp["logits"], stream)
            m.permute(inp["x"], stream)
            e[1].record(stream)
            m.fc1(inp["W_gate"], inp["W_up"], stream)
            e[2].record(stream)
            m.fc2(inp["W_down"], stream)
            e[3].record(stream)
            m.combine(stream)
            e[4].record(stream)
            marks.append(e)
        torch.cuda.synchronize(dev)
        barrier(dev)
        clk = clocks.stop()

        seg = {"route_permute": [], "fc1": [], "fc2": [], "combine": [], "step": []}
        for e in marks:
            seg["route_permute"].append(e[0].elapsed_time(e[1]))
            seg["fc1"].append(e[1].elapsed_time(e[2]))
            seg["fc2"].append(e[2].elapsed_time(e[3]))
            seg["combine"].append(e[3].elapsed_time(e[4]))
            seg["step"].append(e[0].elapsed_time(e[4]))
        ms_step = max_over_ranks(statistics.mean(seg["step"]), dev)
        mean = {k: statistics.mean(v) for k, v in seg.items()}
        if m.ws.read_error(stream) != 0:
            raise RuntimeError("device error word set during the timed steps")

        # separate route / permute split (same launches, timed apart once per step)
        rp = []
        for _ in range(max(3, args.steps // 2)):
            flush.fill_(1.0)
            e = [ev() for _ in range(3)]
            e[0].record(stream)
            m.route(inp["logits"], stream)
            e[1].record(stream)
            m.permute(inp["x"], stream)
            e[2].record(stream)
            rp.append((e[0], e[1], e[2]))
        torch.cuda.synchronize(dev)
        t_route = statistics.mean(a.elapsed_time(b) for a, b, _ in rp)
        t_perm = statistics.mean(b.elapsed_time(c) for _, b, c in rp)

        # ---------------- end to end through the public API with host buffers
        x_h = inp["x"].cpu().pin_memory()
        lg_h = inp["logits"].cpu().pin_memory()
        out_h = torch.empty(shape.T, shape.H, dtype=torch.bfloat16).pin_memory()
        x_d = torch.empty_like(inp["x"])
        lg_d = torch.empty_like(inp["logits"])
        e2e_times = []
        for it in range(args.warmup + args.steps):
            flush.fill_(2.0)
            e0, e1 = ev(), ev()
            e0.record(stream)
            x_d.copy_(x_h, non_blocking=True)
            lg_d.copy_(lg_h, non_blocking=True)
            m(x_d, lg_d, inp["W_gate"], inp["W_up"], inp["W_down"], stream=stream)
            out_h.copy_(m.out, non_blocking=True)
            e1.record(stream)
            if it >= args.warmup:
                e2e_times.append((e0, e1))
        torch.cuda.synchronize(dev)
        ms_e2e = max_over_ranks(statistics.mean(a.elapsed_time(b) for a, b in e2e_times), dev)

    tokens = shape.T * world
    value = tokens / (ms_step / 1e3)
    fc1_tflops = W["fc1_flop"] / (mean["fc1"] / 1e3) / 1e12
    ffn_tflops = (W["fc1_flop"] + W["fc2_flop"]) / ((mean["fc1"] + mean["fc2"]) / 1e3) / 1e12
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded, BASELINE shapes and distributions)",
        "config": {"workload": shape.name, "T": shape.T, "H": shape.H, "F": shape.F, "E": shape.E,
                   "k": shape.k, "l2": "flushed between steps (256 MiB write outside the timed events)"},
        "breakdown_ms": {"route": t_route, "permute": t_perm, "fc1_swiglu": mean["fc1"], "fc2": mean["fc2"],
                         "combine": mean["combine"]},
        "ffn_tflops": ffn_tflops,
        "ffn_frac_of_bf16_peak": ffn_tflops / peaks["bf16_tflops"],
        "permute_gbs": W["permute_bytes"] / (t_perm / 1e3) / 1e9,
        "combine_gbs": W["combine_bytes"] / (mean["combine"] / 1e3) / 1e9,
        "roofline": {"kernel": "grouped_gemm FC1_SWIGLU", "bound": "tensor", "achieved": fc1_tflops,
                     "peak": peaks["bf16_tflops"], "unit": "TFLOP/s", "frac": fc1_tflops / peaks["bf16_tflops"],
                     "peak_source": f"{peaks['source']} bf16 dense burst",
                     "traffic": profiled_traffic(shape.name),
                     "algorithmic_bytes": W["fc1_bytes"]},
        "clocks": clk,
        "gpu_launches": 7 * args.steps,
        "e2e": {"value": tokens / (ms_e2e / 1e3), "unit": UNIT,
                "h2d_bytes_per_step": shape.T * shape.H * 2 + shape.T * shape.E * 4,
                "d2h_bytes_per_step": shape.T * shape.H * 2},
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        c = cpu_inputs({k: v for k, v in inp.items()})
        rate, done, spent, cores = oracle_sample_rate(shape, c, args.cpu_seconds)
        line["cpu_baseline"] = {"value": rate, "unit": UNIT, "cores": cores, "kind": "oracle",
                                "sample": f"{done} of {shape.T} tokens through the per-token fp64 oracle in "
                                          f"{spent:.1f} s (routing + permutation over all tokens), scaled to T"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--config", default="fine_grained")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--ref-tokens", type=int, default=64)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args(argv)
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
