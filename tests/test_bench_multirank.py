"""Host logic of bench.py's multi-rank (torchrun) mode on CPU: world size 2
over gloo.  Each rank runs an independent replica, so the only cross-rank
steps are the barriers around the timed region and the max over ranks of the
step time; the reference arm runs on rank 0 alone."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist
    ws, r = bench.init_dist("gloo")
    step_ms = [1.25, 3.5][rank]             # rank 1 is the slow one
    bench.barrier()
    worst = bench.max_over_ranks(step_ms)
    bench.barrier()
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump({"ws": ws, "rank": r, "max": worst}, f)
    dist.destroy_process_group()


def test_max_over_ranks_and_barrier_gloo_world2(tmp_path):
    port = _free_port()
    mp.start_processes(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True, start_method="spawn")
    got = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(2)]
    assert [g["rank"] for g in got] == [0, 1]
    assert all(g["ws"] == 2 for g in got)
    assert all(g["max"] == 3.5 for g in got)   # every rank sees the slowest rank's time


def test_max_over_ranks_without_process_group_is_identity():
    assert bench.max_over_ranks(2.75) == 2.75
    bench.barrier()   # no process group: a no-op


def test_reference_arm_runs_on_rank0_only(tmp_path):
    """Under torchrun the reference arm's non-zero ranks exit 0 at once, printing nothing."""
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1", MASTER_ADDR="127.0.0.1",
               MASTER_PORT=str(_free_port()))
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--steps", "1", "--warmup", "3"], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""


def test_bench_refuses_cpu_only_run():
    """The GPU arm has no CPU fallback."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    with pytest.raises(RuntimeError, match="needs a CUDA GPU"):
        bench.main(["--steps", "1", "--warmup", "3"])
