"""Host-side logic of the N > 1 path on CPU: two ranks over gloo.

Replicas only: every rank runs the whole layer on its own batch, so the
multi-rank logic is the timing reduction (the slowest replica sets the job's
time), the whole-job throughput, and the reference arm's rank handling under
torchrun (rank 0 alone runs and prints; the other ranks exit 0 without work).
"""
import importlib.util
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    import torch.distributed as dist
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    b = _bench()
    ms = b.max_over_ranks(10.0 + 5.0 * rank, world)          # rank 1 is the slow replica
    e2e = b.max_over_ranks(30.0 - 7.0 * rank, world)         # rank 0 is the slow one here
    tok = b.job_tokens_per_s(100, world, ms)
    with open(os.path.join(out_dir, f"r{rank}.json"), "w") as f:
        json.dump({"ms": ms, "e2e": e2e, "tok": tok}, f)
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_and_job_throughput_gloo(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       join=True, start_method="spawn")
    res = [json.load(open(tmp_path / f"r{r}.json")) for r in range(world)]
    for r in res:
        assert r["ms"] == 15.0                    # both ranks see the slowest replica's time
        assert r["e2e"] == 30.0
        assert r["tok"] == pytest.approx(100 * world / 15e-3)


def test_single_rank_needs_no_process_group():
    b = _bench()
    assert b.max_over_ranks(12.5, 1) == 12.5
    assert b.job_tokens_per_s(64, 1, 2.0) == pytest.approx(32000.0)


@pytest.mark.timeout(600)
def test_reference_arm_under_torchrun_prints_once():
    """The driver's launch of the reference arm for N = 2, on CPU."""
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes", "1", "--nproc-per-node",
           "2", "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl",
           "reference", "--workload", "tiny", "--gpus", "2", "--steps", "1", "--warmup", "0",
           "--cpu-budget-s", "2"]
    env = dict(os.environ, OMP_NUM_THREADS="2")
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=540, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2
    assert d["cpu_baseline"]["kind"] == "oracle" and d["value"] > 0
