"""The multi-GPU path is replicas only: each rank decodes its own request and
the ranks meet only to time the job (a barrier and a max over ranks).  These
tests run that host logic as world_size-2 gloo process groups on the CPU."""
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


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, ws, port, values, out):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    dist.barrier()
    got = bench.max_over_ranks(values[rank], "cpu")
    out[rank] = got
    dist.destroy_process_group()


def test_max_over_ranks_gloo_world_size_2():
    ws, port = 2, _free_port()
    values = [12.5, 40.25]
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.start_processes(_rank_main, args=(ws, port, values, out), nprocs=ws, start_method="spawn", join=True)
        assert dict(out) == {0: 40.25, 1: 40.25}


def test_max_over_ranks_single_process():
    assert bench.max_over_ranks(3.5, "cpu") == 3.5


def test_job_throughput_is_weak_scaling_aggregate():
    # two replicas, 256 tokens each per step, the slowest taking 250 ms: 2048 tokens/s for the job
    assert bench.job_tokens_per_s(2, 256, 250.0) == pytest.approx(2048.0)
    assert bench.job_tokens_per_s(1, 256, 250.0) == pytest.approx(1024.0)


def test_reference_arm_under_torchrun_prints_once():
    """`bench.py --impl reference` launched as 2 ranks: rank 0 alone runs the
    oracle and prints one JSON line; rank 1 exits 0 without work."""
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--workload", "tiny", "--gpus", "2", "--steps", "1", "--warmup", "0"]
    env = dict(os.environ, OMP_NUM_THREADS="2")
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["n_gpus"] == 2 and rec["value"] > 0
    assert rec["cpu_baseline"]["kind"] == "oracle"
