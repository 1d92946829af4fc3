"""The multi-process side of bench.py, on CPU with the gloo backend.

With N > 1 the bench runs N independent replicas (sequences shard across
ranks with no exchange) and reports the slowest rank's time with the work of
all ranks; under torchrun the reference arm runs on rank 0 only.  These
tests run world-size-2 process groups over 127.0.0.1 without a GPU."""
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


def _ranks_agree(rank, world, port, values, out):
    import torch.distributed as dist
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        out[rank] = bench.max_over_ranks(values[rank], world)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_takes_the_slowest_rank():
    port, values = _free_port(), [3.25, 7.5]
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_ranks_agree, args=(2, port, values, out), nprocs=2, join=True)
        assert dict(out) == {0: 7.5, 1: 7.5}


def test_whole_job_rate_counts_every_rank():
    # 32 tokens per rank per step on 2 ranks, slowest rank 0.5 ms per step
    assert bench.whole_job_rate(32, 2, 0.5) == pytest.approx(128000.0)
    assert bench.whole_job_rate(32, 1, 0.5) == pytest.approx(64000.0)
    assert bench.max_over_ranks(1.25, 1) == 1.25


def test_reference_arm_under_torchrun_prints_once():
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="", PYTHONPATH=ROOT)
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr=127.0.0.1", f"--master-port={_free_port()}", os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--workload", "tiny", "--gpus", "2", "--steps", "1", "--warmup", "0"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"
