"""The benchmark's N > 1 host logic on CPU, without a GPU: world-size-2 gloo
process groups for the max-over-ranks timing and the whole-job value, and a
torchrun launch of the reference arm (the CPU oracle), where rank 0 alone
prints its JSON line and the other rank exits 0 without work.  Replicas need
no collective on the data path; the only one is the timing reduction."""

import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, q):
    import torch
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    t = bench.max_over_ranks(times[rank], torch.device("cpu"))
    v = bench.job_value(256, world, t)
    dist.barrier()
    dist.destroy_process_group()
    q.put((rank, t, v))


def test_max_over_ranks_and_job_value_with_gloo():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    times = [0.061, 0.075]
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, times, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, t, v in out:
        assert t == pytest.approx(0.075)                 # every rank sees the slowest
        assert v == pytest.approx(2 * 256 / 0.075e-3)    # all ranks' rows over that time


def test_single_process_needs_no_group():
    import torch
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(0.06, torch.device("cpu")) == 0.06
    assert bench.job_value(256, 1, 0.064) == pytest.approx(4.0e6)


def test_reference_arm_under_torchrun_prints_once():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py",
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"
