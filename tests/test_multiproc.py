"""The N > 1 path of the benchmark on CPU: world-size-2 gloo ranks.

The attention path has no exchange step, so N GPUs run N independent replicas; what
crosses ranks is only the timing: the step time is the maximum over ranks and the value
counts every rank's work.  The reference arm prints from rank 0 only.
"""
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, ms, out):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    total, value = bench.aggregate(ms[rank], 1e12, 10, world)
    out[rank] = (total, value)
    dist.barrier()
    dist.destroy_process_group()


def test_aggregate_takes_the_slowest_rank():
    world = 2
    mgr = mp.Manager()
    out = mgr.dict()
    ms = [100.0, 250.0]            # rank 1 is slower
    mp.spawn(_worker, args=(world, _free_port(), ms, out), nprocs=world, join=True)
    for r in range(world):
        total, value = out[r]
        assert total == 250.0
        # 2 ranks x 10 steps x 1e12 FLOP in 0.25 s
        assert value == pytest.approx(2 * 10 * 1e12 / 0.25 / 1e12)


def test_single_rank_aggregate():
    sys.path.insert(0, ROOT)
    import bench
    total, value = bench.aggregate(50.0, 2e12, 5, 1)
    assert total == 50.0 and value == pytest.approx(5 * 2e12 / 0.05 / 1e12)


@pytest.mark.skipif(not os.path.exists("/usr/bin/python3") and not sys.executable, reason="no interpreter")
def test_reference_arm_prints_from_rank_zero_only():
    """torchrun with 2 CPU ranks: rank 0 times the oracle sample, rank 1 exits 0 silently."""
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr=127.0.0.1", f"--master-port={port}", os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0", "--workload", "tiny_causal"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    import json
    j = json.loads(lines[0])
    assert j["impl"] == "reference" and j["n_gpus"] == 2 and j["value"] > 0
    assert j["cpu_baseline"]["kind"] == "oracle"
    assert j["e2e"]["h2d_bytes_per_step"] == 0
