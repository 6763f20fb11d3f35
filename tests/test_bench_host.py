"""Host logic of bench.py: strategy parsing, the replica aggregation used
under torchrun (sum of work, max of time over ranks) on two gloo ranks, and
the reference arm's JSON line. No GPU."""
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


def test_parse_strategy():
    assert bench.parse_strategy("sync") == dict(strategy="sync", depth=1, tile=(0, 0))
    assert bench.parse_strategy("etb8") == dict(strategy="etb", depth=8, tile=(0, 0))
    assert bench.parse_strategy("ba4@32x16") == dict(strategy="ba", depth=4, tile=(32, 16))
    with pytest.raises(ValueError):
        bench.parse_strategy("gs3")


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    units, secs = bench.aggregate(1000.0 * (rank + 1), 0.5 + rank)
    q.put((rank, units, secs))
    dist.destroy_process_group()


def test_aggregate_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, units, secs in out:
        assert units == 3000.0 and secs == 1.5


def test_aggregate_single_process_is_identity():
    assert bench.aggregate(7.0, 2.0) == (7.0, 2.0)


def test_reference_arm_line():
    """--impl reference times the oracle on a bounded sample and prints one
    JSON line with the contract's keys."""
    res = subprocess.run(
        [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
         "--workload", "n512_r1_point", "--steps", "1", "--warmup", "0",
         "--cpu-sample-sweeps", "16"],
        capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert res.returncode == 0, res.stderr
    line = json.loads(res.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "GLUP/s"
    assert line["value"] > 0 and line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0
