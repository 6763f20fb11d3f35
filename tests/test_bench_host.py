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


def test_headline_is_shortest_time_to_solution():
    """Block-async needs more sweeps, so its GLUP/s can exceed that of a
    strategy that reaches the solution sooner; the headline follows time."""
    results = {
        "sync": {"ms_per_solve_median": 160.0, "glups": 430.0},
        "etb8": {"ms_per_solve_median": 44.5, "glups": 1550.0},
        "ba16": {"ms_per_solve_median": 79.6, "glups": 2311.0},
    }
    assert bench.headline(results) == "etb8"


def test_kernel_names_follow_default_shapes():
    assert bench.kernel_name("etb4").startswith("k_etbr")
    assert bench.kernel_name("etb2").startswith("k_etb ")
    assert bench.kernel_name("etb8@112x48").startswith("k_etb ")
    assert bench.kernel_name("etb8@112x92").startswith("k_etbr")
    assert bench.kernel_name("etb16@96x64").startswith("k_etbr")
    assert bench.kernel_name("ba8").startswith("k_bar")
    assert bench.kernel_name("ba8@32x16").startswith("k_ba ")
    assert bench.kernel_name("ba8o4").startswith("k_ba ")


def test_persistent_token():
    kw = bench.parse_strategy("etb8p")
    assert kw["strategy"] == "etb" and kw["depth"] == 8
    assert kw["control"] == "persistent"
    assert bench.kernel_name("etb8p").startswith("k_etbp")


def test_roofline_bound_follows_l2_residency():
    """In L2 the sweep launches do not reach HBM: the record takes the FP32
    pipe as the bound (8 operations per lattice update against 128 lanes x
    SMs x clock); out of L2 it takes the measured HBM copy bandwidth with the
    algorithmic 12 B per point per launch."""
    kw = bench.parse_strategy("etb8")
    interior = 2046 ** 2
    args = (kw, interior, 0.027, 50_331_648)
    rest = (152, 6774.9, "measured", 2070.0, "measured")
    in_l2 = bench.roofline_record(*args, 132_120_576, *rest)
    assert in_l2["bound"] == "alu" and in_l2["l2_resident"]
    assert in_l2["peak"] == pytest.approx(128 * 152 * 2070e6 / 1e12)
    assert in_l2["achieved"] == pytest.approx(8 * interior * 8 / 0.027e-3 / 1e12)
    assert in_l2["frac"] == pytest.approx(in_l2["achieved"] / in_l2["peak"])
    assert in_l2["hbm"]["achieved"] == pytest.approx(12 * interior / 0.027e-3 / 1e9)
    out = bench.roofline_record(*args, 40_000_000, *rest)
    assert out["bound"] == "hbm" and out["unit"] == "GB/s"
    assert out["frac"] == pytest.approx(out["hbm"]["achieved"] / 6774.9)
    unfused = bench.roofline_record(bench.parse_strategy("syncu"), interior, 0.027,
                                    50_331_648, 40_000_000, *rest)
    assert unfused["alg_bytes_per_launch"] == 16 * interior


def test_spawned_replicas_aggregate_on_two_gloo_ranks(capfd):
    """--gpus N without a torchrun environment starts N ranks itself
    (bench.spawn_ranks); the ranks' work is summed and their time maxed."""
    rc = bench.spawn_ranks(2, [], script=os.path.join(ROOT, "tests", "replica_rank.py"))
    out = capfd.readouterr().out
    assert rc == 0, out
    lines = [json.loads(x) for x in out.splitlines() if x.startswith("{")]
    assert len(lines) == 1
    # (1e9 + 2e9) updates over max(0.5, 1.5) s
    assert lines[0]["n_gpus"] == 2 and lines[0]["value"] == pytest.approx(2.0)


def test_gpus_flag_spawns_the_reference_arm_once():
    """bench.py --gpus 2 outside torchrun runs two ranks; only rank 0 prints
    the reference line, and it declares both GPUs."""
    res = subprocess.run(
        [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
         "--gpus", "2", "--workload", "n512_r1_point", "--steps", "1",
         "--warmup", "0", "--cpu-sample-sweeps", "8"],
        capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert res.returncode == 0, res.stderr
    lines = [json.loads(x) for x in res.stdout.splitlines() if x.startswith("{")]
    assert len(lines) == 1 and lines[0]["impl"] == "reference"
    assert lines[0]["n_gpus"] == 2


def test_gpus_flag_must_match_the_launcher():
    res = subprocess.run(
        [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
         "--gpus", "2", "--workload", "n512_r1_point"],
        capture_output=True, text=True, timeout=120, cwd=ROOT,
        env={**os.environ, "WORLD_SIZE": "1", "RANK": "0", "LOCAL_RANK": "0"})
    assert res.returncode != 0 and "WORLD_SIZE" in res.stderr


def test_kernel_name_follows_the_resolved_tile():
    """tile_y = 0 is the column-streamed kernel (the D = 8 default on large
    grids); the solver reports the tile it resolved."""
    assert bench.kernel_name("etb8", (112, 0)).startswith("k_etbs")
    assert bench.kernel_name("etb8@112x0").startswith("k_etbs")
    assert bench.kernel_name("etb8", (112, 92)).startswith("k_etbr")


def test_cpu_baseline_times_the_whole_solve_when_it_is_small(monkeypatch):
    """cpu_baseline runs the oracle's whole ten-step solve when the solve
    needs at most FULL_SOLVE_LUPS lattice updates, and otherwise a sample of
    about 1e10; the oracle itself is replaced by a recorder here."""
    import types
    calls = []

    class FakeSample:
        def __init__(self, n, r, source, threads=1):
            self.n, self.threads = n, threads

        def __call__(self, sweeps):
            calls.append((self.n, self.threads, sweeps))
            return 1.0, 2.0, sweeps

    monkeypatch.setattr(bench, "OracleSample", FakeSample)
    args = types.SimpleNamespace(workload="n2048_r10_gauss", cpu_sample_sweeps=0)
    rec = bench.cpu_baseline(args, 4064)  # 4064 * 2046^2 = 1.7e10 updates
    assert [c[2] for c in calls] == [4064, 4064]
    assert rec["time_to_solution_s"] == 2.0 and "whole ten-step solve" in rec["sample"]
    assert rec["cores"] == 1 and rec["all_cores"]["cores"] >= 1
    calls.clear()
    args = types.SimpleNamespace(workload="n18432_r10_point", cpu_sample_sweeps=0)
    rec = bench.cpu_baseline(args, 2256)  # 7.7e11 updates: a sample
    sweeps = calls[0][2]
    assert sweeps % 8 == 0 and 0.5e10 <= sweeps * 18430 ** 2 <= 2e10
    assert rec["time_to_solution_s"] is None and rec["sample"].startswith("first")
    calls.clear()
    bench.cpu_baseline(args, None)  # no GPU sweep count: a sample
    assert calls[0][2] == sweeps
