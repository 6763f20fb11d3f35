#!/usr/bin/env python3
"""Benchmark of the five-point Jacobi solver for implicit 2-D diffusion.

One bench step = one full run of the method on one synthetic workload: u⁰
reset, then ten backward-Euler time steps (fused right-hand side, Jacobi
sweeps of the chosen strategy, residual every check interval, stop
decision), timed with CUDA events on the solver's stream, checks included
("Synchronous vs block-async Jacobi on one RTX 5050", sections 01-03).

Default workload: the largest grid, N = 18432 (ring included; 1.36 GB per
field, far beyond L2), r = 10, point source 1000 at the centre, 10 time
steps, tol 1e-5, M = 8; strategies SYNC, EXACT_TEMPORAL_BLOCKED D = 8 and
BLOCK_ASYNC D = 8; convergence loop on the device (--control host: one host
round trip per check instead). `value` is the GLUP/s (interior points ×
sweeps ÷ time) of the strategy with the shortest ten-step time-to-solution;
every strategy's figures are under "strategies". SYNC and
EXACT_TEMPORAL_BLOCKED perform the same sweeps (exact temporal blocking is
bit-identical to SYNC, which the line re-checks on the final fields), so
their GLUP/s compare time-to-solution directly; BLOCK_ASYNC needs s times
the sweeps, its GLUP/s counts them, and its final field is checked against
the SYNC field within 5e-4 ||b||inf.

Besides the headline kernel's roofline the line carries the synchronous
sweep's HBM roofline on the same grid ("roofline_sync") and at N = 8192
("roofline_sync_n8192").

Usage:
  python bench.py [--steps K] [--warmup W] [--workload NAME]
                  [--strategies sync,etb8,ba8] [--impl ours|reference]
                  [--gpus N]
Multi-GPU: independent replicas of the same solve, one process per GPU, no
data exchange; value = all ranks' lattice updates ÷ max time. Under torchrun
the ranks come from the environment; with --gpus N > 1 and no torchrun
environment bench.py starts the N ranks itself through torch.distributed.run.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from temporal_blocked_jacobi_gb300 import problem as P  # noqa: E402

METRIC = "Jacobi GLUP/s, HBM GB/s vs peak, 10-step time-to-solution per strategy"
UNIT = "GLUP/s"

WORKLOADS = {
    # name: (N, r, source, default strategies)
    "n512_r1_point": (512, 1.0, "point", "sync,etb2,etb4,etb8"),
    "n2048_r10_gauss": (2048, 10.0, "gauss", "sync,syncu,etb2,etb4,etb8"),
    "n8192_r100_gauss": (8192, 100.0, "gauss", "sync,syncu,etb4,etb8,etb16"),
    "n18432_r10_point": (18432, 10.0, "point", "sync,etb8,ba8"),
    "n4096_r1_gauss": (4096, 1.0, "gauss",
                         "sync,syncu,etb2,etb4,etb8,etb16,ba2,ba4,ba8,ba16,gasc8,gdesc8,gfb8"),
    "n4096_r10_gauss": (4096, 10.0, "gauss",
                         "sync,syncu,etb2,etb4,etb8,etb16,ba2,ba4,ba8,ba16,gasc8,gdesc8,gfb8"),
    "n4096_r100_gauss": (4096, 100.0, "gauss",
                         "sync,syncu,etb2,etb4,etb8,etb16,ba2,ba4,ba8,ba16,gasc8,gdesc8,gfb8"),
}
DEFAULT_WORKLOAD = "n18432_r10_point"
TIME_STEPS = 10
L2_FLUSH_BYTES = 512 << 20  # > 129 MB L2


def parse_strategy(tok: str):
    """'sync' | 'syncu' | 'etbD' | 'etbDp' | 'baD' | 'baDoO' | 'gascD' |
    'gdescD' | 'gfbD', each optionally '@TXxTY' -> kwargs for jacobi.Solver.
    'etbDp': EXACT_TEMPORAL_BLOCKED under persistent control (one cooperative
    launch per time step); 'syncu':
    SYNC with the unfused right-hand side; 'baDoO': BLOCK_ASYNC on subdomains
    overlapping by O cells in both directions; 'gasc', 'gdesc', 'gfb':
    BLOCK_ASYNC with that depth controller and D up to the given depth (host
    control)."""
    tok = tok.strip()
    tile = (0, 0)
    if "@" in tok:
        tok, t = tok.split("@")
        tx, ty = t.lower().split("x")
        tile = (int(tx), int(ty))
    if tok == "sync":
        return dict(strategy="sync", depth=1, tile=tile)
    if tok == "syncu":
        return dict(strategy="sync", depth=1, tile=tile, rhs="unfused")
    for prefix, adapt in (("gasc", "g_asc"), ("gdesc", "g_desc"), ("gfb", "g_fb")):
        if tok.startswith(prefix):
            return dict(strategy="ba", depth=int(tok[len(prefix):]), tile=tile,
                        adapt=adapt, control="host")
    if tok.startswith("ba") and "o" in tok:  # 'baDoO': overlap O both ways
        depth, ov = tok[2:].split("o")
        return dict(strategy="ba", depth=int(depth), tile=tile,
                    overlap=(int(ov), int(ov)))
    if tok.startswith("etb") and tok.endswith("p"):  # 'etbDp': persistent control
        return dict(strategy="etb", depth=int(tok[3:-1]), tile=tile,
                    control="persistent")
    for prefix, name in (("etb", "etb"), ("ba", "ba")):
        if tok.startswith(prefix):
            return dict(strategy=name, depth=int(tok[len(prefix):]), tile=tile)
    raise ValueError(f"unknown strategy {tok!r}")


def bytes_per_point(kw):
    """Algorithmic bytes per interior point per launch: read u, read b (u^n
    and g when the right-hand side is unfused), write u'."""
    return 16.0 if kw.get("rhs") == "unfused" else 12.0


def sweeps_per_launch(kw):
    return 1 if kw["strategy"] == "sync" else kw["depth"]


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def sm_max_mhz():
    """Maximum SM clock: MEASURED_PEAKS.json's figure, else GB300's 2070 MHz."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["sm_max_mhz"]), "measured"
    except (OSError, ValueError, KeyError):
        return 2070.0, "nominal"


# FP32 pipe operations one lattice update needs at least: the 5 of the update
# (W+E, N+S, their sum, r*s, b + r*s) and the 3 of a correctly rounded
# division by the fixed d (q0 = x*y, rho = fma(q0, d, -x), q = fma(-rho, y,
# q0)). Each SM's FP32 pipe issues 128 of them per clock.
FP32_OPS_PER_LUP = 8
FP32_LANES_PER_SM = 128


def roofline_record(kw, interior, launch_ms, working_set, l2_bytes, sms,
                    hbm_peak, hbm_how, mhz, mhz_how):
    """Roofline of one sweep launch of strategy `kw` taking launch_ms.

    HBM view: the algorithmic bytes of a launch (12 B per interior point, 16
    with the unfused right-hand side) over its duration, against the measured
    copy bandwidth. ALU view: FP32_OPS_PER_LUP operations per lattice update
    (D updates per point per launch) against 128 lanes x SMs x the SM clock.
    When u, u_alt and b fit in L2 the launches of a solve do not go to HBM,
    so the bound reported is the FP32 pipe ("alu"); otherwise it is HBM."""
    per = sweeps_per_launch(kw)
    sec = launch_ms * 1e-3
    alg_bytes = bytes_per_point(kw) * interior
    gbs = alg_bytes / sec / 1e9
    lups = interior * per / sec
    ops = FP32_OPS_PER_LUP * lups / 1e12
    alu_peak = FP32_LANES_PER_SM * sms * mhz * 1e6 / 1e12
    hbm = {"achieved": gbs, "peak": hbm_peak, "unit": "GB/s", "frac": gbs / hbm_peak,
           "peak_source": (f"{hbm_how} (MEASURED_PEAKS.json hbm_gbs)"
                           if hbm_how == "measured" else hbm_how)}
    alu = {"achieved": ops, "peak": alu_peak, "unit": "Top/s", "frac": ops / alu_peak,
           "peak_source": (f"{FP32_LANES_PER_SM} FP32 lanes x {sms} SMs x {mhz:.0f} MHz "
                           f"(maximum SM clock, {mhz_how})"),
           "ops_per_lup": FP32_OPS_PER_LUP,
           # the same with the division counted as one operation (7 flops
           # per lattice update: 3 adds, 1 multiply, 1 add, 1 division)
           "frac_at_7_flops_per_lup": 7 * lups / 1e12 / alu_peak}
    l2_resident = working_set < l2_bytes
    bound = "alu" if l2_resident else "hbm"
    main = alu if bound == "alu" else hbm
    return {"bound": bound, "achieved": main["achieved"], "peak": main["peak"],
            "unit": main["unit"], "frac": main["frac"], "peak_source": main["peak_source"],
            "hbm": hbm, "alu": alu,
            "working_set_bytes": working_set, "l2_bytes": l2_bytes,
            "l2_resident": l2_resident, "alg_bytes_per_launch": alg_bytes,
            "launch_us": launch_ms * 1e3, "sweeps_per_launch": per, "lups_per_s": lups}


# ---------------------------------------------------------------------------
# Multi-process plumbing (replicas): max of the elapsed time and sum of the
# work over ranks. Works with any torch.distributed backend.
# ---------------------------------------------------------------------------
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def aggregate(local_units: float, local_seconds: float, device=None):
    """(sum of units over ranks, max of seconds over ranks)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return local_units, local_seconds
    t = torch.tensor([local_units], dtype=torch.float64, device=device)
    s = torch.tensor([local_seconds], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    dist.all_reduce(s, op=dist.ReduceOp.MAX)
    return float(t.item()), float(s.item())


def replica_glups(local_lups: float, local_seconds: float, device=None):
    """Whole-job GLUP/s of independent replicas: every rank's lattice
    updates over the slowest rank's time."""
    units, seconds = aggregate(local_lups, local_seconds, device=device)
    return units / seconds / 1e9


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


# ---------------------------------------------------------------------------
# Clock sampling during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if not self.path or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), parts[4:9]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        reasons = set()
        for _, _, flags in rows:
            for name, flag in zip(names, flags[1:]):
                if flag.lower() == "active":
                    reasons.add(name)
        sm = [r[0] for r in rows]
        busy = [s for s in sm if s > 0.5 * max(sm)] or sm
        return {"sm_mhz": statistics.median(busy), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": sorted(reasons), "samples": len(rows)}


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------
def run_ours(args):
    import torch

    from temporal_blocked_jacobi_gb300 import jacobi

    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group(args.dist_backend)
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    n, r, source, default_strats = WORKLOADS[args.workload]
    strategies = [s for s in (args.strategies or default_strats).split(",") if s]
    ld = P.padded_ld(n)
    interior = (n - 2) ** 2

    u0_host = P.initial_field(n, ld)
    g_host = P.source_term(n, ld, source)
    stream = torch.cuda.Stream(dev)
    u0 = torch.from_numpy(u0_host).to(dev)
    g = torch.from_numpy(g_host).to(dev)
    u, u_alt, b = jacobi.allocate(n, ld, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    torch.cuda.synchronize(dev)

    results = {}
    solvers = {}
    with torch.cuda.stream(stream):
        for tok in strategies:
            kw = parse_strategy(tok)
            kw.setdefault("control", args.control)
            u.copy_(u0)
            solvers[tok] = jacobi.Solver(u, u_alt, b, r, stream=stream, **kw)

        def one_step(tok):
            """Reset u⁰ (setup, untimed) and run the ten time steps (timed)."""
            s = solvers[tok]
            flush.fill_(1.0)  # evict the working set from L2
            u.copy_(u0)
            start = torch.cuda.Event(enable_timing=True)
            end = torch.cuda.Event(enable_timing=True)
            l0 = s.launch_count
            start.record(stream)
            counts = s.run(g, TIME_STEPS)
            end.record(stream)
            end.synchronize()
            return start.elapsed_time(end), counts, s.launch_count - l0

        for tok in strategies:
            for _ in range(args.warmup):
                one_step(tok)

        barrier()
        torch.cuda.synchronize(dev)
        t_wall0 = time.perf_counter()
        with ClockSampler(dev.index if dev.index is not None else 0) as clocks:
            for tok in strategies:
                times, launches, counts = [], 0, None
                for _ in range(args.steps):
                    ms, counts, nl = one_step(tok)
                    times.append(ms)
                    launches += nl
                sweeps = sum(counts)
                ms_med = statistics.median(times)
                kw = parse_strategy(tok)
                results[tok] = dict(
                    sweeps=sweeps, sweeps_per_step=counts,
                    ms_per_solve_median=ms_med, ms_per_solve_mean=sum(times) / len(times),
                    ms_per_solve_all=[round(t, 3) for t in times],
                    glups=interior * sweeps / (ms_med * 1e-3) / 1e9,
                    sync_equiv_gbs=12.0 * interior * sweeps / (ms_med * 1e-3) / 1e9,
                    # (D varies under a depth controller: not defined there)
                    alg_gbs=None if kw.get("adapt") else
                    bytes_per_point(kw) * interior * sweeps
                    / sweeps_per_launch(kw) / (ms_med * 1e-3) / 1e9,
                    launches=launches, total_ms=sum(times))
        torch.cuda.synchronize(dev)
        barrier()
        wall = time.perf_counter() - t_wall0

        # --- after the timed region: the answers of the strategies
        checks = answer_checks(solvers, strategies, u, u0, g, stream, n)

    best = headline(results)
    base = results.get("sync")
    for tok, res in results.items():
        if base:
            res["speedup_vs_sync"] = base["ms_per_solve_median"] / res["ms_per_solve_median"]
            res["sweep_ratio_s"] = res["sweeps"] / base["sweeps"]
            # cost per sweep relative to a synchronous sweep: S = 1/(c*s)
            res["cost_per_sweep_c"] = 1.0 / (res["speedup_vs_sync"] * res["sweep_ratio_s"])
        if tok in checks:
            res["answer_check"] = checks[tok]
    if base and "syncu" in results:
        # section 05, Table VI: T_unfused / T_fused of the synchronous sweep
        results["syncu"]["t_unfused_over_fused"] = (
            results["syncu"]["ms_per_solve_median"] / base["ms_per_solve_median"])
    total_ms = sum(res["total_ms"] for res in results.values())
    total_lups = sum(interior * res["sweeps"] * args.steps for res in results.values())
    value = replica_glups(float(interior * results[best]["sweeps"] * args.steps),
                          results[best]["total_ms"] * 1e-3,
                          device=dev if world > 1 else None)

    # --- dominant kernel: the headline strategy's sweep kernel, timed alone
    roof = kernel_roofline(solvers[best], best, u, u0, stream, interior, args.workload)
    roof_sync = None
    if "sync" in solvers and best != "sync":
        roof_sync = kernel_roofline(solvers["sync"], "sync", u, u0, stream, interior,
                                    args.workload)

    # --- end to end through the public API with host buffers
    e2e = end_to_end(solvers[best], u, g, u0_host, g_host, stream, interior, args)

    for s in solvers.values():
        s.close()
    del u, u_alt, b, g, u0, flush
    torch.cuda.synchronize(dev)
    torch.cuda.empty_cache()
    roof_8192 = None
    if n != SYNC_ROOFLINE_N and not args.no_sync_n8192:
        roof_8192 = sync_roofline_at(SYNC_ROOFLINE_N, dev)

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": results[best]["ms_per_solve_median"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic",
        "config": {"workload": args.workload, "n": n, "r": r, "source": source,
                   "interior_points": interior, "time_steps": TIME_STEPS,
                   "tol": 1e-5, "check_every": 8, "strategy": best,
                   "control": args.control,
                   "strategies_timed": strategies,
                   "l2": "flushed (512 MiB write) before every timed solve",
                   "parallelism": f"replicas x{world}"},
        "roofline": roof, "e2e": e2e,
        "gpu_launches": sum(res["launches"] for res in results.values()),
        "clocks": clocks.summary(),
        "wall_s_timed_region": wall, "device_ms_all_strategies": total_ms,
        "lups_all_strategies": total_lups,
        "strategies": results,
    }
    if roof_sync is not None:
        line["roofline_sync"] = roof_sync
    if roof_8192 is not None:
        line["roofline_sync_n8192"] = roof_8192
    if base:
        etbs = [t for t in results if parse_strategy(t)["strategy"] == "etb"]
        if etbs:
            fastest = min(etbs, key=lambda t: results[t]["ms_per_solve_median"])
            line["etb_over_sync"] = {
                "strategy": fastest,
                "time_to_solution_ratio": results[fastest]["speedup_vs_sync"]}
    if rank == 0:
        if not args.no_cpu_baseline and world == 1:
            exact = [v["sweeps"] for t, v in results.items()
                     if parse_strategy(t)["strategy"] in ("sync", "etb")]
            line["cpu_baseline"] = cpu_baseline(args, exact[0] if exact else None)
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# The grid on which the synchronous sweep's HBM fraction is also reported
# (section 05 "Results beyond L2": 805 MB per sweep, far beyond L2).
SYNC_ROOFLINE_N = 8192


def answer_checks(solvers, strategies, u, u0, g, stream, n):
    """After the timed region, one more ten-step run of each strategy from u⁰:
    EXACT_TEMPORAL_BLOCKED must give SYNC's sweep counts and field bit for
    bit -- SYNC checked at the same interval, lcm(8, D) sweeps (D = 16: every
    16) --; BLOCK_ASYNC must lie within 5e-4 ||b||inf of SYNC's field,
    ||b||inf being the norm of SYNC's last right-hand side (section 02).
    Compared on the device. Without a SYNC strategy there is nothing to
    compare with."""
    import math

    import torch

    from temporal_blocked_jacobi_gb300 import jacobi
    if "sync" not in solvers:
        return {}
    s = solvers["sync"]
    refs = {}  # check interval -> (sweep counts, field) of SYNC

    def sync_ref(interval):
        if interval not in refs:
            u.copy_(u0)
            if interval == 8:
                counts = s.run(g, TIME_STEPS)
            else:
                with jacobi.Solver(u, s.u_alt, s.b, s.r, stream=stream,
                                   check_every=interval, control="device") as s2:
                    counts = s2.run(g, TIME_STEPS)
            refs[interval] = (counts, u.clone())
        return refs[interval]

    sync_counts, ref = sync_ref(8)
    u.copy_(ref)
    _, bmax = s.residual()
    out = {}
    for tok in strategies:
        kw = parse_strategy(tok)
        if tok == "sync":
            continue
        interval = 8 * sweeps_per_launch(kw) // math.gcd(8, sweeps_per_launch(kw))
        if kw["strategy"] == "etb" and interval != 8:
            want_counts, want = sync_ref(interval)
        else:
            want_counts, want = sync_counts, ref
        u.copy_(u0)
        counts = solvers[tok].run(g, TIME_STEPS)
        torch.cuda.current_stream().wait_stream(stream)
        diff = (u[1:n - 1, 1:n - 1] - ref[1:n - 1, 1:n - 1]).abs().max().item()
        rec = {"max_abs_diff_vs_sync": diff, "bmax": float(bmax)}
        if kw["strategy"] in ("etb", "sync"):
            same = bool(torch.equal(u.view(torch.int32), want.view(torch.int32)))
            rec.update(kind=f"bit-exact vs sync checked every {interval} sweeps",
                       same_counts=counts == want_counts, bit_identical=same,
                       ok=same and counts == want_counts)
        else:
            bound = 5e-4 * float(bmax)
            rec.update(kind="within 5e-4 ||b||inf of sync", bound=bound,
                       diff_over_bmax=diff / float(bmax) if bmax else None,
                       ok=diff <= bound)
        out[tok] = rec
    refs.clear()
    return out


def sync_roofline_at(n, dev):
    """The synchronous sweep's HBM roofline on an N x N Gaussian problem (r =
    100), launched back to back on a fresh solver after the timed region."""
    import torch

    from temporal_blocked_jacobi_gb300 import jacobi
    ld = P.padded_ld(n)
    interior = (n - 2) ** 2
    stream = torch.cuda.Stream(dev)
    with torch.cuda.stream(stream):
        u0 = torch.from_numpy(P.initial_field(n, ld)).to(dev)
        g = torch.from_numpy(P.source_term(n, ld, "gauss")).to(dev)
        u, u_alt, b = jacobi.allocate(n, ld, device=dev)
        u.copy_(u0)
        with jacobi.Solver(u, u_alt, b, 100.0, stream=stream) as s:
            s.rhs(g)
            rec = kernel_roofline(s, "sync", u, u0, stream, interior,
                                  f"n{n}_r100_gauss")
    rec["workload"] = f"n{n}_r100_gauss"
    del u0, g, u, u_alt, b
    torch.cuda.synchronize(dev)
    torch.cuda.empty_cache()
    return rec


def headline(results):
    """The strategy with the shortest ten-step time-to-solution. Block-async
    strategies sweep more often than SYNC (sweep ratio s > 1), so their
    GLUP/s is not a time-to-solution ranking."""
    return min(results, key=lambda t: results[t]["ms_per_solve_median"])


def kernel_roofline(solver, tok, u, u0, stream, interior, workload):
    """Average duration of the strategy's sweep kernel, launched back to back
    on the solver's stream (no checks) and timed there with CUDA events, as a
    roofline record (roofline_record) with the DRAM traffic of the committed
    ncu capture."""
    import torch
    kw = parse_strategy(tok)
    per = sweeps_per_launch(kw)
    launches = max(8, 256 // per)
    u.copy_(u0)
    solver.sweeps(launches)  # warm
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(stream)
    solver.sweeps(launches)
    end.record(stream)
    end.synchronize()
    ms = start.elapsed_time(end) / launches
    props = torch.cuda.get_device_properties(u.device)
    hbm_peak, hbm_how = measured_peaks()
    mhz, mhz_how = sm_max_mhz()
    # u, u_alt and b
    rec = roofline_record(kw, interior, ms, 3 * u.numel() * 4, props.L2_cache_size,
                          props.multi_processor_count, hbm_peak, hbm_how, mhz, mhz_how)
    rec["kernel"] = kernel_name(tok, solver.tile)
    rec["tile"] = list(solver.tile)
    rec["launches_timed"] = launches
    rec["traffic"] = load_traffic(tok, workload)
    return rec


# Tile sizes (with (0, 0), the default) of the register-resident shapes of
# exact temporal blocking, per depth.
ETBR_TILES = {4: ((0, 0), (120, 88), (120, 40)), 8: ((0, 0), (112, 80), (112, 92)),
              16: ((0, 0), (96, 64), (96, 76))}


def kernel_name(tok, tile=None):
    """The sweep kernel of strategy `tok`; `tile`: the tile the solver
    resolved (Solver.tile), which tells the column-streamed kernel apart."""
    kw = parse_strategy(tok)
    if kw["strategy"] == "sync":
        return "k_sweep_sync" + (" (unfused rhs)" if kw.get("rhs") == "unfused" else "")
    if kw["strategy"] == "etb":
        if (tile or kw.get("tile", (0, 0)))[1] == 0 and (tile or kw.get("tile"))[0] > 0:
            return f"k_etbs (D={kw['depth']}, column-streamed)"
        # default shapes: bands in registers for D = 4, 8 and 16, box in
        # shared memory for D = 2; explicit tiles of the band shapes likewise
        name = ("k_etbr" if kw.get("tile", (0, 0)) in ETBR_TILES.get(kw["depth"], ())
                else "k_etb")
        if kw.get("control") == "persistent":
            name = "k_etbp"  # the whole step in one cooperative launch
        return f"{name} (D={kw['depth']})"
    if kw.get("tile", (0, 0)) in ((0, 0), (32, 8)) and not kw.get("overlap"):
        return f"k_bar (D={kw['depth']})"  # 32 x 8 tiles held in registers
    return f"k_ba / k_block_async (D={kw['depth']})"


def load_traffic(tok, workload):
    """DRAM bytes per launch of this kernel from a committed ncu summary
    (profiles/traffic.json), or None if it was not captured for the current
    kernel source."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    try:
        d = json.load(open(path))
        return d.get(workload, {}).get(tok)
    except (ValueError, OSError):
        return None


def end_to_end(solver, u, g, u0_host, g_host, stream, interior, args):
    """Same metric through the public C ABI with host buffers
    (jacobi_run_host): `steps` problems, each copying u⁰ and g from pinned
    host memory, running the ten time steps and copying the final field
    back; the library overlaps each problem's copies with its neighbours'
    solves. Timed with the host clock around the call, after a warm-up
    call of `warmup` problems."""
    import torch
    u0_pin = torch.from_numpy(u0_host).pin_memory()
    g_pin = torch.from_numpy(g_host).pin_memory()
    outs = [torch.empty_like(u0_pin).pin_memory() for _ in range(2)]

    def call(k):
        return solver.run_host([u0_pin] * k, [g_pin] * k,
                               [outs[i % 2] for i in range(k)], TIME_STEPS)

    call(args.warmup)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    counts = call(args.steps)
    dt = time.perf_counter() - t0
    sweeps = sum(sum(c) for c in counts)
    nbytes = u0_pin.numel() * 4
    return {"value": interior * sweeps / dt / 1e9, "unit": UNIT,
            "h2d_bytes_per_step": 2 * nbytes, "d2h_bytes_per_step": nbytes,
            "ms_per_step": dt / args.steps * 1e3, "clock": "host wall clock",
            "api": "jacobi_run_host (host buffers; copies overlapped with "
                   "the neighbouring problems' solves)",
            "sweeps_per_problem": sum(counts[0])}


# ---------------------------------------------------------------------------
# CPU oracle legs (test infrastructure, timed as a reported baseline)
# ---------------------------------------------------------------------------
class OracleSample:
    """The oracle (single-threaded C; `threads` > 1: its row-parallel form,
    bit-identical) timed on a bounded sample of the ten-step solve: the first
    `sweeps` sweeps, right-hand sides and residual checks included,
    continuing into later time steps as each one converges. The inputs are
    built once, outside the timed calls."""

    def __init__(self, n, r, source, threads=1):
        self.threads = threads
        import oracle
        self.oracle = oracle
        self.n, self.r = n, r
        self.u0 = P.initial_field(n)
        self.g = P.source_term(n, kind=source)
        oracle.rhs(self.u0[:3, :4].copy(), self.g[:3, :4].copy(), 3)  # load the library

    def __call__(self, sample_sweeps):
        oracle = self.oracle
        u = self.u0.copy()
        done, steps = 0, 0
        t0 = time.perf_counter()
        while done < sample_sweeps and steps < TIME_STEPS:
            b = oracle.rhs(u, self.g)
            k, _, _ = oracle.solve_step(u, b, self.r, max_sweeps=sample_sweeps - done,
                                        threads=self.threads)
            done += (sample_sweeps - done) if k < 0 else k
            steps += 1
        dt = time.perf_counter() - t0
        return (self.n - 2) ** 2 * done / dt / 1e9, dt, done


def oracle_sample(n, r, source, sample_sweeps):
    """One timed oracle sample of `sample_sweeps` sweeps: (GLUP/s, s, sweeps)."""
    return OracleSample(n, r, source)(sample_sweeps)


# The oracle's whole ten-step solve is timed when it needs at most this many
# lattice updates (about 30 s on one host core); otherwise a sample of 1e10.
FULL_SOLVE_LUPS = 2.5e10


def cpu_baseline(args, solve_sweeps=None):
    """The oracle timed on the host: the whole ten-step solve when
    `solve_sweeps` (the GPU's sweep count of the synchronous solve, which
    the oracle reproduces) times the interior points is at most
    FULL_SOLVE_LUPS, else its first ~1e10 lattice updates (10-15 s)."""
    n, r, source, _ = WORKLOADS[args.workload]
    points = (n - 2) ** 2
    full = (not args.cpu_sample_sweeps and solve_sweeps is not None
            and points * solve_sweeps <= FULL_SOLVE_LUPS)
    if full:
        sweeps = solve_sweeps
    else:
        sweeps = args.cpu_sample_sweeps or max(8, int(8 * round(1.0e10 / points / 8)))
    sample = OracleSample(n, r, source)
    glups, dt, done = sample(sweeps)
    cores = os.cpu_count() or 1
    sample.threads = cores
    glups_all, dt_all, _ = sample(sweeps)
    what = (f"the whole ten-step solve ({done} sweeps, checks every 8)" if full
            else f"first {done} sweeps of the ten-step solve (checks every 8)")
    return {"value": glups, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"{what}, single-threaded C oracle, {dt:.1f} s",
            "time_to_solution_s": dt if full else None,
            "host_cpus": cores,
            # the same sample with the oracle's rows split over every host
            # core (bit-identical results)
            "all_cores": {"value": glups_all, "unit": UNIT, "cores": cores,
                          "seconds": dt_all}}


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    n, r, source, _ = WORKLOADS[args.workload]
    # about 1e9 lattice updates per bench step (at least one check interval)
    sweeps = args.cpu_sample_sweeps or max(8, int(8 * round(1.0e9 / (n - 2) ** 2 / 8)))
    sample = OracleSample(n, r, source)
    for _ in range(args.warmup):
        sample(sweeps)
    vals, secs = [], []
    for _ in range(args.steps):
        v, dt, done = sample(sweeps)
        vals.append(v)
        secs.append(dt)
    value = statistics.median(vals)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": statistics.median(secs) * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic",
            "config": {"workload": args.workload, "n": n, "r": r, "source": source,
                       "strategy": "sync (oracle)", "parallelism": "single host core"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                             "sample": f"first {sweeps} sweeps of the ten-step solve per "
                                       "bench step, single-threaded C oracle"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def spawn_ranks(nproc, argv, script=None):
    """Start `nproc` ranks of `script` (default: this file) through
    torch.distributed.run on 127.0.0.1, one process per GPU, and return the
    launcher's exit code. The ranks see WORLD_SIZE and do not spawn again."""
    import socket
    with socket.socket() as sock:
        sock.bind(("127.0.0.1", 0))
        port = sock.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
           f"--nproc-per-node={nproc}", "--master-addr=127.0.0.1",
           f"--master-port={port}", script or os.path.abspath(__file__), *argv]
    return subprocess.call(cmd)


def main(argv=None):
    argv = sys.argv[1:] if argv is None else list(argv)
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WORKLOADS))
    ap.add_argument("--strategies", default=None,
                    help="comma list: sync, etbD, baD, baD@TXxTY (default per workload)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--control", default="device", choices=["device", "host"],
                    help="convergence loop on the device (one graph per time "
                         "step) or on the host (one round trip per check)")
    ap.add_argument("--dist-backend", default="nccl",
                    help="torch.distributed backend of the replicas' two scalar "
                         "reductions")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-sync-n8192", action="store_true",
                    help="skip the extra synchronous-sweep roofline at N = 8192")
    ap.add_argument("--cpu-sample-sweeps", type=int, default=0)
    args = ap.parse_args(argv)
    if args.gpus < 1:
        ap.error("--gpus must be at least 1")
    if args.warmup < 3 and args.impl == "ours":
        ap.error("--warmup must be at least 3")
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        sys.exit(spawn_ranks(args.gpus, argv))
    world, _, _ = dist_env()
    if world != args.gpus:
        ap.error(f"--gpus {args.gpus} but WORLD_SIZE={world}")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
