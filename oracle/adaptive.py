"""Oracle for the adaptive-depth block-asynchronous solve.

TEST INFRASTRUCTURE ONLY (same rule as the rest of this package: imported by
tests/ and nothing in the product path).

Source: "Synchronous vs block-async Jacobi on one RTX 5050", section 02
(D is a kernel argument and may change between launches; G-asc and G-desc
move D up or down as rho passes 1e-2, 1e-3 and 1e-4, latched; G-fb climbs
from D = 1 on the measured convergence rate -ln(rho_k / rho_{k-1}) per ms,
doubling while the rate holds, halving on a drop of more than 10 %, and
skipping the residual bump right after each change).

Readings, where the page leaves a step open:
  * depths are 1, 2, 4, ... up to depth_max; G-desc starts at depth_max;
  * "latched": the number of thresholds rho has ever been below, within the
    time step, only grows; every time step starts the controller afresh;
  * G-fb compares each measured rate with the previous measured one (the
    first one always counts as holding), the time of a check interval is its
    device time, and the settling window is one measurement;
  * rho is rmax / bmax of the stopping rule's own check, and D changes only
    at checks.

Pins (tests/test_oracle_adaptive.py): hand-worked controller sequences from
the rules above, monotonicity and range invariants on random sequences, the
constant schedule reducing to the fixed-depth block-asynchronous solve of
oracle.solve_step, and D = 1 reducing to synchronous sweeps.
"""
from __future__ import annotations

import math

import numpy as np

from . import ba_launch, residual

THRESHOLDS = (1e-2, 1e-3, 1e-4)


class Controller:
    """One time step's depth controller. `depth` is the D of the next check
    interval; `observe(rho, ms)` is called after each check."""

    def __init__(self, policy: str, depth_max: int):
        if depth_max not in (2, 4, 8, 16):
            raise ValueError("depth_max must be 2, 4, 8 or 16")
        if policy not in ("g_asc", "g_desc", "g_fb"):
            raise ValueError(f"unknown policy {policy!r}")
        self.policy = policy
        self.depth_max = depth_max
        # the ladder of depths, smallest first
        self.ladder = [1 << k for k in range(depth_max.bit_length())]
        self.crossed = 0            # G-asc / G-desc: latched threshold count
        self.last_rho = None        # G-fb
        self.last_rate = None       # G-fb
        self.skip = 0               # G-fb: measurements left to ignore
        self.depth = depth_max if policy == "g_desc" else 1
        self.changes = 0

    def _move_to(self, d):
        d = min(max(d, 1), self.depth_max)
        if d != self.depth:
            self.depth = d
            self.changes += 1
            if self.policy == "g_fb":
                self.skip = 1

    def observe(self, rho: float, ms: float) -> int:
        if self.policy in ("g_asc", "g_desc"):
            now = sum(1 for t in THRESHOLDS if rho < t)
            self.crossed = max(self.crossed, now)
            rung = min(self.crossed, len(self.ladder) - 1)
            if self.policy == "g_asc":
                self._move_to(self.ladder[rung])
            else:
                self._move_to(self.ladder[len(self.ladder) - 1 - rung])
            return self.depth
        # G-fb
        prev, self.last_rho = self.last_rho, rho
        if (prev is None or not (prev > 0) or not (rho > 0) or not (ms > 0)
                or math.isinf(prev) or math.isinf(rho)):
            return self.depth
        rate = -math.log(rho / prev) / ms
        if self.skip:
            self.skip -= 1
            return self.depth
        ref, self.last_rate = self.last_rate, rate
        if ref is None or rate >= 0.9 * ref:
            self._move_to(2 * self.depth)
        else:
            self._move_to(self.depth // 2)
        return self.depth


def depths(policy, depth_max, rhos, mss):
    """D before the first check, then after each (rho, ms)."""
    c = Controller(policy, depth_max)
    out = [c.depth]
    for rho, ms in zip(rhos, mss):
        out.append(c.observe(rho, ms))
    return out


def solve_step(u, b, r, *, policy, depth_max, tile_x=32, tile_y=8, m=8,
               tol=1e-5, max_sweeps=1 << 22, ms=None, schedule=None):
    """One time step of the block-asynchronous solve with a depth controller,
    in place on u (float32, grid layout).

    Each check interval runs lcm(m, D) sweeps as block-asynchronous launches
    of depth D (oracle.ba_launch), then the residual check of section 01.
    G-fb needs the time of each interval: `ms` is a list (the i-th check's
    time) or a callable (check index, D) -> ms. With `schedule` (a list of D
    per check interval) the controller is bypassed.

    Returns (k, trace) with k the sweep count (negative: -3 not converged,
    -4 non-finite) and trace a list of (D, k, rmax, bmax) per check.
    """
    ctl = None if schedule is not None else Controller(policy, depth_max)
    k, trace, i = 0, [], 0
    while True:
        d = schedule[i] if schedule is not None else ctl.depth
        interval = m * d // math.gcd(m, d)
        for _ in range(interval // d):
            u[...] = ba_launch(u, b, r, tile_x, tile_y, d)
        k += interval
        rmax, bmax = residual(u, b, r)
        trace.append((d, k, rmax, bmax))
        rm, bm = float(rmax), float(bmax)
        if not (np.isfinite(rm) and np.isfinite(bm)):
            return -4, trace
        if rm == 0.0 or rm < tol * bm:
            return k, trace
        if k >= max_sweeps:
            return -3, trace
        if ctl is not None:
            t = ms(i, d) if callable(ms) else (ms[i] if ms is not None else 0.0)
            ctl.observe(rm / bm if bm > 0 else math.inf, t)
        i += 1
