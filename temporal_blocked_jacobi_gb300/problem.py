"""Synthetic inputs for the implicit-diffusion Jacobi solver.

This module only builds input arrays: the initial field u⁰ with its Dirichlet
ring and the source term g = Δt·f. It holds none of the method's arithmetic
(no sweep, right-hand side or residual), so both the CUDA path and the oracle
can take their inputs from it.

Problem statement: "Synchronous vs block-async Jacobi on one RTX 5050",
section 01 "The problem": an N×N unit square, top boundary held at 100 and
the other three at 0, and a source that is either a point at the centre or a
Gaussian with σ = N/16; ten float32 time steps from u⁰ = 0 in the interior.

Readings where that section is not explicit:
  * N counts the ring: the array is N×N and the (N−2)² interior cells are the
    unknowns.
  * Row 0 is the top; all of row 0, corners included, is 100. Corners are
    never read by the five-point stencil.
  * The centre is cell (N//2, N//2) (integer division).
  * The Gaussian is g_ij = 100·exp(−((i−c)² + (j−c)²)/(2σ²)), σ = N/16,
    evaluated once in float64 on the host and rounded to float32, on interior
    cells only, so every consumer sees identical bits.
  * The point source puts Δt·f = 1000 on the centre cell.

Arrays are numpy float32 of shape (N, ld) with ld ≥ N a multiple of 4
(16-byte rows); columns N..ld−1 are padding that no computation reads.
"""
from __future__ import annotations

import numpy as np

TOP_BOUNDARY = 100.0
POINT_AMPLITUDE = 1000.0
GAUSS_AMPLITUDE = 100.0


def padded_ld(n: int, align: int = 4) -> int:
    """Smallest row pitch ≥ n that is a multiple of `align` floats."""
    return (n + align - 1) // align * align


def initial_field(n: int, ld: int | None = None, *, top: float = TOP_BOUNDARY,
                  pad_value: float = 0.0, dtype=np.float32) -> np.ndarray:
    """u⁰: interior 0, row 0 (incl. corners) = `top`, other ring cells 0."""
    if n < 3:
        raise ValueError("n must be at least 3")
    ld = padded_ld(n) if ld is None else ld
    if ld < n:
        raise ValueError("ld must be >= n")
    u = np.zeros((n, ld), dtype=dtype)
    u[0, :n] = top
    if ld > n:
        u[:, n:] = pad_value
    return u


def source_term(n: int, ld: int | None = None, kind: str = "point", *,
                amplitude: float | None = None,
                center: tuple[float, float] | None = None,
                sigma: float | None = None, dtype=np.float32) -> np.ndarray:
    """g = Δt·f on the interior (ring and padding are 0).

    kind = "point": `amplitude` (default 1000) on the centre cell.
    kind = "gauss": amplitude (default 100) · exp(−r²/(2σ²)), σ = N/16,
    computed in float64 and rounded once.
    kind = "zero": no source.
    `center` defaults to (N//2, N//2); odd-N symmetry tests pass
    ((N−1)/2, (N−1)/2).
    """
    ld = padded_ld(n) if ld is None else ld
    g = np.zeros((n, ld), dtype=dtype)
    ci, cj = (n // 2, n // 2) if center is None else center
    if kind == "zero":
        return g
    if kind == "point":
        amp = POINT_AMPLITUDE if amplitude is None else amplitude
        i, j = int(ci), int(cj)
        if not (1 <= i <= n - 2 and 1 <= j <= n - 2):
            raise ValueError("point source must lie in the interior")
        g[i, j] = amp
        return g
    if kind == "gauss":
        amp = GAUSS_AMPLITUDE if amplitude is None else amplitude
        sig = n / 16.0 if sigma is None else float(sigma)
        idx = np.arange(1, n - 1, dtype=np.float64)
        di = (idx - ci) ** 2
        dj = (idx - cj) ** 2
        val = amp * np.exp(-(di[:, None] + dj[None, :]) / (2.0 * sig * sig))
        g[1:n - 1, 1:n - 1] = val.astype(dtype)
        return g
    raise ValueError(f"unknown source kind {kind!r}")


def random_field(n: int, ld: int | None = None, seed: int = 0, *,
                 lo: float = 0.0, hi: float = 100.0,
                 dtype=np.float32) -> np.ndarray:
    """Seeded uniform interior values with the standard ring (for kernel-level
    tests that need a generic iterate or right-hand side)."""
    rng = np.random.default_rng(seed)
    u = initial_field(n, ld, dtype=dtype)
    u[1:n - 1, 1:n - 1] = rng.uniform(lo, hi, size=(n - 2, n - 2)).astype(dtype)
    return u


# The workloads the solver is measured on. Each is fully synthetic and
# deterministic: u⁰ from initial_field, g from source_term.
WORKLOADS = {
    "n512_r1_point": dict(n=512, r=1.0, source="point"),
    "n2048_r10_gauss": dict(n=2048, r=10.0, source="gauss"),
    "n8192_r100_gauss": dict(n=8192, r=100.0, source="gauss"),
    "n18432_r10_point": dict(n=18432, r=10.0, source="point"),
    "n4096_r1_gauss": dict(n=4096, r=1.0, source="gauss"),
    "n4096_r10_gauss": dict(n=4096, r=10.0, source="gauss"),
    "n4096_r100_gauss": dict(n=4096, r=100.0, source="gauss"),
}


def make_workload(n: int, source: str, ld: int | None = None):
    """(u⁰, g) for an N×N grid with the given source kind."""
    ld = padded_ld(n) if ld is None else ld
    return initial_field(n, ld), source_term(n, ld, source)
