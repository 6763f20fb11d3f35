"""Oracle: a plain, slow, single-threaded CPU restatement of the Jacobi solver.

TEST INFRASTRUCTURE ONLY. Only tests/, `__graft_entry__.smoke()` and the
CPU-baseline / reference legs of bench.py may import this package. The CUDA
library shares no code with it and never calls it; the product path has no
CPU fallback.

Source: "Synchronous vs block-async Jacobi on one RTX 5050"
(stencil-jacobian.vercel.app), sections 01 "The problem" and 02 "Method".
The arithmetic lives in oracle_body.h (instantiated in float32 and float64 by
oracle.c) and is compiled with -ffp-contract=off and without fast-math.

Functions and what pins them (tests/test_oracle_pins.py):
  rhs            b = u + g             -- pinned: exact float32 sum (closed form)
  sweep          one Jacobi sweep      -- pinned: float64 dense direct solve,
                                          maximum principle, mirror symmetry,
                                          contraction bound, N=3 closed form,
                                          r=0 special case
  residual       difference-form norms -- pinned: float64 residual of the same
                                          iterate within its rounding bound;
                                          zero at the exact fixed point
  solve_step     stopping rule loop    -- pinned: dense solve within rho·‖b‖,
                                          zero-source first-check stop,
                                          sweep counts per step (section 01)
  ba_launch      block-async launch    -- pinned: depth 1 equals one sweep; one
                                          tile covering the grid equals depth
                                          sweeps; frozen-halo brute force on a
                                          2x2 tiling; mirror symmetry of a
                                          mirror-symmetric tiling
  ba_overlap_launch  overlapping      -- pinned: overlap 0 equals ba_launch;
                 subdomains ("Hierarchical Jacobi Iteration for Structured
                 Matrices on GPUs using Shared Memory")
                                          depth 1 equals one sweep; strips
                                          brute-forced from synchronous sweeps
                                          of each subdomain with its frozen
                                          halo as the ring; mirror symmetry;
                                          fewer sweeps with overlap
  run            ten-step driver       -- pinned through the above
  threads > 1    row-parallel sweeps   -- pinned: bit-identical to one thread
                 and residuals            (tests/test_oracle_threads.py); one
                                          thread stays the oracle of record
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = [os.path.join(_HERE, "oracle.c"), os.path.join(_HERE, "oracle_body.h")]
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_CFLAGS = ["-O2", "-std=c11", "-Wall", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", "-pthread"]
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile liboracle.so beside the sources (gcc, host architecture)."""
    stale = force or not os.path.exists(_LIB_PATH) or any(
        os.path.getmtime(s) > os.path.getmtime(_LIB_PATH) for s in _SRC)
    if stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cc = os.environ.get("CC", "gcc")
        subprocess.check_call([cc, *_CFLAGS, "-o", tmp, _SRC[0], "-lm", "-lpthread"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        f32p = np.ctypeslib.ndpointer(np.float32, flags="C_CONTIGUOUS")
        f64p = np.ctypeslib.ndpointer(np.float64, flags="C_CONTIGUOUS")
        i64p = np.ctypeslib.ndpointer(np.int64, flags="C_CONTIGUOUS")
        c_int, c_ll, c_d = ctypes.c_int, ctypes.c_longlong, ctypes.c_double
        for sfx, rp, real in (("f32", f32p, ctypes.c_float),
                              ("f64", f64p, ctypes.c_double)):
            preal = ctypes.POINTER(real)
            f = getattr(lib, f"oracle_rhs_{sfx}")
            f.argtypes = [c_int, c_ll, rp, rp, rp]
            f.restype = None
            f = getattr(lib, f"oracle_sweep_{sfx}")
            f.argtypes = [c_int, c_ll, real, rp, rp, rp]
            f.restype = None
            f = getattr(lib, f"oracle_residual_{sfx}")
            f.argtypes = [c_int, c_ll, real, rp, rp, preal, preal]
            f.restype = None
            f = getattr(lib, f"oracle_ba_launch_{sfx}")
            f.argtypes = [c_int, c_ll, real, c_int, c_int, c_int, rp, rp, rp]
            f.restype = c_int
            f = getattr(lib, f"oracle_ba_overlap_launch_{sfx}")
            f.argtypes = [c_int, c_ll, real, c_int, c_int, c_int, c_int, c_int,
                          rp, rp, rp]
            f.restype = c_int
            f = getattr(lib, f"oracle_solve_step_{sfx}")
            f.argtypes = [c_int, c_ll, real, c_int, c_d, c_ll, c_int, c_int,
                          c_int, c_int, c_int, rp, rp, rp, preal, preal]
            f.restype = c_ll
            f = getattr(lib, f"oracle_solve_step_mt_{sfx}")
            f.argtypes = [c_int, c_ll, real, c_int, c_d, c_ll, c_int, c_int,
                          c_int, c_int, c_int, rp, rp, rp, preal, preal, c_int]
            f.restype = c_ll
            f = getattr(lib, f"oracle_run_{sfx}")
            f.argtypes = [c_int, c_ll, real, c_int, c_d, c_ll, c_int, c_int,
                          c_int, c_int, c_int, c_int, rp, rp, rp, rp, i64p]
            f.restype = c_ll
            f = getattr(lib, f"oracle_run_mt_{sfx}")
            f.argtypes = [c_int, c_ll, real, c_int, c_d, c_ll, c_int, c_int,
                          c_int, c_int, c_int, c_int, rp, rp, rp, rp, i64p, c_int]
            f.restype = c_ll
        _lib = lib
        return lib


def _sfx(a: np.ndarray) -> str:
    if a.dtype == np.float32:
        return "f32"
    if a.dtype == np.float64:
        return "f64"
    raise TypeError("oracle arrays must be float32 or float64")


def _check(*arrs):
    a0 = arrs[0]
    for a in arrs:
        if a.ndim != 2 or not a.flags.c_contiguous or a.dtype != a0.dtype \
                or a.shape != a0.shape:
            raise ValueError("oracle arrays must be C-contiguous (n, ld) of one dtype")
    return a0.shape[1]


def _real(a):
    return np.float32 if a.dtype == np.float32 else np.float64


def rhs(u, g, n=None):
    """b = u + g on the interior; ring of b is 0."""
    ld = _check(u, g)
    n = u.shape[0] if n is None else n
    b = np.zeros_like(u)
    getattr(_load(), f"oracle_rhs_{_sfx(u)}")(n, ld, u, g, b)
    return b


def sweep(u, b, r, n=None):
    """One synchronous Jacobi sweep; returns a new array with u's ring."""
    ld = _check(u, b)
    n = u.shape[0] if n is None else n
    out = u.copy()
    getattr(_load(), f"oracle_sweep_{_sfx(u)}")(n, ld, _real(u)(r), u, b, out)
    return out


def sweeps(u, b, r, count, n=None):
    """`count` synchronous sweeps from u."""
    cur = u
    for _ in range(count):
        cur = sweep(cur, b, r, n)
    return cur if count else u.copy()


def residual(u, b, r, n=None):
    """(rmax, bmax) over the interior: rmax = max d·|J(u)−u| (the difference
    form of |b − Au|), bmax = max |b_I|, where b_I = b + r·(the cell's
    Dirichlet-ring neighbours) is the right-hand side of the system in the
    unknowns."""
    ld = _check(u, b)
    n = u.shape[0] if n is None else n
    real = ctypes.c_float if u.dtype == np.float32 else ctypes.c_double
    rm, bm = real(), real()
    getattr(_load(), f"oracle_residual_{_sfx(u)}")(
        n, ld, _real(u)(r), u, b, ctypes.byref(rm), ctypes.byref(bm))
    return _real(u)(rm.value), _real(u)(bm.value)


def ba_launch(u, b, r, tile_x, tile_y, depth, n=None):
    """One block-asynchronous launch of `depth` in-tile sweeps."""
    ld = _check(u, b)
    n = u.shape[0] if n is None else n
    out = u.copy()
    rc = getattr(_load(), f"oracle_ba_launch_{_sfx(u)}")(
        n, ld, _real(u)(r), tile_x, tile_y, depth, u, b, out)
    if rc:
        raise ValueError(f"oracle_ba_launch failed ({rc})")
    return out


def ba_overlap_launch(u, b, r, tile_x, tile_y, overlap_x, overlap_y, depth,
                      n=None):
    """One block-asynchronous launch on overlapping subdomains (tiles start
    every tile - overlap cells; shared cells split half and half)."""
    ld = _check(u, b)
    n = u.shape[0] if n is None else n
    out = u.copy()
    rc = getattr(_load(), f"oracle_ba_overlap_launch_{_sfx(u)}")(
        n, ld, _real(u)(r), tile_x, tile_y, overlap_x, overlap_y, depth, u, b, out)
    if rc:
        raise ValueError(f"oracle_ba_overlap_launch failed ({rc})")
    return out


def solve_step(u, b, r, *, m=8, tol=1e-5, max_sweeps=1 << 22, depth=0,
               tile_x=32, tile_y=8, overlap=(0, 0), n=None, threads=1):
    """Solve one step in place from the warm start u. Returns
    (status_or_sweeps, rmax, bmax). depth 0 = synchronous sweeps; depth ≥ 1 =
    block-asynchronous launches on tile_x×tile_y tiles (overlapping by
    `overlap` = (ox, oy) cells when not zero). threads > 1 splits the rows of
    each synchronous sweep and residual among POSIX threads (same bits; the
    single-threaded form is the oracle of record)."""
    ld = _check(u, b)
    n = u.shape[0] if n is None else n
    work = u.copy()
    real = ctypes.c_float if u.dtype == np.float32 else ctypes.c_double
    rm, bm = real(), real()
    if threads <= 1:
        k = getattr(_load(), f"oracle_solve_step_{_sfx(u)}")(
            n, ld, _real(u)(r), m, tol, max_sweeps, depth, tile_x, tile_y,
            overlap[0], overlap[1], u, work, b, ctypes.byref(rm), ctypes.byref(bm))
    else:
        k = getattr(_load(), f"oracle_solve_step_mt_{_sfx(u)}")(
            n, ld, _real(u)(r), m, tol, max_sweeps, depth, tile_x, tile_y,
            overlap[0], overlap[1], u, work, b, ctypes.byref(rm), ctypes.byref(bm),
            int(threads))
    return int(k), _real(u)(rm.value), _real(u)(bm.value)


def run(u0, g, r, *, steps=10, m=8, tol=1e-5, max_sweeps=1 << 22, depth=0,
        tile_x=32, tile_y=8, overlap=(0, 0), n=None, threads=1):
    """Run `steps` backward-Euler steps from u⁰. Returns (u_final, sweeps per
    step as a list, b of the last step). Raises on a negative status.
    threads > 1: row-parallel synchronous sweeps and residuals (same bits)."""
    ld = _check(u0, g)
    n = u0.shape[0] if n is None else n
    u = u0.copy()
    work = u0.copy()
    b = np.zeros_like(u0)
    counts = np.zeros(steps, dtype=np.int64)
    if threads <= 1:
        rc = getattr(_load(), f"oracle_run_{_sfx(u)}")(
            n, ld, _real(u)(r), m, tol, max_sweeps, depth, tile_x, tile_y,
            overlap[0], overlap[1], steps, u, g, work, b, counts)
    else:
        rc = getattr(_load(), f"oracle_run_mt_{_sfx(u)}")(
            n, ld, _real(u)(r), m, tol, max_sweeps, depth, tile_x, tile_y,
            overlap[0], overlap[1], steps, u, g, work, b, counts, int(threads))
    if rc < 0:
        raise RuntimeError(f"oracle run failed with status {rc}: {counts.tolist()}")
    return u, counts.tolist(), b


def check_interval(m: int, sweeps_per_launch: int) -> int:
    """Sweeps between residual checks: lcm(m, sweeps per launch)."""
    import math
    return m * sweeps_per_launch // math.gcd(m, sweeps_per_launch)
