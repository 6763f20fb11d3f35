"""The row-parallel oracle (threads > 1) against the single-threaded oracle of
record. A synchronous sweep reads only the previous iterate, so its cells can
be computed in any order by any thread with the same code, and the residual's
maxima do not depend on the order in which they are taken: the threaded run
must reproduce the single-threaded one bit for bit, sweep counts included.
It exists to check full ten-step solves on large grids in reasonable time.
No GPU."""
import numpy as np
import pytest

import oracle
from temporal_blocked_jacobi_gb300 import problem as P


def bits(a):
    return np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)


@pytest.mark.parametrize("n,r,source", [(17, 1.0, "point"), (64, 10.0, "gauss"),
                                        (130, 100.0, "gauss"), (131, 10.0, "point")])
@pytest.mark.parametrize("threads", [2, 3, 7])
def test_threaded_run_matches_one_thread(n, r, source, threads):
    u0 = P.initial_field(n)
    g = P.source_term(n, kind=source)
    want_u, want_k, want_b = oracle.run(u0, g, r, steps=3)
    got_u, got_k, got_b = oracle.run(u0, g, r, steps=3, threads=threads)
    assert got_k == want_k
    assert np.array_equal(bits(got_u), bits(want_u))
    assert np.array_equal(bits(got_b), bits(want_b))


def test_more_threads_than_rows():
    u0 = P.initial_field(5)
    g = P.source_term(5, kind="point")
    want_u, want_k, _ = oracle.run(u0, g, 10.0, steps=2)
    got_u, got_k, _ = oracle.run(u0, g, 10.0, steps=2, threads=64)
    assert got_k == want_k and np.array_equal(bits(got_u), bits(want_u))


@pytest.mark.parametrize("row", [1, 40, 62])
def test_threaded_residual_propagates_nan_from_any_rows(row):
    """A NaN in the rows of any thread reaches the norm: solve_step stops with
    the non-finite status at the first check, as with one thread."""
    n = 64
    u = P.random_field(n, seed=3)
    b = P.random_field(n, seed=4)
    u[row, 17] = np.nan
    one = oracle.solve_step(u.copy(), b, 10.0, max_sweeps=8)
    many = oracle.solve_step(u.copy(), b, 10.0, max_sweeps=8, threads=5)
    assert one[0] == many[0] == -4


def test_threaded_solve_step_norms_match():
    n = 96
    u = P.random_field(n, seed=5)
    b = P.random_field(n, seed=6)
    u1, u2 = u.copy(), u.copy()
    k1, rm1, bm1 = oracle.solve_step(u1, b, 100.0, max_sweeps=64)
    k2, rm2, bm2 = oracle.solve_step(u2, b, 100.0, max_sweeps=64, threads=4)
    assert k1 == k2 == -3  # not converged in 64 sweeps at r = 100
    assert bits(np.float32(rm1)) == bits(np.float32(rm2))
    assert bits(np.float32(bm1)) == bits(np.float32(bm2))
    assert np.array_equal(bits(u1), bits(u2))
