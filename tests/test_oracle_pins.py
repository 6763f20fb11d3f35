"""Pins of the oracle against facts fixed by the page and by mathematics.

The oracle restates "Synchronous vs block-async Jacobi on one RTX 5050",
sections 01 "The problem" and 02 "Method". None of these checks re-types its
arithmetic: each compares it with something independent of it -- a float64
dense direct solve of the backward-Euler system, an invariant of the exact
iteration (maximum principle, mirror symmetry, contraction), a closed form,
brute force on tiny inputs, or the sweep counts the page prints.
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
from temporal_blocked_jacobi_gb300 import problem as P

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden",
                                     "page_numbers.json")))
EPS32 = 2.0 ** -24


# ---------------------------------------------------------------------------
# Independent float64 statement of the linear system (section 01): for every
# interior cell (1+4r) u_ij - r * (sum of interior neighbours) = b_ij + r *
# (sum of Dirichlet neighbours). Assembled as a dense matrix and solved with
# LAPACK (numpy.linalg.solve).
# ---------------------------------------------------------------------------
def dense_system(u, b, r):
    n = u.shape[0]
    m = n - 2
    idx = lambda i, j: (i - 1) * m + (j - 1)
    A = np.zeros((m * m, m * m))
    rhs = np.zeros(m * m)
    for i in range(1, n - 1):
        for j in range(1, n - 1):
            k = idx(i, j)
            A[k, k] = 1.0 + 4.0 * r
            rhs[k] = float(b[i, j])
            for (a, c) in ((i - 1, j), (i + 1, j), (i, j - 1), (i, j + 1)):
                if 1 <= a <= n - 2 and 1 <= c <= n - 2:
                    A[k, idx(a, c)] = -r
                else:
                    rhs[k] += r * float(u[a, c])
    return A, rhs


def interior(a):
    n = a.shape[0]
    return np.asarray(a[1:n - 1, 1:n - 1], dtype=np.float64)


def exact_solution(u, b, r):
    A, rhs = dense_system(u, b, r)
    m = u.shape[0] - 2
    return np.linalg.solve(A, rhs).reshape(m, m), A, rhs


def true_residual64(u, b, r):
    """b_I - A u in float64 from the (float32) iterate u."""
    A, rhs = dense_system(u, b, r)
    return rhs - A @ interior(u).ravel(), rhs


def problem(n, r, kind, seed=None, center=None, ld=None):
    u0 = P.initial_field(n, ld)
    g = P.source_term(n, ld, kind, center=center)
    if seed is not None:  # a generic warm start uⁿ
        u0 = P.random_field(n, ld, seed)
    return u0, g


# ---------------------------------------------------------------------------
# 1. Dense direct solve
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("n", [16, 17, 32])
@pytest.mark.parametrize("r", [0.5, 1.0, 10.0, 100.0])
@pytest.mark.parametrize("kind", ["point", "gauss"])
def test_float64_oracle_matches_dense_solve(n, r, kind):
    u0, g = problem(n, r, kind, seed=n)
    u = u0.astype(np.float64)
    b = oracle.rhs(u, g.astype(np.float64))
    ustar, _, _ = exact_solution(u, b, r)
    k, rmax, bmax = oracle.solve_step(u, b, r, tol=1e-13)
    assert k > 0
    err = np.abs(interior(u) - ustar).max()
    assert err <= 1e-10 * np.abs(ustar).max()


@pytest.mark.parametrize("n", [16, 31])
@pytest.mark.parametrize("r", [1.0, 10.0, 100.0])
@pytest.mark.parametrize("kind", ["point", "gauss"])
def test_float32_oracle_error_bounded_by_residual(n, r, kind):
    """A is strictly diagonally dominant with every row sum >= 1, so
    ||A^-1||inf <= 1 and ||u - u*|| <= ||b - Au|| (section 01). The float32
    stopping rule leaves rho < 1e-5; the exact residual of the float32 iterate
    differs from the float32 difference form by the rounding of J."""
    u0, g = problem(n, r, kind)
    b = oracle.rhs(u0, g)
    u = u0.copy()
    k, rmax, bmax = oracle.solve_step(u, b, r)
    assert k > 0 and k % 8 == 0
    assert float(rmax) < 1e-5 * float(bmax) or rmax == 0
    ustar, _, _ = exact_solution(u0.astype(np.float64), b.astype(np.float64), r)
    err = np.abs(interior(u) - ustar).max()
    d = 1 + 4 * r
    rounding = d * 8 * EPS32 * max(np.abs(ustar).max(), 100.0)
    assert err <= float(rmax) + rounding


# ---------------------------------------------------------------------------
# 2. Maximum principle and contraction of the exact iteration
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("r", [1.0, 10.0, 100.0])
@pytest.mark.parametrize("kind", ["point", "gauss"])
def test_maximum_principle_every_sweep(r, kind):
    """J(u) is a weighted mean of b and the four neighbours with weights
    1/(1+4r) and r/(1+4r); with b >= 0 every iterate stays in
    [0, max(100, max b)] (rounding is monotone; allow 4 ulp at the top)."""
    n = 40
    u0, g = problem(n, r, kind)
    b = oracle.rhs(u0, g)
    top = max(100.0, float(b.max()))
    u = u0
    for _ in range(60):
        u = oracle.sweep(u, b, r)
        inner = interior(u)
        assert inner.min() >= 0.0
        assert inner.max() <= top * (1 + 4 * EPS32)


@pytest.mark.parametrize("r", [0.25, 1.0, 10.0, 100.0])
def test_contraction_bound_float64(r):
    """||u_{k+1} - u*||inf <= (4r/(1+4r)) ||u_k - u*||inf (section 01)."""
    n = 20
    u0, g = problem(n, r, "gauss", seed=3)
    u = u0.astype(np.float64)
    b = oracle.rhs(u, g.astype(np.float64))
    ustar, _, _ = exact_solution(u, b, r)
    q = 4 * r / (1 + 4 * r)
    prev = np.abs(interior(u) - ustar).max()
    for _ in range(40):
        u = oracle.sweep(u, b, r)
        cur = np.abs(interior(u) - ustar).max()
        assert cur <= q * prev * (1 + 1e-12) + 1e-12
        prev = cur


# ---------------------------------------------------------------------------
# 3. Mirror symmetry of centred problems
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("n", [33, 65])
@pytest.mark.parametrize("kind", ["point", "gauss"])
@pytest.mark.parametrize("r", [1.0, 100.0])
def test_left_right_mirror_bitwise(n, kind, r):
    """The top boundary, the other edges and a source centred at column
    (N-1)/2 are symmetric under j -> N-1-j; the neighbour sum pairs W with E,
    so every sweep maps bit for bit under the mirror."""
    c = (n - 1) / 2
    u0, g = problem(n, r, kind, center=(c, c), ld=n)
    assert np.array_equal(g, g[:, ::-1])
    b = oracle.rhs(u0, g)
    u = u0
    for _ in range(24):
        u = oracle.sweep(u, b, r)
        assert np.array_equal(u, u[:, ::-1])
    uf, counts, _ = oracle.run(u0, g, r, steps=3)
    assert np.array_equal(uf, uf[:, ::-1])


# ---------------------------------------------------------------------------
# 4. Closed forms and special cases
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("r", [1.0, 10.0, 100.0, 0.3])
@pytest.mark.parametrize("g_val", [0.0, 1000.0, 7.25])
def test_single_unknown_closed_form(r, g_val):
    """N = 3 has one unknown whose neighbours are all ring cells (top 100):
    (1+4r) x = b + 100 r. One sweep reaches the float32 fixed point, which is
    the correctly rounded quotient of the rounded numerator."""
    n = 3
    u0 = P.initial_field(n, 4)
    g = np.zeros_like(u0)
    g[1, 1] = g_val
    b = oracle.rhs(u0, g)
    assert b[1, 1] == np.float32(g_val)
    r32 = np.float32(r)
    d = Fraction(1) + Fraction(4) * Fraction(float(r32))
    num = Fraction(float(b[1, 1])) + Fraction(100) * Fraction(float(r32))
    x_exact = num / d
    u1 = oracle.sweep(u0, b, r)
    x = u1[1, 1]
    ulp = np.spacing(np.float32(x))
    # within 1 ulp + the rounding of the numerator (relative 2^-24)
    assert abs(Fraction(float(x)) - x_exact) <= Fraction(float(ulp)) + x_exact * Fraction(1, 1 << 23)
    u2 = oracle.sweep(u1, b, r)
    assert u2[1, 1] == x
    rmax, bmax = oracle.residual(u1, b, r)
    assert rmax == 0.0
    k, rm, bm = oracle.solve_step(u0.copy(), b, r)
    assert k == 8 and rm == 0.0


@pytest.mark.parametrize("r", [1.0, 10.0, 100.0])
def test_linear_field_is_exact_fixed_point(r):
    """A field linear in i and j has zero discrete Laplacian, so with g = 0
    (b = u) it solves (1+4r)u - r*sum(nbrs) = u exactly; with small integer
    values every float32 operation is exact, so one sweep returns it bit for
    bit and the residual is exactly 0. A dropped or duplicated neighbour
    breaks this."""
    n = 24
    ii, jj = np.meshgrid(np.arange(n), np.arange(n), indexing="ij")
    u = (3 * ii + 2 * jj + 5).astype(np.float32)
    b = oracle.rhs(u, np.zeros_like(u))
    u1 = oracle.sweep(u, b, r)
    assert np.array_equal(u1, u)
    rmax, bmax = oracle.residual(u, b, r)
    assert rmax == 0.0


def test_r_zero_gives_b_after_one_sweep():
    n = 19
    u0 = P.random_field(n, 20, seed=7)
    g = P.random_field(n, 20, seed=8)
    b = oracle.rhs(u0, g)
    u1 = oracle.sweep(u0, b, 0.0)
    assert np.array_equal(interior(u1), interior(b))


def test_zero_problem_converges_at_first_check():
    n = 30
    u0 = P.initial_field(n, top=0.0)
    g = P.source_term(n, kind="zero")
    b = oracle.rhs(u0, g)
    k, rmax, bmax = oracle.solve_step(u0, b, 10.0)
    assert k == 8 and rmax == 0.0 and bmax == 0.0
    assert not interior(u0).any()


def test_rhs_is_elementwise_float32_sum():
    n = 37
    u = P.random_field(n, 40, seed=1)
    g = P.random_field(n, 40, seed=2)
    b = oracle.rhs(u, g)
    assert np.array_equal(interior(b), interior(u + g))
    assert not b[0].any() and not b[-1].any()


# ---------------------------------------------------------------------------
# 5. Residual in the difference form
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("r", [1.0, 10.0, 100.0])
@pytest.mark.parametrize("sweeps", [0, 5, 40])
def test_residual_matches_float64_definition(r, sweeps):
    """rmax = ||b_I - A u||inf of the float32 iterate, up to the rounding of
    J (5 roundings, |J| <= max|u|) scaled by d; bmax = ||b_I||inf where b_I
    carries the Dirichlet neighbours, up to one rounding."""
    n = 26
    u0, g = problem(n, r, "gauss", seed=11)
    b = oracle.rhs(u0, g)
    u = oracle.sweeps(u0, b, r, sweeps)
    rmax, bmax = oracle.residual(u, b, r)
    res64, rhs64 = true_residual64(u, b, r)
    d = 1 + 4 * r
    bound = d * 8 * EPS32 * max(float(np.abs(u).max()), float(np.abs(b).max()))
    assert abs(float(rmax) - np.abs(res64).max()) <= bound
    assert abs(float(bmax) - np.abs(rhs64).max()) <= 2 * EPS32 * np.abs(rhs64).max()


def test_residual_zero_at_fixed_point_and_nan_propagates():
    n = 12
    u0, g = problem(n, 1.0, "point")
    b = oracle.rhs(u0, g)
    u = u0.copy()
    # iterate to the float32 fixed point
    for _ in range(2000):
        nu = oracle.sweep(u, b, 1.0)
        if np.array_equal(nu, u):
            break
        u = nu
    rmax, _ = oracle.residual(u, b, 1.0)
    assert rmax == 0.0
    g[5, 5] = np.nan
    bn = oracle.rhs(u0, g)
    rmax, bmax = oracle.residual(u0, bn, 1.0)
    assert math.isnan(rmax) and math.isnan(bmax)
    k, _, _ = oracle.solve_step(u0.copy(), bn, 1.0)
    assert k == -4


def test_sweep_cap_reports_not_converged():
    u0, g = problem(64, 100.0, "point")
    b = oracle.rhs(u0, g)
    k, _, _ = oracle.solve_step(u0.copy(), b, 100.0, max_sweeps=16)
    assert k == -3


# ---------------------------------------------------------------------------
# 6. Sweep counts per step, printed in section 01
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("n", [256, 512])
@pytest.mark.parametrize("r,key,rel", [(1.0, "r1", 0.10), (10.0, "r10", 0.02),
                                       (100.0, "r100", 0.02)])
def test_sweeps_per_step_match_page(n, r, key, rel):
    """About 35 / 226 / 1417 sweeps per step for r = 1 / 10 / 100,
    independent of N. With the point source and ||b|| taken over the
    interior system's right-hand side, the oracle gives 32.8 / 225.6 / 1412
    (N=256) and 1416 (N=512). The r = 1 figure is given to ~2 digits and the
    counts are multiples of M = 8, hence the wider band."""
    if n == 512 and r != 100.0:
        pytest.skip("N-independence at r=1, 10 is covered by N=256 vs the page")
    u0, g = problem(n, r, "point")
    _, counts, _ = oracle.run(u0, g, r)
    assert all(c % 8 == 0 for c in counts)
    mean = sum(counts) / len(counts)
    target = GOLDEN["sweeps_per_step"][key]
    assert abs(mean - target) <= rel * target, (counts, mean, target)


def test_sweep_counts_grow_with_r_not_n():
    means = {}
    for n in (128, 256):
        u0, g = problem(n, 10.0, "point")
        _, counts, _ = oracle.run(u0, g, 10.0)
        means[n] = sum(counts) / len(counts)
    assert abs(means[128] - means[256]) <= 8


# ---------------------------------------------------------------------------
# 7. Block-asynchronous emulator (section 02 "Block-asynchronous")
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("n,tx,ty", [(70, 32, 8), (37, 8, 4), (70, 32, 16)])
def test_ba_depth1_is_one_sync_sweep(n, tx, ty):
    u = P.random_field(n, None, seed=n)
    b = oracle.rhs(u, P.random_field(n, None, seed=n + 1))
    assert np.array_equal(oracle.ba_launch(u, b, 10.0, tx, ty, 1),
                          oracle.sweep(u, b, 10.0))


@pytest.mark.parametrize("depth", [2, 4, 8])
def test_ba_single_tile_equals_depth_sync_sweeps(depth):
    """One tile covering the whole interior has only ring cells as halo,
    which are fixed anyway: D in-tile sweeps are D synchronous sweeps."""
    n = 30
    u = P.random_field(n, 32, seed=depth)
    b = oracle.rhs(u, P.random_field(n, 32, seed=99))
    got = oracle.ba_launch(u, b, 1.0, 64, 64, depth)
    assert np.array_equal(got, oracle.sweeps(u, b, 1.0, depth))


def test_ba_frozen_halo_brute_force():
    """4x4 interior cut into 2x2 tiles, two in-tile sweeps. Each tile sees its
    halo as the values at launch. Written out cell by cell with float32
    scalar operations in the section's update (b + r*sum)/(1+4r)."""
    n, r, D = 6, np.float32(2.5), 2
    u = P.random_field(n, 8, seed=5)
    b = oracle.rhs(u, P.random_field(n, 8, seed=6))
    f = np.float32
    d = f(f(1) + f(f(4) * r))
    expect = u.copy()
    for ty0 in (1, 3):
        for tx0 in (1, 3):
            cur = {(i, j): u[i, j] for i in range(ty0 - 1, ty0 + 3)
                   for j in range(tx0 - 1, tx0 + 3)}
            for _ in range(D):
                new = dict(cur)
                for i in (ty0, ty0 + 1):
                    for j in (tx0, tx0 + 1):
                        s = f(f(cur[i, j - 1] + cur[i, j + 1])
                              + f(cur[i - 1, j] + cur[i + 1, j]))
                        new[i, j] = f(f(b[i, j] + f(r * s)) / d)
                cur = new
            for i in (ty0, ty0 + 1):
                for j in (tx0, tx0 + 1):
                    expect[i, j] = cur[i, j]
    got = oracle.ba_launch(u, b, float(r), 2, 2, D)
    assert np.array_equal(got, expect)
    assert not np.array_equal(got, oracle.sweeps(u, b, float(r), D))


def test_ba_mirror_symmetric_tiling():
    """Interior width 64 = 2 tiles of 32: the tiling is mirror symmetric, so
    a centred Gaussian keeps the iterates mirror symmetric bit for bit."""
    n = 66
    c = (n - 1) / 2
    u0 = P.initial_field(n, n)
    g = P.source_term(n, n, "gauss", center=(c, c))
    b = oracle.rhs(u0, g)
    u = u0
    for _ in range(6):
        u = oracle.ba_launch(u, b, 10.0, 32, 8, 4)
        assert np.array_equal(u, u[:, ::-1])


def test_ba_sweep_ratio_matches_page():
    """D8 on 32x16 tiles at r = 10 needs 1.738x the synchronous sweeps
    (section 05); D1 needs exactly as many (section 04)."""
    n, r = 512, 10.0
    u0, g = problem(n, r, "point")
    _, c_sync, _ = oracle.run(u0, g, r)
    _, c_ba, _ = oracle.run(u0, g, r, depth=8, tile_x=32, tile_y=16)
    s = sum(c_ba) / sum(c_sync)
    target = GOLDEN["block_async_sweep_ratio_d8_32x16_r10"]["value"]
    assert abs(s - target) <= 0.015 * target, s
    assert all(c % 8 == 0 for c in c_ba)


def test_ba_depth1_solve_equals_sync_solve():
    n, r = 64, 10.0
    u0, g = problem(n, r, "gauss")
    u_s, c_s, _ = oracle.run(u0, g, r)
    u_b, c_b, _ = oracle.run(u0, g, r, depth=1, tile_x=32, tile_y=8)
    assert c_s == c_b and np.array_equal(u_s, u_b)


def test_check_interval_for_deep_launches():
    """A 16-sweep launch cannot stop after 8 sweeps: the residual is read
    every lcm(8, 16) = 16 sweeps, and synchronous sweeps checked every 16
    give the same counts and field."""
    assert oracle.check_interval(8, 16) == 16
    assert oracle.check_interval(8, 4) == 8
    n, r = 48, 10.0
    u0, g = problem(n, r, "point")
    _, c16, _ = oracle.run(u0, g, r, m=16)
    assert all(c % 16 == 0 for c in c16)
