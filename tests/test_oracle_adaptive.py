"""Pins of the adaptive-depth oracle, and the library's depth controller
(host code, no GPU) against it.

Source: "Synchronous vs block-async Jacobi on one RTX 5050", section 02
(G-asc, G-desc: D stepped as rho passes 1e-2, 1e-3, 1e-4, latched; G-fb:
start at D = 1, double while -ln(rho_k/rho_{k-1}) per ms holds, halve on a
drop of more than 10 %, skip the bump right after each change).
"""
import math

import numpy as np
import pytest

import oracle
from oracle import adaptive
from temporal_blocked_jacobi_gb300 import problem as P


# -- hand-worked sequences ------------------------------------------------
RHOS = [0.5, 0.02, 0.009, 0.05, 0.0009, 0.00009, 0.5]


@pytest.mark.parametrize("policy,dmax,want", [
    # rho falls below 1e-2 at the third check, 1e-3 at the fifth, 1e-4 at the
    # sixth; the rise to 0.05 and 0.5 changes nothing (latched)
    ("g_asc", 8, [1, 1, 1, 2, 2, 4, 8, 8]),
    ("g_desc", 8, [8, 8, 8, 4, 4, 2, 1, 1]),
    # a shorter ladder saturates; a longer one is not reached by 3 thresholds
    ("g_asc", 4, [1, 1, 1, 2, 2, 4, 4, 4]),
    ("g_desc", 16, [16, 16, 16, 8, 8, 4, 2, 2]),
    ("g_asc", 16, [1, 1, 1, 2, 2, 4, 8, 8]),
])
def test_threshold_controllers_hand_worked(policy, dmax, want):
    assert adaptive.depths(policy, dmax, RHOS, [1.0] * len(RHOS)) == want


def test_threshold_controller_skips_levels():
    # one check from 0.5 straight to 5e-5 crosses all three thresholds
    assert adaptive.depths("g_asc", 8, [0.5, 5e-5], [1, 1]) == [1, 1, 8]
    assert adaptive.depths("g_desc", 8, [0.5, 5e-5], [1, 1]) == [8, 8, 1]
    # exactly at a threshold is not below it
    assert adaptive.depths("g_asc", 8, [1e-2], [1]) == [1, 1]


def rhos_from_rates(rates, rho0=0.5, ms=1.0):
    """rho_k with -ln(rho_k / rho_{k-1}) / ms = rates[k-1]."""
    out, rho = [rho0], rho0
    for rate in rates:
        rho = rho * math.exp(-rate * ms)
        out.append(rho)
    return out


def test_feedback_controller_hand_worked():
    # check 1 has no rate; then the rates below, 1 ms per interval
    rates = [1.0, 5.0, 1.0, 0.1, 0.8, 3.0, 0.95, 2.0, 1.0, 7.0, 1.0, 0.5]
    rhos = rhos_from_rates(rates)
    got = adaptive.depths("g_fb", 8, rhos, [1.0] * len(rhos))
    want = [1,      # start
            1,      # first check: nothing to compare
            2,      # first rate: double
            2,      # settling (5.0 ignored)
            4,      # 1.0 >= 0.9 * 1.0: holds, double
            4,      # settling
            2,      # 0.8 < 0.9 * 1.0: drop, halve
            2,      # settling
            4,      # 0.95 >= 0.9 * 0.8: holds
            4,      # settling
            8,      # 1.0 >= 0.9 * 0.95: holds
            8,      # settling
            8,      # holds, but 16 > depth_max: stays, no settling
            4]      # 0.5 < 0.9: halve
    assert got == want


def test_feedback_controller_time_matters():
    # the same rho sequence with the second interval twice as long: its rate
    # per ms halves, a drop
    rhos = rhos_from_rates([1.0, 9.0, 1.0])
    assert adaptive.depths("g_fb", 8, rhos, [1.0, 1.0, 1.0, 1.0]) == [1, 1, 2, 2, 4]
    assert adaptive.depths("g_fb", 8, rhos, [1.0, 1.0, 1.0, 2.0]) == [1, 1, 2, 2, 1]


def test_feedback_controller_rising_residual_halves():
    # rates ln2 (double), skipped, ln2 (holds: double), skipped, -ln2 (drop)
    rhos = [0.5, 0.25, 0.2, 0.1, 0.2, 0.4]
    assert adaptive.depths("g_fb", 8, rhos, [1] * 6) == [1, 1, 2, 2, 4, 4, 2]


def test_feedback_controller_ignores_unmeasurable_checks():
    assert adaptive.depths("g_fb", 8, [0.5, 0.0, 0.1], [1, 1, 1]) == [1, 1, 1, 1]
    assert adaptive.depths("g_fb", 8, [0.5, 0.25], [1, 0.0]) == [1, 1, 1]
    assert adaptive.depths("g_fb", 8, [0.5, float("nan"), 0.25], [1, 1, 1]) == [1, 1, 1, 1]


# -- invariants on random sequences ---------------------------------------
def random_sequence(seed, n=200):
    rng = np.random.default_rng(seed)
    rhos = 10.0 ** rng.uniform(-6, 0, n)
    mss = rng.uniform(0.01, 2.0, n)
    return rhos.tolist(), mss.tolist()


@pytest.mark.parametrize("seed", range(20))
@pytest.mark.parametrize("dmax", [2, 4, 8, 16])
def test_controller_invariants(seed, dmax):
    rhos, mss = random_sequence(seed)
    ladder = {1 << k for k in range(dmax.bit_length())}
    asc = adaptive.depths("g_asc", dmax, rhos, mss)
    desc = adaptive.depths("g_desc", dmax, rhos, mss)
    fb = adaptive.depths("g_fb", dmax, rhos, mss)
    assert all(a <= b for a, b in zip(asc, asc[1:]))
    assert all(a >= b for a, b in zip(desc, desc[1:]))
    for seq in (asc, desc, fb):
        assert set(seq) <= ladder
    # G-fb moves one rung at a time, and never twice in a row
    for a, b in zip(fb, fb[1:]):
        assert b in (a, 2 * a, a // 2)
    for a, b, c in zip(fb, fb[1:], fb[2:]):
        assert not (a != b and b != c)


# -- the library's controller (host code) equals the oracle's --------------
@pytest.fixture(scope="module")
def lib():
    from temporal_blocked_jacobi_gb300 import _build, jacobi
    _build.build()
    return jacobi


@pytest.mark.parametrize("seed", range(30))
@pytest.mark.parametrize("policy", ["g_asc", "g_desc", "g_fb"])
@pytest.mark.parametrize("dmax", [2, 8, 16])
def test_library_controller_matches_oracle(lib, seed, policy, dmax):
    rhos, mss = random_sequence(100 + seed)
    if seed % 3 == 0:   # smooth decay with noise: the usual shape in a solve
        rng = np.random.default_rng(seed)
        rates = np.abs(rng.normal(1.0, 0.15, 200))
        rhos = rhos_from_rates(rates.tolist(), ms=0.3)[1:]
        mss = [0.3] * len(rhos)
    assert lib.adapt_depths(policy, dmax, rhos, mss) == \
        adaptive.depths(policy, dmax, rhos, mss)


def test_library_controller_rejects_bad_arguments(lib):
    with pytest.raises(lib.JacobiError):
        lib.adapt_depths("g_fb", 3, [], [])
    with pytest.raises(lib.JacobiError):
        lib.adapt_depths(7, 8, [], [])


# -- the adaptive solve reduces to the fixed-depth one ---------------------
def problem(n, source, r):
    u0 = P.initial_field(n)
    g = P.source_term(n, kind=source)
    return u0, oracle.rhs(u0, g)


@pytest.mark.parametrize("depth", [1, 2, 4, 8])
@pytest.mark.parametrize("tile", [(32, 8), (8, 4)])
def test_constant_schedule_is_fixed_depth_solve(depth, tile):
    n, r = 40, 10.0
    u0, b = problem(n, "gauss", r)
    u_fixed = u0.copy()
    k_fixed, _, _ = oracle.solve_step(u_fixed, b, r, depth=depth,
                                      tile_x=tile[0], tile_y=tile[1])
    u = u0.copy()
    k, trace = adaptive.solve_step(u, b, r, policy="g_fb", depth_max=8,
                                   tile_x=tile[0], tile_y=tile[1],
                                   schedule=[depth] * 100000)
    assert k == k_fixed
    assert np.array_equal(u.view(np.uint32), u_fixed.view(np.uint32))
    assert [t[1] for t in trace] == list(range(8, k + 1, 8))


def test_depth_one_schedule_is_synchronous():
    n, r = 33, 1.0
    u0, b = problem(n, "point", r)
    u_sync = u0.copy()
    k_sync, _, _ = oracle.solve_step(u_sync, b, r)
    u = u0.copy()
    k, _ = adaptive.solve_step(u, b, r, policy="g_asc", depth_max=8,
                               schedule=[1] * 100000)
    assert k == k_sync
    assert np.array_equal(u.view(np.uint32), u_sync.view(np.uint32))


@pytest.mark.parametrize("policy", ["g_asc", "g_desc"])
def test_adaptive_solve_follows_its_controller(policy):
    """The solve's depth sequence is the controller's answer to the solve's
    own residuals, and the answer satisfies the stopping rule."""
    n, r = 48, 10.0
    u0, b = problem(n, "gauss", r)
    u = u0.copy()
    k, trace = adaptive.solve_step(u, b, r, policy=policy, depth_max=8)
    assert k > 0
    rhos = [float(rm) / float(bm) for _, _, rm, bm in trace]
    want = adaptive.depths(policy, 8, rhos[:-1], [0.0] * (len(rhos) - 1))
    assert [t[0] for t in trace] == want
    rm, bm = oracle.residual(u, b, r)
    assert float(rm) < 1e-5 * float(bm)
