"""JACOBI_CONTROL_PERSISTENT: a whole time step of exact temporal blocking as
one cooperative launch, rounds of D sweeps separated by grid-wide barriers
("Synchronous vs block-async Jacobi on one RTX 5050", sections 01-02: the
synchronization that costs time is moved onto the device). Same iterates,
sweep counts and statuses as the oracle and as the other controls."""
import numpy as np
import pytest

import oracle
from temporal_blocked_jacobi_gb300 import problem as P
from tests.gpu_helpers import gpu_run, mismatch, same_bits, to_dev, workload

pytestmark = pytest.mark.gpu


def _jacobi():
    from temporal_blocked_jacobi_gb300 import jacobi
    return jacobi


@pytest.mark.parametrize("n", [17, 70, 300])
@pytest.mark.parametrize("depth", [4, 8, 16])
def test_persistent_run_bit_exact(n, depth):
    """Grids of one tile, a few tiles and many ragged tiles: the field and
    the sweep counts of three steps equal the oracle's."""
    u0, g = workload(n, "gauss")
    ref_u, ref_k, _ = oracle.run(u0, g, 10.0, steps=3, m=max(8, depth))
    got_u, got_k, _ = gpu_run(u0, g, 10.0, steps=3, strategy="etb", depth=depth,
                              control="persistent")
    assert got_k == ref_k
    assert same_bits(got_u, ref_u), mismatch(got_u, ref_u)


@pytest.mark.parametrize("depth,tile", [(4, (120, 88)), (8, (112, 80)), (8, (112, 92)),
                                        (16, (96, 64)), (16, (96, 76))])
def test_persistent_register_shapes_bit_exact(depth, tile):
    """Every register-resident tile shape, selected by its size, on a grid of
    many ragged tiles."""
    u0, g = workload(300, "gauss")
    ref_u, ref_k, _ = oracle.run(u0, g, 10.0, steps=2, m=max(8, depth))
    got_u, got_k, _ = gpu_run(u0, g, 10.0, steps=2, strategy="etb", depth=depth,
                              tile=tile, control="persistent")
    assert got_k == ref_k
    assert same_bits(got_u, ref_u), mismatch(got_u, ref_u)


@pytest.mark.parametrize("depth", [4, 8])
def test_persistent_n2048_r10_gauss_bit_exact(depth):
    u0, g = workload(2048, "gauss")
    ref_u, ref_k, _ = oracle.run(u0, g, 10.0)
    got_u, got_k, _ = gpu_run(u0, g, 10.0, strategy="etb", depth=depth,
                              control="persistent")
    assert got_k == ref_k
    assert same_bits(got_u, ref_u), mismatch(got_u, ref_u)


@pytest.mark.parametrize("depth", [4, 8])
def test_persistent_solve_step_matches_device_loop(depth):
    """jacobi_solve_step (one step graph) and jacobi_run (one run graph)
    agree with the device-side WHILE loop, step by step."""
    import torch
    jacobi = _jacobi()
    n, r = 300, 1.0
    u0, g = workload(n, "point")
    results = {}
    for control in ("device", "persistent"):
        u, u_alt, b = jacobi.allocate(n, u0.shape[1])
        u.copy_(to_dev(u0))
        ks = []
        with jacobi.Solver(u, u_alt, b, r, strategy="etb", depth=depth,
                           control=control) as s:
            for _ in range(3):
                s.rhs(to_dev(g))
                ks.append(s.solve_step())
            ks += s.run(to_dev(g), 2)
        torch.cuda.synchronize()
        results[control] = (ks, u.cpu().numpy())
    assert results["device"][0] == results["persistent"][0]
    assert same_bits(results["device"][1], results["persistent"][1])


def test_persistent_unsupported_combinations():
    jacobi = _jacobi()
    n = 70
    u0, _ = workload(n, "gauss")
    u, u_alt, b = jacobi.allocate(n, u0.shape[1])
    u.copy_(to_dev(u0))
    for kw in ({"strategy": "sync", "depth": 1}, {"strategy": "ba", "depth": 4},
               {"strategy": "etb", "depth": 2},
               {"strategy": "etb", "depth": 4, "tile": (120, 56)}):
        with pytest.raises(jacobi.JacobiError) as ei:
            jacobi.Solver(u, u_alt, b, 1.0, control="persistent", **kw)
        assert ei.value.status == jacobi.ERR_UNSUPPORTED


def test_persistent_nan_source_reports_nonfinite():
    jacobi = _jacobi()
    n = 64
    u0, g = workload(n, "gauss")
    g[10, 12] = np.nan
    u, u_alt, b = jacobi.allocate(n, u0.shape[1])
    u.copy_(to_dev(u0))
    with jacobi.Solver(u, u_alt, b, 1.0, strategy="etb", depth=4,
                       control="persistent") as s:
        s.rhs(to_dev(g))
        assert s.solve_step(raise_on_error=False) == jacobi.ERR_NONFINITE


@pytest.mark.parametrize("depth", [4, 8])
def test_persistent_run_stops_at_failing_step(depth):
    """Step 2's right-hand side overflows: step 1 converges, step 2 reports
    JACOBI_ERR_NONFINITE with u at its last checked iterate, later steps are
    skipped on the device, and the handle works afterwards."""
    import ctypes
    import torch
    jacobi = _jacobi()
    n, r = 40, 1.0
    u0 = P.initial_field(n)
    g = P.source_term(n, kind="zero")
    g[20, 20] = np.float32(2e38)
    ref = u0.copy()
    ref_k = []
    for _ in range(4):
        bb = oracle.rhs(ref, g)
        k, _, _ = oracle.solve_step(ref, bb, r)
        ref_k.append(k)
        if k < 0:
            break
    assert ref_k[0] > 0 and ref_k[1] == jacobi.ERR_NONFINITE
    u, u_alt, b = jacobi.allocate(n, u0.shape[1])
    u.copy_(to_dev(u0))
    g_dev = to_dev(g)
    with jacobi.Solver(u, u_alt, b, r, strategy="etb", depth=depth,
                       control="persistent") as s:
        counts = (ctypes.c_longlong * 4)()
        total = jacobi.load().jacobi_run(s.handle, ctypes.c_void_p(g_dev.data_ptr()),
                                         4, counts)
        assert total == jacobi.ERR_NONFINITE
        assert [counts[0], counts[1]] == ref_k
        torch.cuda.synchronize()
        got = u.cpu().numpy()
        bad = ~np.isfinite(ref)
        assert bad.any()
        assert np.array_equal(~np.isfinite(got), bad)
        assert np.array_equal(got.view(np.uint32)[~bad], ref.view(np.uint32)[~bad])
        u.copy_(to_dev(u0))
        assert sum(s.run(to_dev(P.source_term(n, kind="gauss")), 2)) > 0


def test_persistent_max_sweeps_reports_not_converged():
    jacobi = _jacobi()
    n = 130
    u0, g = workload(n, "gauss")
    u, u_alt, b = jacobi.allocate(n, u0.shape[1])
    u.copy_(to_dev(u0))
    ref = u0.copy()
    bb = oracle.rhs(ref, g)
    k, _, _ = oracle.solve_step(ref, bb, 100.0, max_sweeps=64)
    assert k == jacobi.ERR_NOT_CONVERGED
    with jacobi.Solver(u, u_alt, b, 100.0, strategy="etb", depth=8,
                       control="persistent", max_sweeps=64) as s:
        s.rhs(to_dev(g))
        assert s.solve_step(raise_on_error=False) == jacobi.ERR_NOT_CONVERGED
    got = u.cpu().numpy()
    assert same_bits(got, ref), mismatch(got, ref)
