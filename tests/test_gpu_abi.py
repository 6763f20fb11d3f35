"""Status codes of the C ABI: bad arguments are rejected, the sweep cap and
non-finite residuals are reported, and the handle stays usable after."""
import numpy as np
import pytest

import oracle
from temporal_blocked_jacobi_gb300 import problem as P
from tests.gpu_helpers import mismatch, same_bits, to_dev, workload

pytestmark = pytest.mark.gpu


def _jacobi():
    from temporal_blocked_jacobi_gb300 import jacobi
    return jacobi


def test_invalid_arguments_rejected():
    import torch
    jacobi = _jacobi()
    u, u_alt, b = jacobi.allocate(32, 32)
    with pytest.raises(jacobi.JacobiError) as e:  # ld not a multiple of 4
        x = torch.zeros((32, 34), device="cuda")
        jacobi.Solver(x, x.clone(), x.clone(), 1.0)
    assert e.value.status == jacobi.ERR_INVALID_ARG
    with pytest.raises(jacobi.JacobiError) as e:  # n < 3
        x = torch.zeros((2, 4), device="cuda")
        jacobi.Solver(x, x.clone(), x.clone(), 1.0)
    assert e.value.status == jacobi.ERR_INVALID_ARG
    with pytest.raises(jacobi.JacobiError) as e:  # aliased buffers
        jacobi.Solver(u, u, b, 1.0)
    assert e.value.status == jacobi.ERR_INVALID_ARG
    with pytest.raises(jacobi.JacobiError) as e:  # negative r
        jacobi.Solver(u, u_alt, b, -1.0)
    assert e.value.status == jacobi.ERR_INVALID_ARG
    with pytest.raises(jacobi.JacobiError) as e:  # bad depth
        jacobi.Solver(u, u_alt, b, 1.0, strategy="etb", depth=3)
    assert e.value.status == jacobi.ERR_INVALID_ARG
    with pytest.raises(jacobi.JacobiError) as e:  # box wider than TMA allows
        jacobi.Solver(u, u_alt, b, 1.0, strategy="etb", depth=16, tile=(248, 8))
    assert e.value.status == jacobi.ERR_UNSUPPORTED
    with pytest.raises(jacobi.JacobiError) as e:  # tile_x not a multiple of 4
        jacobi.Solver(u, u_alt, b, 1.0, strategy="ba", depth=4, tile=(30, 8))
    assert e.value.status == jacobi.ERR_INVALID_ARG
    for kw in (dict(strategy="ba", depth=4, overlap=(3, 0)),      # odd
               dict(strategy="ba", depth=4, tile=(8, 8), overlap=(8, 0)),  # >= tile
               dict(strategy="etb", depth=4, overlap=(2, 2)),     # not BA
               dict(strategy="ba", depth=4, overlap=(-2, 0))):
        with pytest.raises(jacobi.JacobiError) as e:
            jacobi.Solver(u, u_alt, b, 1.0, **kw)
        assert e.value.status == jacobi.ERR_INVALID_ARG, kw
    # misaligned (4-byte offset) view
    big = torch.zeros(32 * 32 + 4, device="cuda")
    mis = big[1:1 + 32 * 32].view(32, 32)
    with pytest.raises(jacobi.JacobiError) as e:
        jacobi.Solver(mis, u_alt, b, 1.0)
    assert e.value.status == jacobi.ERR_INVALID_ARG


def test_rhs_mode_checked():
    """The unfused right-hand side is SYNC-only; a solve whose b was prepared
    for the other mode is refused until jacobi_rhs runs again."""
    jacobi = _jacobi()
    n = 40
    u0, g = workload(n, "gauss")
    u, u_alt, b = jacobi.allocate(n, u0.shape[1])
    u.copy_(to_dev(u0))
    with pytest.raises(jacobi.JacobiError) as e:
        jacobi.Solver(u, u_alt, b, 1.0, strategy="etb", depth=4, rhs="unfused")
    assert e.value.status == jacobi.ERR_UNSUPPORTED
    with pytest.raises(jacobi.JacobiError) as e:
        jacobi.Solver(u, u_alt, b, 1.0, rhs=7)
    assert e.value.status == jacobi.ERR_INVALID_ARG
    g_dev = to_dev(g)
    with jacobi.Solver(u, u_alt, b, 1.0) as s:
        s.rhs(g_dev)
        s.set_strategy(rhs="unfused")
        with pytest.raises(jacobi.JacobiError) as e:
            s.solve_step()
        assert e.value.status == jacobi.ERR_INVALID_ARG
        s.rhs(g_dev)
        k_unfused = s.solve_step()
    u.copy_(to_dev(u0))
    with jacobi.Solver(u, u_alt, b, 1.0) as s:
        s.rhs(g_dev)
        assert s.solve_step() == k_unfused


def test_host_buffers_rejected():
    import ctypes
    jacobi = _jacobi()
    lib = jacobi.load()
    hosts = [np.zeros((16, 16), dtype=np.float32) for _ in range(3)]
    h = ctypes.c_void_p()
    p = [a.ctypes.data_as(ctypes.c_void_p) for a in hosts]
    rc = lib.jacobi_create(ctypes.byref(h), 16, 16, 1.0, None, p[0], p[1],
                           p[2], None)
    assert rc == jacobi.ERR_INVALID_ARG
    assert not h.value


@pytest.mark.parametrize("control", ["host", "device"])
@pytest.mark.parametrize("strategy,depth", [("sync", 1), ("etb", 8), ("ba", 4)])
def test_sweep_cap_not_converged_then_recovers(control, strategy, depth):
    import torch
    import oracle
    jacobi = _jacobi()
    n, r = 128, 100.0
    u0, g = workload(n, "point")
    u, u_alt, b = jacobi.allocate(n, u0.shape[1])
    u.copy_(to_dev(u0))
    with jacobi.Solver(u, u_alt, b, r, max_sweeps=24, strategy=strategy,
                       depth=depth, control=control) as s:
        s.rhs(to_dev(g))
        k = s.solve_step(raise_on_error=False)
        assert k == jacobi.ERR_NOT_CONVERGED
        assert "not converged" in s.last_error
        # u holds the iterate at the cap (24 sweeps), as the oracle's does
        if strategy != "ba":
            ref = oracle.sweeps(u0, oracle.rhs(u0, g), r, 24)
            assert np.array_equal(u.cpu().numpy(), ref)
        s.set_strategy(strategy, depth, max_sweeps=1 << 22, control=control)
        assert s.solve_step() > 0
    torch.cuda.synchronize()


@pytest.mark.parametrize("strategy,depth", [("sync", 1), ("etb", 4), ("etb", 8), ("ba", 8)])
def test_device_run_stops_at_failing_step(strategy, depth):
    """jacobi_run under device control is one graph for all steps. With a
    source so large that step 2's right-hand side overflows, step 1
    converges and step 2 reports JACOBI_ERR_NONFINITE with u holding its last
    checked iterate, as the oracle's run leaves it; later steps do nothing
    and the handle works afterwards."""
    import ctypes
    import torch
    import oracle
    jacobi = _jacobi()
    n, r = 40, 1.0
    u0 = P.initial_field(n)
    g = P.source_term(n, kind="zero")
    g[20, 20] = np.float32(2e38)
    ref = u0.copy()
    ref_k = []
    for _ in range(4):
        bb = oracle.rhs(ref, g)
        k, _, _ = oracle.solve_step(ref, bb, r, depth=depth if strategy == "ba" else 0)
        ref_k.append(k)
        if k < 0:
            break
    assert ref_k[0] > 0 and ref_k[1] == jacobi.ERR_NONFINITE
    u, u_alt, b = jacobi.allocate(n, u0.shape[1])
    u.copy_(to_dev(u0))
    g_dev = to_dev(g)
    with jacobi.Solver(u, u_alt, b, r, strategy=strategy, depth=depth,
                       control="device") as s:
        counts = (ctypes.c_longlong * 4)()
        total = jacobi.load().jacobi_run(s.handle, ctypes.c_void_p(g_dev.data_ptr()),
                                         4, counts)
        assert total == jacobi.ERR_NONFINITE
        assert [counts[0], counts[1]] == ref_k
        assert "not finite" in s.last_error
        torch.cuda.synchronize()
        got = u.cpu().numpy()
        # Non-finite at the same cells, every finite cell bit for bit. (Which
        # non-finite value a cell holds may differ: the verified fixed-divisor
        # division is IEEE-exact for finite numerators but turns an infinite
        # one into NaN; NaN payloads differ between GPU and host too.)
        bad = ~np.isfinite(ref)
        assert bad.any()
        assert np.array_equal(~np.isfinite(got), bad)
        assert np.array_equal(got.view(np.uint32)[~bad], ref.view(np.uint32)[~bad])
        u.copy_(to_dev(u0))
        assert sum(s.run(to_dev(P.source_term(n, kind="gauss")), 2)) > 0


def test_device_run_graph_follows_source_and_step_count():
    """The run graph is rebuilt when the source buffer or the number of steps
    changes; each run matches the oracle."""
    import torch
    import oracle
    jacobi = _jacobi()
    n, r = 70, 10.0
    u0, g = workload(n, "gauss")
    g2 = (g * np.float32(0.5)).astype(np.float32)
    u, u_alt, b = jacobi.allocate(n, u0.shape[1])
    u.copy_(to_dev(u0))
    ref = u0.copy()
    with jacobi.Solver(u, u_alt, b, r, strategy="etb", depth=8,
                       control="device") as s:
        for src, steps in ((g, 3), (g2, 3), (g2, 2), (g, 1)):
            got_k = s.run(to_dev(src), steps)
            ref, ref_k, _ = oracle.run(ref, src, r, steps=steps, m=8)
            assert got_k == ref_k
        torch.cuda.synchronize()
        assert np.array_equal(u.cpu().numpy(), ref)


def test_nan_source_reports_nonfinite():
    jacobi = _jacobi()
    n = 64
    u0, g = workload(n, "gauss")
    g[10, 12] = np.nan
    u, u_alt, b = jacobi.allocate(n, u0.shape[1])
    u.copy_(to_dev(u0))
    for kw in ({}, {"strategy": "etb", "depth": 4}, {"strategy": "ba", "depth": 2},
               {"control": "device"}, {"strategy": "etb", "depth": 8, "control": "device"},
               {"strategy": "ba", "depth": 2, "control": "device"}):
        u.copy_(to_dev(u0))
        with jacobi.Solver(u, u_alt, b, 1.0, **kw) as s:
            s.rhs(to_dev(g))
            assert s.solve_step(raise_on_error=False) == jacobi.ERR_NONFINITE


@pytest.mark.parametrize("control", ["host", "device"])
def test_zero_problem_converges_at_first_check(control):
    jacobi = _jacobi()
    n = 50
    u0 = P.initial_field(n, top=0.0)
    g = P.source_term(n, kind="zero")
    u, u_alt, b = jacobi.allocate(n, u0.shape[1])
    u.copy_(to_dev(u0))
    with jacobi.Solver(u, u_alt, b, 10.0, strategy="etb", depth=8, control=control) as s:
        s.rhs(to_dev(g))
        assert s.solve_step() == 8
        assert s.residual() == (0.0, 0.0)


def test_launch_count_grows():
    jacobi = _jacobi()
    n = 40
    u0, g = workload(n, "point")
    u, u_alt, b = jacobi.allocate(n, u0.shape[1])
    u.copy_(to_dev(u0))
    with jacobi.Solver(u, u_alt, b, 1.0) as s:
        c0 = s.launch_count
        s.rhs(to_dev(g))
        k = s.solve_step()
        # rhs + k sweeps + one residual per check interval of 8
        assert s.launch_count - c0 == 1 + k + k // 8


@pytest.mark.parametrize("strategy,depth", [("sync", 1), ("etb", 4), ("etb", 8)])
def test_device_control_launch_count(strategy, depth):
    """Device control: one graph per step holding a reset kernel, the bmax
    kernel and the loop body (its sweep launches and one loop-condition
    kernel); launches after the stop are counted (they run and return)."""
    jacobi = _jacobi()
    n = 64
    u0, g = workload(n, "point")
    u, u_alt, b = jacobi.allocate(n, u0.shape[1])
    u.copy_(to_dev(u0))
    with jacobi.Solver(u, u_alt, b, 10.0, strategy=strategy, depth=depth,
                       control="device") as s:
        s.rhs(to_dev(g))
        c0 = s.launch_count
        k = s.solve_step()
        per = 1 if strategy == "sync" else depth
        L = 8 // per if per <= 8 else 1
        checks = k // 8 + 1
        body = 1 if L >= 8 else 8 // L  # check intervals per loop iteration
        if L % 2 and body % 2:
            body += 1
        iters = -(-checks // body)
        copy = 1 if (L % 2 and checks % 2 == 0) else 0
        assert s.launch_count - c0 == 2 + iters * (body * L + 1) + copy


def test_run_host_matches_the_oracle_problem_by_problem():
    """jacobi_run_host: independent problems given as host buffers, each
    equal to the oracle's ten-step solve of its own inputs (different
    sources and boundary rows), whatever the copies' overlap; pinned and
    pageable host memory; odd and even problem counts (odd problems run on
    the handle's second pair of fields), after which u holds the last
    problem's result; and a second call after a change of strategy."""
    import torch
    from temporal_blocked_jacobi_gb300 import jacobi
    n, r, steps = 130, 10.0, 3
    ld = P.padded_ld(n)
    cases = []
    for k, (src, top) in enumerate((("point", 100.0), ("gauss", 50.0),
                                    ("gauss", 100.0), ("point", 0.0))):
        u0 = P.initial_field(n, ld, top=top)
        g = P.source_term(n, ld, src, amplitude=1000.0 * (k + 1) if src == "point" else None)
        cases.append((u0, g, *oracle.run(u0, g, r, steps=steps)[:2]))
    def check(s, sel, pinned, kw):
        u0s = [torch.from_numpy(cases[i][0]) for i in sel]
        gs = [torch.from_numpy(cases[i][1]) for i in sel]
        outs = [torch.full((n, ld), float("nan")) for _ in sel]
        if pinned:
            u0s = [t.pin_memory() for t in u0s]
            gs = [t.pin_memory() for t in gs]
            outs = [t.pin_memory() for t in outs]
        counts = s.run_host(u0s, gs, outs, steps)
        for i, got, k in zip(sel, outs, counts):
            ref_u, ref_k = cases[i][2], cases[i][3]
            assert k == ref_k, (kw, pinned, k, ref_k)
            assert same_bits(got.numpy()[:, :n], ref_u[:, :n]), (kw, pinned, mismatch(got.numpy(), ref_u))
        torch.cuda.synchronize()
        assert same_bits(s.u.cpu().numpy()[:, :n], cases[sel[-1]][2][:, :n]), (kw, pinned)

    for pinned in (True, False):
        for kw in ({"strategy": "etb", "depth": 8, "control": "device"},
                   {"strategy": "etb", "depth": 8, "tile": (112, 0), "control": "device"},
                   {"strategy": "sync", "control": "host"}):
            u, u_alt, b = jacobi.allocate(n, ld)
            with jacobi.Solver(u, u_alt, b, r, **kw) as s:
                check(s, [0, 1, 2, 3], pinned, kw)
                check(s, [3, 0, 2], pinned, kw)
                s.set_strategy("sync", 1, control="device")
                check(s, [1, 2], pinned, kw)
