"""Adaptive-depth block-asynchronous solves through the C ABI against the
oracle ("Synchronous vs block-async Jacobi on one RTX 5050", section 02:
G-asc, G-desc, G-fb).

G-asc and G-desc decide from the residuals alone, so the GPU's depth
sequence, sweep counts and fields must equal the oracle's bit for bit. G-fb
also uses the measured interval times; the oracle is given the times the GPU
recorded (jacobi_check_trace) and must then make the same decisions and
reach the same field bit for bit.
"""
import numpy as np
import pytest

import oracle
from oracle import adaptive
from tests.gpu_helpers import interior, mismatch, same_bits, to_dev, workload

pytestmark = pytest.mark.gpu


def run_steps(u0, g, r, steps, **kw):
    """GPU: `steps` steps one at a time; per step (k, trace)."""
    import torch
    from temporal_blocked_jacobi_gb300 import jacobi
    n, ld = u0.shape
    u, u_alt, b = jacobi.allocate(n, ld)
    u.copy_(to_dev(u0))
    g_dev = to_dev(g)
    out = []
    with jacobi.Solver(u, u_alt, b, r, strategy="ba", control="host", **kw) as s:
        for _ in range(steps):
            s.rhs(g_dev)
            k = s.solve_step()
            out.append((k, s.check_trace()))
    torch.cuda.synchronize()
    return u.cpu().numpy(), out


@pytest.mark.parametrize("policy", ["g_asc", "g_desc"])
@pytest.mark.parametrize("n,r,source,dmax,tile", [
    (70, 10.0, "gauss", 8, (32, 8)),
    (130, 100.0, "point", 8, (32, 8)),
    (259, 10.0, "gauss", 16, (32, 16)),
    (66, 1.0, "point", 4, (8, 4)),
])
def test_threshold_controllers_bit_exact(policy, n, r, source, dmax, tile):
    u0, g = workload(n, source)
    got_u, steps = run_steps(u0, g, r, 3, depth=dmax, tile=tile, adapt=policy)
    u = u0.copy()
    for k_gpu, trace in steps:
        b = oracle.rhs(u, g)
        k, ref = adaptive.solve_step(u, b, r, policy=policy, depth_max=dmax,
                                     tile_x=tile[0], tile_y=tile[1])
        assert k_gpu == k
        assert [t["depth"] for t in trace] == [t[0] for t in ref]
        assert [t["sweeps"] for t in trace] == [t[1] for t in ref]
        for t, (_, _, rm, bm) in zip(trace, ref):
            assert same_bits(np.float32(t["rmax"]), rm)
            assert same_bits(np.float32(t["bmax"]), bm)
        assert all(t["ms"] > 0 for t in trace)
    assert same_bits(got_u, u), mismatch(got_u, u)


@pytest.mark.parametrize("n,r,source,dmax,tile", [
    (70, 10.0, "gauss", 8, (32, 8)),
    (130, 100.0, "gauss", 8, (32, 8)),
    (258, 10.0, "point", 16, (32, 16)),
])
def test_feedback_controller_replays_on_oracle(n, r, source, dmax, tile):
    u0, g = workload(n, source)
    got_u, steps = run_steps(u0, g, r, 3, depth=dmax, tile=tile, adapt="g_fb")
    u = u0.copy()
    changes = 0
    for k_gpu, trace in steps:
        b = oracle.rhs(u, g)
        ms = [t["ms"] for t in trace]
        k, ref = adaptive.solve_step(u, b, r, policy="g_fb", depth_max=dmax,
                                     tile_x=tile[0], tile_y=tile[1], ms=ms)
        depths = [t["depth"] for t in trace]
        assert k_gpu == k
        assert depths == [t[0] for t in ref]
        changes += sum(1 for a, c in zip(depths, depths[1:]) if a != c)
    assert changes > 0  # the controller did move
    assert same_bits(got_u, u), mismatch(got_u, u)


@pytest.mark.parametrize("policy", ["g_asc", "g_desc", "g_fb"])
def test_adaptive_within_tolerance_of_sync(policy):
    """Ten steps, final field within 5e-4 ||b||inf of the synchronous answer
    (the tolerance block-asynchronous solves are held to)."""
    from tests.gpu_helpers import gpu_run
    n, r = 200, 10.0
    u0, g = workload(n, "gauss")
    got_u, got_k, _ = gpu_run(u0, g, r, strategy="ba", depth=8, adapt=policy,
                              control="host")
    sync_u, _, sync_b = oracle.run(u0, g, r)
    _, bmax = oracle.residual(sync_u, sync_b, r)
    diff = np.abs(interior(got_u).astype(np.float64) - interior(sync_u)).max()
    assert diff <= 5e-4 * float(bmax)


def test_adaptive_config_checked():
    from temporal_blocked_jacobi_gb300 import jacobi
    n = 40
    u0, _ = workload(n, "gauss")
    u, u_alt, b = jacobi.allocate(n, u0.shape[1])
    u.copy_(to_dev(u0))
    cases = [
        (dict(strategy="etb", depth=8, adapt="g_fb"), jacobi.ERR_INVALID_ARG),
        (dict(strategy="ba", depth=1, adapt="g_asc"), jacobi.ERR_INVALID_ARG),
        (dict(strategy="ba", depth=8, adapt=9), jacobi.ERR_INVALID_ARG),
        (dict(strategy="ba", depth=8, adapt="g_fb", control="device"),
         jacobi.ERR_UNSUPPORTED),
    ]
    for kw, status in cases:
        with pytest.raises(jacobi.JacobiError) as e:
            jacobi.Solver(u, u_alt, b, 10.0, **kw)
        assert e.value.status == status, kw


def test_switching_controller_between_steps():
    """set_strategy moves between fixed and adaptive depth; each step's
    answer matches the oracle for the configuration it ran with."""
    import torch
    from temporal_blocked_jacobi_gb300 import jacobi
    n, r = 100, 10.0
    u0, g = workload(n, "point")
    u, u_alt, b = jacobi.allocate(n, u0.shape[1])
    u.copy_(to_dev(u0))
    g_dev = to_dev(g)
    ref = u0.copy()
    plan = [dict(strategy="ba", depth=8, adapt="g_asc"),
            dict(strategy="sync", depth=1),
            dict(strategy="ba", depth=4, adapt="g_fb"),
            dict(strategy="ba", depth=8)]
    with jacobi.Solver(u, u_alt, b, r) as s:
        for cfg in plan:
            s.set_strategy(control="host", **cfg)
            s.rhs(g_dev)
            k = s.solve_step()
            trace = s.check_trace()
            bb = oracle.rhs(ref, g)
            if cfg.get("adapt"):
                kr, _ = adaptive.solve_step(
                    ref, bb, r, policy=cfg["adapt"], depth_max=cfg["depth"],
                    ms=[t["ms"] for t in trace])
            else:
                depth = 0 if cfg["strategy"] == "sync" else cfg["depth"]
                kr, _, _ = oracle.solve_step(ref, bb, r, depth=depth)
            assert k == kr, cfg
    torch.cuda.synchronize()
    assert same_bits(u.cpu().numpy(), ref)
