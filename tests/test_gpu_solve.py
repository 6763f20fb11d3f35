"""Solve-level parity: ten backward-Euler steps through the C ABI against the
oracle -- same sweep counts and the same field bit for bit for SYNC and
EXACT_TEMPORAL_BLOCKED; BLOCK_ASYNC bit for bit against the oracle's
block-asynchronous emulator and within 5e-4 ||b||inf of the synchronous
answer ("Synchronous vs block-async Jacobi on one RTX 5050", sections 01-02).

Workloads follow the measured configurations: N = 512 (r = 1, point source),
N = 2048 (r = 10, Gaussian), N = 4096 (r = 1, 10, 100, Gaussian), N = 8192
(r = 100, Gaussian) and N = 18432 (r = 10, point source). Where the full
ten-step oracle would take too long (N >= 4096), the oracle checks the first
check interval of the first step bit for bit at full size, the final field's
residual is recomputed by the oracle from the GPU's field, and SYNC and
EXACT_TEMPORAL_BLOCKED are required to agree bit for bit with each other.
"""
import numpy as np
import pytest

import oracle
from temporal_blocked_jacobi_gb300 import problem as P
from tests.gpu_helpers import gpu_run, interior, mismatch, same_bits, to_dev, workload

pytestmark = pytest.mark.gpu


CONTROLS = ["host", "device"]


@pytest.mark.parametrize("control", CONTROLS)
def test_n512_r1_point_sync_bit_exact(control):
    u0, g = workload(512, "point")
    ref_u, ref_k, _ = oracle.run(u0, g, 1.0)
    got_u, got_k, _ = gpu_run(u0, g, 1.0, control=control)
    assert got_k == ref_k
    assert same_bits(got_u, ref_u), mismatch(got_u, ref_u)


@pytest.fixture(scope="module")
def n2048_reference():
    u0, g = workload(2048, "gauss")
    ref_u, ref_k, ref_b = oracle.run(u0, g, 10.0)
    return u0, g, ref_u, ref_k


@pytest.mark.parametrize("control", CONTROLS)
@pytest.mark.parametrize("strategy,depth", [("sync", 1), ("etb", 2), ("etb", 4), ("etb", 8)])
def test_n2048_r10_gauss_bit_exact(n2048_reference, strategy, depth, control):
    u0, g, ref_u, ref_k = n2048_reference
    got_u, got_k, _ = gpu_run(u0, g, 10.0, strategy=strategy, depth=depth,
                              control=control)
    assert got_k == ref_k
    assert same_bits(got_u, ref_u), mismatch(got_u, ref_u)


# Every compiled tile shape of exact temporal blocking, selected by its tile
# size (the defaults depend on N; those of N = 2048 run in the test above).
ETB_SHAPES = [(2, (120, 60)), (2, (248, 60)), (4, (120, 56)), (4, (248, 56)),
              (4, (120, 40)), (8, (112, 80)), (8, (112, 48)), (8, (112, 112)),
              (8, (240, 48)), (8, (112, 92)), (8, (112, 0)), (16, (96, 64)), (16, (96, 96)),
              (16, (224, 64)), (16, (96, 76))]


@pytest.mark.parametrize("depth,tile", ETB_SHAPES)
def test_etb_tile_shapes_device_loop_bit_exact(depth, tile):
    """Every compiled tile shape through the device-side loop, whose first
    launch per check interval also reduces the residual: same sweep counts and
    field as the oracle on a grid of several tiles with ragged edges."""
    u0, g = workload(300, "gauss")
    ref_u, ref_k, _ = oracle.run(u0, g, 10.0, steps=2, m=max(8, depth))
    got_u, got_k, _ = gpu_run(u0, g, 10.0, steps=2, strategy="etb", depth=depth,
                              tile=tile, control="device")
    assert got_k == ref_k
    assert same_bits(got_u, ref_u), mismatch(got_u, ref_u)


@pytest.mark.parametrize("control", CONTROLS)
def test_n2048_r10_gauss_unfused_sync_bit_exact(n2048_reference, control):
    """The unfused right-hand side (section 05, Table VI) changes the
    traffic, not the answer."""
    u0, g, ref_u, ref_k = n2048_reference
    got_u, got_k, _ = gpu_run(u0, g, 10.0, rhs="unfused", control=control)
    assert got_k == ref_k
    assert same_bits(got_u, ref_u), mismatch(got_u, ref_u)


@pytest.mark.parametrize("control", CONTROLS)
@pytest.mark.parametrize("n,r,source", [(130, 100.0, "gauss"), (70, 10.0, "point")])
def test_etb16_checks_every_16_sweeps(n, r, source, control):
    """A 16-sweep launch is checked every lcm(8, 16) = 16 sweeps; it equals
    synchronous sweeps checked every 16."""
    u0, g = workload(n, source)
    ref_u, ref_k, _ = oracle.run(u0, g, r, m=16)
    got_u, got_k, _ = gpu_run(u0, g, r, strategy="etb", depth=16, control=control)
    assert got_k == ref_k and all(k % 16 == 0 for k in got_k)
    assert same_bits(got_u, ref_u), mismatch(got_u, ref_u)


@pytest.mark.parametrize("control", CONTROLS)
@pytest.mark.parametrize("n,r,source,depth,tile", [
    (256, 10.0, "point", 4, (32, 8)),
    (256, 1.0, "gauss", 2, (32, 8)),
    (70, 100.0, "gauss", 8, (32, 16)),
    (258, 10.0, "point", 8, (32, 16)),
    (130, 10.0, "gauss", 16, (128, 64)),
])
def test_block_async_solve(n, r, source, depth, tile, control):
    u0, g = workload(n, source)
    ref_u, ref_k, _ = oracle.run(u0, g, r, depth=depth, tile_x=tile[0], tile_y=tile[1])
    got_u, got_k, got_b = gpu_run(u0, g, r, strategy="ba", depth=depth, tile=tile,
                                  control=control)
    assert got_k == ref_k
    assert same_bits(got_u, ref_u), mismatch(got_u, ref_u)
    # within 5e-4 ||b||inf of the synchronous answer
    sync_u, _, sync_b = oracle.run(u0, g, r)
    _, bmax = oracle.residual(sync_u, sync_b, r)
    assert np.abs(interior(got_u).astype(np.float64) - interior(sync_u)).max() <= 5e-4 * float(bmax)


@pytest.mark.parametrize("control", CONTROLS)
@pytest.mark.parametrize("n,r,source,depth,tile,overlap", [
    (130, 10.0, "gauss", 8, (32, 32), (4, 4)),
    (259, 100.0, "point", 16, (32, 16), (4, 2)),
    (70, 1.0, "gauss", 4, (16, 8), (2, 2)),
])
def test_block_async_overlap_solve(n, r, source, depth, tile, overlap, control):
    u0, g = workload(n, source)
    ref_u, ref_k, _ = oracle.run(u0, g, r, depth=depth, tile_x=tile[0],
                                 tile_y=tile[1], overlap=overlap)
    got_u, got_k, _ = gpu_run(u0, g, r, strategy="ba", depth=depth, tile=tile,
                              overlap=overlap, control=control)
    assert got_k == ref_k
    assert same_bits(got_u, ref_u), mismatch(got_u, ref_u)
    sync_u, _, sync_b = oracle.run(u0, g, r)
    _, bmax = oracle.residual(sync_u, sync_b, r)
    assert np.abs(interior(got_u).astype(np.float64) - interior(sync_u)).max() <= 5e-4 * float(bmax)


def test_block_async_depth1_equals_sync():
    u0, g = workload(200, "gauss")
    a_u, a_k, _ = gpu_run(u0, g, 10.0, strategy="ba", depth=1)
    s_u, s_k, _ = gpu_run(u0, g, 10.0)
    assert a_k == s_k and same_bits(a_u, s_u)


def test_strategy_change_between_steps():
    """D is only a launch parameter: switching SYNC -> ETB(4) -> ETB(8)
    between steps leaves the answer and the counts unchanged."""
    from temporal_blocked_jacobi_gb300 import jacobi
    import torch
    n, r = 300, 10.0
    u0, g = workload(n, "point")
    ref_u, ref_k, _ = oracle.run(u0, g, r, steps=6)
    u, u_alt, b = jacobi.allocate(n, u0.shape[1])
    u.copy_(to_dev(u0))
    g_dev = to_dev(g)
    counts = []
    with jacobi.Solver(u, u_alt, b, r) as s:
        for step, (strategy, depth, control) in enumerate(
                [("sync", 1, "host"), ("etb", 4, "device"), ("etb", 8, "device"),
                 ("sync", 1, "device"), ("etb", 2, "host"), ("etb", 8, "host")]):
            s.set_strategy(strategy, depth, control=control)
            s.rhs(g_dev)
            counts.append(s.solve_step())
    torch.cuda.synchronize()
    assert counts == ref_k
    assert same_bits(u.cpu().numpy(), ref_u)


def test_mirror_symmetry_on_gpu():
    n = 65
    c = (n - 1) / 2
    u0 = P.initial_field(n, 68)
    g = P.source_term(n, 68, "gauss", center=(c, c))
    for kw in ({}, {"strategy": "etb", "depth": 8}, {"control": "device"}):
        got_u, _, _ = gpu_run(u0, g, 100.0, **kw)
        inner = got_u[:, :n]
        assert same_bits(inner, inner[:, ::-1])


# --------------------------------------------------------------------------
# Full-size workloads
# --------------------------------------------------------------------------
def first_interval_matches_oracle(n, r, source, strategy, depth):
    """The first check interval of step 1 at full size, bit for bit."""
    from temporal_blocked_jacobi_gb300 import jacobi
    import torch
    u0, g = workload(n, source)
    b_ref = oracle.rhs(u0, g)
    interval = oracle.check_interval(8, depth)
    ref = oracle.sweeps(u0, b_ref, r, interval)
    rm_ref, bm_ref = oracle.residual(ref, b_ref, r)
    u, u_alt, b = jacobi.allocate(n, u0.shape[1])
    u.copy_(to_dev(u0))
    with jacobi.Solver(u, u_alt, b, r, strategy=strategy, depth=depth) as s:
        s.rhs(to_dev(g))
        s.sweeps(interval // depth)
        rm, bm = s.residual()
    torch.cuda.synchronize()
    got = u.cpu().numpy()
    del u, u_alt, b
    assert same_bits(got, ref), mismatch(got, ref)
    assert same_bits(np.float32(rm), rm_ref) and same_bits(np.float32(bm), bm_ref)


def full_solve_properties(n, r, source, variants):
    """All variants give identical counts and fields; the oracle recomputes
    the final residual from the GPU's field and confirms the stopping rule."""
    u0, g = workload(n, source)
    results = []
    for kw in variants:
        got_u, got_k, got_b = gpu_run(u0, g, r, **kw)
        results.append((kw, got_u, got_k, got_b))
    kw0, u_s, k_s, b_s = results[0]
    for kw, got_u, got_k, _ in results[1:]:
        assert got_k == k_s, (kw, got_k, k_s)
        assert same_bits(got_u, u_s), (kw, mismatch(got_u, u_s))
    rm, bm = oracle.residual(u_s, b_s, r)
    assert float(rm) < 1e-5 * float(bm) or rm == 0
    return k_s


@pytest.mark.parametrize("r", [1.0, 10.0, 100.0])
def test_n4096_gauss(r):
    first_interval_matches_oracle(4096, r, "gauss", "sync", 1)
    first_interval_matches_oracle(4096, r, "gauss", "etb", 8)
    full_solve_properties(4096, r, "gauss", [
        {"strategy": "sync", "depth": 1}, {"strategy": "etb", "depth": 2},
        {"strategy": "etb", "depth": 4}, {"strategy": "etb", "depth": 8},
        {"strategy": "sync", "depth": 1, "control": "device"},
        {"strategy": "etb", "depth": 4, "control": "device"},
        {"strategy": "etb", "depth": 8, "control": "device"},
        {"strategy": "etb", "depth": 8, "tile": (112, 92), "control": "device"},
        {"strategy": "sync", "depth": 1, "rhs": "unfused", "control": "device"}])


@pytest.mark.parametrize("n", [3530, 3585, 3586, 4097])
def test_etb8_default_around_the_streamed_threshold(n):
    """Sizes on both sides of where the D = 8 default turns from the
    register-band to the column-streamed kernel (64 rows per warp): two time
    steps of the default ETB(8) under device control equal SYNC's, sweep
    counts and fields bit for bit (SYNC being pinned to the oracle)."""
    import torch
    from temporal_blocked_jacobi_gb300 import jacobi
    u0, g = workload(n, "gauss")
    ref_u, ref_k, _ = gpu_run(u0, g, 10.0, steps=2, control="device")
    got_u, got_k, _ = gpu_run(u0, g, 10.0, steps=2, strategy="etb", depth=8,
                              control="device")
    assert got_k == ref_k
    assert same_bits(got_u, ref_u), mismatch(got_u, ref_u)
    u, u_alt, b = jacobi.allocate(n, u0.shape[1])
    with jacobi.Solver(u, u_alt, b, 10.0, strategy="etb", depth=8) as s:
        streamed = s.tile == (112, 0)
    torch.cuda.synchronize()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    strips = -(-(n - 1) // 112)
    assert streamed == ((n - 2) * strips >= 64 * 12 * sms)


def test_n8192_r100_gauss():
    first_interval_matches_oracle(8192, 100.0, "gauss", "etb", 4)
    full_solve_properties(8192, 100.0, "gauss", [
        {"strategy": "sync", "depth": 1}, {"strategy": "etb", "depth": 4},
        {"strategy": "etb", "depth": 8},
        {"strategy": "etb", "depth": 4, "control": "device"}])
    full_solve_properties(8192, 100.0, "gauss", [
        {"strategy": "sync", "depth": 1, "check_every": 16},
        {"strategy": "etb", "depth": 16},
        {"strategy": "etb", "depth": 16, "control": "device"}])


def test_n18432_r10_point():
    first_interval_matches_oracle(18432, 10.0, "point", "etb", 8)
    full_solve_properties(18432, 10.0, "point", [
        {"strategy": "sync", "depth": 1}, {"strategy": "etb", "depth": 8},
        {"strategy": "etb", "depth": 8, "control": "device"}])
