"""Full-size checks of the measured configurations that the solve-level
parity tests (test_gpu_solve.py) cover only through their first check
interval or through GPU self-consistency.

* BLOCK_ASYNC at the sizes it is measured on ("Synchronous vs block-async
  Jacobi on one RTX 5050", section 02 "Block-asynchronous"; sections 04-05):
  N = 4096 with r = 1, 10, 100 and D = 2, 4, 8, 16, and N = 18432, r = 10,
  D = 8. The first launch (32 x 8 tiles held in registers) is compared bit
  for bit with the oracle's block-asynchronous emulator at full size; the
  ten-step field must lie within 5e-4 ||b||inf of the synchronous answer,
  ||b||inf being the norm of SYNC's last right-hand side. The SYNC field is
  the GPU's, which is bit-exact to the oracle (below and in
  test_gpu_solve.py).
* Ten full time steps of SYNC and EXACT_TEMPORAL_BLOCKED(8) at N = 4096
  (r = 1 and 10) and at N = 18432 (r = 10, point source) against the oracle
  run on all host cores (row-parallel, bit for bit equal to the
  single-threaded oracle: test_oracle_threads.py).
* The first check interval at N = 8192, r = 100 for SYNC and
  EXACT_TEMPORAL_BLOCKED with D = 4, 8 and 16 (D = 16: one 16-sweep launch).
"""
import os

import numpy as np
import pytest

import oracle
from tests.gpu_helpers import gpu_run, interior, mismatch, same_bits, to_dev, workload

pytestmark = pytest.mark.gpu

BA_TILE = (32, 8)  # the default block-asynchronous tile


def first_ba_launch_matches_oracle(u0, g, r, depth):
    """One block-asynchronous launch from u⁰ after the right-hand side."""
    import torch
    from temporal_blocked_jacobi_gb300 import jacobi
    b_ref = oracle.rhs(u0, g)
    ref = oracle.ba_launch(u0, b_ref, r, BA_TILE[0], BA_TILE[1], depth)
    n, ld = u0.shape
    u, u_alt, b = jacobi.allocate(n, ld)
    u.copy_(to_dev(u0))
    with jacobi.Solver(u, u_alt, b, r, strategy="ba", depth=depth) as s:
        s.rhs(to_dev(g))
        assert s.sweeps(1) == depth
    torch.cuda.synchronize()
    got = u.cpu().numpy()
    del u, u_alt, b
    assert same_bits(got, ref), mismatch(got, ref)


def within_bound_of_sync(got_u, sync_u, bmax):
    diff = float(np.abs(interior(got_u).astype(np.float64)
                        - interior(sync_u).astype(np.float64)).max())
    assert diff <= 5e-4 * float(bmax), (diff, 5e-4 * float(bmax))
    return diff


_sync_4096 = {}


def sync_4096(r):
    """(u0, g, GPU SYNC field, counts, bmax of SYNC's last right-hand side)
    at N = 4096, Gaussian source, cached per r."""
    if r not in _sync_4096:
        u0, g = workload(4096, "gauss")
        u, k, b = gpu_run(u0, g, r, control="device")
        _, bmax = oracle.residual(u, b, r)
        _sync_4096[r] = (u0, g, u, k, bmax)
    return _sync_4096[r]


@pytest.mark.parametrize("r", [1.0, 10.0, 100.0])
@pytest.mark.parametrize("depth", [2, 4, 8, 16])
def test_n4096_block_async_full_size(r, depth):
    u0, g, sync_u, sync_k, bmax = sync_4096(r)
    first_ba_launch_matches_oracle(u0, g, r, depth)
    got_u, got_k, _ = gpu_run(u0, g, r, strategy="ba", depth=depth, control="device")
    interval = oracle.check_interval(8, depth)
    assert all(k > 0 and k % interval == 0 for k in got_k), got_k
    within_bound_of_sync(got_u, sync_u, bmax)


def test_n18432_r10_point_block_async():
    u0, g = workload(18432, "point")
    first_ba_launch_matches_oracle(u0, g, 10.0, 8)
    sync_u, sync_k, sync_b = gpu_run(u0, g, 10.0, control="device")
    _, bmax = oracle.residual(sync_u, sync_b, 10.0)
    del sync_b
    got_u, got_k, _ = gpu_run(u0, g, 10.0, strategy="ba", depth=8, control="device")
    assert all(k > 0 and k % 8 == 0 for k in got_k), got_k
    within_bound_of_sync(got_u, sync_u, bmax)


def host_threads():
    return max(1, min(64, os.cpu_count() or 1))


@pytest.mark.parametrize("r", [1.0, 10.0])
def test_n4096_ten_steps_bit_exact_to_threaded_oracle(r):
    u0, g = workload(4096, "gauss")
    ref_u, ref_k, _ = oracle.run(u0, g, r, threads=host_threads())
    for kw in ({"strategy": "sync", "depth": 1, "control": "device"},
               {"strategy": "etb", "depth": 8, "control": "device"},
               {"strategy": "etb", "depth": 8, "control": "host"}):
        got_u, got_k, _ = gpu_run(u0, g, r, **kw)
        assert got_k == ref_k, (kw, got_k, ref_k)
        assert same_bits(got_u, ref_u), (kw, mismatch(got_u, ref_u))


def test_n8192_first_interval_every_strategy():
    from tests.test_gpu_solve import first_interval_matches_oracle
    for strategy, depth in (("sync", 1), ("etb", 4), ("etb", 8), ("etb", 16)):
        first_interval_matches_oracle(8192, 100.0, "gauss", strategy, depth)


def test_default_d8_kernel_follows_the_grid():
    """At D = 8 the default is the column-streamed kernel (tile 112 x 0) on
    grids with enough rows per warp and a register-band shape on small ones;
    persistent control always gets a register-band shape."""
    import torch
    from temporal_blocked_jacobi_gb300 import jacobi
    for n, want in ((2048, (112, 92)), (8192, (112, 0)), (18432, (112, 0))):
        u, u_alt, b = jacobi.allocate(n)
        with jacobi.Solver(u, u_alt, b, 10.0, strategy="etb", depth=8,
                           control="device") as s:
            assert s.tile == want, (n, s.tile)
        if n == 8192:
            with jacobi.Solver(u, u_alt, b, 10.0, strategy="etb", depth=8,
                               control="persistent") as s:
                assert s.tile[1] > 0
        del u, u_alt, b
        torch.cuda.empty_cache()


def test_n18432_ten_steps_bit_exact_to_threaded_oracle():
    """The default bench configuration (N = 18432, r = 10, point source):
    all ten time steps of SYNC and of EXACT_TEMPORAL_BLOCKED(8) (the
    column-streamed kernel at this N) against the oracle run on all host
    cores, fields and sweep counts bit for bit. About 8e11 lattice updates
    on the host."""
    u0, g = workload(18432, "point")
    ref_u, ref_k, _ = oracle.run(u0, g, 10.0, threads=host_threads())
    for kw in ({"strategy": "etb", "depth": 8, "control": "device"},
               {"strategy": "sync", "depth": 1, "control": "device"}):
        got_u, got_k, _ = gpu_run(u0, g, 10.0, **kw)
        assert got_k == ref_k, (kw, got_k, ref_k)
        assert same_bits(got_u, ref_u), (kw, mismatch(got_u, ref_u))
        del got_u
