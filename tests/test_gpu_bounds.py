"""The bounds-checked library (libtbjacobi_checked.so; include/jacobi.h,
"Bounds-checked build") on the GPU, standing in for a memory checker.

Every tiled kernel shape -- exact temporal blocking in all compiled shapes
and block-async in the register, streaming (one and two chunks per lane) and
generic kernels, with and without overlapping subdomains -- solves two time
steps on grids of N = 17, 70, 130 and 259 (smaller than one tile, a few
tiles, ragged edges) with every access range-checked, shared memory and the
destination's interior poisoned with NaN before each launch. No check may
fire (a fired check raises JACOBI_ERR_CUDA), and the result must equal the
oracle's bit for bit, as with the unchecked library. The checker itself is
shown to refuse out-of-range accesses by jacobi_bounds_selftest.
"""
import numpy as np
import pytest

import oracle
from tests.gpu_helpers import mismatch, same_bits, to_dev, workload

pytestmark = pytest.mark.gpu

SIZES = [17, 70, 130, 259]


def run_checked(u0, g, r, steps=2, **kw):
    import torch
    from temporal_blocked_jacobi_gb300 import jacobi
    n, ld = u0.shape
    u, u_alt, b = jacobi.allocate(n, ld)
    u.copy_(to_dev(u0))
    with jacobi.Solver(u, u_alt, b, r, checked=True, **kw) as s:
        counts = s.run(to_dev(g), steps)
    torch.cuda.synchronize()
    return u.cpu().numpy(), counts


def test_checker_refuses_out_of_range_accesses():
    import torch
    from temporal_blocked_jacobi_gb300 import jacobi
    u0, _ = workload(40, "point")
    u, u_alt, b = jacobi.allocate(40)
    u.copy_(to_dev(u0))
    with jacobi.Solver(u, u_alt, b, 1.0, checked=True) as s:
        assert s.bounds_selftest() == 0x7  # refused: 0, 1, 2; allowed: 3, 4
        assert s.bounds_selftest() == 0x7
    torch.cuda.synchronize()
    assert same_bits(u.cpu().numpy(), u0)  # the test stores changed nothing
    with jacobi.Solver(u, u_alt, b, 1.0) as s:
        with pytest.raises(jacobi.JacobiError):
            s.bounds_selftest()  # the unchecked library has no checker


ETB = [(2, (0, 0)), (4, (0, 0)), (8, (0, 0)), (16, (0, 0)),
       (2, (120, 60)), (2, (248, 60)), (2, (120, 92)), (4, (120, 56)),
       (4, (248, 56)), (4, (120, 40)), (4, (120, 88)), (8, (112, 80)),
       (8, (112, 48)), (8, (112, 112)), (8, (240, 48)), (8, (112, 92)), (8, (112, 0)),
       (16, (96, 64)), (16, (96, 96)), (16, (224, 64)), (16, (96, 76))]


@pytest.mark.parametrize("n", SIZES)
@pytest.mark.parametrize("depth,tile", ETB)
def test_etb_shapes_checked(depth, tile, n):
    u0, g = workload(n, "gauss")
    ref_u, ref_k, _ = oracle.run(u0, g, 10.0, steps=2, m=max(8, depth))
    for control in ("device", "host"):
        got_u, got_k = run_checked(u0, g, 10.0, strategy="etb", depth=depth,
                                   tile=tile, control=control)
        assert got_k == ref_k, (control, got_k, ref_k)
        assert same_bits(got_u, ref_u), (control, mismatch(got_u, ref_u))


# (depth, tile, overlap): the register kernel (32 x 8), the streaming kernel
# with one float4 chunk per lane (32 x 16, 4 x 3) and two (84 x 8, 128 x 64),
# and the generic kernel (taller than 64 cells, overlap)
BA = [(8, (32, 8), (0, 0)), (4, (32, 8), (0, 0)), (8, (32, 16), (0, 0)),
      (4, (4, 3), (0, 0)), (8, (84, 8), (0, 0)), (8, (128, 64), (0, 0)),
      (4, (8, 72), (0, 0)), (16, (128, 128), (0, 0)), (8, (32, 32), (4, 4)),
      (4, (16, 8), (2, 2))]


@pytest.mark.parametrize("n", SIZES)
@pytest.mark.parametrize("depth,tile,overlap", BA)
def test_block_async_shapes_checked(depth, tile, overlap, n):
    u0, g = workload(n, "point")
    ref_u, ref_k, _ = oracle.run(u0, g, 10.0, steps=2, depth=depth, tile_x=tile[0],
                                 tile_y=tile[1], overlap=overlap)
    for control in ("device", "host"):
        got_u, got_k = run_checked(u0, g, 10.0, strategy="ba", depth=depth,
                                   tile=tile, overlap=overlap, control=control)
        assert got_k == ref_k, (control, got_k, ref_k)
        assert same_bits(got_u, ref_u), (control, mismatch(got_u, ref_u))


@pytest.mark.parametrize("n", SIZES)
def test_sync_and_persistent_checked(n):
    u0, g = workload(n, "gauss")
    ref_u, ref_k, _ = oracle.run(u0, g, 1.0, steps=2)
    for kw in ({"strategy": "sync"}, {"strategy": "etb", "depth": 8,
                                      "control": "persistent"}):
        got_u, got_k = run_checked(u0, g, 1.0, **kw)
        assert got_k == ref_k and same_bits(got_u, ref_u), (kw, mismatch(got_u, ref_u))
