"""jacobi_residual_noalloc: the residual norms for callers that cannot
allocate device memory (inside stream capture, in loops that must not pay
for cudaMalloc's device-wide synchronisation, or under an application's own
allocator). It keeps its reduction scratch in a fixed array in the library
instead of in a solver handle. These tests call it through the C ABI and
compare it with the handle-based jacobi_residual, bit for bit (the tolerance
every residual test here uses), on two calls in a row -- the second call
must not be disturbed by what the first left in the shared scratch.

This file is collected last on purpose: it must pass both alone in a fresh
process and after every other test.
"""
import ctypes

import numpy as np
import pytest

from temporal_blocked_jacobi_gb300 import problem as P
from tests.gpu_helpers import same_bits, to_dev

pytestmark = pytest.mark.gpu


def handle_residual(u0, g, r):
    """Norms from the existing entry point (solver handle)."""
    import torch
    from temporal_blocked_jacobi_gb300 import jacobi
    n, ld = u0.shape
    u, u_alt, b = jacobi.allocate(n, ld)
    u.copy_(to_dev(u0))
    with jacobi.Solver(u, u_alt, b, r) as s:
        s.rhs(to_dev(g))
        rm, bm = s.residual()
    torch.cuda.synchronize()
    return np.float32(rm), np.float32(bm), u, b


@pytest.mark.parametrize("n,r,seed", [(515, 10.0, 3), (70, 100.0, 4), (1030, 1.0, 5)])
def test_noalloc_matches_handle_residual_twice(n, r, seed):
    import torch
    from temporal_blocked_jacobi_gb300 import jacobi
    ld = P.padded_ld(n) + 4
    fields = []
    for k in range(2):  # two different inputs, one call each, back to back
        u0 = P.random_field(n, ld, seed + 10 * k)
        g = P.random_field(n, ld, seed + 10 * k + 1)
        fields.append(handle_residual(u0, g, r))
    norms = torch.full((2,), float("nan"), dtype=torch.float32, device="cuda")
    for rm, bm, u, b in fields:
        norms.fill_(float("nan"))
        assert jacobi.residual_noalloc(u, b, r, norms) == jacobi.OK
        torch.cuda.synchronize()
        got = norms.cpu().numpy()
        assert same_bits(got[0], rm) and same_bits(got[1], bm), (got, rm, bm)


def test_noalloc_through_raw_c_abi_on_a_side_stream():
    import torch
    from temporal_blocked_jacobi_gb300 import jacobi
    lib = jacobi.load()
    n, r = 260, 10.0
    u0 = P.initial_field(n)
    g = P.source_term(n, kind="gauss")
    rm, bm, u, b = handle_residual(u0, g, r)
    norms = torch.zeros(2, dtype=torch.float32, device="cuda")
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    for _ in range(2):
        rc = lib.jacobi_residual_noalloc(n, u.shape[1], r, ctypes.c_void_p(u.data_ptr()),
                                         ctypes.c_void_p(b.data_ptr()),
                                         ctypes.c_void_p(norms.data_ptr()),
                                         ctypes.c_void_p(side.cuda_stream))
        assert rc == jacobi.OK
        side.synchronize()
        got = norms.cpu().numpy()
        assert same_bits(got[0], rm) and same_bits(got[1], bm)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    """N beyond JACOBI_RESIDUAL_NOALLOC_MAX_N is refused before anything is
    launched (so small placeholder buffers are never touched)."""
    import torch
    from temporal_blocked_jacobi_gb300 import jacobi
    lib = jacobi.load()
    small = torch.zeros(64, dtype=torch.float32, device="cuda")
    p = ctypes.c_void_p(small.data_ptr())
    assert lib.jacobi_residual_noalloc(23172, 23172, 1.0, p, p, p, None) == jacobi.ERR_UNSUPPORTED
    assert lib.jacobi_residual_noalloc(2, 4, 1.0, p, p, p, None) == jacobi.ERR_INVALID_ARG
    assert lib.jacobi_residual_noalloc(16, 18, 1.0, p, p, p, None) == jacobi.ERR_INVALID_ARG
    assert lib.jacobi_residual_noalloc(16, 16, -1.0, p, p, p, None) == jacobi.ERR_INVALID_ARG
