"""jacobi_residual_noalloc: the residual norms for callers that cannot
allocate device memory (inside stream capture, in loops that must not pay
for cudaMalloc's device-wide synchronisation, or under an application's own
allocator). It keeps its reduction scratch in a fixed array in the library
instead of in a solver handle. These tests call it through the C ABI and
compare it with the handle-based jacobi_residual and with the oracle's
residual, bit for bit (the tolerance every residual test here uses; a NaN
norm only has to be NaN, since NaN payloads differ between GPU and host), on
two calls in a row -- the second call must not be disturbed by what the
first left in the shared scratch -- and replayed from a captured CUDA graph.

This file is collected last on purpose: it must pass both alone in a fresh
process and after every other test.
"""
import ctypes

import numpy as np
import pytest

import oracle
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


def oracle_norms_match(got, u_host, b_host, r):
    rm, bm = oracle.residual(u_host, b_host, r)
    for g, w in ((got[0], rm), (got[1], bm)):
        if np.isnan(w):
            assert np.isnan(g), (got, rm, bm)
        else:
            assert same_bits(g, w), (got, rm, bm)


@pytest.mark.parametrize("case", ["random", "nan_in_b", "nan_in_u", "inf_in_b",
                                  "n3", "n4", "zero"])
def test_noalloc_matches_oracle(case):
    """Against the oracle's difference-form residual on the host, two calls
    in a row on different inputs."""
    import torch
    from temporal_blocked_jacobi_gb300 import jacobi
    n = {"n3": 3, "n4": 4}.get(case, 261)
    r = 10.0 if case != "zero" else 1.0
    ld = P.padded_ld(n) + 4
    norms = torch.full((2,), float("nan"), dtype=torch.float32, device="cuda")
    for call in range(2):
        u = P.random_field(n, ld, seed=20 + call)
        b = P.random_field(n, ld, seed=30 + call)
        u[:, n:] = np.nan  # padding is never read
        b[:, n:] = np.nan
        if case == "nan_in_b":
            b[n // 2, n // 3] = np.nan
        elif case == "nan_in_u":
            u[n // 3, n // 2 + call] = np.nan
        elif case == "inf_in_b":
            b[1, n - 2] = -np.inf
        elif case == "zero":
            u[:] = 0.0
            b[:] = 0.0
        norms.fill_(float("nan"))
        ud, bd = to_dev(u), to_dev(b)
        assert jacobi.residual_noalloc(ud, bd, r, norms) == jacobi.OK
        torch.cuda.synchronize()
        oracle_norms_match(norms.cpu().numpy(), u, b, r)


def test_noalloc_replayed_from_a_captured_graph():
    """A call captured into a CUDA graph (after one plain call that looks the
    scratch up) gives the oracle's norms on every replay, for whatever the
    captured buffers hold at replay time."""
    import torch
    from temporal_blocked_jacobi_gb300 import jacobi
    n, r = 300, 100.0
    ld = P.padded_ld(n)
    ud = torch.zeros((n, ld), dtype=torch.float32, device="cuda")
    bd = torch.zeros_like(ud)
    norms = torch.zeros(2, dtype=torch.float32, device="cuda")
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        assert jacobi.residual_noalloc(ud, bd, r, norms, stream=side) == jacobi.OK
    side.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        rc = jacobi.residual_noalloc(ud, bd, r, norms,
                                     stream=torch.cuda.current_stream())
    assert rc == jacobi.OK
    for seed in (41, 42, 43):
        u = P.random_field(n, ld, seed=seed)
        b = P.random_field(n, ld, seed=seed + 100)
        ud.copy_(to_dev(u))
        bd.copy_(to_dev(b))
        norms.fill_(float("nan"))
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        oracle_norms_match(norms.cpu().numpy(), u, b, r)


def test_noalloc_wrapper_rejects_mixed_devices():
    import torch
    from temporal_blocked_jacobi_gb300 import jacobi
    u = torch.zeros((8, 8), dtype=torch.float32, device="cuda")
    with pytest.raises(ValueError):
        jacobi.residual_noalloc(u, u, 1.0, torch.zeros(2))  # norms on the host
