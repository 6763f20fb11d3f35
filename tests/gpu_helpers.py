"""Shared helpers for the GPU parity tests (CUDA path through the C ABI)."""
import numpy as np

from temporal_blocked_jacobi_gb300 import problem as P


def to_dev(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def interior(a):
    n = a.shape[0]
    return a[1:n - 1, 1:n - 1]


def same_bits(a, b):
    """Bitwise equality of float32 arrays (NaN payloads included)."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    b = np.ascontiguousarray(b, dtype=np.float32)
    return a.shape == b.shape and np.array_equal(a.view(np.uint32), b.view(np.uint32))


def mismatch(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    diff = np.argwhere(a != b)
    if len(diff) == 0:
        return "identical"
    i, j = diff[0]
    return (f"{len(diff)} cells differ; first at {tuple(diff[0])}: {a[i, j]!r} vs "
            f"{b[i, j]!r}; max |diff| {np.nanmax(np.abs(a - b))}")


def gpu_run(u0, g, r, steps=10, **solver_kw):
    """Run `steps` time steps on the GPU from u0 (numpy) with source g.
    Returns (final u as numpy, sweeps per step, last b as numpy)."""
    import torch
    from temporal_blocked_jacobi_gb300 import jacobi
    n, ld = u0.shape
    u, u_alt, b = jacobi.allocate(n, ld)
    u.copy_(to_dev(u0))
    g_dev = to_dev(g)
    with jacobi.Solver(u, u_alt, b, r, **solver_kw) as s:
        counts = s.run(g_dev, steps)
    torch.cuda.synchronize()
    return u.cpu().numpy(), counts, b.cpu().numpy()


def workload(n, source, ld=None):
    return P.initial_field(n, ld), P.source_term(n, ld, source)
