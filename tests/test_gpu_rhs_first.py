"""The run graph's step that starts with the column-streamed kernel forming
the right-hand side itself ("Synchronous vs block-async Jacobi on one RTX
5050", section 01: b = u^n + dt f is fixed within a step; section 05 on
fusing the right-hand side into the sweep).

Under device control, with exact temporal blocking at D = 8 in whole columns
(tile 112 x 0) and one launch per check interval, each step of jacobi_run is
reset -> bmax of the ring-adjacent cells -> the first sweep launch, which
forms b = fl(u^n + g) from the u^n it reads, writes it, and reduces |b| over
the other cells -> the device-side loop from its output. A step starts from
whichever buffer holds the previous step's answer (an if/else graph node),
and only the run's answer is moved into u. The sweep counts, fields and the
last step's b must equal the oracle's, bit for bit, whatever cell holds
max |b_I| and whichever buffer each step ends in; errors and launch counts
behave as on the ordinary path.
"""
import ctypes

import numpy as np
import pytest

import oracle
from temporal_blocked_jacobi_gb300 import problem as P
from tests.gpu_helpers import gpu_run, interior, mismatch, same_bits, to_dev, workload

pytestmark = pytest.mark.gpu

STREAMED = dict(strategy="etb", depth=8, tile=(112, 0), control="device")


@pytest.mark.parametrize("n,r,source", [(3, 10.0, "point"), (17, 1.0, "point"),
                                        (70, 10.0, "gauss"), (70, 10.0, "zero"),
                                        (131, 1.0, "point"), (300, 10.0, "gauss"),
                                        (1030, 1.0, "gauss")])
def test_first_launch_forms_the_right_hand_side(n, r, source):
    u0, g = workload(n, source)
    ref_u, ref_k, ref_b = oracle.run(u0, g, r, steps=3)
    got_u, got_k, got_b = gpu_run(u0, g, r, steps=3, **STREAMED)
    assert got_k == ref_k
    assert same_bits(got_u, ref_u), mismatch(got_u, ref_u)
    assert same_bits(interior(got_b), interior(ref_b)), \
        mismatch(interior(got_b), interior(ref_b))


# Where max |b_I| sits: on a cell next to the top, right or bottom ring, the
# interior's corner, or deep inside (positive or negative). The spike sets
# the convergence threshold, so a bmax that missed it would change the
# sweep counts.
SPIKES = {"top": (1, 30, 1e4), "right": (33, 68, 1e4), "bottom": (68, 12, -1e4),
          "corner": (68, 68, 1e4), "deep": (35, 35, 1e4),
          "deep_negative": (20, 40, -1e4)}


@pytest.mark.parametrize("where", sorted(SPIKES))
def test_bmax_wherever_it_sits(where):
    n, r = 70, 10.0
    u0 = P.initial_field(n)
    g = P.source_term(n, kind="gauss")
    i, j, v = SPIKES[where]
    g[i, j] = np.float32(v)
    ref_u, ref_k, ref_b = oracle.run(u0, g, r, steps=3)
    got_u, got_k, got_b = gpu_run(u0, g, r, steps=3, **STREAMED)
    assert got_k == ref_k
    assert same_bits(got_u, ref_u), mismatch(got_u, ref_u)
    assert same_bits(interior(got_b), interior(ref_b))


def test_failing_step_stops_the_run():
    """Step 2's right-hand side overflows at one cell: step 1 converges, step 2
    reports JACOBI_ERR_NONFINITE at its first check with u holding that
    check's iterate (finite cells bit for bit as the oracle leaves them),
    later steps do nothing, and the handle works afterwards."""
    import torch
    from temporal_blocked_jacobi_gb300 import jacobi
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
    with jacobi.Solver(u, u_alt, b, r, **STREAMED) as s:
        counts = (ctypes.c_longlong * 4)()
        total = jacobi.load().jacobi_run(s.handle, ctypes.c_void_p(to_dev(g).data_ptr()),
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
        g2 = P.source_term(n, kind="gauss")
        ref_u, ref_k2, _ = oracle.run(u0, g2, r, steps=2)
        assert s.run(to_dev(g2), 2) == ref_k2
        torch.cuda.synchronize()
        assert same_bits(u.cpu().numpy(), ref_u)


def test_sweep_cap_reports_not_converged():
    """A cap below the first check: the step's first check (after the launch
    that formed b) stops it with JACOBI_ERR_NOT_CONVERGED and 8 sweeps, as
    on the ordinary path."""
    from temporal_blocked_jacobi_gb300 import jacobi
    n, r = 70, 100.0
    u0, g = workload(n, "point")
    u, u_alt, b = jacobi.allocate(n, u0.shape[1])
    u.copy_(to_dev(u0))
    with jacobi.Solver(u, u_alt, b, r, max_sweeps=4, **STREAMED) as s:
        counts = (ctypes.c_longlong * 2)()
        total = jacobi.load().jacobi_run(s.handle, ctypes.c_void_p(to_dev(g).data_ptr()),
                                         2, counts)
        assert total == jacobi.ERR_NOT_CONVERGED
        assert "not converged after 8 sweeps" in s.last_error


@pytest.mark.parametrize("n", [64, 1030])
def test_launch_count(n):
    """Per step: the reset, the branch choice (steps after the first: the
    step starts from the buffer holding the previous answer), the ring part
    of bmax, the first launch, then loop iterations of `body` launches and
    one loop-condition kernel until the check that stops (the first launch
    covered the unchecked first interval); at the end one kernel moves the
    run's answer into u."""
    import torch
    from temporal_blocked_jacobi_gb300 import jacobi
    u0, g = workload(n, "point")
    u, u_alt, b = jacobi.allocate(n, u0.shape[1])
    u.copy_(to_dev(u0))
    with jacobi.Solver(u, u_alt, b, 10.0, **STREAMED) as s:
        c0 = s.launch_count
        counts = s.run(to_dev(g), 3)
        body = 16 if n >= 1024 else 8
        expected = 1 + sum(3 + (s > 0) + -(-(k // 8) // body) * (body + 1)
                           for s, k in enumerate(counts))
        assert s.launch_count - c0 == expected
    torch.cuda.synchronize()
