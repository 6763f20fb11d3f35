"""Kernel-level parity: each CUDA kernel, run once through the C ABI, against
the oracle on the same seeded inputs, bit for bit.

Sizes span several tiles and ragged tails (N = 70 leaves partial tiles at the
edges, as in "Synchronous vs block-async Jacobi on one RTX 5050", section
02), the row pitch is padded, and the padding is filled with NaN so any read
of it into a result shows up.
"""
import numpy as np
import pytest

import oracle
from temporal_blocked_jacobi_gb300 import problem as P
from tests.gpu_helpers import interior, mismatch, same_bits, to_dev

pytestmark = pytest.mark.gpu

SIZES = [3, 4, 5, 16, 17, 33, 70, 127, 128, 130, 259, 520]
RS = [1.0, 10.0, 100.0, 0.3]


def fields(n, pad, seed):
    ld = P.padded_ld(n) + pad
    u0 = P.random_field(n, ld, seed)
    g = P.random_field(n, ld, seed + 1000)
    if pad or ld > n:
        u0[:, n:] = np.nan
        g[:, n:] = np.nan
    return u0, g


def make_solver(u0, r, **kw):
    from temporal_blocked_jacobi_gb300 import jacobi
    n, ld = u0.shape
    u, u_alt, b = jacobi.allocate(n, ld)
    u.copy_(to_dev(u0))
    return jacobi.Solver(u, u_alt, b, r, **kw), u, b


@pytest.mark.parametrize("n", SIZES)
@pytest.mark.parametrize("pad", [0, 12])
@pytest.mark.parametrize("division", ["auto", "ieee"])
def test_rhs_sweep_residual_sync(n, pad, division):
    r = RS[n % len(RS)]
    u0, g = fields(n, pad, seed=n)
    s, u, b = make_solver(u0, r, division=division)
    with s:
        s.rhs(to_dev(g))
        b_ref = oracle.rhs(u0, g)
        assert same_bits(interior(b.cpu().numpy()), interior(b_ref))
        rm, bm = s.residual()
        rm_ref, bm_ref = oracle.residual(u0, b_ref, r)
        assert same_bits(np.float32(rm), rm_ref) and same_bits(np.float32(bm), bm_ref)
        ref = u0
        for launches in (1, 2, 5):
            s.sweeps(launches)
            ref = oracle.sweeps(ref, b_ref, r, launches)
            got = u.cpu().numpy()
            assert same_bits(interior(got), interior(ref)), mismatch(got, ref)
        # ring and padding untouched
        got = u.cpu().numpy()
        assert same_bits(got[0], u0[0]) and same_bits(got[-1], u0[-1])
        assert same_bits(got[:, 0], u0[:, 0]) and same_bits(got[:, n - 1], u0[:, n - 1])
        assert np.isnan(got[:, n:]).all()
        rm, bm = s.residual()
        rm_ref, bm_ref = oracle.residual(ref, b_ref, r)
        assert same_bits(np.float32(rm), rm_ref) and same_bits(np.float32(bm), bm_ref)


@pytest.mark.parametrize("n", [3, 5, 17, 70, 130, 259])
@pytest.mark.parametrize("pad", [0, 12])
@pytest.mark.parametrize("division", ["auto", "ieee"])
def test_unfused_rhs_sweep_residual(n, pad, division):
    """Unfused right-hand side (section 02; section 05, Table VI): b keeps
    u^n and every sweep and residual forms fl(u^n + g) itself, the value the
    fused b holds, so sweeps and norms match the oracle bit for bit."""
    r = RS[(n + 1) % len(RS)]
    u0, g = fields(n, pad, seed=7 * n + 1)
    s, u, b = make_solver(u0, r, rhs="unfused", division=division)
    with s:
        s.rhs(to_dev(g))
        assert same_bits(interior(b.cpu().numpy()), interior(u0))
        b_ref = oracle.rhs(u0, g)
        rm, bm = s.residual()
        rm_ref, bm_ref = oracle.residual(u0, b_ref, r)
        assert same_bits(np.float32(rm), rm_ref) and same_bits(np.float32(bm), bm_ref)
        ref = u0
        for launches in (1, 3):
            s.sweeps(launches)
            ref = oracle.sweeps(ref, b_ref, r, launches)
            got = u.cpu().numpy()
            assert same_bits(interior(got), interior(ref)), mismatch(got, ref)
        assert np.isnan(got[:, n:]).all()
        rm, bm = s.residual()
        rm_ref, bm_ref = oracle.residual(ref, b_ref, r)
        assert same_bits(np.float32(rm), rm_ref) and same_bits(np.float32(bm), bm_ref)


# Compiled tile shapes of the exact-temporal-blocking kernel, per depth
# ((0, 0) selects the default).
ETB_TILES = {2: [(0, 0), (120, 60), (248, 60)],
             4: [(0, 0), (120, 56), (248, 56), (120, 40)],
             8: [(0, 0), (112, 80), (112, 48), (112, 112), (240, 48), (112, 92),
                 (112, 0)],  # (112, 0): whole columns, streamed (k_etbs)
             16: [(0, 0), (96, 64), (96, 96), (224, 64), (96, 76)]}
ETB_CASES = [(dd, t) for dd, ts in ETB_TILES.items() for t in ts]


@pytest.mark.parametrize("n", [17, 70, 130, 259, 520, 1030])
@pytest.mark.parametrize("depth,tile", ETB_CASES)
@pytest.mark.parametrize("division", ["auto", "ieee"])
def test_etb_launch_equals_depth_sync_sweeps(n, depth, tile, division):
    """Exact temporal blocking: one launch = D synchronous sweeps, bit for
    bit (section 02, ghost-zone technique), for every compiled tile shape and
    both division paths."""
    r = 10.0 if depth != 16 else 100.0
    u0, g = fields(n, 8, seed=3 * n + depth)
    s, u, b = make_solver(u0, r, strategy="etb", depth=depth, tile=tile,
                          division=division)
    with s:
        s.rhs(to_dev(g))
        b_ref = oracle.rhs(u0, g)
        s.sweeps(1)
        ref = oracle.sweeps(u0, b_ref, r, depth)
        got = u.cpu().numpy()
        assert same_bits(interior(got), interior(ref)), mismatch(got, ref)
        s.sweeps(2)
        ref = oracle.sweeps(ref, b_ref, r, 2 * depth)
        got = u.cpu().numpy()
        assert same_bits(interior(got), interior(ref)), mismatch(got, ref)
        assert np.isnan(got[:, n:]).all()


@pytest.mark.parametrize("n", [17, 70, 130, 259])
@pytest.mark.parametrize("depth", [1, 2, 4, 8, 16, 32])
@pytest.mark.parametrize("tile", [(32, 8), (32, 16), (64, 32), (4, 3), (128, 64)])
def test_block_async_launch_matches_emulator(n, depth, tile):
    """Block-asynchronous launch: tiles swept D times against halos frozen at
    launch (section 02), bit for bit against the oracle's emulator."""
    r = 1.0 if depth < 8 else 10.0
    u0, g = fields(n, 4, seed=5 * n + depth)
    s, u, b = make_solver(u0, r, strategy="ba", depth=depth, tile=tile)
    with s:
        s.rhs(to_dev(g))
        b_ref = oracle.rhs(u0, g)
        ref = u0
        for _ in range(2):
            s.sweeps(1)
            ref = oracle.ba_launch(ref, b_ref, r, tile[0], tile[1], depth)
            got = u.cpu().numpy()
            assert same_bits(interior(got), interior(ref)), mismatch(got, ref)
        if depth == 1:
            assert same_bits(interior(ref), interior(oracle.sweeps(u0, b_ref, r, 2)))


@pytest.mark.parametrize("n", [17, 70, 131, 259])
@pytest.mark.parametrize("depth", [1, 4, 8, 16, 32])
@pytest.mark.parametrize("tile,overlap", [
    ((32, 8), (2, 2)), ((32, 8), (4, 0)), ((32, 32), (4, 4)),
    ((16, 16), (6, 2)), ((8, 4), (2, 2)), ((64, 32), (30, 8)), ((4, 3), (2, 2)),
])
def test_block_async_overlap_matches_oracle(n, depth, tile, overlap):
    """Overlapping subdomains ("Hierarchical Jacobi Iteration for Structured
    Matrices on GPUs using Shared Memory"): tiles start every tile - overlap
    cells and write back their half of each shared band; bit for bit against
    the oracle's launch."""
    r = 1.0 if depth < 8 else 10.0
    u0, g = fields(n, 4, seed=11 * n + depth)
    s, u, b = make_solver(u0, r, strategy="ba", depth=depth, tile=tile,
                          overlap=overlap)
    with s:
        s.rhs(to_dev(g))
        b_ref = oracle.rhs(u0, g)
        ref = u0
        for _ in range(2):
            s.sweeps(1)
            ref = oracle.ba_overlap_launch(ref, b_ref, r, tile[0], tile[1],
                                           overlap[0], overlap[1], depth)
            got = u.cpu().numpy()
            assert same_bits(interior(got), interior(ref)), mismatch(got, ref)
        assert np.isnan(got[:, n:]).all()


@pytest.mark.parametrize("r", [1.0, 10.0, 100.0])
def test_fixed_divisor_division_enabled_for_page_couplings(r):
    """For d = 5, 41, 401 the fixed-divisor division passes its exhaustive
    check against IEEE division, so the fast path is the one that runs;
    forcing IEEE division is honoured."""
    u0, _ = fields(40, 0, seed=2)
    s, _, _ = make_solver(u0, r)
    with s:
        assert s.division_mode == 1
    s, _, _ = make_solver(u0, r, division="ieee")
    with s:
        assert s.division_mode == 0


def test_residual_propagates_nan():
    n = 40
    u0, g = fields(n, 0, seed=1)
    g[7, 9] = np.nan
    s, u, b = make_solver(u0, 1.0)
    with s:
        s.rhs(to_dev(g))
        rm, bm = s.residual()
        assert np.isnan(rm) and np.isnan(bm)


def test_no_fused_multiply_add():
    """Inputs where fl(b + fl(r*s)) differs from fma(r, s, b): the kernels
    must give the two-rounding result (the oracle's), not the fused one."""
    n = 6
    rng = np.random.default_rng(12)
    found = 0
    for _ in range(200):
        u0 = P.initial_field(n, 8)
        u0[1:n - 1, 1:n - 1] = rng.uniform(0, 1, (n - 2, n - 2)).astype(np.float32)
        g = np.zeros_like(u0)
        g[1:n - 1, 1:n - 1] = rng.uniform(0, 1, (n - 2, n - 2)).astype(np.float32)
        r = float(np.float32(rng.uniform(0.1, 3)))
        b_ref = oracle.rhs(u0, g)
        ref = oracle.sweep(u0, b_ref, r)
        # does a fused evaluation differ anywhere?
        r64 = np.float64(np.float32(r))
        uu = u0.astype(np.float64)
        s_ = ((uu[1:-1, :-2].astype(np.float32) + uu[1:-1, 2:].astype(np.float32))
              + (uu[:-2, 1:-1].astype(np.float32) + uu[2:, 1:-1].astype(np.float32)))
        fused = (b_ref[1:-1, 1:-1].astype(np.float64) + r64 * s_.astype(np.float64)).astype(np.float32)
        plain = (b_ref[1:-1, 1:-1] + np.float32(r) * s_).astype(np.float32)
        if np.array_equal(fused, plain):
            continue
        found += 1
        s, u, b = make_solver(u0, r)
        with s:
            s.rhs(to_dev(g))
            s.sweeps(1)
            assert same_bits(interior(u.cpu().numpy()), interior(ref))
        if found >= 5:
            break
    assert found >= 1
