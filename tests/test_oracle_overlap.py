"""Pins of the oracle's block-asynchronous launch on overlapping subdomains
("Hierarchical Jacobi Iteration for Structured Matrices on GPUs using Shared
Memory", overlapping subdomains in 1-D and 2-D: neighbouring subdomains
share an even number of interior points; each shared point is written back by
the subdomain in which it lies further from the edge).

The brute force here builds the result differently from the oracle: each
subdomain is an independent small grid whose fixed border is its frozen
halo, swept with whole-array float32 arithmetic (checked against the pinned
synchronous oracle sweep), and every cell takes the value of the subdomain
whose edges are furthest from it in both directions.
"""
import numpy as np
import pytest

import oracle
from temporal_blocked_jacobi_gb300 import problem as P


def subdomain_starts(ni, t, o):
    """Interior offsets of the subdomains covering ni cells (the page's
    (N - o) / (tpb - o) blocks, enough to reach the end)."""
    starts = [0]
    while starts[-1] + t < ni:
        starts.append(starts[-1] + t - o)
    return starts


def owner(x, starts, t, ni):
    """Index of the subdomain in which interior offset x lies furthest from
    the subdomain's edges: the one whose (nominal, uncut) centre is nearest.
    With even overlaps two centres are never equally near an integer x."""
    best, best_dist = None, None
    for k, s in enumerate(starts):
        if s <= x < s + t:
            dist = abs(x - (s + (t - 1) / 2))
            assert best_dist is None or dist != best_dist
            if best_dist is None or dist < best_dist:
                best, best_dist = k, dist
    return best


def box_sweeps(box, bbox, r, depth):
    """`depth` Jacobi sweeps of a rectangular float32 box whose border is held
    fixed (numpy float32: one rounding per operation, no fused multiply-add),
    ((W + E) + (N + S)) * r + b, divided by 1 + 4r."""
    r = np.float32(r)
    d = np.float32(1) + np.float32(4) * r
    cur = box.copy()
    for _ in range(depth):
        nxt = cur.copy()
        s = (cur[1:-1, :-2] + cur[1:-1, 2:]) + (cur[:-2, 1:-1] + cur[2:, 1:-1])
        nxt[1:-1, 1:-1] = (bbox[1:-1, 1:-1] + r * s) / d
        cur = nxt
    return cur


def test_box_sweeps_is_the_oracle_sweep():
    u, b = fields(19, seed=3, ld=19)
    assert same(box_sweeps(u, b, 10.0, 3), oracle.sweeps(u, b, 10.0, 3))


def brute_force(u, b, r, tx, ty, ox, oy, depth):
    n = u.shape[0]
    ni = n - 2
    sx, sy = subdomain_starts(ni, tx, ox), subdomain_starts(ni, ty, oy)
    results = {}
    for q, y0 in enumerate(sy):
        for p, x0 in enumerate(sx):
            h, w = min(ty, ni - y0), min(tx, ni - x0)
            # grid rows 1 + y0 - 1 .. 1 + y0 + h: the subdomain and its halo
            box = np.ascontiguousarray(u[y0:y0 + h + 2, x0:x0 + w + 2])
            bbox = np.ascontiguousarray(b[y0:y0 + h + 2, x0:x0 + w + 2])
            results[(q, p)] = box_sweeps(box, bbox, r, depth)
    out = u.copy()
    for i in range(ni):
        q = owner(i, sy, ty, ni)
        for j in range(ni):
            p = owner(j, sx, tx, ni)
            out[1 + i, 1 + j] = results[(q, p)][1 + i - sy[q], 1 + j - sx[p]]
    return out


def fields(n, seed, ld=None):
    ld = P.padded_ld(n) if ld is None else ld
    u = P.random_field(n, ld, seed)
    g = P.random_field(n, ld, seed + 1)
    return u, oracle.rhs(u, g)


def same(a, b):
    return np.array_equal(a.view(np.uint32), b.view(np.uint32))


@pytest.mark.parametrize("n,tx,ty,ox,oy,depth", [
    (20, 8, 8, 2, 2, 4), (20, 8, 4, 4, 2, 3), (23, 12, 8, 6, 0, 5),
    (17, 4, 4, 2, 2, 2), (30, 16, 8, 0, 4, 8), (26, 8, 6, 6, 4, 6),
    (12, 32, 32, 4, 4, 8), (40, 12, 10, 10, 8, 4),
])
def test_overlap_launch_matches_brute_force(n, tx, ty, ox, oy, depth):
    u, b = fields(n, seed=n + tx + ox)
    r = 10.0
    got = oracle.ba_overlap_launch(u, b, r, tx, ty, ox, oy, depth)
    want = brute_force(u, b, r, tx, ty, ox, oy, depth)
    assert same(got[:n, :n], want[:n, :n])


@pytest.mark.parametrize("tile", [(32, 8), (8, 4), (12, 12)])
@pytest.mark.parametrize("depth", [1, 2, 8])
def test_zero_overlap_is_plain_block_async(tile, depth):
    u, b = fields(37, seed=depth)
    got = oracle.ba_overlap_launch(u, b, 1.0, tile[0], tile[1], 0, 0, depth)
    assert same(got, oracle.ba_launch(u, b, 1.0, tile[0], tile[1], depth))


@pytest.mark.parametrize("ov", [(2, 2), (6, 0), (0, 4)])
def test_depth_one_is_one_sweep(ov):
    u, b = fields(29, seed=5)
    got = oracle.ba_overlap_launch(u, b, 100.0, 8, 8, ov[0], ov[1], 1)
    assert same(got, oracle.sweep(u, b, 100.0))


def test_single_subdomain_is_synchronous():
    u, b = fields(18, seed=9)
    got = oracle.ba_overlap_launch(u, b, 10.0, 16, 16, 4, 4, 6)
    assert same(got, oracle.sweeps(u, b, 10.0, 6))


def test_mirror_symmetric_tiling_keeps_symmetry():
    # ni = 20 = 8 + 2 * (8 - 2): three subdomains per row, symmetric
    n = 22
    c = (n - 1) / 2
    u = P.initial_field(n, 24)
    g = P.source_term(n, 24, "gauss", center=(c, c))
    b = oracle.rhs(u, g)
    for _ in range(5):
        u = oracle.ba_overlap_launch(u, b, 10.0, 8, 4, 2, 2, 4)
        inner = u[:, :n]
        assert same(np.ascontiguousarray(inner), np.ascontiguousarray(inner[:, ::-1]))


def test_overlap_reduces_sweeps():
    """Overlap improves the values near subdomain edges, so fewer sweeps
    reach the tolerance (the page's cycle counts fall with overlap)."""
    n, r = 66, 10.0
    u0 = P.initial_field(n)
    b = oracle.rhs(u0, P.source_term(n, kind="gauss"))
    counts = []
    for ov in (0, 4, 8):
        u = u0.copy()
        k, _, _ = oracle.solve_step(u, b, r, depth=16, tile_x=16, tile_y=16,
                                    overlap=(ov, ov))
        counts.append(k)
    assert counts[0] > counts[1] > counts[2] > 0


def test_bad_overlap_rejected():
    u, b = fields(20, seed=1)
    for ox, oy in ((1, 0), (0, 3), (8, 0), (-2, 0)):
        with pytest.raises(ValueError):
            oracle.ba_overlap_launch(u, b, 1.0, 8, 8, ox, oy, 2)
