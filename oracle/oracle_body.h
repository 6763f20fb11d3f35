/*
 * Body of the oracle, written once and instantiated twice by oracle.c:
 * REAL = float  (suffix f32) -- the precision the method runs in;
 * REAL = double (suffix f64) -- used only to pin the float32 oracle.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the product path may include, link or
 * call this code; the CUDA library shares no code with it.
 *
 * Source: "Synchronous vs block-async Jacobi on one RTX 5050"
 * (stencil-jacobian.vercel.app), sections 01 "The problem" and 02 "Method".
 *
 * Layout: an n-by-n grid including the Dirichlet ring, row-major with row
 * pitch ld (>= n) elements; A[i][j] is row i (i = 0 is the top), column j,
 * stored at A[i*ld + j]. Unknowns are the (n-2)^2 interior cells.
 *
 * Arithmetic: every operation below is one IEEE round-to-nearest operation in
 * REAL. The file is compiled with -ffp-contract=off so no multiply-add is
 * fused, and without fast-math so subnormals are kept.
 */

#define CAT2(a, b) a##_##b
#define CAT(a, b) CAT2(a, b)
#define FN(name) CAT(name, SFX)

/*
 * One Jacobi update of cell (i, j) for the backward-Euler system
 *   (1+4r) u_ij - r (uN + uS + uE + uW) = b_ij        (section 01)
 * with the iterate's neighbours on the right-hand side (section 02,
 * "Synchronous"):  J(u)_ij = (b_ij + r * s_ij) / d,  d = 1 + 4r.
 * Neighbour sum order: s = (uW + uE) + (uN + uS); the page fixes one
 * arithmetic definition for all kernels without printing the order, and this
 * pairing maps bit-for-bit under a left-right mirror.
 */
static REAL FN(jacobi_point)(REAL uw, REAL ue, REAL un, REAL us, REAL bij,
                             REAL r, REAL d) {
    REAL horiz = uw + ue;
    REAL vert = un + us;
    REAL s = horiz + vert;
    REAL rs = r * s;
    REAL num = bij + rs;
    return num / d;
}

static REAL FN(diag)(REAL r) {
    REAL four_r = (REAL)4 * r;
    return (REAL)1 + four_r;
}

/* Fused right-hand side, formed once per time step (section 02):
 * b = u + g on the interior. The ring of b is left
 * untouched (it is never read). */
void FN(oracle_rhs)(int n, long long ld, const REAL *u, const REAL *g,
                    REAL *b) {
    for (int i = 1; i < n - 1; ++i)
        for (int j = 1; j < n - 1; ++j) {
            long long p = (long long)i * ld + j;
            b[p] = u[p] + g[p];
        }
}

/* Rows i0 <= i < i1 (interior rows only) of one synchronous sweep. */
static void FN(sweep_rows)(int n, long long ld, REAL r, const REAL *u,
                           const REAL *b, REAL *out, int i0, int i1) {
    REAL d = FN(diag)(r);
    for (int i = i0; i < i1; ++i)
        for (int j = 1; j < n - 1; ++j) {
            long long p = (long long)i * ld + j;
            out[p] = FN(jacobi_point)(u[p - 1], u[p + 1], u[p - ld],
                                      u[p + ld], b[p], r, d);
        }
}

/* One synchronous sweep u -> out over all interior cells. The ring of out is
 * not written: the caller keeps both buffers' rings equal. */
void FN(oracle_sweep)(int n, long long ld, REAL r, const REAL *u,
                      const REAL *b, REAL *out) {
    FN(sweep_rows)(n, ld, r, u, b, out, 1, n - 1);
}

/* Is cell (i, j) on the Dirichlet ring? */
static int FN(on_ring)(int n, int i, int j) {
    return i == 0 || j == 0 || i == n - 1 || j == n - 1;
}

/*
 * Residual norms in the difference form of section 01 (chosen there because
 * forming b - Au directly loses digits to float32 cancellation). Per cell
 *   e_ij = d * |J(u)_ij - u_ij|,
 * which equals |b - A u|_ij in exact arithmetic because
 * d (J(u) - u) = b + r s - d u. J is evaluated exactly as in the sweep.
 *
 * ||b||inf is the norm of the right-hand side of the linear system in the
 * unknowns (section 01: every backward-Euler step is a linear solve):
 * the Dirichlet values are known, so they move to the right-hand side, and
 *   bI_ij = b_ij + r * q_ij,  q_ij = (qW + qE) + (qN + qS),
 * where qX is the neighbour's value when that neighbour is a ring cell and 0
 * otherwise. With this norm the stopping rule reproduces the section's sweep
 * counts per step (about 35, 226 and 1417 for r = 1, 10, 100).
 *
 * rmax = max e_ij, bmax = max |bI_ij| over the interior. A NaN anywhere makes
 * the corresponding norm NaN.
 */
/* Partial norms over rows i0 <= i < i1: the largest non-NaN e and |bI| seen
 * (from 0) and whether a NaN was seen. The maximum of a set does not depend
 * on the order it is taken in, so partials over any split of the rows combine
 * (max of the maxima, OR of the flags) to exactly the whole-grid result. */
static void FN(residual_rows)(int n, long long ld, REAL r, const REAL *u,
                              const REAL *b, int i0, int i1, REAL *rmax_out,
                              REAL *bmax_out, int *r_nan_out,
                              int *b_nan_out) {
    REAL d = FN(diag)(r);
    REAL rmax = 0, bmax = 0;
    int r_nan = 0, b_nan = 0;
    for (int i = i0; i < i1; ++i)
        for (int j = 1; j < n - 1; ++j) {
            long long p = (long long)i * ld + j;
            REAL ju = FN(jacobi_point)(u[p - 1], u[p + 1], u[p - ld],
                                       u[p + ld], b[p], r, d);
            REAL diff = ju - u[p];
            REAL e = d * (diff < 0 ? -diff : diff);
            REAL qw = FN(on_ring)(n, i, j - 1) ? u[p - 1] : (REAL)0;
            REAL qe = FN(on_ring)(n, i, j + 1) ? u[p + 1] : (REAL)0;
            REAL qn = FN(on_ring)(n, i - 1, j) ? u[p - ld] : (REAL)0;
            REAL qs = FN(on_ring)(n, i + 1, j) ? u[p + ld] : (REAL)0;
            REAL q = (qw + qe) + (qn + qs);
            REAL rq = r * q;
            REAL bi = b[p] + rq;
            REAL bb = bi < 0 ? -bi : bi;
            if (e != e) r_nan = 1;
            else if (e > rmax) rmax = e;
            if (bb != bb) b_nan = 1;
            else if (bb > bmax) bmax = bb;
        }
    *rmax_out = rmax;
    *bmax_out = bmax;
    *r_nan_out = r_nan;
    *b_nan_out = b_nan;
}

void FN(oracle_residual)(int n, long long ld, REAL r, const REAL *u,
                         const REAL *b, REAL *rmax_out, REAL *bmax_out) {
    REAL rmax, bmax;
    int r_nan, b_nan;
    FN(residual_rows)(n, ld, r, u, b, 1, n - 1, &rmax, &bmax, &r_nan, &b_nan);
    *rmax_out = r_nan ? (REAL)NAN : rmax;
    *bmax_out = b_nan ? (REAL)NAN : bmax;
}

/*
 * Row-parallel forms of the sweep and the residual, for checking large grids
 * in reasonable time. Every cell is computed by the same code as above, and a
 * sweep's cells are independent of each other (Jacobi reads only the previous
 * iterate), so splitting the interior rows among threads gives the same bits
 * as one thread; the residual's partial maxima combine exactly (see
 * residual_rows). threads <= 1 calls the single-threaded functions.
 */
typedef struct {
    int kind; /* 0 sweep, 1 residual */
    int n;
    long long ld;
    REAL r;
    const REAL *u, *b;
    REAL *out;
    int i0, i1;
    REAL rmax, bmax;
    int r_nan, b_nan;
} FN(rows_job);

static void *FN(rows_worker)(void *arg) {
    FN(rows_job) *j = (FN(rows_job) *)arg;
    if (j->kind == 0)
        FN(sweep_rows)(j->n, j->ld, j->r, j->u, j->b, j->out, j->i0, j->i1);
    else
        FN(residual_rows)(j->n, j->ld, j->r, j->u, j->b, j->i0, j->i1,
                          &j->rmax, &j->bmax, &j->r_nan, &j->b_nan);
    return NULL;
}

#define ORACLE_MAX_THREADS 256

/* Run `proto` over the interior rows split into `threads` contiguous ranges
 * (job 0 on the calling thread). Returns 0, or -2 if a thread could not be
 * started (all started threads are joined first). */
static int FN(run_rows)(int threads, const FN(rows_job) *proto,
                        FN(rows_job) *jobs) {
    int rows = proto->n - 2;
    if (threads > rows) threads = rows;
    if (threads < 1) threads = 1;
    pthread_t tid[ORACLE_MAX_THREADS];
    int started[ORACLE_MAX_THREADS];
    int rc = 0;
    for (int t = 0; t < threads; ++t) {
        jobs[t] = *proto;
        jobs[t].i0 = 1 + (int)((long long)rows * t / threads);
        jobs[t].i1 = 1 + (int)((long long)rows * (t + 1) / threads);
        started[t] = 0;
    }
    for (int t = 1; t < threads; ++t) {
        if (pthread_create(&tid[t], NULL, FN(rows_worker), &jobs[t]) == 0)
            started[t] = 1;
        else
            rc = -2;
    }
    if (rc == 0) FN(rows_worker)(&jobs[0]);
    for (int t = 1; t < threads; ++t)
        if (started[t]) pthread_join(tid[t], NULL);
    return rc;
}

static int FN(sweep_mt)(int threads, int n, long long ld, REAL r,
                        const REAL *u, const REAL *b, REAL *out) {
    if (threads <= 1) {
        FN(oracle_sweep)(n, ld, r, u, b, out);
        return 0;
    }
    FN(rows_job) proto = {0, n, ld, r, u, b, out, 0, 0, 0, 0, 0, 0};
    FN(rows_job) jobs[ORACLE_MAX_THREADS];
    return FN(run_rows)(threads, &proto, jobs);
}

static int FN(residual_mt)(int threads, int n, long long ld, REAL r,
                           const REAL *u, const REAL *b, REAL *rmax_out,
                           REAL *bmax_out) {
    if (threads <= 1) {
        FN(oracle_residual)(n, ld, r, u, b, rmax_out, bmax_out);
        return 0;
    }
    FN(rows_job) proto = {1, n, ld, r, u, b, NULL, 0, 0, 0, 0, 0, 0};
    FN(rows_job) jobs[ORACLE_MAX_THREADS];
    int nt = threads > n - 2 ? n - 2 : threads;
    if (FN(run_rows)(threads, &proto, jobs)) return -2;
    REAL rmax = 0, bmax = 0;
    int r_nan = 0, b_nan = 0;
    for (int t = 0; t < nt; ++t) {
        r_nan |= jobs[t].r_nan;
        b_nan |= jobs[t].b_nan;
        if (jobs[t].rmax > rmax) rmax = jobs[t].rmax;
        if (jobs[t].bmax > bmax) bmax = jobs[t].bmax;
    }
    *rmax_out = r_nan ? (REAL)NAN : rmax;
    *bmax_out = b_nan ? (REAL)NAN : bmax;
    return 0;
}

/*
 * Stopping rule (section 01): rho = ||b - Au||inf / ||b||inf < tol. The test
 * is made as rmax < tol * bmax in double, which needs no division and also
 * accepts rmax == 0 (covers bmax == 0).
 * Returns 1 converged, 0 not yet, -1 non-finite norms.
 */
static int FN(converged)(REAL rmax, REAL bmax, double tol) {
    double rm = (double)rmax, bm = (double)bmax;
    if (!isfinite(rm) || !isfinite(bm)) return -1;
    if (rm == 0.0) return 1;
    return rm < tol * bm ? 1 : 0;
}

static void FN(copy_interior)(int n, long long ld, const REAL *src, REAL *dst) {
    for (int i = 1; i < n - 1; ++i)
        memcpy(dst + (long long)i * ld + 1, src + (long long)i * ld + 1,
               (size_t)(n - 2) * sizeof(REAL));
}

/*
 * One block-asynchronous launch (section 02, "Block-asynchronous", after
 * Anzt et al.): the interior is cut into tiles of tx-by-ty cells whose first
 * tile starts at interior cell (1,1); tiles at the right and bottom edges are
 * partial. Each tile copies its cells plus a one-cell halo from u (the state
 * at launch), then sweeps its own cells depth times with Jacobi updates,
 * reading the halo as frozen values; only the tile's cells are written to
 * out. Inside a tile each sweep reads the previous in-tile iterate (two local
 * buffers), so the result does not depend on the order of cells.
 * With depth = 1 this is exactly one synchronous sweep.
 */
int FN(oracle_ba_launch)(int n, long long ld, REAL r, int tx, int ty,
                         int depth, const REAL *u, const REAL *b, REAL *out) {
    if (tx < 1 || ty < 1 || depth < 1) return -1;
    REAL d = FN(diag)(r);
    int lw = tx + 2, lh = ty + 2;
    REAL *cur = (REAL *)malloc(sizeof(REAL) * (size_t)lw * (size_t)lh);
    REAL *nxt = (REAL *)malloc(sizeof(REAL) * (size_t)lw * (size_t)lh);
    if (!cur || !nxt) { free(cur); free(nxt); return -2; }
    for (int y0 = 1; y0 < n - 1; y0 += ty) {
        int h = (y0 + ty <= n - 1) ? ty : (n - 1 - y0);
        for (int x0 = 1; x0 < n - 1; x0 += tx) {
            int w = (x0 + tx <= n - 1) ? tx : (n - 1 - x0);
            /* local (a, c) <-> grid (y0 - 1 + a, x0 - 1 + c) */
            for (int a = 0; a < h + 2; ++a)
                for (int c = 0; c < w + 2; ++c) {
                    REAL v = u[(long long)(y0 - 1 + a) * ld + (x0 - 1 + c)];
                    cur[a * lw + c] = v;
                    nxt[a * lw + c] = v;
                }
            for (int sweep = 0; sweep < depth; ++sweep) {
                for (int a = 1; a <= h; ++a)
                    for (int c = 1; c <= w; ++c) {
                        long long p = (long long)(y0 - 1 + a) * ld + (x0 - 1 + c);
                        nxt[a * lw + c] = FN(jacobi_point)(
                            cur[a * lw + c - 1], cur[a * lw + c + 1],
                            cur[(a - 1) * lw + c], cur[(a + 1) * lw + c],
                            b[p], r, d);
                    }
                REAL *t = cur; cur = nxt; nxt = t;
            }
            for (int a = 1; a <= h; ++a)
                for (int c = 1; c <= w; ++c)
                    out[(long long)(y0 - 1 + a) * ld + (x0 - 1 + c)] =
                        cur[a * lw + c];
        }
    }
    free(cur);
    free(nxt);
    return 0;
}

/*
 * Number of subdomains of t cells that start every t - o cells and together
 * cover ni cells ("Hierarchical Jacobi Iteration for Structured Matrices on
 * GPUs using Shared Memory", Eqs. 8-9: (N - o) / (tpb - o) blocks, rounded up
 * so that the last one reaches the end; one subdomain when t >= ni).
 */
static int FN(subdomains)(int ni, int t, int o) {
    if (ni <= t) return 1;
    return (ni - o + (t - o) - 1) / (t - o);
}

/*
 * One block-asynchronous launch on overlapping subdomains (same page, the
 * sections on overlapping subdomains in 1-D and 2-D, Eqs. 15-16).
 * Subdomain (p, q) holds the tx-by-ty interior cells starting at interior
 * column p*(tx-ox) and row q*(ty-oy) (cut at the grid's edge), plus a
 * one-cell halo. It is swept `depth` times against that halo frozen at its
 * value at launch, exactly as in oracle_ba_launch. Two neighbouring
 * subdomains share ox columns (oy rows); of these the left (upper) one
 * contributes the left (upper) half to `out` and the right (lower) one the
 * other half, the half that lies further from each one's edge. ox, oy even,
 * 0 <= ox < tx, 0 <= oy < ty; with ox = oy = 0 this is oracle_ba_launch.
 */
int FN(oracle_ba_overlap_launch)(int n, long long ld, REAL r, int tx, int ty,
                                 int ox, int oy, int depth, const REAL *u,
                                 const REAL *b, REAL *out) {
    if (tx < 1 || ty < 1 || depth < 1 || ox < 0 || oy < 0 || ox % 2 ||
        oy % 2 || ox >= tx || oy >= ty)
        return -1;
    const int ni = n - 2;
    const int kx = FN(subdomains)(ni, tx, ox), ky = FN(subdomains)(ni, ty, oy);
    REAL d = FN(diag)(r);
    int lw = tx + 2, lh = ty + 2;
    REAL *cur = (REAL *)malloc(sizeof(REAL) * (size_t)lw * (size_t)lh);
    REAL *nxt = (REAL *)malloc(sizeof(REAL) * (size_t)lw * (size_t)lh);
    if (!cur || !nxt) { free(cur); free(nxt); return -2; }
    for (int q = 0; q < ky; ++q) {
        int y0 = 1 + q * (ty - oy);
        int h = (y0 + ty <= n - 1) ? ty : (n - 1 - y0);
        /* rows this subdomain writes: [wy0, wy1) */
        int wy0 = y0 + (q > 0 ? oy / 2 : 0);
        int wy1 = (q < ky - 1) ? y0 + ty - oy / 2 : y0 + h;
        for (int p = 0; p < kx; ++p) {
            int x0 = 1 + p * (tx - ox);
            int w = (x0 + tx <= n - 1) ? tx : (n - 1 - x0);
            int wx0 = x0 + (p > 0 ? ox / 2 : 0);
            int wx1 = (p < kx - 1) ? x0 + tx - ox / 2 : x0 + w;
            for (int a = 0; a < h + 2; ++a)
                for (int c = 0; c < w + 2; ++c) {
                    REAL v = u[(long long)(y0 - 1 + a) * ld + (x0 - 1 + c)];
                    cur[a * lw + c] = v;
                    nxt[a * lw + c] = v;
                }
            for (int sweep = 0; sweep < depth; ++sweep) {
                for (int a = 1; a <= h; ++a)
                    for (int c = 1; c <= w; ++c) {
                        long long pp = (long long)(y0 - 1 + a) * ld + (x0 - 1 + c);
                        nxt[a * lw + c] = FN(jacobi_point)(
                            cur[a * lw + c - 1], cur[a * lw + c + 1],
                            cur[(a - 1) * lw + c], cur[(a + 1) * lw + c],
                            b[pp], r, d);
                    }
                REAL *t = cur; cur = nxt; nxt = t;
            }
            for (int gy = wy0; gy < wy1; ++gy)
                for (int gx = wx0; gx < wx1; ++gx)
                    out[(long long)gy * ld + gx] =
                        cur[(gy - y0 + 1) * lw + (gx - x0 + 1)];
        }
    }
    free(cur);
    free(nxt);
    return 0;
}

static long long FN(gcd)(long long a, long long b) {
    while (b) { long long t = a % b; a = b; b = t; }
    return a;
}

/*
 * Solve one backward-Euler step from the warm start u (= uⁿ; section 01
 * keeps uⁿ fixed inside b while the iterate moves): repeat launches of the chosen
 * strategy, and after every check interval evaluate the residual and stop
 * when the stopping rule holds.
 *   depth == 0 : synchronous sweeps, one sweep per launch.
 *   depth >= 1 : block-asynchronous launches of `depth` sweeps on tx-by-ty
 *                tiles (depth 1 reproduces the synchronous iterates).
 * The check interval is lcm(m, sweeps per launch) sweeps: a launch of several
 * sweeps cannot stop part-way, so with m = 8 and 16 sweeps per launch the
 * residual is read every 16 sweeps. Exact temporal blocking with depth D is,
 * by its definition, D synchronous sweeps; it is modelled here as depth == 0
 * with m = lcm(8, D).
 * On return u holds the last iterate (both buffers must carry the same ring;
 * work is scratch of the same shape). Returns the sweep count, or
 * -3 when max_sweeps is reached without convergence, -4 on non-finite norms,
 * -1 on bad arguments.
 */
long long FN(oracle_solve_step_mt)(int n, long long ld, REAL r, int m,
                                   double tol, long long max_sweeps,
                                   int depth, int tx, int ty, int ox, int oy,
                                   REAL *u, REAL *work, const REAL *b,
                                   REAL *rmax_out, REAL *bmax_out,
                                   int threads) {
    if (n < 3 || ld < n || m < 1 || depth < 0) return -1;
    if (threads > ORACLE_MAX_THREADS) threads = ORACLE_MAX_THREADS;
    long long per_launch = depth == 0 ? 1 : depth;
    long long interval = (long long)m / FN(gcd)(m, per_launch) * per_launch;
    long long launches_per_check = interval / per_launch;
    REAL *cur = u, *nxt = work;
    long long k = 0;
    long long status = 0;
    REAL rmax = 0, bmax = 0;
    for (;;) {
        for (long long l = 0; l < launches_per_check; ++l) {
            if (depth == 0) {
                if (FN(sweep_mt)(threads, n, ld, r, cur, b, nxt)) return -2;
            } else if (ox == 0 && oy == 0) {
                if (FN(oracle_ba_launch)(n, ld, r, tx, ty, depth, cur, b, nxt))
                    return -1;
            } else if (FN(oracle_ba_overlap_launch)(n, ld, r, tx, ty, ox, oy,
                                                    depth, cur, b, nxt))
                return -1;
            REAL *t = cur; cur = nxt; nxt = t;
        }
        k += interval;
        if (FN(residual_mt)(threads, n, ld, r, cur, b, &rmax, &bmax)) return -2;
        int c = FN(converged)(rmax, bmax, tol);
        if (c < 0) { status = -4; break; }
        if (c > 0) { status = k; break; }
        if (k >= max_sweeps) { status = -3; break; }
    }
    if (cur != u) FN(copy_interior)(n, ld, cur, u);
    if (rmax_out) *rmax_out = rmax;
    if (bmax_out) *bmax_out = bmax;
    return status;
}

/* The oracle of record: one thread. */
long long FN(oracle_solve_step)(int n, long long ld, REAL r, int m,
                                double tol, long long max_sweeps, int depth,
                                int tx, int ty, int ox, int oy, REAL *u,
                                REAL *work, const REAL *b, REAL *rmax_out,
                                REAL *bmax_out) {
    return FN(oracle_solve_step_mt)(n, ld, r, m, tol, max_sweeps, depth, tx,
                                    ty, ox, oy, u, work, b, rmax_out,
                                    bmax_out, 1);
}

/*
 * Ten (or `steps`) backward-Euler steps from u = u⁰ (section 01: a run is
 * ten successive time steps): b = u + g, then solve to the stopping
 * rule warm-started from uⁿ; the converged iterate becomes uⁿ⁺¹ in place.
 * sweeps[s] receives each step's count (or its negative status, after which
 * the run stops). Returns 0, or the first negative status.
 */
long long FN(oracle_run_mt)(int n, long long ld, REAL r, int m, double tol,
                            long long max_sweeps, int depth, int tx, int ty,
                            int ox, int oy, int steps, REAL *u, const REAL *g,
                            REAL *work, REAL *b, long long *sweeps,
                            int threads) {
    for (int s = 0; s < steps; ++s) {
        FN(oracle_rhs)(n, ld, u, g, b);
        long long k = FN(oracle_solve_step_mt)(n, ld, r, m, tol, max_sweeps,
                                               depth, tx, ty, ox, oy, u, work,
                                               b, 0, 0, threads);
        sweeps[s] = k;
        if (k < 0) return k;
    }
    return 0;
}

long long FN(oracle_run)(int n, long long ld, REAL r, int m, double tol,
                         long long max_sweeps, int depth, int tx, int ty,
                         int ox, int oy, int steps, REAL *u, const REAL *g,
                         REAL *work, REAL *b, long long *sweeps) {
    return FN(oracle_run_mt)(n, ld, r, m, tol, max_sweeps, depth, tx, ty, ox,
                             oy, steps, u, g, work, b, sweeps, 1);
}

#undef FN
#undef CAT
#undef CAT2
