/*
 * jacobi.h -- C ABI of the GB300 (sm_103a) five-point Jacobi solver for
 * implicit 2-D diffusion.
 *
 * The method is the one of "Synchronous vs block-async Jacobi on one
 * RTX 5050" (stencil-jacobian.vercel.app):
 *   section 01 "The problem": du/dt = alpha Lap u + f on an N x N unit square,
 *     backward Euler; each step solves (1+4r) u_ij - r (uN+uS+uE+uW) = b_ij,
 *     r = alpha dt / h^2, top boundary 100, the others 0, float32; a step
 *     converges when ||b - Au||inf / ||b||inf < 1e-5, checked every M = 8
 *     sweeps, the residual taken in a cancellation-free difference form;
 *   section 02 "Method": the synchronous sweep, the fused right-hand side
 *     b = u^n + dt f, the block-asynchronous kernel (tiles swept D times
 *     against frozen one-cell halos) and exact temporal blocking (a D-deep
 *     halo, shrinking valid region, bit-identical to D synchronous sweeps).
 *
 * Grid layout (all buffers): N x N float32 cells INCLUDING the Dirichlet ring,
 * row-major with row pitch `ld` floats; cell (i, j) -- row i, i = 0 the top,
 * column j -- lives at ptr[i * ld + j]. Requirements: N >= 3, ld >= N,
 * ld % 4 == 0 (16-byte rows), every base pointer 16-byte aligned. Columns
 * N..ld-1 are padding and are never read into a result or written.
 *
 * Arithmetic: every kernel evaluates
 *   J(u)_ij = ((uW + uE) + (uN + uS)) * r  added to b_ij, divided by d,
 *   d = 1 + 4r,
 * as float32 round-to-nearest operations in exactly that order, with no
 * fused multiply-add and with subnormals kept.
 *
 * Errors: every entry point returns a status (0 or a negative
 * jacobi_status_t); none aborts or traps. Device-side waits are bounded and
 * report JACOBI_ERR_CUDA through the handle when they give up.
 *
 * Threading: a handle is bound to one CUDA stream and must be used from one
 * host thread at a time. All work is enqueued on that stream.
 */
#ifndef TEMPORAL_BLOCKED_JACOBI_GB300_JACOBI_H
#define TEMPORAL_BLOCKED_JACOBI_GB300_JACOBI_H

#ifdef __cplusplus
extern "C" {
#endif

/* Strategies of section 02 "Method". */
typedef enum {
    JACOBI_SYNC = 0,                   /* one launch per sweep, ping-pong buffers */
    JACOBI_EXACT_TEMPORAL_BLOCKED = 1, /* D sweeps per launch, bit-identical to SYNC */
    JACOBI_BLOCK_ASYNC = 2             /* D in-tile sweeps per launch, frozen halos */
} jacobi_strategy_t;

typedef enum {
    JACOBI_OK = 0,
    JACOBI_ERR_INVALID_ARG = -1,  /* bad size, pitch, alignment, pointer or config */
    JACOBI_ERR_CUDA = -2,         /* a CUDA call failed or a device wait gave up */
    JACOBI_ERR_NOT_CONVERGED = -3,/* max_sweeps reached; u holds the last iterate */
    JACOBI_ERR_NONFINITE = -4,    /* a residual norm is NaN or Inf */
    JACOBI_ERR_UNSUPPORTED = -5   /* valid but not provided (e.g. tile too large) */
} jacobi_status_t;

/* How the convergence loop is driven. */
typedef enum {
    /* One CUDA graph per check interval; its last node copies (rmax, bmax)
     * to pinned host memory and the host makes the stop/continue decision,
     * as in section 02 where the reduction's two norms go back to the host. */
    JACOBI_CONTROL_HOST = 0,
    /* The check interval runs inside a device-side conditional WHILE graph
     * node, so a whole time step is one graph launch and one host
     * synchronisation. The first launch of each interval also reduces the
     * residual norms of its input iterate (its first sweep evaluates J(u)
     * anyway) and its last block applies the stopping rule and sets the loop
     * condition; launches queued after the stop return at once. Same
     * iterates, same sweep counts, same statuses as JACOBI_CONTROL_HOST. */
    JACOBI_CONTROL_DEVICE = 1,
    /* EXACT_TEMPORAL_BLOCKED only, with a register-resident tile shape (the
     * default tiles of D = 4, 8 and 16; other shapes return
     * JACOBI_ERR_UNSUPPORTED): a whole time step is one cooperative kernel
     * launch. Its blocks sweep the tiles D sweeps at a time and meet at a
     * grid-wide barrier between those rounds instead of at a kernel
     * boundary; the first round of each check interval reduces the residual
     * of its input and the last block to reach the following barrier applies
     * the stopping rule. Every barrier wait gives up after about a second
     * and the step then returns JACOBI_ERR_CUDA. Same iterates, sweep counts
     * and statuses as the other controls. */
    JACOBI_CONTROL_PERSISTENT = 2
} jacobi_control_t;

/* How the kernels divide by d = 1 + 4r. Both give the correctly rounded
 * float32 quotient for every finite numerator, so results are identical. */
typedef enum {
    /* Use a fixed-divisor division (one multiply and two fused multiply-adds
     * with the precomputed RN(1/d)) if an exhaustive check against IEEE
     * division over all finite float32 numerators passes for this d (run
     * once per distinct d and cached for the process, about 7 ms on
     * GB300); otherwise IEEE division. */
    JACOBI_DIVISION_AUTO = 0,
    /* Always the IEEE division instruction sequence. */
    JACOBI_DIVISION_IEEE = 1
} jacobi_division_t;

/* Where the right-hand side u^n + dt f is formed (section 02 and section 05,
 * Table VI: the fused form is the fair synchronous baseline). Both give the
 * same b_ij = fl(u^n_ij + g_ij) bit for bit, hence identical iterates. */
typedef enum {
    /* jacobi_rhs writes b = u^n + g once per time step; a sweep reads u and
     * b: 12 bytes per cell. */
    JACOBI_RHS_FUSED = 0,
    /* jacobi_rhs keeps u^n in b and a copy of g in a buffer the handle
     * allocates (N*ld floats); every sweep reads u, u^n and g and adds
     * u^n + g itself: 16 bytes per cell. SYNC only. */
    JACOBI_RHS_UNFUSED = 1
} jacobi_rhs_t;

/* Depth controllers for BLOCK_ASYNC (section 02: D is only a kernel
 * argument, so it may change between launches). D changes only at a residual
 * check, from the check's rho = rmax / bmax; the depths used are the powers
 * of two 1, 2, 4, ... up to the config's `depth`. The controller starts
 * afresh at every time step (jacobi_solve_step). */
typedef enum {
    JACOBI_ADAPT_NONE = 0,  /* fixed D = depth */
    /* G-asc: D = 1 while rho >= 1e-2, then doubled each time rho first falls
     * below 1e-2, 1e-3 and 1e-4; latched: a later rise of rho never lowers
     * it again within the step. */
    JACOBI_ADAPT_G_ASC = 1,
    /* G-desc: the mirror image, D = depth halved at each of the same
     * crossings (latched), never below 1. */
    JACOBI_ADAPT_G_DESC = 2,
    /* G-fb, hill climbing on the convergence rate per unit time: start at
     * D = 1; at each check measure rate = -ln(rho_k / rho_{k-1}) / t_k, t_k
     * the device time of the check interval in ms. The first measured rate
     * doubles D; afterwards D doubles while the rate stays at or above 90%
     * of the previously measured one and halves when it falls below (a drop
     * of more than 10%); every measured rate becomes the next comparison
     * point. After each change of D one measurement is skipped (settling:
     * the residual bump the change causes). D stays within [1, depth]. */
    JACOBI_ADAPT_G_FB = 3
} jacobi_adapt_t;

typedef struct {
    int strategy;         /* jacobi_strategy_t */
    int depth;            /* D: SYNC 1; EXACT_TEMPORAL_BLOCKED 2,4,8,16; BLOCK_ASYNC 1,2,4,8,16,32 */
    int tile_x, tile_y;   /* tile shape in cells; 0 = library default for the strategy.
                             tile_x a multiple of 4 for both tiled strategies;
                             BLOCK_ASYNC default 32 x 8 (section 02).
                             EXACT_TEMPORAL_BLOCKED defaults depend on n: the
                             register-resident shape that leaves each SM the
                             fewest box rows (D = 4: 120 x 88; D = 8: 112 x 80
                             or 112 x 92; D = 16: 96 x 64 or 96 x 76); D = 2:
                             120 x 92. At D = 8, on grids with enough rows
                             per warp (n from about 6000 on GB300; not under
                             JACOBI_CONTROL_PERSISTENT), the default is
                             112 x 0: tile_y = 0 selects the column-streamed
                             kernel, in which each warp sweeps a 112-column
                             strip D times as a pipeline down its rows (D = 8
                             only). Any shape gives the same bits. */
    int check_every;      /* M: residual checked every lcm(M, sweeps per launch) sweeps; default 8 */
    double tol;           /* stop when rmax < tol * bmax (or rmax == 0); default 1e-5 */
    long long max_sweeps; /* give up (JACOBI_ERR_NOT_CONVERGED) at this many sweeps; default 1<<22 */
    int control;          /* jacobi_control_t; default JACOBI_CONTROL_HOST */
    int division;         /* jacobi_division_t; default JACOBI_DIVISION_AUTO */
    int rhs;              /* jacobi_rhs_t; default JACOBI_RHS_FUSED */
    int adapt;            /* jacobi_adapt_t; default JACOBI_ADAPT_NONE. Other
                             values: BLOCK_ASYNC with depth 2, 4, 8 or 16 (the
                             largest D) and JACOBI_CONTROL_HOST only */
    int overlap_x, overlap_y; /* BLOCK_ASYNC overlapping subdomains ("Hierarchical
                             Jacobi Iteration for Structured Matrices on GPUs
                             using Shared Memory", overlapping subdomains in
                             1-D and 2-D): tiles start every tile_x - overlap_x
                             columns and tile_y - overlap_y rows, so
                             neighbours share overlap_x columns (overlap_y
                             rows); each tile sweeps all its cells against its
                             frozen one-cell halo and writes back the cells
                             of each shared band on its own side of the
                             band's middle. Even, 0 <= overlap < tile size;
                             default 0 (plain tiles). */
} jacobi_config_t;

typedef struct jacobi_handle jacobi_handle_t;

/* Fill *cfg with the defaults (SYNC, D 1, M 8, tol 1e-5, 1<<22 sweeps). */
int jacobi_config_default(jacobi_config_t *cfg);

/*
 * Create a solver over caller-owned device buffers.
 *   n, ld      grid side (ring included) and row pitch, see "Grid layout".
 *   r          alpha dt / h^2 (section 01), finite and >= 0.
 *   cfg        strategy and control; NULL = defaults.
 *   u          N*ld floats: on entry u^n with its ring filled; the solution
 *              of each step is left here.
 *   u_alt      N*ld floats of scratch for ping-pong; its ring is overwritten
 *              with u's ring here and never written again.
 *   b          N*ld floats that receive the right-hand side (interior only).
 *   cuda_stream a cudaStream_t (NULL = the legacy default stream).
 * The caller keeps ownership of u, u_alt, b and must keep them alive and
 * unmoved until jacobi_destroy. The handle owns its graphs, tensor maps,
 * reduction scratch and pinned host words. On failure *out is NULL.
 */
int jacobi_create(jacobi_handle_t **out, int n, long long ld, float r,
                  const jacobi_config_t *cfg, float *u, float *u_alt,
                  float *b, void *cuda_stream);

/*
 * Right-hand side of the next time step. With JACOBI_RHS_FUSED (section 02:
 * u^n + dt f is formed once per time step instead of inside every sweep):
 * b_ij = u_ij + g_ij on the interior, one float32 add per cell. With
 * JACOBI_RHS_UNFUSED: b receives a copy of u (= u^n) and the handle's own
 * buffer a copy of g, both on the interior; the sweeps form u^n + g. g is a
 * device buffer in the grid layout (g = dt f); it may be freed or changed
 * once this call's work has run. Asynchronous on the handle's stream. Call it
 * again after changing the rhs mode with jacobi_set_strategy: a solve whose b
 * was prepared for the other mode returns JACOBI_ERR_INVALID_ARG.
 */
int jacobi_rhs(jacobi_handle_t *h, const float *g);

/*
 * Solve one backward-Euler step from the warm start u = u^n (section 01:
 * u^n stays fixed inside b while the iterate changes), using b from jacobi_rhs: launches of
 * the configured strategy until the stopping rule holds at a check.
 * Returns the number of sweeps (>= 0, a multiple of the check interval;
 * for BLOCK_ASYNC launches x D) or a negative jacobi_status_t. On return
 * (success or NOT_CONVERGED / NONFINITE) u holds the last checked iterate.
 * Synchronises the stream.
 */
long long jacobi_solve_step(jacobi_handle_t *h);

/*
 * Run `launches` launches of the configured strategy on u with no residual
 * check (for kernel-level tests and timing). Returns the sweeps performed
 * (launches x sweeps per launch) or a negative status; the result is left
 * in u. Asynchronous.
 */
long long jacobi_sweeps(jacobi_handle_t *h, long long launches);

/*
 * Residual norms of the current u (section 01): rmax = max over the
 * interior of d |J(u) - u| (the difference form of |b - Au|), bmax = the
 * max-norm of the right-hand side of the system in the unknowns,
 * |b_ij + r (sum of the cell's Dirichlet-ring neighbours)|. NaN propagates
 * into the norm. Host pointers; synchronises the stream.
 */
int jacobi_residual(jacobi_handle_t *h, float *rmax, float *bmax);

/*
 * Residual norms without any allocation. The page has no counterpart for
 * this call; it exists for callers that cannot call cudaMalloc when they need
 * the norms: code running while a stream is being captured into a CUDA
 * graph, loops that must not pay for the device-wide synchronisation that
 * cudaMalloc/cudaFree imply, and applications whose device memory is handed
 * out only by their own allocator.
 *
 * It computes what jacobi_residual computes, for any u and b in the grid
 * layout, without a handle: norms[0] = rmax = max over the interior of
 * d |J(u) - u|, norms[1] = bmax = max |b_ij + r (sum of the cell's
 * Dirichlet-ring neighbours)|, d = 1 + 4r. u, b: device, N*ld floats,
 * 16-byte aligned. norms: device, 2 floats, written asynchronously on
 * cuda_stream (a stream of the current device; NULL = legacy default).
 *
 * Scratch: a fixed array in the library's device memory, reserved on every
 * GPU that loads the library until the process exits (about 256 KiB). All
 * calls share it, so calls that could overlap on the GPU (other streams,
 * other host threads) race and must be serialised by the caller. The first
 * call on each device looks up the array's device address; make that first
 * call before any stream capture. Every later call enqueues one kernel and
 * nothing else: the kernel's last block leaves the array ready for the next
 * call. Only the first call after a call on the same device that returned
 * JACOBI_ERR_CUDA also enqueues a 4-byte memset of the array's counter. It
 * calls no allocating routine.
 *
 * Returns JACOBI_OK, JACOBI_ERR_INVALID_ARG (sizes, pitch, r, NULL or
 * misaligned pointers), JACOBI_ERR_UNSUPPORTED when N exceeds
 * JACOBI_RESIDUAL_NOALLOC_MAX_N (the scratch holds partial maxima for at most
 * JACOBI_RESIDUAL_NOALLOC_MAX_BLOCKS reduction blocks; nothing is launched),
 * or JACOBI_ERR_CUDA.
 */
#define JACOBI_RESIDUAL_NOALLOC_MAX_BLOCKS 32768
#define JACOBI_RESIDUAL_NOALLOC_MAX_N 23168
int jacobi_residual_noalloc(int n, long long ld, float r, const float *u,
                            const float *b, float *norms, void *cuda_stream);

/*
 * Change strategy, depth, tile, tolerance or control between steps
 * (section 02: D is a launch parameter, so switching it costs nothing).
 * Rebuilds the handle's graphs. u must hold the current iterate.
 */
int jacobi_set_strategy(jacobi_handle_t *h, const jacobi_config_t *cfg);

/*
 * The time-step loop (section 01: a run is ten successive time steps): for each of
 * `steps` steps, jacobi_rhs(g) then jacobi_solve_step; u^{n+1} replaces u^n
 * in u. sweeps_per_step (host, `steps` entries, may be NULL) receives each
 * step's count. Returns the total sweep count or the first negative status.
 * b holds the last step's right-hand side afterwards. Under device control
 * with the column-streamed ETB(8) kernel and one launch per check interval,
 * each step's first sweep launch forms b = u^n + g itself (section 05 on
 * fusing the right-hand side); the results are the same bits.
 */
long long jacobi_run(jacobi_handle_t *h, const float *g, int steps,
                     long long *sweeps_per_step);

/*
 * Independent problems on host data (the time-step loop of section 01 for
 * each of `count` problems of the handle's size, r and configuration):
 * problem i starts from u0_host[i] (host, N*ld floats with its Dirichlet
 * ring), has source g_host[i] (host, N*ld floats) and runs `steps` time
 * steps as jacobi_run does; its final field is written to u_host[i] (host,
 * N*ld floats). sweeps (host, count * steps entries, may be NULL) receives
 * the sweeps of every step, problem by problem. Returns the total sweep
 * count or the first negative status (later problems are not run).
 *
 * The host-device copies overlap the solves: problem i + 1's inputs are
 * copied in, and problem i - 1's result out, while problem i is solved, on
 * a stream of the handle's own. Problems alternate between the handle's
 * fields and a second pair of fields solved by a twin handle (same
 * configuration, b and stream), so inputs and results move straight
 * between host memory and the fields that are solved. Host buffers should
 * be pinned (cudaHostAlloc or equivalent) for the copies to be
 * asynchronous. u, u_alt are overwritten (u holds the last problem's result
 * on return), and b receives the right-hand sides. On first use the handle
 * allocates four device buffers of N*ld floats (the twin's two fields and
 * the two sources), the twin handle, a stream and two events, kept until
 * jacobi_destroy. Synchronous: returns when every result is in host memory.
 */
long long jacobi_run_host(jacobi_handle_t *h, int count,
                          const float *const *u0_host,
                          const float *const *g_host, float *const *u_host,
                          int steps, long long *sweeps);

/*
 * One residual check of the last jacobi_solve_step, in order. depth: D of the
 * launches of that check interval; sweeps: sweeps done when the check was
 * taken; rmax, bmax: its norms; ms: device time of the interval (its launches
 * and the residual) from CUDA events, recorded under an adaptive depth
 * controller only (0 otherwise).
 */
typedef struct {
    int depth;
    int pad;
    long long sweeps;
    float rmax, bmax;
    float ms;
    float pad2;
} jacobi_check_record_t;

/*
 * Copy up to `cap` records of the last jacobi_solve_step's checks into rec
 * (host memory; may be NULL when cap is 0). Returns the number of checks of
 * that step (possibly more than cap) or a negative status. Recorded under
 * JACOBI_CONTROL_HOST; under JACOBI_CONTROL_DEVICE the step's checks run on
 * the device and 0 is returned.
 */
long long jacobi_check_trace(const jacobi_handle_t *h, jacobi_check_record_t *rec,
                             long long cap);

/*
 * The depth controller alone (host code; no GPU needed), as an adaptive
 * BLOCK_ASYNC solve runs it: jacobi_adapt_init starts it for one time step;
 * after each check jacobi_adapt_next takes the check's rho = rmax / bmax and
 * the interval's device time in ms and returns the D for the next interval
 * (>= 1) or a negative status (bad state). The state is plain data.
 */
typedef struct {
    int policy;        /* jacobi_adapt_t */
    int depth;         /* D of the next interval */
    int depth_max;     /* the config's depth */
    int level;         /* G-asc / G-desc: thresholds crossed so far (latched) */
    int settle;        /* G-fb: measurements still to skip */
    int have_prev;     /* G-fb: rho_prev holds the previous check's rho */
    int have_ref;      /* G-fb: rate_ref holds the previous measured rate */
    int changes;       /* changes of D so far */
    double rho_prev;
    double rate_ref;
} jacobi_adapt_state_t;

int jacobi_adapt_init(jacobi_adapt_state_t *st, int policy, int depth_max);
int jacobi_adapt_next(jacobi_adapt_state_t *st, double rho, double ms);

/* Division the handle's kernels use: 1 = verified fixed-divisor division,
 * 0 = IEEE division, < 0 = error (NULL handle). */
int jacobi_division_mode(const jacobi_handle_t *h);

/* The tile the handle's tiled kernel uses (the default resolved), into
 * *tile_x, *tile_y (host ints); 0 x 0 for SYNC. For EXACT_TEMPORAL_BLOCKED,
 * tile_y = 0 is the column-streamed kernel (see jacobi_config_t). Returns
 * JACOBI_OK or JACOBI_ERR_INVALID_ARG (NULL argument). */
int jacobi_tile(const jacobi_handle_t *h, int *tile_x, int *tile_y);

/*
 * Bounds-checked build. The pages have no counterpart for these calls; they
 * serve testing. The same sources built with JACOBI_BOUNDS_CHECK give
 * libtbjacobi_checked.so, with the same entry points and results, in which
 * the tiled kernels (exact temporal blocking and block-async, all tile
 * shapes) check every shared-memory access, plain global load, global store
 * and TMA box load against its range. An access out of range is not
 * performed; the launch's error word records it and the next call that
 * reads that word (solve, residual) returns JACOBI_ERR_CUDA with the message
 * "bounds check: ...". Nothing traps. Stores are allowed on interior cells
 * only (rows and columns 1 .. N-2), never on the Dirichlet ring or the row
 * padding. The checked build also fills each block's dynamic shared memory
 * with NaN at kernel entry, and the destination field's interior with NaN
 * before every sweep launch (not under JACOBI_CONTROL_PERSISTENT), so a
 * value read before it was written, or an interior cell that a launch does
 * not write, turns the result into NaN. It is slower and not meant for
 * timing.
 *
 * jacobi_bounds_checked: 1 in the checked library, 0 otherwise.
 * jacobi_bounds_selftest: runs the checker on five accesses of its own on
 * the handle's u (one thread; synchronises the stream; allocates and frees
 * 20 bytes of device memory): a shared-memory load past the region declared
 * to the checker (bit 0), stores to a ring row (bit 1) and a ring column
 * (bit 2) of u, a shared load inside the region (bit 3) and a store to
 * interior cell (1, 1) (bit 4). Every store writes back the value the cell
 * holds. Returns the mask of the accesses that were refused -- 0x7 when the
 * checker works -- or a negative status; JACOBI_ERR_UNSUPPORTED in the
 * unchecked library.
 */
int jacobi_bounds_checked(void);
int jacobi_bounds_selftest(jacobi_handle_t *h);

/* Number of kernels this handle has launched so far (graph nodes included). */
long long jacobi_launch_count(const jacobi_handle_t *h);

/* Release library-owned state only; the caller's buffers are untouched. */
void jacobi_destroy(jacobi_handle_t *h);

/* Text of the last error on this handle ("" if none); valid until the next
 * call on the handle. For h == NULL, the last jacobi_create failure. */
const char *jacobi_last_error(const jacobi_handle_t *h);

/* Static name of a status code. */
const char *jacobi_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* TEMPORAL_BLOCKED_JACOBI_GB300_JACOBI_H */
