// Exact temporal blocking, column-streamed ("Synchronous vs block-async
// Jacobi on one RTX 5050", section 02 "Exact temporal blocking"): one launch
// performs D synchronous sweeps and is bit-identical to D launches of the
// synchronous sweep, like k_etbr, but with no block-level cooperation.
//
// A warp owns a strip of 128 grid columns (lane l holds columns
// bxo + 4l .. bxo + 4l + 3, bxo = s*TX - HX) and streams down it, one input
// row per step, holding D levels of a software pipeline in registers: level
// k is the field after k sweeps. When input row r arrives, level 1 computes
// row r-1 from level 0's rows r-2, r-1, r; level 2 computes row r-2 from
// level 1's rows r-3, r-2, r-1 (the last one computed a moment ago); ...;
// level D computes row r-D, which is final. Each level keeps the two rows it
// last received, in registers; b is read, per level, from the rows staged in
// shared memory. West and east neighbours come from the adjacent lanes by
// shuffle. Cells move out of
// the exact region one column per level at the strip's two edges, so after
// D levels the TX = 128 - 2*HX columns in the middle (HX = D rounded up to a
// multiple of 4 >= D) are exact: the strip's output. Rows need no halo
// beyond the D rows streamed before and after a run of output rows.
//
// So every warp sweeps its own strip with no barrier and no shared-memory
// exchange, and the only redundant cells are the strip's 2*HX halo columns
// (about 1.14x at D = 8) and the 2*D rows that fill and drain the pipeline
// per run. Work is handed out dynamically: the grid's rows are cut into
// bands and each band into one run per strip; the warps of the persistent
// grid take runs from a counter in band order, so the strips of a band run
// side by side (their shared halo columns come from L2) and a warp that
// finishes early takes more. Bands shrink toward the bottom of the grid
// (guided scheduling: a run is the work left divided by twice the warps, at
// most kBandMax and at least kBandMin rows), so the launch ends with short
// runs instead of a long tail. The last warp to finish resets the counter
// for the next launch. Measured on GB300 at N = 8192 / 12288 / 18432 (us
// per launch, when these settings took 236 / 477 / 959): runs of the work
// left over the warps alone, 64 to 256 rows, 247 / 461 / 978; fixed
// 128-row runs 229 / 474 / 1028; fixed 256 235 / - / 983; one static share
// per warp 272 / - / 1294. With the current source (230 / - / 924 us), a
// largest run of 256, 384, 640, 1024 or 2048 rows instead of 512 takes
// 933, 934, 949, 1002, 1002 us at N = 18432.
//
// Input rows reach the warp through rings of rows of u and b in its slice
// of shared memory, filled with cp.async kAhead rows ahead; a row's b stays
// there while levels 1 .. D still need it (kRing >= D + kAhead + 1).
// Lane l copies and reads back only its own 16 bytes of each row. Rows and
// columns outside the array are zero-filled. Cells that are not interior
// grid cells keep their value at every level (the Dirichlet ring).
//
// Three variants: plain; residual-fused (the device-side loop's launches:
// level 1 also reduces max |J(u) - u| of the launch's input); and
// right-hand-side (a time step's first launch in a whole run: it forms
// b = u^n + g as the rows of u^n arrive).
//
// Compiled for D = 8, the depth it is made for: at D = 4 the register-band
// kernel is already close to the HBM bound, and at D = 16 the 2*D rows of
// pipeline state do not fit in registers.
#include "jacobi_kernels.cuh"

namespace tbj {
namespace {

constexpr unsigned FULL = 0xffffffffu;
constexpr int kWarps = 4;   // warps per block, each independent
constexpr int kRing = 16;   // staged b rows per warp (a power of 2)
constexpr int kURing = 4;   // staged u rows per warp (a power of 2 > kAhead)
constexpr int kAhead = 3;   // rows staged ahead of the one consumed
constexpr int kBandMax = 512, kBandMin = 64;  // rows of a run
constexpr int kGuide = 2;  // a run is the work left / (kGuide x warps)

// Floats of one warp's staging: b twice in kRing slots, u in kURing slots,
// 128 floats (one row of the strip) each.
constexpr int kSliceFloats = (2 * kRing + kURing) * 128;

template <int D>
struct EtbsShape {
    static constexpr int HX = (D + 3) / 4 * 4;  // halo columns per side
    static constexpr int TX = 128 - 2 * HX;     // output columns per strip
};

// One 16-byte asynchronous copy global -> shared from grid `base`; `in` false
// writes zeros and reads nothing. (Checked build: dropped when out of range.)
__device__ __forceinline__ void cp16(float *dst, const float *base,
                                     const float *src, bool in) {
    if (!smem_ok(dst, 16) || (in && !load_ok(base, src, 4))) return;
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(
                     static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
                 "l"(in ? src : base), "r"(in ? 16u : 0u)
                 : "memory");
}
__device__ __forceinline__ void cp_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// One run of output rows [ya, yb) of the strip whose box starts at column
// bxo. sw: this warp's staging slice (kSliceFloats floats).
//
// FUSED: rmf accumulates max |J(u) - u| of the run's cells (level 1).
// RHS (the first launch of a time step): bsrc is the source term g and the
// launch forms the step's right-hand side b = fl(u + g) itself, from its
// input u = u^n, as each row is staged: the levels read it from the b ring
// as usual, the run's output cells of b go to bout, and rmf accumulates
// max |b| over those of them that have no Dirichlet-ring neighbour (for
// them b_I = b; the ring-adjacent cells are reduced by k_bnorm_ring).
template <int D, bool FAST, bool EDGE, bool FUSED, bool RHS>
__device__ __forceinline__ void etbs_run(const float *__restrict__ src,
                                         const float *__restrict__ bsrc,
                                         float *__restrict__ out,
                                         float *__restrict__ bout, float *sw,
                                         int n, long long ld, float r, float d,
                                         float y, int bxo, int ya, int yb,
                                         float &rmf) {
    static_assert(!(FUSED && RHS), "a right-hand-side launch checks nothing");
    using S = EtbsShape<D>;
    const int lane = threadIdx.x & 31;
    const int c0 = bxo + 4 * lane;  // this lane's first grid column
    const int left = (lane + 31) & 31, right = (lane + 1) & 31;
    const bool col_in = c0 >= 0 && c0 + 3 < ld;  // the 16 bytes exist
    unsigned colmask = 0xfu;  // interior columns among the lane's four
    if (EDGE) {
        colmask = 0u;
#pragma unroll
        for (int k = 0; k < 4; ++k)
            colmask |= (c0 + k >= 1 && c0 + k <= n - 2) ? (1u << k) : 0u;
    }
    const bool in_tile = 4 * lane >= S::HX && 4 * lane < S::HX + S::TX;

    static_assert(kRing >= D + kAhead + 1, "b rows must outlive their levels");
    // Input rows ra .. ra + steps - 1 (rows past the run are streamed in, as
    // zeros past the array, and never written). Output rows leave level D
    // at steps t >= 2D; level 1 computes output row ya + t - D - 1.
    const int ra = ya - D;
    const int steps = (yb - ya) + 2 * D;
    // This lane's 16 bytes of the staging rows: u in kURing slots, b in
    // kRing slots stored twice (slot s and s + kRing), so that the b rows
    // that levels 1 .. D read at one step are consecutive slots below one
    // base and need no index arithmetic of their own.
    float *bown = sw + 4 * lane;
    float *uown = sw + 2 * kRing * 128 + 4 * lane;
    int row = ra;  // next row to stage
    const float *pu = src + (long long)ra * ld + c0;
    const float *pb = bsrc + (long long)ra * ld + c0;
    float *po = out + (long long)(ra - D) * ld + c0;  // output row ra + t - D
    float *pbo = RHS ? bout + (long long)ra * ld + c0 : nullptr;  // b, row ra + t
    unsigned deepmask = 0xfu;  // cells of the lane with no ring neighbour
    if (RHS && EDGE) {
        deepmask = 0u;
#pragma unroll
        for (int k = 0; k < 4; ++k)
            deepmask |= (c0 + k >= 2 && c0 + k <= n - 3) ? (1u << k) : 0u;
    }

    auto issue = [&](int t) {  // stage input row ra + t (== row)
        // Interior runs stage rows and columns that all exist (the caller
        // keeps kAhead rows of margin below them), so their copies need no
        // test; edge runs zero-fill what lies outside the array.
        const bool in = !EDGE || (col_in && row >= 0 && row < n);
        cp16(uown + (t & (kURing - 1)) * 128, src, pu, in);
        float *bs = bown + (t & (kRing - 1)) * 128;
        cp16(bs, bsrc, pb, in);
        cp16(bs + kRing * 128, bsrc, pb, in);
        cp_commit();
        ++row;
        pu += ld;
        pb += ld;
    };
#pragma unroll
    for (int t = 0; t < kAhead; ++t) issue(t);

    const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
    float4 wa[D], wb[D];  // level k: rows i-1, i it last received
#pragma unroll
    for (int k = 0; k < D; ++k) {
        wa[k] = z;
        wb[k] = z;
    }

    // Each level's rows rotate through three registers (the two it holds
    // and the one it receives), so three steps per loop iteration let the
    // compiler rename instead of move; more steps per iteration outgrow the
    // instruction cache (measured on GB300: 1294 us per launch at N = 18432
    // with 3, 1434 with 1, 1520 with 2, 1805 with 6, 1733 with 8).
#pragma unroll 3
    for (int t = 0; t < steps; ++t) {
        // Row ra + t + kAhead replaces the row kRing rows before it, whose b
        // the last level used D steps after it arrived.
        issue(t + kAhead);
        cp_wait<kAhead>();  // row ra + t has landed
        float4 fresh = lds4(uown + (t & (kURing - 1)) * 128);  // level 0
        if (RHS) {
            // b of input row ra + t over its g, in both of its slots, before
            // level 1 reads it at the next step.
            float *bs = bown + (t & (kRing - 1)) * 128;
            const float4 gq = lds4(bs);
            const float4 bq = make_float4(
                __fadd_rn(fresh.x, gq.x), __fadd_rn(fresh.y, gq.y),
                __fadd_rn(fresh.z, gq.z), __fadd_rn(fresh.w, gq.w));
            sts4(bs, bq);
            sts4(bs + kRing * 128, bq);
            const int i = ra + t;
            if (in_tile && i >= ya && i < yb && colmask) {
                if (colmask == 0xfu) {
                    gst4(pbo, bq);
                } else {
                    if (colmask & 1u) gst1(pbo + 0, bq.x);
                    if (colmask & 2u) gst1(pbo + 1, bq.y);
                    if (colmask & 4u) gst1(pbo + 2, bq.z);
                    if (colmask & 8u) gst1(pbo + 3, bq.w);
                }
                if (!EDGE) {
                    rmf = max_nan_abs(rmf, bq.x);
                    rmf = max_nan_abs(rmf, bq.y);
                    rmf = max_nan_abs(rmf, bq.z);
                    rmf = max_nan_abs(rmf, bq.w);
                } else if (i >= 2 && i <= n - 3) {
                    if (deepmask & 1u) rmf = max_nan_abs(rmf, bq.x);
                    if (deepmask & 2u) rmf = max_nan_abs(rmf, bq.y);
                    if (deepmask & 4u) rmf = max_nan_abs(rmf, bq.z);
                    if (deepmask & 8u) rmf = max_nan_abs(rmf, bq.w);
                }
            }
            pbo += ld;
        }
        // b of row ra + t - k sits k - 1 slots below bk1 (level 1's)
        const float *bk1 = bown + (((t - 1) & (kRing - 1)) + kRing) * 128;
        const bool out_row = t >= 2 * D;
        const bool res_row = t > D && t <= D + (yb - ya);
#pragma unroll
        for (int k = 1; k <= D; ++k) {
            const int i = ra + t - k;  // row this level computes
            const float4 north = wa[k - 1], cur = wb[k - 1];
            const float wv = __shfl_sync(FULL, cur.w, left);
            const float ev = __shfl_sync(FULL, cur.x, right);
            const float4 bi = lds4(bk1 - (k - 1) * 128);
            float4 nv = update4_we<FAST>(north, cur, fresh, bi, wv, ev, r, d, y);
            const bool row_ok = !EDGE || (i >= 1 && i <= n - 2);
            if (EDGE) nv = hold4(nv, cur, row_ok, colmask);
            if (FUSED && k == 1 && in_tile && res_row && row_ok) {
                const float2 d01 = __fadd2_rn(make_float2(nv.x, nv.y),
                                              make_float2(-cur.x, -cur.y));
                const float2 d23 = __fadd2_rn(make_float2(nv.z, nv.w),
                                              make_float2(-cur.z, -cur.w));
                if (colmask & 1u) rmf = max_nan_abs(rmf, d01.x);
                if (colmask & 2u) rmf = max_nan_abs(rmf, d01.y);
                if (colmask & 4u) rmf = max_nan_abs(rmf, d23.x);
                if (colmask & 8u) rmf = max_nan_abs(rmf, d23.y);
            }
            if (k == D && in_tile && out_row && row_ok && colmask) {
                float *g = po;
                if (colmask == 0xfu) {
                    gst4(g, nv);
                } else {
                    if (colmask & 1u) gst1(g + 0, nv.x);
                    if (colmask & 2u) gst1(g + 1, nv.y);
                    if (colmask & 4u) gst1(g + 2, nv.z);
                    if (colmask & 8u) gst1(g + 3, nv.w);
                }
            }
            wa[k - 1] = cur;
            wb[k - 1] = fresh;
            fresh = nv;
        }
        po += ld;
    }
    cp_wait<0>();  // the rows staged past the run, before the slots are reused
}

// RHS: bsrc is g; the launch also writes the step's b into bout and folds
// max |b| of the cells without ring neighbours into lp.state->bmax.
template <int D, bool FAST, bool FUSED, bool RHS>
__global__ void __launch_bounds__(32 * kWarps, 3)
k_etbs(const float *__restrict__ src, const float *__restrict__ bsrc,
       float *__restrict__ out, float *__restrict__ bout, int n, long long ld,
       float r, float d, float y, int strips, int *work, int bands,
       unsigned *err, const int *stop, LoopParams lp) {
    using S = EtbsShape<D>;
    __shared__ unsigned fin_scratch[33];
    extern __shared__ __align__(16) float smem[];  // kWarps slices
    bounds_begin(smem, 0, out, RHS ? bout : nullptr, src, bsrc, n, ld, err);
    allow_dependents();
    grid_dependency_wait();
    if (stop && *stop) return;  // same value for every thread of the launch
    float rmf = 0.f;
    float *sw = smem + (threadIdx.x >> 5) * kSliceFloats;
    const int lane = threadIdx.x & 31;
    const unsigned runs = (unsigned)bands * (unsigned)strips;
    const int *band_start = work + 2;
    for (;;) {
        unsigned c = 0u;
        if (lane == 0) c = atomicAdd(reinterpret_cast<unsigned *>(work), 1u);
        c = __shfl_sync(FULL, c, 0);
        if (c >= runs) break;  // uniform per warp
        const int s = (int)(c % (unsigned)strips);
        const int band = (int)(c / (unsigned)strips);
        const int ya = band_start[band], yb = band_start[band + 1];
        const int bxo = s * S::TX - S::HX;
        // Interior runs: every cell of the strip's box is an interior grid
        // cell and the kAhead rows staged past the run exist.
        const bool edge = bxo < 1 || bxo + 128 > n - 1 || ya - D < 1 ||
                          yb + D + kAhead > n;
        if (edge)
            etbs_run<D, FAST, true, FUSED, RHS>(src, bsrc, out, bout, sw, n, ld,
                                                r, d, y, bxo, ya, yb, rmf);
        else
            etbs_run<D, FAST, false, FUSED, RHS>(src, bsrc, out, bout, sw, n,
                                                 ld, r, d, y, bxo, ya, yb, rmf);
    }
    // The last warp out re-arms the work list for the next launch (a launch
    // starts only after the previous one has finished, PDL included).
    if (lane == 0) {
        __threadfence();
        const unsigned warps = gridDim.x * kWarps;
        if (atomicAdd(reinterpret_cast<unsigned *>(work) + 1, 1u) == warps - 1) {
            work[0] = 0;
            work[1] = 0;
            __threadfence();
        }
    }
    if (FUSED) fused_block_finish(__float_as_uint(rmf), lp, fin_scratch);
    if (RHS) block_max_into(__float_as_uint(rmf),
                            reinterpret_cast<unsigned *>(&lp.state->bmax),
                            fin_scratch);
}

constexpr size_t kSmemBytes = (size_t)kWarps * kSliceFloats * sizeof(float);

template <int D>
cudaError_t prepare_d(TileConf &tc, int n) {
    int dev = 0, sms = 0, per_sm = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
            &per_sm, k_etbs<D, true, true, false>, 32 * kWarps, kSmemBytes);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    // As many blocks as run at once; no more warps than strip rows.
    const long long strips = (n - 1 + EtbsShape<D>::TX - 1) / EtbsShape<D>::TX;
    const long long work = strips * (n - 2);
    long long blocks = (long long)sms * per_sm;
    if (blocks * kWarps > work) blocks = (work + kWarps - 1) / kWarps;
    tc.ctas = (int)(blocks < 1 ? 1 : blocks);
    tc.smem = kSmemBytes;
    return cudaSuccess;
}

template <int D>
cudaError_t launch_d(const GridDesc &g, const TileConf &tc, const float *src,
                     const float *b, float *out, unsigned *err,
                     const LaunchCtl &ctl, cudaStream_t stream) {
    if (!tc.work || tc.bands < 1) return cudaErrorInvalidValue;
    const int strips = (g.n - 1 + EtbsShape<D>::TX - 1) / EtbsShape<D>::TX;
    const bool rhs = ctl.rhs_g != nullptr;
    if (rhs && (ctl.fused || !ctl.rhs_b || !ctl.lp.state))
        return cudaErrorInvalidValue;
#define TBJ_K(F, FU, RH)                                                       \
    launch_pdl(k_etbs<D, F, FU, RH>, dim3(tc.ctas), dim3(32 * kWarps),         \
               kSmemBytes, stream, src, RH ? ctl.rhs_g : b, out,               \
               RH ? ctl.rhs_b : nullptr, g.n, g.ld, g.r, g.d, g.y, strips,     \
               tc.work, tc.bands, err, ctl.stop, ctl.lp)
    if (g.fast) {
        if (rhs) return TBJ_K(true, false, true);
        return ctl.fused ? TBJ_K(true, true, false) : TBJ_K(true, false, false);
    }
    if (rhs) return TBJ_K(false, false, true);
    return ctl.fused ? TBJ_K(false, true, false) : TBJ_K(false, false, false);
#undef TBJ_K
}

}  // namespace

bool etbs_configure(int n, int depth, TileConf *tc) {
    (void)n;
    if (depth != 8) return false;
    tc->depth = depth;
    tc->halo_x = (depth + 3) / 4 * 4;
    tc->halo_y = depth;
    tc->box_x = 128;
    tc->box_y = 1;  // (no TMA boxes: rows are copied with cp.async)
    tc->tile_x = 128 - 2 * tc->halo_x;
    tc->tile_y = 0;  // whole columns, cut into one run per warp
    tc->origin = 0;
    tc->threads = 32 * kWarps;
    tc->smem = 0;
    tc->variant = kEtbsVariant;
    tc->ctas = 0;
    tc->stream = tc->ch = tc->sx = tc->sy = tc->grid_x = tc->grid_y = 0;
    tc->work = nullptr;  // set by the handle (etbs_schedule)
    tc->bands = 0;
    return true;
}

int etbs_schedule(const TileConf &tc, int n, int *band_start, int cap) {
    const int tx = tc.tile_x;
    const long long strips = (n - 1 + tx - 1) / tx;
    const long long warps = (long long)tc.ctas * kWarps;
    const int rows = n - 2;
    int bands = 0, y = 0;
    if (cap < 2 || warps < 1) return -1;
    band_start[0] = 1;
    while (y < rows) {
        // the work left over kGuide times the warps, in rows of one run
        long long h = ((long long)(rows - y) * strips + kGuide * warps - 1) /
                      (kGuide * warps);
        if (h > kBandMax) h = kBandMax;
        if (h < kBandMin) h = kBandMin;
        if (h > rows - y) h = rows - y;
        y += (int)h;
        if (++bands + 1 > cap) return -1;
        band_start[bands] = 1 + y;
    }
    return 2 + bands + 1;
}

bool etbs_preferred(int n, int sms) {
    // Rows per warp of the whole launch at 12 warps per SM: below about 64
    // the pipeline's fill and drain (2 D rows per run) and the launch's last
    // runs outweigh the saved halo. Measured on GB300, ten-step solves at
    // D = 8 under device control (this kernel also forms each step's
    // right-hand side there), register-band kernel against this one:
    // N = 3072 (47 rows per warp) 28.0 against 32.8 ms; N = 4096 (83)
    // 42.6 against 40.5 ms at r = 10, 6.71 against 6.04 at r = 1, 310.1
    // against 297.6 at r = 100; N = 6144 88.5 against 80.3.
    const long long strips = (n - 1 + EtbsShape<8>::TX - 1) / EtbsShape<8>::TX;
    return (long long)(n - 2) * strips >= 64LL * 12 * sms;
}

cudaError_t prepare_sweep_etbs(TileConf &tc, int n) {
    if (tc.depth != 8) return cudaErrorInvalidValue;
    const void *kernels[6] = {(const void *)k_etbs<8, true, false, false>,
                              (const void *)k_etbs<8, false, false, false>,
                              (const void *)k_etbs<8, true, true, false>,
                              (const void *)k_etbs<8, false, true, false>,
                              (const void *)k_etbs<8, true, false, true>,
                              (const void *)k_etbs<8, false, false, true>};
    for (const void *k : kernels) {
        cudaError_t e = cudaFuncSetAttribute(
            k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
        if (e != cudaSuccess) return e;
    }
    return prepare_d<8>(tc, n);
}

cudaError_t launch_sweep_etbs(const GridDesc &g, const TileConf &tc,
                              const float *src, const float *b, float *out,
                              unsigned *err, const LaunchCtl &ctl,
                              cudaStream_t stream) {
    if (tc.depth != 8) return cudaErrorInvalidValue;
    return launch_d<8>(g, tc, src, b, out, err, ctl, stream);
}

}  // namespace tbj
