// Row-streaming kernels: fused right-hand side, synchronous sweep, residual
// reduction and the interior copy.
//
// Layout of the work: a warp owns a strip 128 floats wide (32 lanes x one
// float4 each) and ROWS consecutive grid rows. It walks down the strip
// holding rows i-1, i and i+1 in registers, so every float of u is read from
// memory once per strip (plus the two rows above and below it). The west and
// east neighbours of a lane's four cells come from the adjacent lanes through
// warp shuffles; only lanes 0 and 31 read one extra float per row. One sweep
// therefore moves 4 B of u, 4 B of b and 4 B of u' per cell: the 12 B/cell
// of "Synchronous vs block-async Jacobi on one RTX 5050", section 02.
#include "jacobi_kernels.cuh"

namespace tbj {
namespace {

constexpr unsigned FULL = 0xffffffffu;
constexpr int kWarps = 4;  // warps per block, stacked vertically

// Rows per warp: the largest of 32, 16, 8, 4 that still gives at least
// ~54 resident warps' worth of strips per SM on 152 SMs, so small grids
// keep enough loads in flight.
int rows_per_warp(int n) {
    const long long strips = ((n + 3) / 4 + 31) / 32;
    for (int rows : {32, 16, 8}) {
        if (strips * ((n - 2 + rows - 1) / rows) >= 8192) return rows;
    }
    return 4;
}

__device__ __forceinline__ float4 ld4(const float *p) {
    return *reinterpret_cast<const float4 *>(p);
}
__device__ __forceinline__ void st4(float *p, float4 v) {
    *reinterpret_cast<float4 *>(p) = v;
}

// Store the cells of a float4 at column x0 that lie in [1, n-2].
__device__ __forceinline__ void store_interior(float *row, int x0, int n,
                                               float4 v) {
    if (x0 >= 1 && x0 + 3 <= n - 2) {
        st4(row + x0, v);
    } else {
        if (x0 + 0 >= 1 && x0 + 0 <= n - 2) row[x0 + 0] = v.x;
        if (x0 + 1 >= 1 && x0 + 1 <= n - 2) row[x0 + 1] = v.y;
        if (x0 + 2 >= 1 && x0 + 2 <= n - 2) row[x0 + 2] = v.z;
        if (x0 + 3 >= 1 && x0 + 3 <= n - 2) row[x0 + 3] = v.w;
    }
}

// One row's inputs for a lane: the centre float4 of u and the extra float
// that lane 0 (west) or lane 31 (east) needs from beyond the warp's strip.
struct RowIn {
    float4 bot;   // u[i+1][x0..x0+3]
    float4 bb;    // b[i][x0..x0+3]
    float edge;   // lane 0: u[i][x0-1]; lane 31: u[i][x0+4]; others unused
};

// UNF: b holds u^n and the right-hand side is formed here as fl(u^n + g)
// (section 02: the unfused form reads both arrays on every sweep).
template <bool UNF>
__device__ __forceinline__ RowIn load_row(const float *__restrict__ u,
                                          const float *__restrict__ b,
                                          const float *__restrict__ g,
                                          long long ld, int n, int i, int x0,
                                          int lane, bool active) {
    RowIn in;
    in.bot = make_float4(0.f, 0.f, 0.f, 0.f);
    in.bb = in.bot;
    in.edge = 0.f;
    if (active) {
        const long long row = (long long)i * ld;
        in.bot = ld4(u + row + ld + x0);
        in.bb = ld4(b + row + x0);
        if (UNF) {
            const float4 gg = ld4(g + row + x0);
            in.bb.x = __fadd_rn(in.bb.x, gg.x);
            in.bb.y = __fadd_rn(in.bb.y, gg.y);
            in.bb.z = __fadd_rn(in.bb.z, gg.z);
            in.bb.w = __fadd_rn(in.bb.w, gg.w);
        }
        if (lane == 0 && x0 > 0) in.edge = u[row + x0 - 1];
        if (lane == 31 && x0 + 4 < n) in.edge = u[row + x0 + 4];
    }
    return in;
}

// ---------------------------------------------------------------------------
// Synchronous sweep u -> out (section 02 "Synchronous"): every interior cell
// gets J(u); the ring of out is never written. FUSED also reduces the
// residual norms of the input u (see LoopState); `stop`, when given, makes
// the launch a no-op once the device-side loop has stopped.
// ---------------------------------------------------------------------------
template <int ROWS, bool FAST, bool FUSED, bool UNF>
__global__ void __launch_bounds__(32 * kWarps)
k_sweep_sync(const float *__restrict__ u, const float *__restrict__ b,
             const float *__restrict__ g, float *__restrict__ out, int n,
             long long ld, float r, float d, float y, const int *stop,
             LoopParams lp) {
    allow_dependents();
    grid_dependency_wait();     // u, b and the stop flag come from before
    if (stop && *stop) return;  // same value for every thread of the launch
    const int lane = threadIdx.x;
    const int vx = blockIdx.x * 32 + lane;
    const int x0 = vx * 4;
    const bool active = x0 < n;
    const int i0 = 1 + (blockIdx.y * kWarps + threadIdx.y) * ROWS;
    const int i1 = min(i0 + ROWS, n - 1);
    unsigned rm = 0u;  // fused: max |J(u) - u| bits
    if (i0 <= n - 2) {  // uniform across the warp
        float4 top = make_float4(0.f, 0.f, 0.f, 0.f), mid = top;
        if (active) {
            top = ld4(u + (long long)(i0 - 1) * ld + x0);
            mid = ld4(u + (long long)i0 * ld + x0);
        }
        RowIn next = load_row<UNF>(u, b, g, ld, n, i0, x0, lane, active);
        for (int i = i0; i < i1; ++i) {
            const RowIn cur = next;
            if (i + 1 < i1)
                next = load_row<UNF>(u, b, g, ld, n, i + 1, x0, lane, active);
            float west = __shfl_up_sync(FULL, mid.w, 1);
            float east = __shfl_down_sync(FULL, mid.x, 1);
            if (lane == 0) west = cur.edge;
            if (lane == 31) east = cur.edge;
            float4 o;
            o.x = jacobi_update<FAST>(west, mid.y, top.x, cur.bot.x, cur.bb.x, r, d, y);
            o.y = jacobi_update<FAST>(mid.x, mid.z, top.y, cur.bot.y, cur.bb.y, r, d, y);
            o.z = jacobi_update<FAST>(mid.y, mid.w, top.z, cur.bot.z, cur.bb.z, r, d, y);
            o.w = jacobi_update<FAST>(mid.z, east, top.w, cur.bot.w, cur.bb.w, r, d, y);
            if (active) {
                store_interior(out + (long long)i * ld, x0, n, o);
                if (FUSED) {
                    if (x0 + 0 >= 1 && x0 + 0 <= n - 2) rm = max(rm, change_bits(o.x, mid.x));
                    if (x0 + 1 >= 1 && x0 + 1 <= n - 2) rm = max(rm, change_bits(o.y, mid.y));
                    if (x0 + 2 >= 1 && x0 + 2 <= n - 2) rm = max(rm, change_bits(o.z, mid.z));
                    if (x0 + 3 >= 1 && x0 + 3 <= n - 2) rm = max(rm, change_bits(o.w, mid.w));
                }
            }
            top = mid;
            mid = cur.bot;
        }
    }
    if (FUSED) {
        __shared__ unsigned scratch[33];
        fused_block_finish(rm, lp, scratch);
    }
}

// ---------------------------------------------------------------------------
// Residual norms (section 01, difference form). Per interior cell:
//   e  = d * |J(u) - u|
//   bI = b + r * ((qW + qE) + (qN + qS)),  qX = neighbour value if it lies on
//        the Dirichlet ring, else 0 (right-hand side of the system in the
//        unknowns)
// rmax = max e, bmax = max |bI|. Maxima are taken on the IEEE bit patterns
// of non-negative floats, which order like the values and put NaN above
// +Inf, so a NaN anywhere reaches the result. Each block folds its two
// maxima into out->racc / bacc with atomicMax; the last block to finish
// (ticket) moves them to out->rmax / bmax and re-arms the accumulators.
// ---------------------------------------------------------------------------
__device__ __forceinline__ unsigned fbits(float x) {
    return __float_as_uint(fabsf(x));
}

template <bool FAST>
__device__ __forceinline__ void cell_norms(float c, float west, float east,
                                           float north, float south, float bb,
                                           int i, int x, int n, float r,
                                           float d, float y, unsigned &rm,
                                           unsigned &bm) {
    if (x < 1 || x > n - 2) return;
    const float ju = jacobi_update<FAST>(west, east, north, south, bb, r, d, y);
    const float e = __fmul_rn(d, fabsf(__fsub_rn(ju, c)));
    const float qw = (x - 1 == 0) ? west : 0.f;
    const float qe = (x + 1 == n - 1) ? east : 0.f;
    const float qn = (i - 1 == 0) ? north : 0.f;
    const float qs = (i + 1 == n - 1) ? south : 0.f;
    const float q = __fadd_rn(__fadd_rn(qw, qe), __fadd_rn(qn, qs));
    const float bi = __fadd_rn(bb, __fmul_rn(r, q));
    rm = max(rm, fbits(e));
    bm = max(bm, fbits(bi));
}

__device__ __forceinline__ unsigned warp_max(unsigned v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(FULL, v, o));
    return v;
}

template <int ROWS, bool FAST, bool UNF>
__global__ void __launch_bounds__(32 * kWarps)
k_residual(const float *__restrict__ u, const float *__restrict__ b,
           const float *__restrict__ g, int n, long long ld, float r, float d,
           float y, ResidualOut *__restrict__ out) {
    const int lane = threadIdx.x;
    const int vx = blockIdx.x * 32 + lane;
    const int x0 = vx * 4;
    const bool active = x0 < n;
    const int i0 = 1 + (blockIdx.y * kWarps + threadIdx.y) * ROWS;
    const int i1 = min(i0 + ROWS, n - 1);
    unsigned rm = 0u, bm = 0u;
    if (i0 <= n - 2) {
        float4 top = make_float4(0.f, 0.f, 0.f, 0.f), mid = top;
        if (active) {
            top = ld4(u + (long long)(i0 - 1) * ld + x0);
            mid = ld4(u + (long long)i0 * ld + x0);
        }
        RowIn next = load_row<UNF>(u, b, g, ld, n, i0, x0, lane, active);
        for (int i = i0; i < i1; ++i) {
            const RowIn cur = next;
            if (i + 1 < i1)
                next = load_row<UNF>(u, b, g, ld, n, i + 1, x0, lane, active);
            float west = __shfl_up_sync(FULL, mid.w, 1);
            float east = __shfl_down_sync(FULL, mid.x, 1);
            if (lane == 0) west = cur.edge;
            if (lane == 31) east = cur.edge;
            if (active) {
                cell_norms<FAST>(mid.x, west, mid.y, top.x, cur.bot.x, cur.bb.x, i, x0 + 0, n, r, d, y, rm, bm);
                cell_norms<FAST>(mid.y, mid.x, mid.z, top.y, cur.bot.y, cur.bb.y, i, x0 + 1, n, r, d, y, rm, bm);
                cell_norms<FAST>(mid.z, mid.y, mid.w, top.z, cur.bot.z, cur.bb.z, i, x0 + 2, n, r, d, y, rm, bm);
                cell_norms<FAST>(mid.w, mid.z, east, top.w, cur.bot.w, cur.bb.w, i, x0 + 3, n, r, d, y, rm, bm);
            }
            top = mid;
            mid = cur.bot;
        }
    }
    rm = warp_max(rm);
    bm = warp_max(bm);
    __shared__ unsigned s_r[kWarps], s_b[kWarps];
    if (lane == 0) {
        s_r[threadIdx.y] = rm;
        s_b[threadIdx.y] = bm;
    }
    __syncthreads();
    if (threadIdx.y != 0 || lane != 0) return;
    unsigned br = 0u, bbm = 0u;
    for (int w = 0; w < kWarps; ++w) {
        br = max(br, s_r[w]);
        bbm = max(bbm, s_b[w]);
    }
    if (br) atomicMax(&out->racc, br);
    if (bbm) atomicMax(&out->bacc, bbm);
    __threadfence();
    if (atomicAdd(&out->ticket, 1u) != gridDim.x * gridDim.y - 1) return;
    // Last block: every other block's maxima are in.
    __threadfence();
    out->rmax = __uint_as_float(atomicExch(&out->racc, 0u));
    out->bmax = __uint_as_float(atomicExch(&out->bacc, 0u));
    out->ticket = 0u;
}

// ---------------------------------------------------------------------------
// bmax of a time step: max over the interior of |b_I|, b_I = b (+ g when the
// right-hand side is unfused) + r * (the cell's Dirichlet-ring neighbours),
// exactly as k_residual forms it. b is fixed within a step, so the
// device-side loop takes it once per step. One block per row (grid-stride),
// one atomicMax per block into st->bmax.
// ---------------------------------------------------------------------------
template <bool UNF>
__global__ void __launch_bounds__(256)
k_bnorm(const float *__restrict__ u, const float *__restrict__ b,
        const float *__restrict__ g, int n, long long ld, float r,
        LoopState *st) {
    unsigned bm = 0u;
    for (int i = 1 + blockIdx.x; i <= n - 2; i += gridDim.x) {
        const long long row = (long long)i * ld;
        for (int x = 1 + threadIdx.x; x <= n - 2; x += blockDim.x) {
            const long long p = row + x;
            float bb = b[p];
            if (UNF) bb = __fadd_rn(bb, g[p]);
            const float qw = (x == 1) ? u[p - 1] : 0.f;
            const float qe = (x == n - 2) ? u[p + 1] : 0.f;
            const float qn = (i == 1) ? u[p - ld] : 0.f;
            const float qs = (i == n - 2) ? u[p + ld] : 0.f;
            const float q = __fadd_rn(__fadd_rn(qw, qe), __fadd_rn(qn, qs));
            bm = max(bm, abs_bits(__fadd_rn(bb, __fmul_rn(r, q))));
        }
    }
    bm = warp_max(bm);
    __shared__ unsigned s_b[8];
    if ((threadIdx.x & 31) == 0) s_b[threadIdx.x >> 5] = bm;
    __syncthreads();
    if (threadIdx.x != 0) return;
    for (int w = 1; w < (int)(blockDim.x >> 5); ++w) bm = max(bm, s_b[w]);
    if (bm) atomicMax(reinterpret_cast<unsigned *>(&st->bmax), bm);
}

// ---------------------------------------------------------------------------
// The ring-adjacent part of bmax (rows 1 and n-2, columns 1 and n-2 of the
// interior), for a step whose first sweep launch forms b = u + g and reduces
// |b| over the other interior cells. Per cell the same b_I as k_bnorm, with
// b = fl(u + g) formed here from u^n and the source g. Cells at a corner of
// the interior are visited twice, which a maximum does not mind.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256)
k_bnorm_ring(const float *__restrict__ u, const float *__restrict__ g, int n,
             long long ld, float r, LoopState *st) {
    const int m = n - 2;  // interior cells per side
    unsigned bm = 0u;
    for (int idx = blockIdx.x * blockDim.x + threadIdx.x; idx < 4 * m;
         idx += gridDim.x * blockDim.x) {
        const int side = idx / m, pos = 1 + idx % m;
        const int i = side == 0 ? 1 : side == 1 ? n - 2 : pos;
        const int x = side == 2 ? 1 : side == 3 ? n - 2 : pos;
        const long long p = (long long)i * ld + x;
        const float bb = __fadd_rn(u[p], g[p]);
        const float qw = (x == 1) ? u[p - 1] : 0.f;
        const float qe = (x == n - 2) ? u[p + 1] : 0.f;
        const float qn = (i == 1) ? u[p - ld] : 0.f;
        const float qs = (i == n - 2) ? u[p + ld] : 0.f;
        const float q = __fadd_rn(__fadd_rn(qw, qe), __fadd_rn(qn, qs));
        bm = max(bm, abs_bits(__fadd_rn(bb, __fmul_rn(r, q))));
    }
    bm = warp_max(bm);
    __shared__ unsigned s_b[8];
    if ((threadIdx.x & 31) == 0) s_b[threadIdx.x >> 5] = bm;
    __syncthreads();
    if (threadIdx.x != 0) return;
    for (int w = 1; w < (int)(blockDim.x >> 5); ++w) bm = max(bm, s_b[w]);
    if (bm) atomicMax(reinterpret_cast<unsigned *>(&st->bmax), bm);
}

// ---------------------------------------------------------------------------
// Fused right-hand side b = u + g and the interior copy dst = src: one float4
// per thread, grid-stride over rows.
// ---------------------------------------------------------------------------
__global__ void k_rhs(const float *__restrict__ u, const float *__restrict__ g,
                      float *__restrict__ b, int n, long long ld) {
    const int x0 = (blockIdx.x * blockDim.x + threadIdx.x) * 4;
    if (x0 >= n) return;
    for (int i = 1 + blockIdx.y * blockDim.y + threadIdx.y; i <= n - 2;
         i += gridDim.y * blockDim.y) {
        const long long row = (long long)i * ld;
        const float4 a = ld4(u + row + x0);
        const float4 c = ld4(g + row + x0);
        float4 o;
        o.x = __fadd_rn(a.x, c.x);
        o.y = __fadd_rn(a.y, c.y);
        o.z = __fadd_rn(a.z, c.z);
        o.w = __fadd_rn(a.w, c.w);
        store_interior(b + row, x0, n, o);
    }
}

// The Dirichlet ring of src into dst: rows 0 and n-1, columns 0 and n-1.
__global__ void k_copy_ring(const float *__restrict__ src, float *__restrict__ dst,
                            int n, long long ld) {
    for (int idx = blockIdx.x * blockDim.x + threadIdx.x; idx < 4 * n;
         idx += gridDim.x * blockDim.x) {
        const int side = idx / n, pos = idx % n;
        const long long p = side == 0   ? (long long)pos
                            : side == 1 ? (long long)(n - 1) * ld + pos
                            : side == 2 ? (long long)pos * ld
                                        : (long long)pos * ld + (n - 1);
        dst[p] = src[p];
    }
}

__global__ void k_copy_interior(const float *__restrict__ src,
                                float *__restrict__ dst, int n, long long ld) {
    const int x0 = (blockIdx.x * blockDim.x + threadIdx.x) * 4;
    if (x0 >= n) return;
    for (int i = 1 + blockIdx.y * blockDim.y + threadIdx.y; i <= n - 2;
         i += gridDim.y * blockDim.y) {
        const long long row = (long long)i * ld;
        store_interior(dst + row, x0, n, ld4(src + row + x0));
    }
}

// Bounds-checked build: NaN into every interior cell of dst ahead of a sweep
// launch, which must write all of them. It honours the stop flag as the
// sweep kernels do, so an answer that a device-side stop left in dst is
// kept.
__global__ void k_poison_interior(float *__restrict__ dst, int n, long long ld,
                                  const int *stop) {
    if (stop && *stop) return;
    const float q = __int_as_float(0x7fc0bad0);
    for (int i = 1 + blockIdx.y * blockDim.y + threadIdx.y; i <= n - 2;
         i += gridDim.y * blockDim.y)
        for (int j = 1 + blockIdx.x * blockDim.x + threadIdx.x; j <= n - 2;
             j += gridDim.x * blockDim.x)
            dst[(long long)i * ld + j] = q;
}

// Bounds-checked build: the checker's own test (launch_bounds_selftest).
// One thread runs five accesses, each against its own error word; the
// refused ones would be harmless even if performed: the shared load stays
// inside the block's allocation (past the part declared to the checker),
// and every store writes back the value the cell holds.
__global__ void k_bounds_selftest(float *grid, int n, long long ld,
                                  unsigned *flags) {
    extern __shared__ __align__(16) float sm[];  // 256 bytes
    bounds_begin(sm, 128, grid, nullptr, nullptr, nullptr, n, ld, flags);
#if defined(JACOBI_BOUNDS_CHECK)
    if (threadIdx.x != 0) return;
    volatile float sink = 0.f;
    g_bounds.err = flags + 0;
    sink = lds1(sm + 40);  // byte 160 of a 128-byte region
    g_bounds.err = flags + 1;
    gst1(grid + 2, grid[2]);  // row 0: the ring
    g_bounds.err = flags + 2;
    gst1(grid + ld + (n - 1), grid[ld + (n - 1)]);  // column n-1: the ring
    g_bounds.err = flags + 3;
    sink = lds1(sm + 4);  // inside the region
    g_bounds.err = flags + 4;
    gst1(grid + ld + 1, grid[ld + 1]);  // interior cell (1, 1)
    (void)sink;
#endif
}

// Reset a step's loop state. In a graph of several time steps `prev` is the
// previous step's state: if that step did not converge, this step is marked
// skipped (stopped before it starts), so every later kernel of it returns at
// entry.
__global__ void k_loop_reset(LoopState *st, const LoopState *prev,
                             long long k0, int keep_where) {
    st->rmax = 0.f;
    st->bmax = 0.f;
    st->err = 0u;
    st->ticket = 0u;
    st->k = k0;
    st->result_k = 0;
    st->stop = 0;
    st->status = 0;
    st->where = 0;
    st->rbits = 0u;
    st->bar_arrive = 0u;
    st->bar_epoch = 0u;
    if (prev && prev->status != 0) {
        st->status = kStepSkipped;
        st->stop = 1;
        // The run's answer stays where the failed step left it.
        if (keep_where) st->where = prev->where;
    }
}

// Condition of a step's if/else node in a run whose steps start from
// wherever the previous step's answer is: 1 (first branch) when it is in u.
__global__ void k_branch_on_where(const LoopState *prev,
                                  cudaGraphConditionalHandle cond) {
    cudaGraphSetConditional(cond, prev->where == 0 ? 1u : 0u);
}

// End of a time step in a multi-step graph: if the answer sits in u_alt
// (LoopState::where), copy its interior into u, so that the next step's
// right-hand side and sweeps start from u.
__global__ void k_settle(const LoopState *st, const float *__restrict__ src,
                         float *__restrict__ dst, int n, long long ld) {
    if (st->where != 1) return;  // same value for every thread
    const int x0 = (blockIdx.x * blockDim.x + threadIdx.x) * 4;
    if (x0 >= n) return;
    for (int i = 1 + blockIdx.y * blockDim.y + threadIdx.y; i <= n - 2;
         i += gridDim.y * blockDim.y) {
        const long long row = (long long)i * ld;
        store_interior(dst + row, x0, n, ld4(src + row + x0));
    }
}

// The loop condition starts at 1 with every launch of the step's graph, so
// only the stop needs setting.
__global__ void k_loop_condition(const LoopState *st,
                                 cudaGraphConditionalHandle cond) {
    if (st->stop) cudaGraphSetConditional(cond, 0u);
}

dim3 strip_grid(int n, int rows) {
    const int nvec = (n + 3) / 4;
    const int per_block = kWarps * rows;
    return dim3((nvec + 31) / 32, (n - 2 + per_block - 1) / per_block);
}

dim3 elementwise_grid(int n) {
    const int nvec = (n + 3) / 4;
    const int gy = min((n - 2 + 7) / 8, 1024);
    return dim3((nvec + 31) / 32, gy);
}

}  // namespace

cudaError_t launch_rhs(const GridDesc &g, const float *u, const float *src,
                       float *b, cudaStream_t stream) {
    k_rhs<<<elementwise_grid(g.n), dim3(32, 8), 0, stream>>>(u, src, b, g.n,
                                                              g.ld);
    return cudaGetLastError();
}

cudaError_t launch_poison_interior(const GridDesc &g, float *dst,
                                  const int *stop, cudaStream_t stream) {
    k_poison_interior<<<elementwise_grid(g.n), dim3(32, 8), 0, stream>>>(
        dst, g.n, g.ld, stop);
    return cudaGetLastError();
}

cudaError_t launch_bounds_selftest(float *grid, int n, long long ld,
                                   unsigned *flags, cudaStream_t stream) {
    k_bounds_selftest<<<1, 32, 256, stream>>>(grid, n, ld, flags);
    return cudaGetLastError();
}

cudaError_t launch_copy_ring(const GridDesc &g, const float *src, float *dst,
                             cudaStream_t stream) {
    const int blocks = (4 * g.n + 255) / 256 < 152 ? (4 * g.n + 255) / 256 : 152;
    k_copy_ring<<<blocks, 256, 0, stream>>>(src, dst, g.n, g.ld);
    return cudaGetLastError();
}

cudaError_t launch_copy_interior(const GridDesc &g, const float *src,
                                 float *dst, cudaStream_t stream) {
    k_copy_interior<<<elementwise_grid(g.n), dim3(32, 8), 0, stream>>>(
        src, dst, g.n, g.ld);
    return cudaGetLastError();
}

cudaError_t launch_sweep_sync(const GridDesc &g, const float *u,
                              const float *b, float *out, const LaunchCtl &ctl,
                              cudaStream_t stream) {
    const int rows = rows_per_warp(g.n);
    const dim3 grid = strip_grid(g.n, rows), block(32, kWarps);
#define TBJ_SWEEP(R, F, FU, UN)                                               \
    launch_pdl(k_sweep_sync<R, F, FU, UN>, grid, block, 0, stream, u, b,      \
               g.g2, out, g.n, g.ld, g.r, g.d, g.y, ctl.stop, ctl.lp)
#define TBJ_SWEEP_F(R, F)                                                     \
    if (g.g2)                                                                 \
        return ctl.fused ? TBJ_SWEEP(R, F, true, true)                        \
                         : TBJ_SWEEP(R, F, false, true);                      \
    return ctl.fused ? TBJ_SWEEP(R, F, true, false)                           \
                     : TBJ_SWEEP(R, F, false, false);
#define TBJ_SWEEP_R(R)                                                        \
    case R:                                                                   \
        if (g.fast) {                                                         \
            TBJ_SWEEP_F(R, true)                                              \
        }                                                                     \
        TBJ_SWEEP_F(R, false)
    switch (rows) {
        TBJ_SWEEP_R(4)
        TBJ_SWEEP_R(8)
        TBJ_SWEEP_R(16)
        TBJ_SWEEP_R(32)
    }
#undef TBJ_SWEEP_R
#undef TBJ_SWEEP_F
#undef TBJ_SWEEP
    return cudaErrorInvalidValue;
}

int sweep_sync_blocks(const GridDesc &g) {
    const dim3 grid = strip_grid(g.n, rows_per_warp(g.n));
    return (int)(grid.x * grid.y);
}

cudaError_t launch_loop_reset(LoopState *st, const LoopState *prev,
                              cudaStream_t stream, long long k0,
                              bool keep_where) {
    k_loop_reset<<<1, 1, 0, stream>>>(st, prev, k0, keep_where ? 1 : 0);
    return cudaGetLastError();
}

cudaError_t launch_settle(const GridDesc &g, const LoopState *st,
                          const float *src, float *dst, cudaStream_t stream) {
    k_settle<<<elementwise_grid(g.n), dim3(32, 8), 0, stream>>>(st, src, dst,
                                                                g.n, g.ld);
    return cudaGetLastError();
}

cudaError_t launch_branch_on_where(const LoopState *prev,
                                  cudaGraphConditionalHandle cond,
                                  cudaStream_t stream) {
    k_branch_on_where<<<1, 1, 0, stream>>>(prev, cond);
    return cudaGetLastError();
}

cudaError_t launch_loop_condition(const LoopState *st,
                                  cudaGraphConditionalHandle cond,
                                  cudaStream_t stream) {
    k_loop_condition<<<1, 1, 0, stream>>>(st, cond);
    return cudaGetLastError();
}

cudaError_t launch_residual(const GridDesc &g, const float *u, const float *b,
                            ResidualOut *out, cudaStream_t stream) {
    const int rows = rows_per_warp(g.n);
    const dim3 grid = strip_grid(g.n, rows), block(32, kWarps);
#define TBJ_RESID_K(R, F, UN)                                                 \
    k_residual<R, F, UN><<<grid, block, 0, stream>>>(u, b, g.g2, g.n, g.ld,   \
                                                     g.r, g.d, g.y, out)
#define TBJ_RESID(R)                                                          \
    case R:                                                                   \
        if (g.fast) {                                                         \
            if (g.g2) TBJ_RESID_K(R, true, true);                             \
            else TBJ_RESID_K(R, true, false);                                 \
        } else {                                                              \
            if (g.g2) TBJ_RESID_K(R, false, true);                            \
            else TBJ_RESID_K(R, false, false);                                \
        }                                                                     \
        break;
    switch (rows) {
        TBJ_RESID(4)
        TBJ_RESID(8)
        TBJ_RESID(16)
        TBJ_RESID(32)
    }
#undef TBJ_RESID
#undef TBJ_RESID_K
    return cudaGetLastError();
}

cudaError_t launch_bnorm_ring(const GridDesc &g, const float *u,
                              const float *src, LoopState *st,
                              cudaStream_t stream) {
    const long long cells = 4LL * (g.n - 2);
    const int blocks = (int)((cells + 255) / 256 < 152 ? (cells + 255) / 256 : 152);
    k_bnorm_ring<<<blocks, 256, 0, stream>>>(u, src, g.n, g.ld, g.r, st);
    return cudaGetLastError();
}

cudaError_t launch_bnorm(const GridDesc &g, const float *u, const float *b,
                         LoopState *st, cudaStream_t stream) {
    const int blocks = g.n - 2 < 2048 ? g.n - 2 : 2048;
    if (g.g2)
        k_bnorm<true><<<blocks, 256, 0, stream>>>(u, b, g.g2, g.n, g.ld, g.r, st);
    else
        k_bnorm<false><<<blocks, 256, 0, stream>>>(u, b, nullptr, g.n, g.ld, g.r, st);
    return cudaGetLastError();
}

}  // namespace tbj
