// Internal declarations shared by the CUDA translation units of the solver.
// Not part of the public ABI (include/jacobi.h is).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

namespace tbj {

// ---------------------------------------------------------------------------
// Correctly rounded division by the fixed diagonal d.
//
// All kernels divide by the same d = 1 + 4r. With y = RN(1/d) the quotient
// is refined once from q0 = RN(x*y) using the exact remainder (P. Markstein,
// "Computation of elementary functions on the IBM RISC System/6000
// processor", IBM J. Res. Dev. 34(1), 1990; the remainder of a faithful
// quotient is exact in one fused multiply-add):
//     q0  = RN(x * y)
//     rho = RN(q0 * d - x)        (exact)
//     q   = RN(q0 - rho * y)
// The remainder is formed with its sign flipped so that x = -0 yields -0.
// Whether this equals the IEEE quotient for EVERY finite x depends on d, so
// each handle checks it exhaustively against __fdiv_rn for its own d (all
// finite float32 numerators) before using it (fastdiv_verify); otherwise
// the kernels use __fdiv_rn. A non-finite numerator gives a non-finite
// result either way (NaN where IEEE gives +-Inf).
// ---------------------------------------------------------------------------
__device__ __forceinline__ float div_fixed(float x, float d, float y) {
    const float q0 = __fmul_rn(x, y);
    const float rho = __fmaf_rn(q0, d, -x);
    return __fmaf_rn(-rho, y, q0);
}

// The same three steps on two numerators at once, with the packed float32
// instructions of sm_100-class GPUs (per component numerically identical to
// the scalar round-to-nearest operations).
__device__ __forceinline__ float2 div2_fixed(float2 x, float2 d2, float2 y2) {
    const float2 q0 = __fmul2_rn(x, y2);
    const float2 rho = __ffma2_rn(q0, d2, make_float2(-x.x, -x.y));
    return __ffma2_rn(make_float2(-rho.x, -rho.y), y2, q0);
}

template <bool FAST>
__device__ __forceinline__ float div_d(float x, float d, float y) {
    if (FAST) return div_fixed(x, d, y);
    return __fdiv_rn(x, d);
}

// ---------------------------------------------------------------------------
// The update of "Synchronous vs block-async Jacobi on one RTX 5050",
// sections 01-02: J(u)_ij = (b_ij + r * ((uW + uE) + (uN + uS))) / d,
// d = 1 + 4r. Round-to-nearest intrinsics fix the order and keep the
// compiler from fusing the multiply into the add; the division is the
// correctly rounded quotient.
// ---------------------------------------------------------------------------
template <bool FAST = false>
__device__ __forceinline__ float jacobi_update(float uw, float ue, float un,
                                               float us, float b, float r,
                                               float d, float y = 0.f) {
    float horiz = __fadd_rn(uw, ue);
    float vert = __fadd_rn(un, us);
    float s = __fadd_rn(horiz, vert);
    float rs = __fmul_rn(r, s);
    float num = __fadd_rn(b, rs);
    return div_d<FAST>(num, d, y);
}

// ---------------------------------------------------------------------------
// Row-chunk forms used by the tiled kernels: one lane holds a float4 chunk
// of a row.
// ---------------------------------------------------------------------------
// J for the four cells of a float4 chunk: n4, c4, s4 the rows above, at and
// below, w/e the cells west of .x and east of .w.
// PACKDIV: the division's three steps on pairs of cells (packed) or one
// cell at a time; the results are the same bits. Which is faster depends on
// the kernel's instruction mix (measured on GB300: packed for the
// column-streamed kernel, 3.5 % slower per launch with scalar division;
// scalar for the register-band and block-async kernels, 2-6 % faster).
template <bool FAST, bool PACKDIV = true>
__device__ __forceinline__ float4 update4_we(float4 n4, float4 c4, float4 s4,
                                             float4 b4, float w, float e,
                                             float r, float d, float y) {
    if (FAST) {
        // Same operations, same order, mostly two cells per instruction:
        // ((W+E) + (N+S)) * r + b, then the fixed-divisor division. The
        // product r * s is formed with scalar round-to-nearest multiplies:
        // a packed multiply feeding a packed add can be fused into one
        // multiply-add by the compiler, which would change the rounding.
        // (Measured on GB300: the packed-multiply intrinsic, an inline
        // mul.rn.f32x2 and a packed fma with a -0 addend all gave fields
        // that differ from the synchronous sweep's.)
        const float2 d2 = make_float2(d, d), y2 = make_float2(y, y);
        const float2 h01 = make_float2(__fadd_rn(w, c4.y), __fadd_rn(c4.x, c4.z));
        const float2 h23 = make_float2(__fadd_rn(c4.y, c4.w), __fadd_rn(c4.z, e));
        const float2 v01 = __fadd2_rn(make_float2(n4.x, n4.y), make_float2(s4.x, s4.y));
        const float2 v23 = __fadd2_rn(make_float2(n4.z, n4.w), make_float2(s4.z, s4.w));
        const float2 s01 = __fadd2_rn(h01, v01), s23 = __fadd2_rn(h23, v23);
        const float2 rs01 = make_float2(__fmul_rn(r, s01.x), __fmul_rn(r, s01.y));
        const float2 rs23 = make_float2(__fmul_rn(r, s23.x), __fmul_rn(r, s23.y));
        const float2 num01 = __fadd2_rn(make_float2(b4.x, b4.y), rs01);
        const float2 num23 = __fadd2_rn(make_float2(b4.z, b4.w), rs23);
        if (!PACKDIV)
            return make_float4(div_fixed(num01.x, d, y), div_fixed(num01.y, d, y),
                               div_fixed(num23.x, d, y), div_fixed(num23.y, d, y));
        const float2 q01 = div2_fixed(num01, d2, y2);
        const float2 q23 = div2_fixed(num23, d2, y2);
        return make_float4(q01.x, q01.y, q23.x, q23.y);
    }
    float4 o;
    o.x = jacobi_update<false>(w, c4.y, n4.x, s4.x, b4.x, r, d, y);
    o.y = jacobi_update<false>(c4.x, c4.z, n4.y, s4.y, b4.y, r, d, y);
    o.z = jacobi_update<false>(c4.y, c4.w, n4.z, s4.z, b4.z, r, d, y);
    o.w = jacobi_update<false>(c4.z, e, n4.w, s4.w, b4.w, r, d, y);
    return o;
}

// Keep the old value where the cell is not an interior grid cell.
__device__ __forceinline__ float4 hold4(float4 nv, float4 old, bool row_ok,
                                        unsigned colmask) {
    float4 o;
    o.x = (row_ok && (colmask & 1u)) ? nv.x : old.x;
    o.y = (row_ok && (colmask & 2u)) ? nv.y : old.y;
    o.z = (row_ok && (colmask & 4u)) ? nv.z : old.z;
    o.w = (row_ok && (colmask & 8u)) ? nv.w : old.w;
    return o;
}

// max(a, |x|) that returns NaN when either is NaN.
__device__ __forceinline__ float max_nan_abs(float a, float x) {
    float o;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(o) : "f"(a), "f"(fabsf(x)));
    return o;
}

// Exhaustive check of div_fixed against __fdiv_rn for one d: counts the
// finite float32 numerators whose quotients differ in any bit. `count` is a
// device word (set to 0 by the caller). Launch fastdiv_verify_launch.
cudaError_t fastdiv_verify_launch(float d, float y, unsigned long long *count,
                                  cudaStream_t stream);
// RN(1/d) in float32, computed exactly on the host.
float reciprocal_rn(float d);

// Error bits written by kernels into the handle's status word.
enum : unsigned {
    ERR_TMA_TIMEOUT = 1u,   // an mbarrier wait for a TMA load gave up
    ERR_SYNC_TIMEOUT = 2u,  // a grid-wide barrier wait gave up
    ERR_BOUNDS = 4u,        // bounds-checked build: an access was out of range
};

// ---------------------------------------------------------------------------
// Bounds-checked build.
//
// Compiled with JACOBI_BOUNDS_CHECK (libtbjacobi_checked.so, a testing aid
// standing in for a memory checker), the tiled kernels -- k_etbs, k_etbr,
// k_etb, k_etbp, k_bar, k_ba, k_block_async -- route every shared-memory
// access, every plain global load of a grid and every global store through
// the accessors below, and check every TMA box load's x coordinate and
// destination. An
// access outside its range is not performed: it sets ERR_BOUNDS in the
// launch's error word (reported as JACOBI_ERR_CUDA) and a load yields NaN.
// Nothing traps. The ranges are
//   * shared memory: the block's dynamic shared memory, [base, base + bytes),
//     with the access aligned to its size;
//   * plain global loads: the N x ld floats of a grid array;
//   * global stores: interior cells of the output grid only (rows and
//     columns 1 .. N-2) -- a store to the Dirichlet ring or the row padding
//     is as wrong as one past the array;
//   * TMA loads: x a multiple of 4 floats (the 16-byte rule), the box inside
//     shared memory.
// The checked build also poisons: bounds_begin() fills the block's dynamic
// shared memory with NaN before anything else, and the host fills the
// destination grid's interior with NaN before every sweep launch, so a cell
// read before it was written, or an interior cell no launch writes, shows up
// as NaN in the result.
//
// Without JACOBI_BOUNDS_CHECK the accessors are plain loads and stores.
// ---------------------------------------------------------------------------
#if defined(JACOBI_BOUNDS_CHECK)
constexpr bool kBoundsChecked = true;
#else
constexpr bool kBoundsChecked = false;
#endif

// The range rules, as pure functions (also compiled and tested on the host).
// off, bytes: byte offset and size of a shared access; limit: the region's
// size in bytes.
__host__ __device__ constexpr bool smem_access_ok(long long off, unsigned bytes,
                                                  unsigned long long limit) {
    return off >= 0 && bytes > 0 && (off % bytes) == 0 &&
           (unsigned long long)off + bytes <= limit;
}
// idx, count: first float and number of floats of a global access to an
// n x ld grid.
__host__ __device__ constexpr bool grid_access_ok(long long idx, int count,
                                                  int n, long long ld) {
    return idx >= 0 && count > 0 && idx + count <= (long long)n * ld;
}
// The same access lies on interior cells only (one row, columns 1 .. n-2).
__host__ __device__ constexpr bool interior_access_ok(long long idx, int count,
                                                      int n, long long ld) {
    return grid_access_ok(idx, count, n, ld) && idx / ld >= 1 &&
           idx / ld <= n - 2 && idx % ld >= 1 && idx % ld + count - 1 <= n - 2;
}
// x coordinate of a TMA load of 4-byte elements.
__host__ __device__ constexpr bool tma_x_ok(int x) { return (x & 3) == 0; }

#if defined(JACOBI_BOUNDS_CHECK)
namespace {
struct BoundsCtx {
    const unsigned char *smem;  // the block's dynamic shared memory
    unsigned smem_bytes;
    const float *out, *out2;    // output grids (stores); out2 may be null
    const float *in0, *in1;     // grids read with plain loads, or null
    long long ld;
    int n;
    unsigned *err;
};
__shared__ BoundsCtx g_bounds;
}  // namespace

__device__ __forceinline__ bool bounds_fail() {
    atomicOr(g_bounds.err, (unsigned)ERR_BOUNDS);
    return false;
}
__device__ __forceinline__ bool smem_ok(const void *p, unsigned bytes) {
    const long long off = reinterpret_cast<const unsigned char *>(p) - g_bounds.smem;
    return smem_access_ok(off, bytes, g_bounds.smem_bytes) || bounds_fail();
}
__device__ __forceinline__ bool store_ok(const float *p, int count) {
    return interior_access_ok(p - g_bounds.out, count, g_bounds.n, g_bounds.ld) ||
           (g_bounds.out2 &&
            interior_access_ok(p - g_bounds.out2, count, g_bounds.n, g_bounds.ld)) ||
           bounds_fail();
}
__device__ __forceinline__ bool load_ok(const float *base, const float *p, int count) {
    const bool known = base == g_bounds.in0 || base == g_bounds.in1;
    return (known && grid_access_ok(p - base, count, g_bounds.n, g_bounds.ld)) ||
           bounds_fail();
}
__device__ __forceinline__ bool tma_ok(const void *dst, unsigned bytes, int x) {
    return (tma_x_ok(x) && smem_access_ok(reinterpret_cast<const unsigned char *>(dst) -
                                              g_bounds.smem,
                                          16, g_bounds.smem_bytes) &&
            smem_access_ok(reinterpret_cast<const unsigned char *>(dst) -
                               g_bounds.smem + bytes - 16,
                           16, g_bounds.smem_bytes)) ||
           bounds_fail();
}
#else
__device__ __forceinline__ bool smem_ok(const void *, unsigned) { return true; }
__device__ __forceinline__ bool store_ok(const float *, int) { return true; }
__device__ __forceinline__ bool load_ok(const float *, const float *, int) { return true; }
__device__ __forceinline__ bool tma_ok(const void *, unsigned, int) { return true; }
#endif

// Start of a tiled kernel (every thread, before anything else). Checked
// build: records what the block may touch -- `smem_bytes` bytes of dynamic
// shared memory from `smem` (0: all of it), the output grids `out`, `out2`
// (null: none), the grids `in0`, `in1` read with plain loads, n, ld, the
// error word -- and fills the dynamic shared memory with NaN. Otherwise
// nothing.
__device__ __forceinline__ void bounds_begin(void *smem, unsigned smem_bytes,
                                             const float *out, const float *out2,
                                             const float *in0, const float *in1,
                                             int n, long long ld, unsigned *err) {
#if defined(JACOBI_BOUNDS_CHECK)
    unsigned dyn;
    asm("mov.u32 %0, %%dynamic_smem_size;" : "=r"(dyn));
    if (smem_bytes == 0 || smem_bytes > dyn) smem_bytes = dyn;
    const int tid = threadIdx.x + blockDim.x * (threadIdx.y + blockDim.y * threadIdx.z);
    const int nt = blockDim.x * blockDim.y * blockDim.z;
    unsigned *w = reinterpret_cast<unsigned *>(smem);
    for (unsigned k = tid; k < dyn / 4; k += nt) w[k] = 0x7fc0dead;  // NaN
    if (tid == 0) {
        g_bounds.smem = reinterpret_cast<const unsigned char *>(smem);
        g_bounds.smem_bytes = smem_bytes;
        g_bounds.out = out;
        g_bounds.out2 = out2;
        g_bounds.in0 = in0;
        g_bounds.in1 = in1;
        g_bounds.ld = ld;
        g_bounds.n = n;
        g_bounds.err = err;
    }
    __syncthreads();
#else
    (void)smem, (void)smem_bytes, (void)out, (void)out2, (void)in0, (void)in1,
        (void)n, (void)ld, (void)err;
#endif
}

// Shared-memory loads and stores of a float4 (16-byte aligned) or a float.
__device__ __forceinline__ float4 lds4(const float *p) {
    if (!smem_ok(p, 16)) {
        const float q = __int_as_float(0x7fc00000);
        return make_float4(q, q, q, q);
    }
    return *reinterpret_cast<const float4 *>(p);
}
__device__ __forceinline__ void sts4(float *p, float4 v) {
    if (smem_ok(p, 16)) *reinterpret_cast<float4 *>(p) = v;
}
__device__ __forceinline__ float lds1(const float *p) {
    return smem_ok(p, 4) ? *p : __int_as_float(0x7fc00000);
}
__device__ __forceinline__ void sts1(float *p, float v) {
    if (smem_ok(p, 4)) *p = v;
}
// Global stores into the output grid's interior.
__device__ __forceinline__ void gst4(float *p, float4 v) {
    if (store_ok(p, 4)) *reinterpret_cast<float4 *>(p) = v;
}
__device__ __forceinline__ void gst1(float *p, float v) {
    if (store_ok(p, 1)) *p = v;
}

// Parameters common to all sweep kernels.
struct GridDesc {
    int n;         // grid side including the ring
    long long ld;  // row pitch in floats
    float r;       // coupling alpha dt / h^2
    float d;       // fl(1 + fl(4 r))
    float y;       // RN(1/d)
    bool fast;     // div_fixed verified equal to IEEE division for this d
    // Unfused right-hand side (synchronous sweep only): when not null, the
    // `b` argument of a launch holds u^n and every read of b_ij becomes
    // fl(u^n_ij + g2_ij), the same value a fused b holds.
    const float *g2 = nullptr;
};

// Result block of a residual reduction (device memory, one per handle).
struct ResidualOut {
    float rmax;
    float bmax;
    unsigned err;       // OR of ERR_* bits seen since the last reset
    unsigned ticket;    // last-block counter, returns to 0 after each use
    unsigned racc, bacc;  // running maxima (bit patterns); 0 between uses
};

// ---------------------------------------------------------------------------
// Device-side convergence loop.
//
// With JACOBI_CONTROL_DEVICE a whole time step is one graph: a reset, the
// right-hand-side norm bmax = max |b_I| of the step (b does not change
// within a step), then a conditional WHILE node that repeats the check
// interval. The first launch of each interval is "fused": besides its sweeps
// it reduces max |J(u) - u| over its INPUT iterate (its first sweep evaluates
// J(u) anyway) into LoopState::rbits with one atomicMax per block, and the
// last of its blocks to finish forms rmax = d * that maximum (the same value
// as the maximum of d|J(u) - u| cell by cell: rounding is monotone), applies
// the stopping rule and updates LoopState. A small kernel at the end of each
// loop iteration clears the loop condition once LoopState::stop is set.
// Every launch first reads LoopState::stop and returns at once when it is
// set, so launches queued after the stop do nothing and the answer (the
// fused launch's input) is left intact.
// ---------------------------------------------------------------------------
struct LoopState {
    float rmax;           // rmax at the last check
    float bmax;           // bmax of the step's right-hand side
    unsigned err;         // ERR_* bits
    unsigned ticket;      // last-block counter of the fused reduction
    long long k;          // sweeps done before the current check interval
    long long result_k;   // sweep count of the answer once stopped
    int stop;             // 1 once the step has finished
    int status;           // 0 converged, or a negative jacobi_status_t
    int where;            // buffer holding the answer: 0 u, 1 u_alt
    unsigned rbits;       // running max of |J(u) - u| (bit pattern) of the
                          // current check; 0 between checks
    unsigned bar_arrive;  // persistent kernel: blocks arrived at its grid
                          // barriers so far (all rounds)
    unsigned bar_epoch;   // persistent kernel: barriers completed
};

struct LoopParams {
    LoopState *state;
    float d;                 // 1 + 4r: rmax = d * max |J(u) - u|
    double tol;
    long long max_sweeps;
    long long interval;      // sweeps per check interval
    cudaGraphConditionalHandle cond;
    int src_is_alt;          // the fused launch reads u_alt (1) or u (0)
};

// Per-launch control: stop flag to honour (nullptr: none) and, for a fused
// launch, where its residual goes.
struct LaunchCtl {
    const int *stop;
    bool fused;
    LoopParams lp;
    // First launch of a time step that forms the right-hand side itself
    // (column-streamed kernel only): g and the b it writes; null otherwise.
    // Its max |b| goes to lp.state->bmax.
    const float *rhs_g;
    float *rhs_b;
};

__device__ __forceinline__ unsigned warp_max_u(unsigned v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// Bit pattern of |x|: non-negative floats order like their bit patterns,
// and a NaN sorts above +Inf, so maxima of these propagate NaN.
__device__ __forceinline__ unsigned abs_bits(float x) {
    return __float_as_uint(fabsf(x));
}

// Stopping rule at the check of the fused launch's input iterate (run by one
// thread of the last block). k == 0 is the start of the step: no check there.
__device__ __forceinline__ void loop_decide(const LoopParams &lp, float rmax,
                                            float bmax) {
    LoopState *st = lp.state;
    st->rmax = rmax;
    st->bmax = bmax;
    const long long k = st->k;
    int stop = 0, status = 0;
    if (st->err) {
        stop = 1;
        status = -2;  // JACOBI_ERR_CUDA
    } else if (k > 0) {
        const double rm = (double)rmax, bm = (double)bmax;
        if (!isfinite(rm) || !isfinite(bm)) {
            stop = 1;
            status = -4;  // JACOBI_ERR_NONFINITE
        } else if (rm == 0.0 || rm < lp.tol * bm) {
            stop = 1;
        } else if (k >= lp.max_sweeps) {
            stop = 1;
            status = -3;  // JACOBI_ERR_NOT_CONVERGED
        }
    }
    if (stop) {
        st->status = status;
        st->where = lp.src_is_alt;
        st->result_k = k;
        st->stop = 1;
    } else {
        st->k = k + lp.interval;
    }
}

// Block-level end of a fused launch: reduce the block's max |J(u) - u| bits
// rm, fold it into LoopState::rbits, and let the last block to finish form
// rmax = d * max and apply the stopping rule with the step's bmax. Every
// block of a fused launch must call this exactly once (blocks with no cells
// pass 0). `scratch` is __shared__ space for 32 + 1 words.
__device__ __forceinline__ void fused_block_finish(unsigned rm,
                                                   const LoopParams &lp,
                                                   unsigned *scratch) {
    const int tid = threadIdx.x + threadIdx.y * blockDim.x;
    const int nthreads = blockDim.x * blockDim.y;
    const int lane = tid & 31, warp = tid >> 5, nwarps = (nthreads + 31) >> 5;
    rm = warp_max_u(rm);
    __syncthreads();  // scratch may alias memory the block used before
    if (lane == 0) scratch[warp] = rm;
    __syncthreads();
    if (tid != 0) return;
    unsigned br = 0u;
    for (int w = 0; w < nwarps; ++w) br = max(br, scratch[w]);
    LoopState *st = lp.state;
    if (br) atomicMax(&st->rbits, br);
    __threadfence();
    const unsigned nblocks = gridDim.x * gridDim.y;
    if (atomicAdd(&st->ticket, 1u) != nblocks - 1) return;
    // Last block: every other block's atomicMax is visible.
    __threadfence();
    const unsigned bits = atomicExch(&st->rbits, 0u);
    st->ticket = 0u;
    // max_i fl(d |x_i|) = fl(d max_i |x_i|): rounding is monotone.
    loop_decide(lp, __fmul_rn(lp.d, __uint_as_float(bits)), st->bmax);
}

// Block-level max of the orderable bit patterns `v` (one per thread) into
// *dst, one atomicMax per block. `scratch` is __shared__ space for 32
// words. Every thread of the block must call it.
__device__ __forceinline__ void block_max_into(unsigned v, unsigned *dst,
                                               unsigned *scratch) {
    const int tid = threadIdx.x + threadIdx.y * blockDim.x;
    const int nthreads = blockDim.x * blockDim.y;
    const int lane = tid & 31, warp = tid >> 5, nwarps = (nthreads + 31) >> 5;
    v = warp_max_u(v);
    __syncthreads();  // scratch may alias memory the block used before
    if (lane == 0) scratch[warp] = v;
    __syncthreads();
    if (tid != 0) return;
    unsigned bv = 0u;
    for (int w = 0; w < nwarps; ++w) bv = max(bv, scratch[w]);
    if (bv) atomicMax(dst, bv);
}

// |J(u) - u| of one cell as an orderable bit pattern (NaN above +Inf).
__device__ __forceinline__ unsigned change_bits(float nv, float c) {
    return abs_bits(__fsub_rn(nv, c));
}

// ---------------------------------------------------------------------------
// Programmatic dependent launch: a sweep kernel may be scheduled while the
// previous kernel on its stream is still draining; it runs its set-up that
// does not depend on that kernel (shared-memory carving, barrier init) and
// then waits in grid_dependency_wait() until the previous grid has finished
// and its writes are visible. It lets its own successor be scheduled early
// with allow_dependents(). Both are no-ops for an ordinary launch.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void grid_dependency_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void allow_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block,
                       size_t smem, cudaStream_t stream, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Launch wrappers (all asynchronous on `stream`). They return the CUDA error
// of the launch.
cudaError_t launch_rhs(const GridDesc &g, const float *u, const float *src,
                       float *b, cudaStream_t stream);
cudaError_t launch_copy_interior(const GridDesc &g, const float *src,
                                 float *dst, cudaStream_t stream);
// The Dirichlet ring (rows 0 and n-1, columns 0 and n-1) of src into dst.
cudaError_t launch_copy_ring(const GridDesc &g, const float *src, float *dst,
                             cudaStream_t stream);
// Bounds-checked build only: NaN into dst's interior unless *stop is set
// (stop may be null).
cudaError_t launch_poison_interior(const GridDesc &g, float *dst,
                                  const int *stop, cudaStream_t stream);
// Bounds-checked build only: exercise the checker on `grid` (n x ld
// floats): flags[k] receives ERR_BOUNDS if check k refused its access.
// Checks 0-2 are out of range (a shared load past the region declared to
// the checker, stores to a ring row and to a ring column of `grid`), 3-4
// in range (a shared load inside it, a store to an interior cell). Every
// store writes the value the cell already holds.
cudaError_t launch_bounds_selftest(float *grid, int n, long long ld,
                                   unsigned *flags, cudaStream_t stream);
cudaError_t launch_sweep_sync(const GridDesc &g, const float *u,
                              const float *b, float *out,
                              const LaunchCtl &ctl, cudaStream_t stream);
int sweep_sync_blocks(const GridDesc &g);
// Status of a step that a multi-step graph skipped because an earlier step
// failed (never returned to callers).
constexpr int kStepSkipped = -100;
// Fresh state for a step; k0: sweeps done before its first loop launch (one
// check interval when the step's first launch runs ahead of the loop).
// keep_where: a step skipped after a failure takes over the failed step's
// LoopState::where (runs whose steps start from either buffer).
cudaError_t launch_loop_reset(LoopState *st, const LoopState *prev,
                              cudaStream_t stream, long long k0 = 0,
                              bool keep_where = false);
// Set the if/else condition `cond` to 1 when the previous step's answer is
// in u (LoopState::where == 0), else 0.
cudaError_t launch_branch_on_where(const LoopState *prev,
                                   cudaGraphConditionalHandle cond,
                                   cudaStream_t stream);
// If st->where == 1, copy the interior of src (u_alt) into dst (u).
cudaError_t launch_settle(const GridDesc &g, const LoopState *st,
                          const float *src, float *dst, cudaStream_t stream);
// End of a loop iteration: clear the loop condition once LoopState::stop is
// set. The sweep kernels only set the flag; keeping the graph call in this
// one small kernel keeps it out of the sweep kernels.
cudaError_t launch_loop_condition(const LoopState *st,
                                  cudaGraphConditionalHandle cond,
                                  cudaStream_t stream);
// Residual norms of u into *out (rmax, bmax; out->racc, bacc and ticket
// must be 0, as they are after every use).
cudaError_t launch_residual(const GridDesc &g, const float *u, const float *b,
                            ResidualOut *out, cudaStream_t stream);
// bmax of the step's right-hand side into st->bmax (which must be 0).
cudaError_t launch_bnorm(const GridDesc &g, const float *u, const float *b,
                         LoopState *st, cudaStream_t stream);
// The part of bmax over the interior cells that have a Dirichlet-ring
// neighbour, with b = fl(u + g) formed on the fly (for a step whose first
// sweep launch forms b and reduces the other cells), folded into st->bmax.
cudaError_t launch_bnorm_ring(const GridDesc &g, const float *u,
                              const float *src, LoopState *st,
                              cudaStream_t stream);

// Tiled strategies (TMA-staged). Box = tile plus halo, read through the
// tensor maps of the source field and of b.
struct TileConf {
    int depth;    // D
    int tile_x;   // TX, multiple of 4
    int tile_y;   // TY
    int halo_x;   // box columns left of the tile (a multiple of 4 for ETB)
    int halo_y;   // box rows above the tile
    int box_x;    // TX + 2 * halo_x  (<= 256)
    int box_y;    // TY + 2 * halo_y  (<= 256)
    int origin;   // grid coordinate of the first tile's first cell (0 or 1)
    int threads;  // block size
    size_t smem;  // dynamic shared memory bytes
    int variant;  // compiled shape (exact temporal blocking)
    int ctas;     // persistent grid size (exact temporal blocking)
    // Block-asynchronous streaming kernel: super-tile sx x sy, ch float4
    // chunks per lane, grid_x x grid_y blocks (stream = 0: generic kernel,
    // one tile per block on a grid_x x grid_y grid).
    int stream, ch, sx, sy, grid_x, grid_y;
    // Block-asynchronous overlapping subdomains (generic kernel only).
    int overlap_x, overlap_y;
    // Column-streamed exact temporal blocking: the handle's work list
    // (device: [0] next run, [1] warps done, [2 ..] band start rows) and its
    // number of row bands.
    int *work;
    int bands;
};

// Exact temporal blocking (section 02 "Exact temporal blocking", after Meng
// and Skadron): halo D deep, valid region shrinking by one cell per sweep.
// streamed: whether the default tile may be the column-streamed kernel
// (not under persistent control, which needs a register-band shape).
int etb_configure(int n, int depth, int tile_x, int tile_y, TileConf *tc,
                  bool streamed = true);
// Raise the kernel's dynamic shared memory limit; call before any launch or
// graph capture that uses `tc`.
// (also sizes the persistent grid, tc.ctas)
cudaError_t prepare_sweep_etb(TileConf &tc, int n);
// src / b: the launch's input iterate and the right-hand side (raw
// pointers, for the column-streamed kernel; the others use the maps).
cudaError_t launch_sweep_etb(const GridDesc &g, const TileConf &tc,
                             const CUtensorMap *map_src,
                             const CUtensorMap *map_b, const float *src,
                             const float *b, float *out, ResidualOut *status,
                             const LaunchCtl &ctl, cudaStream_t stream);

// Column-streamed exact temporal blocking (kernels_etbs.cu): selected with
// tile_x = 128 - 2 * round_up(D, 4) and tile_y = 0, TileConf::variant =
// kEtbsVariant. D = 8 only.
constexpr int kEtbsVariant = 1000;
bool etbs_configure(int n, int depth, TileConf *tc);
cudaError_t prepare_sweep_etbs(TileConf &tc, int n);
// Host: the work list's row bands for `tc` (prepared) on an n x n grid:
// band_start receives bands + 1 row numbers, from 1 to n - 1. Returns the
// number of ints the device work list needs (2 + bands + 1).
int etbs_schedule(const TileConf &tc, int n, int *band_start, int cap);
// Whether the column-streamed kernel is the better D = 8 kernel for this
// grid on `sms` SMs (enough output rows per warp to amortise the pipeline).
bool etbs_preferred(int n, int sms);
cudaError_t launch_sweep_etbs(const GridDesc &g, const TileConf &tc,
                              const float *src, const float *b, float *out,
                              unsigned *err, const LaunchCtl &ctl,
                              cudaStream_t stream);

// Persistent exact temporal blocking (JACOBI_CONTROL_PERSISTENT): one
// cooperative launch runs a whole time step. `tc` must be a register-resident
// shape (etb_persistent_ok). prepare_etb_persistent raises the shared-memory
// limit and sizes the grid to the blocks that fit on the GPU at once.
bool etb_persistent_ok(const TileConf &tc);
cudaError_t prepare_etb_persistent(TileConf &tc, int n);
cudaError_t launch_etb_persistent(const GridDesc &g, const TileConf &tc,
                                  const CUtensorMap *map_u,
                                  const CUtensorMap *map_alt,
                                  const CUtensorMap *map_b, float *u,
                                  float *u_alt, const LoopParams &lp,
                                  long long rounds_per_check,
                                  cudaStream_t stream);

// Block-asynchronous sweep (section 02 "Block-asynchronous"): one-cell
// halo frozen at launch, all tile cells updated D times.
// overlap_x, overlap_y: cells neighbouring tiles share (even, smaller than
// the tile; "Hierarchical Jacobi Iteration for Structured Matrices on GPUs
// using Shared Memory", overlapping subdomains); 0 = plain tiles.
int ba_configure(int n, int depth, int tile_x, int tile_y, int overlap_x,
                 int overlap_y, TileConf *tc);
cudaError_t prepare_sweep_ba(const TileConf &tc);
// src / b: the launch's input iterate and the right-hand side (raw
// pointers, for the register-resident kernel; the others use the maps).
cudaError_t launch_sweep_ba(const GridDesc &g, const TileConf &tc,
                            const CUtensorMap *map_src,
                            const CUtensorMap *map_b, const float *src,
                            const float *b, float *out, ResidualOut *status,
                            const LaunchCtl &ctl, cudaStream_t stream);
// Blocks of one launch of a tiled strategy (size of the fused partials).
int tiled_blocks(const GridDesc &g, const TileConf &tc);
// Register-resident block-asynchronous kernel for 32 x 8 tiles
// (kernels_bar.cu): tc.stream = 2, one warp per strip of four tiles.
bool ba_reg_configure(int n, TileConf *tc);
cudaError_t prepare_sweep_ba_reg();
cudaError_t launch_sweep_ba_reg(const GridDesc &g, const TileConf &tc,
                                const float *src, const float *b, float *out,
                                unsigned *err, const LaunchCtl &ctl,
                                cudaStream_t stream);
// Streaming block-asynchronous kernel (kernels_ba.cu).
bool ba_stream_configure(int n, TileConf *tc);
cudaError_t prepare_sweep_ba_stream(const TileConf &tc);
cudaError_t launch_sweep_ba_stream(const GridDesc &g, const TileConf &tc,
                                   const CUtensorMap *map_src,
                                   const CUtensorMap *map_b, float *out,
                                   unsigned *err, const LaunchCtl &ctl,
                                   cudaStream_t stream);

}  // namespace tbj
