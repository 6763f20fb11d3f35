// Internal declarations shared by the CUDA translation units of the solver.
// Not part of the public ABI (include/jacobi.h is).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

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

// Exhaustive check of div_fixed against __fdiv_rn for one d: counts the
// finite float32 numerators whose quotients differ in any bit. `count` is a
// device word (set to 0 by the caller). Launch fastdiv_verify_launch.
cudaError_t fastdiv_verify_launch(float d, float y, unsigned long long *count,
                                  cudaStream_t stream);
// RN(1/d) in float32, computed exactly on the host.
float reciprocal_rn(float d);

// Error bits written by kernels into the handle's status word.
enum : unsigned {
    ERR_TMA_TIMEOUT = 1u,  // an mbarrier wait for a TMA load gave up
};

// Parameters common to all sweep kernels.
struct GridDesc {
    int n;         // grid side including the ring
    long long ld;  // row pitch in floats
    float r;       // coupling alpha dt / h^2
    float d;       // fl(1 + fl(4 r))
    float y;       // RN(1/d)
    bool fast;     // div_fixed verified equal to IEEE division for this d
};

// Result block of a residual reduction (device memory, one per handle).
struct ResidualOut {
    float rmax;
    float bmax;
    unsigned err;       // OR of ERR_* bits seen since the last reset
    unsigned ticket;    // last-block counter, returns to 0 after each use
};

// Launch wrappers (all asynchronous on `stream`). They return the CUDA error
// of the launch.
cudaError_t launch_rhs(const GridDesc &g, const float *u, const float *src,
                       float *b, cudaStream_t stream);
cudaError_t launch_copy_interior(const GridDesc &g, const float *src,
                                 float *dst, cudaStream_t stream);
cudaError_t launch_sweep_sync(const GridDesc &g, const float *u,
                              const float *b, float *out, cudaStream_t stream);
// partials: 2 * residual_blocks(g) floats of scratch.
int residual_blocks(const GridDesc &g);
cudaError_t launch_residual(const GridDesc &g, const float *u, const float *b,
                            float *partials, ResidualOut *out,
                            cudaGraphConditionalHandle cond, double tol,
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
};

// Exact temporal blocking (section 02 "Exact temporal blocking", after Meng
// and Skadron): halo D deep, valid region shrinking by one cell per sweep.
int etb_configure(int n, int depth, int tile_x, int tile_y, TileConf *tc);
// Raise the kernel's dynamic shared memory limit; call before any launch or
// graph capture that uses `tc`.
cudaError_t prepare_sweep_etb(const TileConf &tc);
cudaError_t launch_sweep_etb(const GridDesc &g, const TileConf &tc,
                             const CUtensorMap *map_src,
                             const CUtensorMap *map_b, float *out,
                             ResidualOut *status, cudaStream_t stream);

// Block-asynchronous sweep (section 02 "Block-asynchronous"): one-cell
// halo frozen at launch, all tile cells updated D times.
int ba_configure(int n, int depth, int tile_x, int tile_y, TileConf *tc);
cudaError_t prepare_sweep_ba(const TileConf &tc);
cudaError_t launch_sweep_ba(const GridDesc &g, const TileConf &tc,
                            const CUtensorMap *map_src,
                            const CUtensorMap *map_b, float *out,
                            ResidualOut *status, cudaStream_t stream);

}  // namespace tbj
