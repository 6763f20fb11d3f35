// Block-asynchronous sweeps ("Synchronous vs block-async Jacobi on one
// RTX 5050", section 02, after Anzt et al.) with the tiles held in
// registers, for the page's BA tile of 32 x 8 cells.
//
// BA tiles start at interior cell (1,1). A warp owns a strip of four tiles
// side by side: grid columns 1 + 128 u .. 128 u + 128 and rows 1 + 8 v ..
// 8 v + 8, lane l holding columns 1 + 128 u + 4 l .. + 3 of every row, so
// lanes 8t .. 8t + 7 hold tile t of the strip and every tile edge falls
// between two lanes. Tiles only see each other through their frozen
// one-cell halo, so a strip needs nothing from any other warp during its D
// sweeps: no shared memory and no barrier.
//
// At launch the warp copies, with cp.async into its slice of shared memory,
// the strip's 8 rows of u plus the rows above and below it (the frozen halo
// in y) over columns 128 u .. 128 u + 131, and its 8 rows of b. Every lane
// then takes into registers its four cells of each row and, per row, the
// cell west and east of them (the frozen halo in x for lanes at a tile's
// first or last column); b stays in shared memory and is read once per row
// and sweep. Each sweep then
// updates the 8 rows in registers, row by row, keeping the previous row's
// old value in a temporary; west/east neighbours inside a tile come from the
// adjacent lanes by shuffle, across a tile edge from the frozen values. The
// last sweep's values are written to the output buffer, cell by cell (the
// strip's columns are not 16-byte aligned).
//
// Cells outside the interior (the Dirichlet ring, columns or rows past it)
// keep their value; rows past the grid are not read.
#include <type_traits>

#include "jacobi_kernels.cuh"

namespace tbj {
namespace {

constexpr unsigned FULL = 0xffffffffu;
constexpr int kTX = 32, kTY = 8;  // the BA tile
constexpr int kWarps = 4;         // strips per block
constexpr int kMinBlocks = 3;     // blocks per SM the registers are sized for


// Columns 4 l + 1 .. 4 l + 4 of an aligned row segment from the two chunks
// that cover columns 4 l .. 4 l + 7.
__device__ __forceinline__ float4 shift1(float4 a, float4 b) {
    return make_float4(a.y, a.z, a.w, b.x);
}

// Asynchronous global -> shared copies of 16 or 4 bytes from grid `base`;
// src_bytes = 0 writes zeros and reads nothing. (Checked build: the copy is
// dropped when its destination or source is out of range.)
__device__ __forceinline__ void cp_async16(float *dst, const float *base,
                                           const float *src,
                                           unsigned src_bytes) {
    if (!smem_ok(dst, 16) || (src_bytes && !load_ok(base, src, 4))) return;
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(
                     static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
                 "l"(src), "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async4(float *dst, const float *base,
                                          const float *src, unsigned src_bytes) {
    if (!smem_ok(dst, 4) || (src_bytes && !load_ok(base, src, 1))) return;
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(
                     static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
                 "l"(src), "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

// Shared memory of one warp: the strip's u rows -1 .. kTY as 33 aligned
// float4 chunks per row (columns 128 u .. 128 u + 131), then b rows 0 ..
// kTY - 1 with lane l's four cells at floats 4 l .. 4 l + 3.
constexpr int kURow = 33 * 4;                  // floats per staged u row
constexpr int kWarpSmem = (kTY + 2) * kURow + kTY * 128;  // floats

template <bool FAST, bool EDGE, bool FUSED>
__device__ __forceinline__ void bar_strip(const float *__restrict__ src,
                                          const float *__restrict__ bsrc,
                                          float *__restrict__ out, float *sw,
                                          int n, long long ld, float r,
                                          float d, float y, int depth, int ux,
                                          int uy, float &rmf) {
    const int lane = threadIdx.x & 31;
    const int c0 = 128 * ux + 4 * lane;  // aligned: one column west of the cells
    const int gx0 = c0 + 1, gy0 = 1 + kTY * uy;
    const bool tile_w = (lane & 7) == 0, tile_e = (lane & 7) == 7;
    const int left = (lane + 31) & 31, right = (lane + 1) & 31;

    // Interior columns among this lane's four cells.
    unsigned colmask = 0xfu;
    if (EDGE) {
        colmask = 0u;
#pragma unroll
        for (int k = 0; k < 4; ++k) colmask |= (gx0 + k <= n - 2) ? (1u << k) : 0u;
    }

    // Stage u rows gy0 - 1 .. gy0 + kTY and b rows gy0 .. gy0 + kTY - 1;
    // rows past the grid and chunks past the row pitch read as zero.
    float *su = sw, *sbl = sw + (kTY + 2) * kURow + 4 * lane;
#pragma unroll
    for (int j = -1; j <= kTY; ++j) {
        const int gy = gy0 + j;
        const bool row_in = !EDGE || gy <= n - 1;
        const float *row = src + (long long)(row_in ? gy : 0) * ld;
        float *srow = su + (j + 1) * kURow;
        const bool a_in = row_in && c0 < ld;
        cp_async16(srow + 4 * lane, src, a_in ? row + c0 : src, a_in ? 16u : 0u);
        if (lane == 31) {
            const bool b_in = row_in && c0 + 4 < ld;
            cp_async16(srow + 128, src, b_in ? row + c0 + 4 : src, b_in ? 16u : 0u);
        }
        if (j >= 0 && j < kTY) {
            const float *brow = bsrc + (long long)(row_in ? gy : 0) * ld;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const bool in = row_in && gx0 + k < ld;
                cp_async4(sbl + 128 * j + k, bsrc, in ? brow + gx0 + k : bsrc,
                          in ? 4u : 0u);
            }
        }
    }
    cp_async_wait_all();
    __syncwarp();  // lane l reads lane l + 1's chunk

    float4 u[kTY], top, bot;
    float fw[kTY], fe[kTY];
    {
        const float4 a = lds4(su + 4 * lane), bb = lds4(su + 4 * lane + 4);
        top = shift1(a, bb);
        const float4 a2 = lds4(su + (kTY + 1) * kURow + 4 * lane);
        const float4 b2 = lds4(su + (kTY + 1) * kURow + 4 * lane + 4);
        bot = shift1(a2, b2);
    }
#pragma unroll
    for (int j = 0; j < kTY; ++j) {
        const float4 a = lds4(su + (j + 1) * kURow + 4 * lane);
        const float4 bb = lds4(su + (j + 1) * kURow + 4 * lane + 4);
        u[j] = shift1(a, bb);
        fw[j] = a.x;
        fe[j] = bb.y;
    }

    auto sweep = [&](auto resid) {
        constexpr bool RESID = decltype(resid)::value;
        float4 prev = top;
#pragma unroll
        for (int j = 0; j < kTY; ++j) {
            const float4 c = u[j];
            const float4 s4 = j + 1 < kTY ? u[j + 1 < kTY ? j + 1 : j] : bot;
            const float wv = __shfl_sync(FULL, c.w, left);
            const float ev = __shfl_sync(FULL, c.x, right);
            const float w = tile_w ? fw[j] : wv;
            const float e = tile_e ? fe[j] : ev;
            const float4 b4 = lds4(sbl + 128 * j);
            float4 nv = update4_we<FAST, false>(prev, c, s4, b4, w, e, r, d, y);
            const bool row_ok = !EDGE || gy0 + j <= n - 2;
            if (RESID && row_ok) {
                const float2 d01 = __fadd2_rn(make_float2(nv.x, nv.y),
                                              make_float2(-c.x, -c.y));
                const float2 d23 = __fadd2_rn(make_float2(nv.z, nv.w),
                                              make_float2(-c.z, -c.w));
                if (colmask & 1u) rmf = max_nan_abs(rmf, d01.x);
                if (colmask & 2u) rmf = max_nan_abs(rmf, d01.y);
                if (colmask & 4u) rmf = max_nan_abs(rmf, d23.x);
                if (colmask & 8u) rmf = max_nan_abs(rmf, d23.y);
            }
            if (EDGE) nv = hold4(nv, c, row_ok, colmask);
            prev = c;
            u[j] = nv;
        }
    };
    if (FUSED)
        sweep(std::true_type{});
    else
        sweep(std::false_type{});
#pragma unroll 1
    for (int s = 1; s < depth; ++s) sweep(std::false_type{});

#pragma unroll
    for (int j = 0; j < kTY; ++j) {
        const int gy = gy0 + j;
        if (EDGE && gy > n - 2) break;
        float *o = out + (long long)gy * ld + gx0;
        if (!EDGE || colmask == 0xfu) {
            gst1(o + 0, u[j].x);
            gst1(o + 1, u[j].y);
            gst1(o + 2, u[j].z);
            gst1(o + 3, u[j].w);
        } else {
            if (colmask & 1u) gst1(o + 0, u[j].x);
            if (colmask & 2u) gst1(o + 1, u[j].y);
            if (colmask & 4u) gst1(o + 2, u[j].z);
            if (colmask & 8u) gst1(o + 3, u[j].w);
        }
    }
}

template <bool FAST, bool FUSED>
__global__ void __launch_bounds__(32 * kWarps, kMinBlocks)
k_bar(const float *__restrict__ src, const float *__restrict__ bsrc,
      float *__restrict__ out, int n, long long ld, float r, float d, float y,
      int depth, int units_x, int units, unsigned *err, const int *stop,
      LoopParams lp) {
    __shared__ unsigned fin_scratch[33];
    extern __shared__ __align__(16) float smem[];  // kWarps slices
    bounds_begin(smem, 0, out, nullptr, src, bsrc, n, ld, err);
    allow_dependents();
    // Everything below reads what the previous kernel wrote.
    grid_dependency_wait();
    if (stop && *stop) return;  // same value for every thread of the launch
    const int unit = blockIdx.x * kWarps + (threadIdx.x >> 5);
    float rmf = 0.f;
    if (unit < units) {  // uniform per warp
        const int ux = unit % units_x, uy = unit / units_x;
        const bool edge = 128 * ux + 128 > n - 2 || kTY * uy + kTY > n - 2;
        float *sw = smem + (threadIdx.x >> 5) * kWarpSmem;
        if (edge)
            bar_strip<FAST, true, FUSED>(src, bsrc, out, sw, n, ld, r, d, y,
                                         depth, ux, uy, rmf);
        else
            bar_strip<FAST, false, FUSED>(src, bsrc, out, sw, n, ld, r, d, y,
                                          depth, ux, uy, rmf);
    }
    if (FUSED) fused_block_finish(__float_as_uint(rmf), lp, fin_scratch);
}

constexpr size_t kSmemBytes = (size_t)kWarps * kWarpSmem * sizeof(float);

}  // namespace

cudaError_t prepare_sweep_ba_reg() {
    const void *kernels[4] = {(const void *)k_bar<true, false>,
                              (const void *)k_bar<false, false>,
                              (const void *)k_bar<true, true>,
                              (const void *)k_bar<false, true>};
    for (const void *k : kernels) {
        cudaError_t e = cudaFuncSetAttribute(
            k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

bool ba_reg_configure(int n, TileConf *tc) {
    if (tc->tile_x != kTX || tc->tile_y != kTY) return false;
    const int units_x = (n - 2 + 127) / 128, units_y = (n - 2 + kTY - 1) / kTY;
    tc->stream = 2;
    tc->ch = 1;
    tc->sx = 128;
    tc->sy = kTY;
    tc->threads = 32 * kWarps;
    tc->smem = kSmemBytes;
    tc->grid_x = (units_x * units_y + kWarps - 1) / kWarps;
    tc->grid_y = 1;
    return true;
}

cudaError_t launch_sweep_ba_reg(const GridDesc &g, const TileConf &tc,
                                const float *src, const float *b, float *out,
                                unsigned *err, const LaunchCtl &ctl,
                                cudaStream_t stream) {
    const int units_x = (g.n - 2 + 127) / 128, units_y = (g.n - 2 + kTY - 1) / kTY;
    const int units = units_x * units_y;
#define TBJ_K(F, FU)                                                         \
    launch_pdl(k_bar<F, FU>, dim3(tc.grid_x), dim3(32 * kWarps), kSmemBytes, \
               stream, src, b, out, g.n, g.ld, g.r, g.d, g.y, tc.depth,      \
               units_x, units, err, ctl.stop, ctl.lp)
    if (g.fast) return ctl.fused ? TBJ_K(true, true) : TBJ_K(true, false);
    return ctl.fused ? TBJ_K(false, true) : TBJ_K(false, false);
#undef TBJ_K
}

}  // namespace tbj
