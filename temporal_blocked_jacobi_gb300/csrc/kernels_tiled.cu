// Block-asynchronous sweeps ("Synchronous vs block-async Jacobi on one
// RTX 5050", section 02, after Anzt et al.), TMA-staged.
//
// A block owns one tile of TX x TY cells. Thread 0 issues three 2-D TMA box
// loads onto one mbarrier: the box (tile plus a one-cell halo) of the source
// field into two shared buffers (the ping-pong pair) and the same box of b.
// The halo is frozen at its value at launch; every one of the D sweeps
// updates all tile cells, alternating buffers, and the last sweep writes the
// tile's cells straight to the destination field in global memory.
//
// Cells on the Dirichlet ring and cells outside the grid (which the TMA load
// fills with zeros) are never updated; no updated cell reads a cell outside
// the grid. The box's left edge is kept on a 16-byte boundary (TMA rule):
// tile k starts at column 1 + k*SX, the box at (k*SX) rounded down to a
// multiple of 4, and the box is TX + 4 columns wide; the extra columns are
// loaded and ignored.
//
// Overlapping subdomains ("Hierarchical Jacobi Iteration for Structured
// Matrices on GPUs using Shared Memory", overlapping subdomains in 1-D and
// 2-D): with overlaps OX, OY (even, smaller than the tile) tiles start every
// SX = TX - OX columns and SY = TY - OY rows, so neighbours share OX columns
// (OY rows). Every tile sweeps all its cells, but writes back only the cells
// it owns: of each shared band the nearer half, i.e. it leaves out OX/2
// columns (OY/2 rows) next to each edge it shares with another tile. With
// OX = OY = 0 this is the plain block-asynchronous launch; with OX even the rounding of the box start shifts the tile at
// most 2 columns into the box, which TX + 4 columns still hold.
#include <cudaTypedefs.h>

#include "jacobi_kernels.cuh"

namespace tbj {
namespace {

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, unsigned count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(count)
                 : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar,
                                                      unsigned bytes) {
    asm volatile(
        "mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(
            smem_addr(bar)),
        "r"(bytes)
        : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, unsigned parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait for phase 0 of the barrier, giving up after ~1 s.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar) {
    if (mbar_try_wait(bar, 0)) return true;
    const uint64_t t0 = global_ns();
    while (!mbar_try_wait(bar, 0)) {
        if (global_ns() - t0 > 1000000000ull) return false;
    }
    return true;
}

__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map,
                                            uint64_t *bar, int x, int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::"
        "complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y),
        "r"(smem_addr(bar))
        : "memory");
}

__host__ __device__ constexpr size_t round128(size_t b) {
    return (b + 127) / 128 * 128;
}

// Shared memory: [barrier | A | B | Bb], every part 128-byte aligned.
__host__ __device__ inline size_t buffer_bytes(int box_x, int box_y) {
    return round128((size_t)box_x * box_y * sizeof(float));
}

// Tile geometry of one launch (see the overlapping-subdomain note above).
struct TileGeom {
    int tx, ty;      // tile size
    int sx, sy;      // distance between tile starts (tile - overlap)
    int ox2, oy2;    // half overlaps: cells left to the neighbour per edge
    int box_x, box_y;
};

template <int D, bool FAST, bool FUSED>
__global__ void __launch_bounds__(512)
k_block_async(const __grid_constant__ CUtensorMap map_src,
              const __grid_constant__ CUtensorMap map_b,
              float *__restrict__ out, int n, long long ld, float r, float d,
              float y, TileGeom tg, unsigned *err, const int *stop,
              LoopParams lp) {
    if (stop && *stop) return;  // same value for every thread of the launch
    __shared__ unsigned fin_scratch[33];
    extern __shared__ __align__(128) unsigned char smem_raw[];
    bounds_begin(smem_raw, 0, out, nullptr, nullptr, nullptr, n, ld, err);
    const int tx = tg.tx, ty = tg.ty, box_x = tg.box_x, box_y = tg.box_y;
    const int gx0 = 1 + blockIdx.x * tg.sx;  // tile's first cell (grid)
    const int gy0 = 1 + blockIdx.y * tg.sy;
    if (gx0 > n - 2 || gy0 > n - 2) {
        if (FUSED) fused_block_finish(0u, lp, fin_scratch);
        return;
    }
    // Box origin: one cell up, and left to a 16-byte boundary.
    const int bxo = (gx0 - 1) & ~3;
    const int byo = gy0 - 1;
    const int hx = gx0 - bxo, hy = 1;  // box position of the tile's first cell
    // Cells this tile writes back (grid coordinates, half-open).
    const int wx0 = gx0 + (blockIdx.x > 0 ? tg.ox2 : 0);
    const int wx1 = gx0 + tx - (blockIdx.x + 1 < gridDim.x ? tg.ox2 : 0);
    const int wy0 = gy0 + (blockIdx.y > 0 ? tg.oy2 : 0);
    const int wy1 = gy0 + ty - (blockIdx.y + 1 < gridDim.y ? tg.oy2 : 0);

    // Offsets from the __shared__ array itself keep every access in the
    // shared address space.
    const unsigned pad = (128u - (smem_addr(smem_raw) & 127u)) & 127u;
    unsigned char *base = smem_raw + pad;
    uint64_t *bar = reinterpret_cast<uint64_t *>(base);
    const size_t buf = buffer_bytes(box_x, box_y);
    float *sA = reinterpret_cast<float *>(base + 128);
    float *sB = reinterpret_cast<float *>(base + 128 + buf);
    float *sBb = reinterpret_cast<float *>(base + 128 + 2 * buf);

    const int tid = threadIdx.x;
    if (tid == 0) {
        mbar_init(bar, 1);
        const unsigned box_bytes = (unsigned)(box_x * box_y * sizeof(float));
        mbar_arrive_expect_tx(bar, 3u * box_bytes);
        // (checked build: a load that fails its check is not issued, and
        // the wait for it runs into its time limit)
        if (tma_ok(sA, box_bytes, bxo)) tma_load_2d(sA, &map_src, bar, bxo, byo);
        if (tma_ok(sB, box_bytes, bxo)) tma_load_2d(sB, &map_src, bar, bxo, byo);
        if (tma_ok(sBb, box_bytes, bxo)) tma_load_2d(sBb, &map_b, bar, bxo, byo);
    }
    __syncthreads();
    const bool ok = mbar_wait_bounded(bar);
    if (__syncthreads_or(!ok)) {
        if (tid == 0) atomicOr(err, (unsigned)ERR_TMA_TIMEOUT);
        // Let any copy still in flight land before the block's shared
        // memory is released (bounded as well).
        mbar_wait_bounded(bar);
        if (FUSED) fused_block_finish(0u, lp, fin_scratch);
        return;
    }

    // Box rows/columns whose grid cell is an interior cell.
    const int vr0 = 1 - byo, vr1 = n - 1 - byo;  // [vr0, vr1)
    const int vc0 = 1 - bxo, vc1 = n - 1 - bxo;
    const int warp = tid >> 5, lane = tid & 31;
    const int nwarps = blockDim.x >> 5;

    unsigned rm = 0u;
#pragma unroll 1
    for (int s = 0; s < D; ++s) {
        const float *src = (s & 1) ? sB : sA;
        float *dst = (s & 1) ? sA : sB;
        const int r0 = max(hy, vr0), r1 = min(hy + ty, vr1);
        const int c0 = max(hx, vc0), c1 = min(hx + tx, vc1);
        const bool last = (s == D - 1);
        for (int by = r0 + warp; by < r1; by += nwarps) {
            const float *row = src + by * box_x;
            const float *brow = sBb + by * box_x;
            const int gy = byo + by;
            const bool own_row = gy >= wy0 && gy < wy1;
            for (int bx = c0 + lane; bx < c1; bx += 32) {
                const float w = lds1(row + bx - 1), e = lds1(row + bx + 1);
                const float nn = lds1(row + bx - box_x), ss = lds1(row + bx + box_x);
                const float v = jacobi_update<FAST>(w, e, nn, ss, lds1(brow + bx), r, d, y);
                const int gx = bxo + bx;
                const bool own = own_row && gx >= wx0 && gx < wx1;
                if (FUSED && s == 0 && own)  // |J(u) - u| of the launch's input
                    rm = max(rm, change_bits(v, lds1(row + bx)));
                if (last) {
                    if (own) gst1(out + (long long)gy * ld + gx, v);
                } else {
                    sts1(dst + by * box_x + bx, v);
                }
            }
        }
        if (!last) __syncthreads();
    }
    if (FUSED) fused_block_finish(rm, lp, fin_scratch);
}

cudaError_t launch_tiled(const GridDesc &g, const TileConf &tc,
                         const CUtensorMap *map_src, const CUtensorMap *map_b,
                         float *out, unsigned *err, const LaunchCtl &ctl,
                         cudaStream_t stream) {
    const dim3 grid(tc.grid_x, tc.grid_y);
    const dim3 block(tc.threads);
    TileGeom tg;
    tg.tx = tc.tile_x;
    tg.ty = tc.tile_y;
    tg.sx = tc.tile_x - tc.overlap_x;
    tg.sy = tc.tile_y - tc.overlap_y;
    tg.ox2 = tc.overlap_x / 2;
    tg.oy2 = tc.overlap_y / 2;
    tg.box_x = tc.box_x;
    tg.box_y = tc.box_y;
#define TBJ_K(DD, F, FU)                                                      \
    k_block_async<DD, F, FU><<<grid, block, tc.smem, stream>>>(               \
        *map_src, *map_b, out, g.n, g.ld, g.r, g.d, g.y, tg, err, ctl.stop,   \
        ctl.lp)
#define TBJ_LAUNCH(DD)                                                        \
    case DD:                                                                  \
        if (g.fast) {                                                         \
            if (ctl.fused) TBJ_K(DD, true, true);                             \
            else TBJ_K(DD, true, false);                                      \
        } else {                                                              \
            if (ctl.fused) TBJ_K(DD, false, true);                            \
            else TBJ_K(DD, false, false);                                     \
        }                                                                     \
        return cudaGetLastError();
    switch (tc.depth) {
        TBJ_LAUNCH(1)
        TBJ_LAUNCH(2)
        TBJ_LAUNCH(4)
        TBJ_LAUNCH(8)
        TBJ_LAUNCH(16)
        TBJ_LAUNCH(32)
        default:
            return cudaErrorInvalidValue;
    }
#undef TBJ_LAUNCH
#undef TBJ_K
}

template <int DD>
cudaError_t prepare_depth(size_t smem) {
    const void *kernels[4] = {(const void *)k_block_async<DD, true, false>,
                              (const void *)k_block_async<DD, false, false>,
                              (const void *)k_block_async<DD, true, true>,
                              (const void *)k_block_async<DD, false, true>};
    for (const void *k : kernels) {
        cudaError_t e = cudaFuncSetAttribute(
            k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t prepare_tiled(const TileConf &tc) {
    switch (tc.depth) {
        case 1: return prepare_depth<1>(tc.smem);
        case 2: return prepare_depth<2>(tc.smem);
        case 4: return prepare_depth<4>(tc.smem);
        case 8: return prepare_depth<8>(tc.smem);
        case 16: return prepare_depth<16>(tc.smem);
        case 32: return prepare_depth<32>(tc.smem);
        default: return cudaErrorInvalidValue;
    }
}

constexpr size_t kMaxSmem = 227 * 1024;

int finish_conf(TileConf *tc) {
    if (tc->box_x > 256 || tc->box_y > 256 || tc->box_x % 4 != 0) return -5;
    tc->smem = 128 + 128 + 3 * buffer_bytes(tc->box_x, tc->box_y);
    if (tc->smem > kMaxSmem) return -5;
    return 0;
}

}  // namespace

// Tiles of t cells starting every t - o cells needed to cover ni cells (at
// least one).
int subdomain_count(int ni, int t, int o) {
    if (ni <= t) return 1;
    return (ni - o + (t - o) - 1) / (t - o);
}

int ba_configure(int n, int depth, int tile_x, int tile_y, int overlap_x,
                 int overlap_y, TileConf *tc) {
    if (depth != 1 && depth != 2 && depth != 4 && depth != 8 && depth != 16 &&
        depth != 32)
        return -1;
    if (tile_x == 0) tile_x = 32;
    if (tile_y == 0) tile_y = 8;
    if (tile_x < 4 || tile_x % 4 != 0 || tile_y < 1) return -1;
    if (overlap_x < 0 || overlap_y < 0 || overlap_x % 2 || overlap_y % 2 ||
        overlap_x >= tile_x || overlap_y >= tile_y)
        return -1;
    tc->depth = depth;
    tc->tile_x = tile_x;
    tc->tile_y = tile_y;
    tc->overlap_x = overlap_x;
    tc->overlap_y = overlap_y;
    tc->halo_x = 1;  // box starts at most 3 columns left of the tile
    tc->halo_y = 1;
    tc->box_x = tile_x + 4;  // tile + 2 halo columns, rounded to 16 bytes
    tc->box_y = tile_y + 2;
    tc->origin = 1;
    const int cells = tile_x * tile_y;
    tc->threads = cells >= 512 ? 512 : (cells + 31) / 32 * 32;
    tc->variant = 0;
    tc->ctas = 0;
    tc->stream = tc->ch = tc->sx = tc->sy = 0;
    tc->work = nullptr;
    tc->bands = 0;
    tc->grid_x = subdomain_count(n - 2, tile_x, overlap_x);
    tc->grid_y = subdomain_count(n - 2, tile_y, overlap_y);
    // Non-overlapping 32 x 8 tiles (the default) are held in registers; the
    // streaming kernel takes every other non-overlapping shape it can fit;
    // the generic one-tile-per-block kernel below is kept for the rest.
    if (overlap_x == 0 && overlap_y == 0 && ba_reg_configure(n, tc)) return 0;
    if (overlap_x == 0 && overlap_y == 0 && ba_stream_configure(n, tc)) return 0;
    return finish_conf(tc);
}

cudaError_t prepare_sweep_ba(const TileConf &tc) {
    if (tc.stream == 2) return prepare_sweep_ba_reg();
    if (tc.stream) return prepare_sweep_ba_stream(tc);
    return prepare_tiled(tc);
}

cudaError_t launch_sweep_ba(const GridDesc &g, const TileConf &tc,
                            const CUtensorMap *map_src,
                            const CUtensorMap *map_b, const float *src,
                            const float *b, float *out, ResidualOut *status,
                            const LaunchCtl &ctl, cudaStream_t stream) {
    unsigned *err = ctl.lp.state ? &ctl.lp.state->err : &status->err;
    if (tc.stream == 2)
        return launch_sweep_ba_reg(g, tc, src, b, out, err, ctl, stream);
    if (tc.stream)
        return launch_sweep_ba_stream(g, tc, map_src, map_b, out, err, ctl,
                                      stream);
    return launch_tiled(g, tc, map_src, map_b, out, err, ctl, stream);
}

int tiled_blocks(const GridDesc &g, const TileConf &tc) {
    (void)g;
    if (tc.ctas > 0) return tc.ctas;  // persistent grid
    return tc.grid_x * tc.grid_y;
}

}  // namespace tbj
