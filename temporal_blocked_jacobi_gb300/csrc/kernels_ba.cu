// Block-asynchronous sweeps ("Synchronous vs block-async Jacobi on one
// RTX 5050", section 02, after Anzt et al.), streaming form.
//
// The interior is cut into BA tiles of TX x TY cells starting at interior
// cell (1,1); each BA tile is swept D times against a one-cell halo frozen at
// its value at launch. A block handles a super-tile of whole BA tiles, SX x SY
// cells (SX a multiple of TX, SY of TY), so that no BA tile spans two blocks.
//
// Layout. The box is the super-tile plus a one-cell halo, loaded by TMA as
// BX = 128*CH columns x (SY + 2) rows starting at grid cell (x0-1, y0-1) --
// x0 - 1 = k*SX is a multiple of 4, as TMA requires; columns past SX + 1 are
// loaded and unused. Box column j is held by lane (j mod 128)/4 of chunk
// j/128; warp w streams the band of box rows 1 + [w*RW, (w+1)*RW).
//
// Three shared buffers: A keeps the box as loaded (the launch snapshot) for
// the whole launch; B and C hold the in-tile iterates (sweep 0 reads A and
// writes B, sweep 1 reads B and writes C, ...). A neighbour that lies in
// another BA tile, or in the halo, is always read from A:
//   * rows: the cell above a BA tile's first row and below its last row;
//   * columns: BA tiles start at box columns that are multiples of TX, i.e.
//     at component .y of a float4 chunk whose column is a multiple of TX; for
//     such chunks the east neighbour of .x and the west neighbour of .y come
//     from A. (West of .x and east of .w are never across a tile edge.)
// Cells of the halo and unused columns are computed but never read through
// B or C, so their values do not matter. In super-tiles that reach the
// Dirichlet ring, ring cells keep their value in every buffer.
#include "jacobi_kernels.cuh"

namespace tbj {
namespace {

constexpr unsigned FULL = 0xffffffffu;
constexpr int kRowsMax = 64;  // SY <= 64

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
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


// J for the four cells of a chunk. ex = east neighbour of .x, wy = west
// neighbour of .y (the chunk's own .y/.x unless a BA tile edge lies between).
template <bool FAST>
__device__ __forceinline__ float4 update4(float4 n4, float4 c4, float4 s4,
                                          float4 b4, float w, float e,
                                          float ex, float wy, float r, float d,
                                          float y) {
    if (FAST) {
        // Packed pairs as in the exact-temporal-blocking kernel; r * s stays
        // scalar so the compiler cannot fuse it into the addition of b.
        const float2 d2 = make_float2(d, d), y2 = make_float2(y, y);
        const float2 h01 = make_float2(__fadd_rn(w, ex), __fadd_rn(wy, c4.z));
        const float2 h23 = make_float2(__fadd_rn(c4.y, c4.w), __fadd_rn(c4.z, e));
        const float2 v01 = __fadd2_rn(make_float2(n4.x, n4.y), make_float2(s4.x, s4.y));
        const float2 v23 = __fadd2_rn(make_float2(n4.z, n4.w), make_float2(s4.z, s4.w));
        const float2 s01 = __fadd2_rn(h01, v01), s23 = __fadd2_rn(h23, v23);
        const float2 rs01 = make_float2(__fmul_rn(r, s01.x), __fmul_rn(r, s01.y));
        const float2 rs23 = make_float2(__fmul_rn(r, s23.x), __fmul_rn(r, s23.y));
        const float2 q01 = div2_fixed(__fadd2_rn(make_float2(b4.x, b4.y), rs01), d2, y2);
        const float2 q23 = div2_fixed(__fadd2_rn(make_float2(b4.z, b4.w), rs23), d2, y2);
        return make_float4(q01.x, q01.y, q23.x, q23.y);
    }
    float4 o;
    o.x = jacobi_update<false>(w, ex, n4.x, s4.x, b4.x, r, d, y);
    o.y = jacobi_update<false>(wy, c4.z, n4.y, s4.y, b4.y, r, d, y);
    o.z = jacobi_update<false>(c4.y, c4.w, n4.z, s4.z, b4.z, r, d, y);
    o.w = jacobi_update<false>(c4.z, e, n4.w, s4.w, b4.w, r, d, y);
    return o;
}

template <int CH, int RW, int NW, bool FAST, bool EDGE, bool FUSED>
__device__ __forceinline__ void ba_sweeps(const float *sA, float *sB, float *sC,
                                          const float4 (&breg)[RW][CH],
                                          float *__restrict__ out, int n,
                                          long long ld, float r, float d,
                                          float y, int depth, int tx, int ty,
                                          int sx, int sy, int bxo, int byo,
                                          unsigned &rm) {
    constexpr int BX = 128 * CH;
    const int lane = threadIdx.x & 31;
    const int r0 = 1 + (threadIdx.x >> 5) * RW;  // first box row of the band
    const int col = 4 * lane;
    const int left = (lane + 31) & 31, right = (lane + 1) & 31;

    // Per chunk: does a BA tile start at its .y? Which of its cells belong to
    // this super-tile (stored), and which are interior grid cells (updated)?
    bool edge_x[CH];
    unsigned keep[CH], interior[CH];
#pragma unroll
    for (int c = 0; c < CH; ++c) {
        const int bx = 128 * c + col;
        edge_x[c] = (bx % tx) == 0 && bx <= sx;
        unsigned km = 0, im = 0;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int gx = bxo + bx + k;
            const bool inside = gx >= 1 && gx <= n - 2;
            im |= inside ? (1u << k) : 0u;
            km |= (inside && bx + k >= 1 && bx + k <= sx) ? (1u << k) : 0u;
        }
        keep[c] = km;
        interior[c] = EDGE ? im : 0xfu;
    }

#pragma unroll 1
    for (int s = 0; s < depth; ++s) {
        const float *src = s == 0 ? sA : ((s & 1) ? sB : sC);
        float *dst = (s & 1) ? sC : sB;
        const bool last = (s == depth - 1);
        if (r0 <= sy) {
            float4 nr[CH], cr[CH];
            // Row above the band: from A if the band starts a BA tile.
            const bool first0 = ((byo + r0 - 1) % ty) == 0;
#pragma unroll
            for (int c = 0; c < CH; ++c) {
                nr[c] = lds4((first0 ? sA : src) + (r0 - 1) * BX + 128 * c + col);
                cr[c] = lds4(src + r0 * BX + 128 * c + col);
            }
#pragma unroll
            for (int j = 0; j < RW; ++j) {
                const int row = r0 + j;
                if (row > sy) break;  // uniform per warp
                const int gy = byo + row;
                const int trow = (gy - 1) % ty;
                const bool tile_last = trow == ty - 1 || row == sy;
                if (j > 0 && trow == 0) {  // first row of a BA tile
#pragma unroll
                    for (int c = 0; c < CH; ++c)
                        nr[c] = lds4(sA + (row - 1) * BX + 128 * c + col);
                }
                float4 nx[CH], sr[CH];
#pragma unroll
                for (int c = 0; c < CH; ++c) {
                    nx[c] = lds4(src + (row + 1) * BX + 128 * c + col);
                    sr[c] = tile_last ? lds4(sA + (row + 1) * BX + 128 * c + col)
                                      : nx[c];
                }
                float wv[CH], ev[CH];
#pragma unroll
                for (int c = 0; c < CH; ++c) {
                    wv[c] = __shfl_sync(FULL, cr[c].w, left);
                    ev[c] = __shfl_sync(FULL, cr[c].x, right);
                }
                const bool row_ok = !EDGE || (gy >= 1 && gy <= n - 2);
#pragma unroll
                for (int c = 0; c < CH; ++c) {
                    const float w = (c > 0 && lane == 0) ? wv[c - 1] : wv[c];
                    const float e = (c < CH - 1 && lane == 31) ? ev[c + 1] : ev[c];
                    float ex = cr[c].y, wy = cr[c].x;
                    if (edge_x[c]) {  // a BA tile edge between .x and .y
                        const float4 a4 = lds4(sA + row * BX + 128 * c + col);
                        ex = a4.y;
                        wy = a4.x;
                    }
                    float4 nv = update4<FAST>(nr[c], cr[c], sr[c], breg[j][c], w, e,
                                              ex, wy, r, d, y);
                    if (FUSED && s == 0 && row_ok) {
                        // |J(u) - u| of the launch's input (sweep 0 reads A,
                        // so nv = J(u)) at this super-tile's cells.
                        const float4 c4 = cr[c];
                        const unsigned m = keep[c];
                        if (m & 1u) rm = max(rm, change_bits(nv.x, c4.x));
                        if (m & 2u) rm = max(rm, change_bits(nv.y, c4.y));
                        if (m & 4u) rm = max(rm, change_bits(nv.z, c4.z));
                        if (m & 8u) rm = max(rm, change_bits(nv.w, c4.w));
                    }
                    if (EDGE) nv = hold4(nv, cr[c], row_ok, interior[c]);
                    if (!last) {
                        sts4(dst + row * BX + 128 * c + col, nv);
                    } else if (row_ok && keep[c]) {
                        float *g = out + (long long)gy * ld + (bxo + 128 * c + col);
                        if (keep[c] == 0xfu) {
                            gst4(g, nv);
                        } else {
                            if (keep[c] & 1u) gst1(g + 0, nv.x);
                            if (keep[c] & 2u) gst1(g + 1, nv.y);
                            if (keep[c] & 4u) gst1(g + 2, nv.z);
                            if (keep[c] & 8u) gst1(g + 3, nv.w);
                        }
                    }
                    nr[c] = cr[c];
                    cr[c] = nx[c];
                }
            }
        }
        if (!last) __syncthreads();
    }
}

template <int CH, int RW, int NW, bool FAST, bool FUSED>
__global__ void __launch_bounds__(32 * NW)
k_ba(const __grid_constant__ CUtensorMap map_src,
     const __grid_constant__ CUtensorMap map_b, float *__restrict__ out, int n,
     long long ld, float r, float d, float y, int depth, int tx, int ty, int sx,
     int sy, unsigned *err, const int *stop, LoopParams lp) {
    constexpr int BX = 128 * CH;
    constexpr int ROWS = kRowsMax + 2;
    __shared__ unsigned fin_scratch[33];
    allow_dependents();
    const int bxo = blockIdx.x * sx;  // grid coords of box cell (0,0)
    const int byo = blockIdx.y * sy;

    extern __shared__ __align__(128) unsigned char smem_raw[];
    bounds_begin(smem_raw, 0, out, nullptr, nullptr, nullptr, n, ld, err);
    const unsigned pad = (128u - (smem_addr(smem_raw) & 127u)) & 127u;
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem_raw + pad);
    float *sA = reinterpret_cast<float *>(smem_raw + pad + 128);
    float *sB = sA + BX * ROWS;
    float *sC = sB + BX * ROWS;

    const int tid = threadIdx.x;
    if (tid == 0) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(bar))
                     : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    // Everything below reads what the previous kernel wrote.
    grid_dependency_wait();
    if (stop && *stop) return;  // same value for every thread of the launch
    if (tid == 0) {
        asm volatile(
            "mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(
                smem_addr(bar)),
            "r"((unsigned)(2 * BX * (sy + 2) * sizeof(float)))
            : "memory");
        const unsigned box = (unsigned)(BX * (sy + 2) * sizeof(float));
        // (checked build: a load that fails its check is not issued, and
        // the wait for it runs into its time limit)
        if (tma_ok(sA, box, bxo)) tma_load_2d(sA, &map_src, bar, bxo, byo);
        if (tma_ok(sC, box, bxo)) tma_load_2d(sC, &map_b, bar, bxo, byo);  // b staged in C
    }
    __syncthreads();
    const bool ok = mbar_wait_bounded(bar);
    if (__syncthreads_or(!ok)) {
        if (tid == 0) atomicOr(err, (unsigned)ERR_TMA_TIMEOUT);
        mbar_wait_bounded(bar);
        if (FUSED) fused_block_finish(0u, lp, fin_scratch);
        return;
    }
    const int lane = tid & 31;
    const int r0 = 1 + (tid >> 5) * RW;
    float4 breg[RW][CH];
#pragma unroll
    for (int j = 0; j < RW; ++j)
#pragma unroll
        for (int c = 0; c < CH; ++c)
            breg[j][c] = r0 + j <= sy ? lds4(sC + (r0 + j) * BX + 128 * c + 4 * lane)
                                      : make_float4(0.f, 0.f, 0.f, 0.f);
    __syncthreads();  // C is first written by sweep 1, after a barrier

    unsigned rm = 0u;
    const bool edge = bxo < 1 || byo < 1 || bxo + BX > n - 1 ||
                      byo + sy + 2 > n - 1;
    if (edge)
        ba_sweeps<CH, RW, NW, FAST, true, FUSED>(sA, sB, sC, breg, out, n, ld, r,
                                                 d, y, depth, tx, ty, sx, sy, bxo,
                                                 byo, rm);
    else
        ba_sweeps<CH, RW, NW, FAST, false, FUSED>(sA, sB, sC, breg, out, n, ld, r,
                                                  d, y, depth, tx, ty, sx, sy, bxo,
                                                  byo, rm);
    if (FUSED) fused_block_finish(rm, lp, fin_scratch);
}

template <int CH>
constexpr size_t smem_bytes() {
    return 256 + 3 * (size_t)(128 * CH) * (kRowsMax + 2) * sizeof(float);
}

template <int CH, int RW, int NW>
cudaError_t launch_ch(const GridDesc &g, const TileConf &tc,
                      const CUtensorMap *map_src, const CUtensorMap *map_b,
                      float *out, unsigned *err, const LaunchCtl &ctl,
                      cudaStream_t stream) {
    const dim3 grid(tc.grid_x, tc.grid_y), block(32 * NW);
    const size_t smem = smem_bytes<CH>();
#define TBJ_K(F, FU)                                                           \
    launch_pdl(k_ba<CH, RW, NW, F, FU>, grid, block, smem, stream, *map_src,   \
               *map_b, out, g.n, g.ld, g.r, g.d, g.y, tc.depth, tc.tile_x,     \
               tc.tile_y, tc.sx, tc.sy, err, ctl.stop, ctl.lp)
    if (g.fast) return ctl.fused ? TBJ_K(true, true) : TBJ_K(true, false);
    return ctl.fused ? TBJ_K(false, true) : TBJ_K(false, false);
#undef TBJ_K
}

template <int CH, int RW, int NW>
cudaError_t prepare_ch() {
    const void *kernels[4] = {(const void *)k_ba<CH, RW, NW, true, false>,
                              (const void *)k_ba<CH, RW, NW, false, false>,
                              (const void *)k_ba<CH, RW, NW, true, true>,
                              (const void *)k_ba<CH, RW, NW, false, true>};
    for (const void *k : kernels) {
        cudaError_t e = cudaFuncSetAttribute(
            k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_bytes<CH>());
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace

// Choose the streaming kernel's super-tile for BA tiles of tx x ty; returns
// false when the shape needs the generic kernel (TY > 64 or TX > 252).
bool ba_stream_configure(int n, TileConf *tc) {
    const int tx = tc->tile_x, ty = tc->tile_y;
    if (ty > kRowsMax || tx > 252 || tx % 4 != 0) return false;
    // Widest super-tile per box width; one chunk per lane if that wastes
    // at most a little more of the warp's columns than two would.
    const int sx1 = (126 / tx) * tx, sx2 = (254 / tx) * tx;
    const double use1 = sx1 / 128.0, use2 = sx2 / 256.0;
    const int ch = (sx1 >= tx && use1 + 0.05 >= use2) ? 1 : 2;
    tc->ch = ch;
    tc->sx = ch == 1 ? sx1 : sx2;
    tc->sy = (kRowsMax / ty) * ty;
    tc->box_x = 128 * ch;
    tc->box_y = tc->sy + 2;
    tc->grid_x = (n - 2 + tc->sx - 1) / tc->sx;
    tc->grid_y = (n - 2 + tc->sy - 1) / tc->sy;
    tc->threads = ch == 1 ? 1024 : 512;
    tc->smem = ch == 1 ? smem_bytes<1>() : smem_bytes<2>();
    tc->stream = 1;
    return true;
}

cudaError_t prepare_sweep_ba_stream(const TileConf &tc) {
    return tc.ch == 1 ? prepare_ch<1, 2, 32>() : prepare_ch<2, 4, 16>();
}

cudaError_t launch_sweep_ba_stream(const GridDesc &g, const TileConf &tc,
                                   const CUtensorMap *map_src,
                                   const CUtensorMap *map_b, float *out,
                                   unsigned *err, const LaunchCtl &ctl,
                                   cudaStream_t stream) {
    if (tc.ch == 1)
        return launch_ch<1, 2, 32>(g, tc, map_src, map_b, out, err, ctl, stream);
    return launch_ch<2, 4, 16>(g, tc, map_src, map_b, out, err, ctl, stream);
}

}  // namespace tbj
