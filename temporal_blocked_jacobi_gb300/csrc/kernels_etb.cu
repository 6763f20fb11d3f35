// Exact temporal blocking ("Synchronous vs block-async Jacobi on one
// RTX 5050", section 02, after Meng and Skadron's ghost zones): one launch
// performs D synchronous sweeps of a tile on chip and is bit-identical to D
// launches of the synchronous sweep.
//
// Layout of a block. The box (tile plus halo) is BX = 128*CH columns by
// BY = NW*RW rows; one warp spans a whole box row (each lane holds CH float4
// chunks, chunk c of lane l covering columns 128c + 4l .. 128c + 4l + 3),
// and warp w owns the band of rows [w*RW, (w+1)*RW). The left/right halo is
// HX = round_up(D, 4) columns (the TMA box must start on a 16-byte
// boundary), the top/bottom halo D rows, so the tile is
// TX = BX - 2*HX by TY = BY - 2*D cells.
//
// Thread 0 loads the box of u and the box of b with two TMA copies onto one
// mbarrier (bounded wait). Each warp keeps its band's b in registers; the
// field ping-pongs between two shared buffers. Sweep s updates rows
// [s+1, BY-1-s) over the full box width: each lane streams down its band
// holding rows i-1, i, i+1 in registers, with west/east neighbours from the
// adjacent lanes by shuffle. Values near the box edge become inexact, but
// inexactness moves inward one cell per sweep, so after D sweeps the tile
// (HX >= D columns and D rows in from the edge) holds exactly the result of
// D synchronous sweeps. The last sweep writes the tile to global memory.
//
// Dirichlet ring cells are never updated: in tiles whose box reaches past
// the interior, a cell keeps its value unless it is an interior grid cell.
#include "jacobi_kernels.cuh"

namespace tbj {
namespace {

constexpr unsigned FULL = 0xffffffffu;

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

template <int D, int CH, int RW, int NW>
struct EtbShape {
    static constexpr int BX = 128 * CH;
    static constexpr int BY = NW * RW;
    static constexpr int HX = (D + 3) / 4 * 4;
    static constexpr int TX = BX - 2 * HX;
    static constexpr int TY = BY - 2 * D;
    static constexpr size_t BUF = (size_t)BX * BY * sizeof(float);
    static constexpr size_t SMEM = 256 + 2 * BUF;
    static_assert(TX >= 4 && TY >= 1, "tile too small for this depth");
    static_assert(BX <= 256 && BY <= 256, "TMA box dimension limit");
};

__device__ __forceinline__ float4 lds4(const float *p) {
    return *reinterpret_cast<const float4 *>(p);
}
__device__ __forceinline__ void sts4(float *p, float4 v) {
    *reinterpret_cast<float4 *>(p) = v;
}

template <bool FAST>
__device__ __forceinline__ float4 update4(float4 n4, float4 c4, float4 s4,
                                          float4 b4, float w, float e, float r,
                                          float d, float y) {
    float4 o;
    o.x = jacobi_update<FAST>(w, c4.y, n4.x, s4.x, b4.x, r, d, y);
    o.y = jacobi_update<FAST>(c4.x, c4.z, n4.y, s4.y, b4.y, r, d, y);
    o.z = jacobi_update<FAST>(c4.y, c4.w, n4.z, s4.z, b4.z, r, d, y);
    o.w = jacobi_update<FAST>(c4.z, e, n4.w, s4.w, b4.w, r, d, y);
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

template <int D, int CH, int RW, int NW, bool FAST, bool EDGE, bool FUSED>
__device__ __forceinline__ void etb_sweeps(const float *sA, float *sB,
                                           const float4 (&breg)[RW][CH],
                                           float *__restrict__ out, int n,
                                           long long ld, float r, float d,
                                           float y, int bxo, int byo,
                                           unsigned &rm, unsigned &bm) {
    using S = EtbShape<D, CH, RW, NW>;
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int band = warp * RW;

    // Columns of this lane's chunks that are interior grid cells (edge tiles).
    unsigned colmask[CH];
    bool in_tile[CH];
#pragma unroll
    for (int c = 0; c < CH; ++c) {
        const int bx = 128 * c + 4 * lane;
        unsigned m = 0;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int gx = bxo + bx + k;
            m |= (gx >= 1 && gx <= n - 2) ? (1u << k) : 0u;
        }
        colmask[c] = EDGE ? m : 0xfu;
        in_tile[c] = bx >= S::HX && bx < S::HX + S::TX;
    }

#pragma unroll 1
    for (int s = 0; s < D; ++s) {
        const float *src = (s & 1) ? sB : sA;
        float *dst = (s & 1) ? const_cast<float *>(sA) : sB;
        const bool last = (s == D - 1);
        const int rlo = max(s + 1, band);
        const int rhi = min(S::BY - 1 - s, band + RW);
        if (rlo < rhi) {
            float4 nr[CH], cr[CH];
#pragma unroll
            for (int c = 0; c < CH; ++c) {
                nr[c] = lds4(src + (rlo - 1) * S::BX + 128 * c + 4 * lane);
                cr[c] = lds4(src + rlo * S::BX + 128 * c + 4 * lane);
            }
#pragma unroll
            for (int j = 0; j < RW; ++j) {
                const int row = band + j;
                if (row < rlo || row >= rhi) continue;  // uniform per warp
                float4 sr[CH];
#pragma unroll
                for (int c = 0; c < CH; ++c)
                    sr[c] = lds4(src + (row + 1) * S::BX + 128 * c + 4 * lane);
                float wv[CH], ev[CH];
#pragma unroll
                for (int c = 0; c < CH; ++c) {
                    wv[c] = __shfl_sync(FULL, cr[c].w, (lane + 31) & 31);
                    ev[c] = __shfl_sync(FULL, cr[c].x, (lane + 1) & 31);
                }
                const int gy = byo + row;
                const bool row_ok = !EDGE || (gy >= 1 && gy <= n - 2);
#pragma unroll
                for (int c = 0; c < CH; ++c) {
                    const float w = (c > 0 && lane == 0) ? wv[c - 1] : wv[c];
                    const float e = (c < CH - 1 && lane == 31) ? ev[c + 1] : ev[c];
                    float4 nv = update4<FAST>(nr[c], cr[c], sr[c], breg[j][c], w,
                                              e, r, d, y);
                    if (FUSED && s == 0 && in_tile[c] && row >= D &&
                        row < D + S::TY && row_ok) {
                        // Residual of the launch's input at the tile's cells.
                        const float4 c4 = cr[c], n4 = nr[c], s4 = sr[c];
                        const float4 b4 = breg[j][c];
                        if (EDGE) {
                            const int gx = bxo + 128 * c + 4 * lane;
                            if (colmask[c] & 1u) cell_residual(nv.x, c4.x, w, c4.y, n4.x, s4.x, b4.x, gy, gx + 0, n, r, d, rm, bm);
                            if (colmask[c] & 2u) cell_residual(nv.y, c4.y, c4.x, c4.z, n4.y, s4.y, b4.y, gy, gx + 1, n, r, d, rm, bm);
                            if (colmask[c] & 4u) cell_residual(nv.z, c4.z, c4.y, c4.w, n4.z, s4.z, b4.z, gy, gx + 2, n, r, d, rm, bm);
                            if (colmask[c] & 8u) cell_residual(nv.w, c4.w, c4.z, e, n4.w, s4.w, b4.w, gy, gx + 3, n, r, d, rm, bm);
                        } else {
                            // No ring cell is next to these cells: b_I = b.
                            rm = max(rm, abs_bits(__fmul_rn(d, fabsf(__fsub_rn(nv.x, c4.x)))));
                            rm = max(rm, abs_bits(__fmul_rn(d, fabsf(__fsub_rn(nv.y, c4.y)))));
                            rm = max(rm, abs_bits(__fmul_rn(d, fabsf(__fsub_rn(nv.z, c4.z)))));
                            rm = max(rm, abs_bits(__fmul_rn(d, fabsf(__fsub_rn(nv.w, c4.w)))));
                            bm = max(bm, abs_bits(b4.x));
                            bm = max(bm, abs_bits(b4.y));
                            bm = max(bm, abs_bits(b4.z));
                            bm = max(bm, abs_bits(b4.w));
                        }
                    }
                    if (EDGE) nv = hold4(nv, cr[c], row_ok, colmask[c]);
                    if (!last) {
                        sts4(dst + row * S::BX + 128 * c + 4 * lane, nv);
                    } else if (in_tile[c] && row_ok) {
                        float *g = out + (long long)gy * ld + (bxo + 128 * c + 4 * lane);
                        if (colmask[c] == 0xfu) {
                            sts4(g, nv);
                        } else {
                            if (colmask[c] & 1u) g[0] = nv.x;
                            if (colmask[c] & 2u) g[1] = nv.y;
                            if (colmask[c] & 4u) g[2] = nv.z;
                            if (colmask[c] & 8u) g[3] = nv.w;
                        }
                    }
                    nr[c] = cr[c];
                    cr[c] = sr[c];
                }
            }
        }
        if (!last) __syncthreads();
    }
}

template <int D, int CH, int RW, int NW, bool FAST, bool FUSED>
__global__ void __launch_bounds__(32 * NW)
k_etb(const __grid_constant__ CUtensorMap map_src,
      const __grid_constant__ CUtensorMap map_b, float *__restrict__ out,
      int n, long long ld, float r, float d, float y, unsigned *err,
      const int *stop, LoopParams lp) {
    using S = EtbShape<D, CH, RW, NW>;
    if (stop && *stop) return;  // same value for every thread of the launch
    __shared__ unsigned fin_scratch[65];
    const int gx0 = blockIdx.x * S::TX;  // tile's first cell (grid coords)
    const int gy0 = blockIdx.y * S::TY;
    if (gx0 > n - 2 || gy0 > n - 2) {  // tile holds no interior cell
        if (FUSED) fused_block_finish(0u, 0u, lp, fin_scratch);
        return;
    }
    const int bxo = gx0 - S::HX;  // grid coords of box cell (0,0)
    const int byo = gy0 - D;

    extern __shared__ unsigned char smem_raw[];
    unsigned char *base = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
    uint64_t *bar = reinterpret_cast<uint64_t *>(base);
    float *sA = reinterpret_cast<float *>(base + 128);
    float *sB = reinterpret_cast<float *>(base + 128 + S::BUF);

    const int tid = threadIdx.x;
    if (tid == 0) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(bar))
                     : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile(
            "mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(
                smem_addr(bar)),
            "r"((unsigned)(2 * S::BUF))
            : "memory");
        tma_load_2d(sA, &map_src, bar, bxo, byo);
        tma_load_2d(sB, &map_b, bar, bxo, byo);  // b staged in the B buffer
    }
    __syncthreads();
    const bool ok = mbar_wait_bounded(bar);
    if (__syncthreads_or(!ok)) {
        if (tid == 0) atomicOr(err, (unsigned)ERR_TMA_TIMEOUT);
        mbar_wait_bounded(bar);
        if (FUSED) fused_block_finish(0u, 0u, lp, fin_scratch);
        return;
    }
    // b of this warp's band into registers; then the B buffer is free.
    const int lane = tid & 31;
    const int band = (tid >> 5) * RW;
    float4 breg[RW][CH];
#pragma unroll
    for (int j = 0; j < RW; ++j)
#pragma unroll
        for (int c = 0; c < CH; ++c)
            breg[j][c] = lds4(sB + (band + j) * S::BX + 128 * c + 4 * lane);
    __syncthreads();

    unsigned rm = 0u, bm = 0u;
    const bool edge = bxo < 1 || byo < 1 || bxo + S::BX > n - 1 ||
                      byo + S::BY > n - 1;
    if (edge)
        etb_sweeps<D, CH, RW, NW, FAST, true, FUSED>(sA, sB, breg, out, n, ld, r,
                                                     d, y, bxo, byo, rm, bm);
    else
        etb_sweeps<D, CH, RW, NW, FAST, false, FUSED>(sA, sB, breg, out, n, ld,
                                                      r, d, y, bxo, byo, rm, bm);
    if (FUSED) fused_block_finish(rm, bm, lp, fin_scratch);
}

// Shapes per depth: {CH, RW, NW}. Index 0 is the default.
struct EtbVariant {
    int depth, ch, rw, nw;
};
constexpr EtbVariant kVariants[] = {
    {2, 1, 4, 16}, {2, 2, 4, 16},
    {4, 1, 4, 16}, {4, 2, 4, 16},
    {8, 1, 8, 16}, {8, 2, 4, 16},
    {16, 2, 4, 24}, {16, 1, 6, 32},
};

template <int D, int CH, int RW, int NW>
cudaError_t launch_variant(const GridDesc &g, const CUtensorMap *map_src,
                           const CUtensorMap *map_b, float *out,
                           unsigned *err, const LaunchCtl &ctl,
                           cudaStream_t stream) {
    using S = EtbShape<D, CH, RW, NW>;
    const dim3 grid((g.n + S::TX - 1) / S::TX, (g.n + S::TY - 1) / S::TY);
#define TBJ_K(F, FU)                                                          \
    k_etb<D, CH, RW, NW, F, FU><<<grid, 32 * NW, S::SMEM, stream>>>(          \
        *map_src, *map_b, out, g.n, g.ld, g.r, g.d, g.y, err, ctl.stop, ctl.lp)
    if (g.fast) {
        if (ctl.fused) TBJ_K(true, true);
        else TBJ_K(true, false);
    } else {
        if (ctl.fused) TBJ_K(false, true);
        else TBJ_K(false, false);
    }
#undef TBJ_K
    return cudaGetLastError();
}

template <int D, int CH, int RW, int NW>
cudaError_t prepare_variant() {
    using S = EtbShape<D, CH, RW, NW>;
    const void *kernels[4] = {
        (const void *)k_etb<D, CH, RW, NW, true, false>,
        (const void *)k_etb<D, CH, RW, NW, false, false>,
        (const void *)k_etb<D, CH, RW, NW, true, true>,
        (const void *)k_etb<D, CH, RW, NW, false, true>};
    for (const void *k : kernels) {
        cudaError_t e = cudaFuncSetAttribute(
            k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)S::SMEM);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

// Dispatch on a variant index (into kVariants).
#define TBJ_ETB_VARIANTS(X)          \
    X(0, 2, 1, 4, 16)                \
    X(1, 2, 2, 4, 16)                \
    X(2, 4, 1, 4, 16)                \
    X(3, 4, 2, 4, 16)                \
    X(4, 8, 1, 8, 16)                \
    X(5, 8, 2, 4, 16)                \
    X(6, 16, 2, 4, 24)               \
    X(7, 16, 1, 6, 32)

}  // namespace

int etb_configure(int n, int depth, int tile_x, int tile_y, TileConf *tc) {
    (void)n;
    int pick = -1;
    for (int v = 0; v < (int)(sizeof(kVariants) / sizeof(kVariants[0])); ++v) {
        const EtbVariant &k = kVariants[v];
        if (k.depth != depth) continue;
        const int hx = (depth + 3) / 4 * 4;
        const int tx = 128 * k.ch - 2 * hx, ty = k.nw * k.rw - 2 * depth;
        if ((tile_x == 0 && tile_y == 0 && pick < 0) ||
            (tile_x == tx && tile_y == ty)) {
            pick = v;
            if (tile_x != 0 || tile_y != 0) break;
        }
    }
    if (depth != 2 && depth != 4 && depth != 8 && depth != 16) return -1;
    if (pick < 0) return -5;
    const EtbVariant &k = kVariants[pick];
    tc->depth = depth;
    tc->halo_x = (depth + 3) / 4 * 4;
    tc->halo_y = depth;
    tc->box_x = 128 * k.ch;
    tc->box_y = k.nw * k.rw;
    tc->tile_x = tc->box_x - 2 * tc->halo_x;
    tc->tile_y = tc->box_y - 2 * depth;
    tc->origin = 0;
    tc->threads = 32 * k.nw;
    tc->smem = 256 + 2 * (size_t)tc->box_x * tc->box_y * sizeof(float);
    tc->variant = pick;
    return 0;
}

cudaError_t prepare_sweep_etb(const TileConf &tc) {
    switch (tc.variant) {
#define TBJ_PREP(I, D, CH, RW, NW) \
    case I:                        \
        return prepare_variant<D, CH, RW, NW>();
        TBJ_ETB_VARIANTS(TBJ_PREP)
#undef TBJ_PREP
        default:
            return cudaErrorInvalidValue;
    }
}

cudaError_t launch_sweep_etb(const GridDesc &g, const TileConf &tc,
                             const CUtensorMap *map_src,
                             const CUtensorMap *map_b, float *out,
                             ResidualOut *status, const LaunchCtl &ctl,
                             cudaStream_t stream) {
    unsigned *err = ctl.lp.state ? &ctl.lp.state->err : &status->err;
    switch (tc.variant) {
#define TBJ_LAUNCH(I, D, CH, RW, NW) \
    case I:                          \
        return launch_variant<D, CH, RW, NW>(g, map_src, map_b, out, err, ctl, stream);
        TBJ_ETB_VARIANTS(TBJ_LAUNCH)
#undef TBJ_LAUNCH
        default:
            return cudaErrorInvalidValue;
    }
}

}  // namespace tbj
