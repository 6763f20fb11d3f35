// Exact-temporal-blocking kernels and their launch templates, shared by the
// translation units kernels_etb.cu (shape selection and dispatch) and
// kernels_etb_part0..3.cu (each instantiates a quarter of the compiled
// shapes, so that they compile in parallel). Everything here has internal
// linkage; a kernel is instantiated only in the part that owns its shape.
//
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
// Two kernels share this layout. Both are persistent: a block walks tiles
// k, k + gridDim.x, ... and thread 0 loads a tile's box of u and of b with
// two TMA copies onto an mbarrier (bounded wait).
//
// k_etb (box in shared memory): with NB = 2 buffer sets the next tile is
// loaded while the current one is swept, with NB = 1 right after it. Each
// warp keeps its band's b in registers; the field ping-pongs between two
// shared buffers,
// each with a spare row above and below the box so that every row of every
// band can be updated without a bounds test. In sweep s each warp updates
// its whole band over the full box width -- bands lying entirely outside the
// rows still needed, [s+1, BY-1-s), are skipped -- streaming down the band
// with rows i-1, i, i+1 in registers and west/east neighbours from the
// adjacent lanes by shuffle. Cells near the box edge (and the spare rows)
// become inexact, but inexactness moves inward one cell per sweep, so after
// D sweeps the tile (HX >= D columns and D rows in from the edge) holds
// exactly the result of D synchronous sweeps. The last sweep writes the tile
// to global memory.
//
// k_etbr (bands in registers) keeps the same band decomposition, skipping and
// inward-moving exactness, but each warp holds its RW rows in registers for
// all D sweeps and trades only its top and bottom rows through shared memory
// (see the comment above k_etbr).
//
// With the verified fixed-divisor division the update of a lane's four
// cells uses packed float32 pairs for everything but the west+east sums.
//
// Dirichlet ring cells are never updated: in tiles whose box reaches past
// the interior, a cell keeps its value unless it is an interior grid cell.
#pragma once

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

__device__ __forceinline__ void mbar_init(uint64_t *bar) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(bar))
                 : "memory");
}

// Wait for the given phase parity of a barrier, giving up after ~1 s.
__device__ __forceinline__ bool mbar_wait_parity(uint64_t *bar, unsigned par) {
    if (mbar_try_wait(bar, par)) return true;
    const uint64_t t0 = global_ns();
    while (!mbar_try_wait(bar, par)) {
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

template <int D, int CH, int RW, int NW, int NB = 2>
struct EtbShape {
    static constexpr int BX = 128 * CH;
    static constexpr int BY = NW * RW;
    static constexpr int HX = (D + 3) / 4 * 4;
    static constexpr int TX = BX - 2 * HX;
    static constexpr int TY = BY - 2 * D;
    // One buffer: the box plus a spare row above and below it. NB sets of
    // two buffers (NB = 2: the current tile and the prefetched next one).
    static constexpr size_t BUF = (size_t)BX * (BY + 2) * sizeof(float);
    static constexpr size_t BOX_BYTES = (size_t)BX * BY * sizeof(float);
    static constexpr size_t SMEM = 256 + 2 * NB * BUF;
    static_assert(TX >= 4 && TY >= 1, "tile too small for this depth");
    static_assert(BX <= 256 && BY <= 256, "TMA box dimension limit");
};


// One sweep of one tile. RESID: also reduce |J(u) - u| (first sweep of a
// fused launch); LAST: write the tile to global memory instead of to dst.
template <int D, int CH, int RW, int NW, bool FAST, bool EDGE, bool RESID,
          bool LAST>
__device__ __forceinline__ void etb_sweep(const float *src, float *dst, int s,
                                          const float4 (&breg)[RW][CH],
                                          float *__restrict__ out, int n,
                                          long long ld, float r, float d,
                                          float y, int bxo, int byo,
                                          const unsigned (&colmask)[CH],
                                          const bool (&in_tile)[CH],
                                          unsigned &rm) {
    using S = EtbShape<D, CH, RW, NW>;
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int band = warp * RW;
    const int col = 4 * lane;
    const int left = (lane + 31) & 31, right = (lane + 1) & 31;
    if (!(band + RW > s + 1 && band < S::BY - 1 - s)) return;
    const float *sp = src + band * S::BX + col;
    float *dp = dst + band * S::BX + col;
    float4 nr[CH], cr[CH];
#pragma unroll
    for (int c = 0; c < CH; ++c) {
        nr[c] = lds4(sp - S::BX + 128 * c);
        cr[c] = lds4(sp + 128 * c);
    }
#pragma unroll
    for (int j = 0; j < RW; ++j) {
        float4 sr[CH];
#pragma unroll
        for (int c = 0; c < CH; ++c) sr[c] = lds4(sp + (j + 1) * S::BX + 128 * c);
        float wv[CH], ev[CH];
#pragma unroll
        for (int c = 0; c < CH; ++c) {
            wv[c] = __shfl_sync(FULL, cr[c].w, left);
            ev[c] = __shfl_sync(FULL, cr[c].x, right);
        }
        const int row = band + j;
        const int gy = byo + row;
        const bool row_ok = !EDGE || (gy >= 1 && gy <= n - 2);
#pragma unroll
        for (int c = 0; c < CH; ++c) {
            const float w = (c > 0 && lane == 0) ? wv[c - 1] : wv[c];
            const float e = (c < CH - 1 && lane == 31) ? ev[c + 1] : ev[c];
            float4 nv = update4_we<FAST, false>(nr[c], cr[c], sr[c], breg[j][c], w, e, r,
                                      d, y);
            if (RESID) {
                const bool tile_row = row >= D && row < D + S::TY;
                if (in_tile[c] && tile_row && row_ok) {
                    const float4 c4 = cr[c];
                    const unsigned m = colmask[c];
                    if (m & 1u) rm = max(rm, change_bits(nv.x, c4.x));
                    if (m & 2u) rm = max(rm, change_bits(nv.y, c4.y));
                    if (m & 4u) rm = max(rm, change_bits(nv.z, c4.z));
                    if (m & 8u) rm = max(rm, change_bits(nv.w, c4.w));
                }
            }
            if (EDGE) nv = hold4(nv, cr[c], row_ok, colmask[c]);
            if (!LAST) {
                sts4(dp + j * S::BX + 128 * c, nv);
            } else {
                const bool tile_row = row >= D && row < D + S::TY;
                if (in_tile[c] && tile_row && row_ok) {
                    float *g = out + (long long)gy * ld + (bxo + 128 * c + col);
                    if (colmask[c] == 0xfu) {
                        gst4(g, nv);
                    } else {
                        if (colmask[c] & 1u) gst1(g + 0, nv.x);
                        if (colmask[c] & 2u) gst1(g + 1, nv.y);
                        if (colmask[c] & 4u) gst1(g + 2, nv.z);
                        if (colmask[c] & 8u) gst1(g + 3, nv.w);
                    }
                }
            }
            nr[c] = cr[c];
            cr[c] = sr[c];
        }
    }
}

// D sweeps of one tile. sA, sB point at box row 0 of the two buffers (rows
// -1 and BY exist); b of this warp's band is in breg.
template <int D, int CH, int RW, int NW, bool FAST, bool EDGE, bool FUSED>
__device__ __forceinline__ void etb_sweeps(float *sA, float *sB,
                                           const float4 (&breg)[RW][CH],
                                           float *__restrict__ out, int n,
                                           long long ld, float r, float d,
                                           float y, int bxo, int byo,
                                           unsigned &rm) {
    using S = EtbShape<D, CH, RW, NW>;
    const int col = 4 * (threadIdx.x & 31);
    unsigned colmask[CH];
    bool in_tile[CH];
#pragma unroll
    for (int c = 0; c < CH; ++c) {
        const int bx = 128 * c + col;
        unsigned m = 0;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int gx = bxo + bx + k;
            m |= (gx >= 1 && gx <= n - 2) ? (1u << k) : 0u;
        }
        colmask[c] = EDGE ? m : 0xfu;
        in_tile[c] = bx >= S::HX && bx < S::HX + S::TX;
    }
    // Sweep 0 (with the residual in a fused launch), sweeps 1 .. D-2, and
    // the last sweep, which writes the tile out.
    etb_sweep<D, CH, RW, NW, FAST, EDGE, FUSED, false>(
        sA, sB, 0, breg, out, n, ld, r, d, y, bxo, byo, colmask, in_tile, rm);
    __syncthreads();
#pragma unroll 1
    for (int s = 1; s < D - 1; ++s) {
        const float *src = (s & 1) ? sB : sA;
        float *dst = (s & 1) ? sA : sB;
        etb_sweep<D, CH, RW, NW, FAST, EDGE, false, false>(
            src, dst, s, breg, out, n, ld, r, d, y, bxo, byo, colmask, in_tile,
            rm);
        __syncthreads();
    }
    // D is even: the last sweep reads sB.
    etb_sweep<D, CH, RW, NW, FAST, EDGE, false, true>(
        sB, sA, D - 1, breg, out, n, ld, r, d, y, bxo, byo, colmask, in_tile,
        rm);
}

// Issue the TMA loads of one tile's box of u (into a) and of b (into bb).
template <class S>
__device__ __forceinline__ void load_tile(const CUtensorMap *map_src,
                                          const CUtensorMap *map_b,
                                          uint64_t *bar, float *a, float *bb,
                                          int tile, int tiles_x, int depth) {
    const int gx0 = (tile % tiles_x) * S::TX, gy0 = (tile / tiles_x) * S::TY;
    asm volatile(
        "mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(
            smem_addr(bar)),
        "r"((unsigned)(2 * S::BOX_BYTES))
        : "memory");
    // (checked build: a load that fails its check is not issued, and the
    // wait for it runs into its time limit)
    if (tma_ok(a, (unsigned)S::BOX_BYTES, gx0 - S::HX))
        tma_load_2d(a, map_src, bar, gx0 - S::HX, gy0 - depth);
    if (tma_ok(bb, (unsigned)S::BOX_BYTES, gx0 - S::HX))
        tma_load_2d(bb, map_b, bar, gx0 - S::HX, gy0 - depth);
}

// Persistent kernel: block k handles tiles k, k + gridDim.x, ... (row-major
// over a tiles_x-wide tile grid). With NB = 2 the TMA engine fills the other
// buffer set with the next tile while the block sweeps the current one; with
// NB = 1 the next tile's load is issued as soon as the current tile is done.
template <int D, int CH, int RW, int NW, int NB, int MINB, bool FAST,
          bool FUSED>
__global__ void __launch_bounds__(32 * NW, MINB)
k_etb(const __grid_constant__ CUtensorMap map_src,
      const __grid_constant__ CUtensorMap map_b, float *__restrict__ out,
      int n, long long ld, float r, float d, float y, unsigned *err,
      const int *stop, LoopParams lp, int tiles_x, int tiles) {
    using S = EtbShape<D, CH, RW, NW, NB>;
    static_assert(S::SMEM <= 227 * 1024, "shared memory per block");
    __shared__ unsigned fin_scratch[33];
    allow_dependents();

    // Offsets from the __shared__ array itself, so that every access stays
    // in the shared address space: [2 barriers | A0 | B0 | A1 | B1] (NB = 2),
    // each buffer = spare row, BY box rows, spare row; rows are 512 or 1024
    // bytes, so every box row is 128-byte aligned.
    extern __shared__ __align__(128) unsigned char smem_raw[];
    bounds_begin(smem_raw, 0, out, nullptr, nullptr, nullptr, n, ld, err);
    const unsigned pad = (128u - (smem_addr(smem_raw) & 127u)) & 127u;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem_raw + pad);
    float *buf0 = reinterpret_cast<float *>(smem_raw + pad + 128);
    constexpr int bufn = S::BX * (S::BY + 2);

    const int tid = threadIdx.x;
    for (int k = tid; k < S::BX; k += 32 * NW)
        for (int q = 0; q < 2 * NB; ++q) {
            sts1(buf0 + q * bufn + k, 0.f);  // spare rows: finite values
            sts1(buf0 + q * bufn + (S::BY + 1) * S::BX + k, 0.f);
        }
    if (tid == 0) {
        mbar_init(&bars[0]);
        mbar_init(&bars[1]);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    // Everything below reads what the previous kernel wrote.
    grid_dependency_wait();
    if (stop && *stop) return;  // same value for every thread of the launch
    if (tid == 0 && (int)blockIdx.x < tiles)
        load_tile<S>(&map_src, &map_b, &bars[0], buf0 + S::BX,
                     buf0 + bufn + S::BX, blockIdx.x, tiles_x, D);
    __syncthreads();

    const int lane = tid & 31;
    const int band = (tid >> 5) * RW;
    unsigned rm = 0u;
    bool failed = false;
    int fail_p = 0;
    unsigned fail_parity = 0u;
    int i = 0;
    for (int t = blockIdx.x; t < tiles; t += gridDim.x, ++i) {
        const int p = NB == 2 ? (i & 1) : 0;
        float *sA = buf0 + (2 * p) * bufn + S::BX;  // box row 0
        float *sB = buf0 + (2 * p + 1) * bufn + S::BX;
        const unsigned parity = NB == 2 ? (unsigned)(i >> 1) & 1u : (unsigned)i & 1u;
        const bool ok = mbar_wait_parity(&bars[p], parity);
        if (__syncthreads_or(!ok)) {
            failed = true;
            fail_p = p;
            fail_parity = parity;
            break;
        }
        float4 breg[RW][CH];
#pragma unroll
        for (int j = 0; j < RW; ++j)
#pragma unroll
            for (int c = 0; c < CH; ++c)
                breg[j][c] = lds4(sB + (band + j) * S::BX + 128 * c + 4 * lane);
        // Everyone is past the previous tile (which used the other set) and
        // holds this tile's b: prefetch the next tile into the other set.
        __syncthreads();
        if (NB == 2 && tid == 0 && t + (int)gridDim.x < tiles) {
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            load_tile<S>(&map_src, &map_b, &bars[p ^ 1],
                         buf0 + (2 * (p ^ 1)) * bufn + S::BX,
                         buf0 + (2 * (p ^ 1) + 1) * bufn + S::BX,
                         t + gridDim.x, tiles_x, D);
        }
        const int gx0 = (t % tiles_x) * S::TX, gy0 = (t / tiles_x) * S::TY;
        const int bxo = gx0 - S::HX, byo = gy0 - D;
        const bool edge = bxo < 1 || byo < 1 || bxo + S::BX > n - 1 ||
                          byo + S::BY > n - 1;
        if (edge)
            etb_sweeps<D, CH, RW, NW, FAST, true, FUSED>(sA, sB, breg, out, n, ld,
                                                         r, d, y, bxo, byo, rm);
        else
            etb_sweeps<D, CH, RW, NW, FAST, false, FUSED>(sA, sB, breg, out, n,
                                                          ld, r, d, y, bxo, byo, rm);
        if (NB == 1 && t + (int)gridDim.x < tiles) {
            __syncthreads();  // everyone is done with the single buffer set
            if (tid == 0) {
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                load_tile<S>(&map_src, &map_b, &bars[0], buf0 + S::BX,
                             buf0 + bufn + S::BX, t + gridDim.x, tiles_x, D);
            }
        }
    }
    if (failed) {
        if (tid == 0) atomicOr(err, (unsigned)ERR_TMA_TIMEOUT);
        // Only the load waited on can be in flight (the next one is issued
        // after it lands): give it one more bounded wait before shared memory
        // is released.
        mbar_wait_parity(&bars[fail_p], fail_parity);
    }
    if (FUSED) fused_block_finish(rm, lp, fin_scratch);
}

// ---------------------------------------------------------------------------
// Register-resident bands. The same exact temporal blocking, but a warp keeps
// the RW rows of its band in registers for all D sweeps of a tile instead of
// ping-ponging the whole box through shared memory. Shared memory holds the
// TMA staging boxes of u and b (read once per tile) and, per sweep parity,
// the top and bottom row of every band: after each sweep a warp publishes
// its two edge rows and, past the barrier, reads the row above and the row
// below its band from its neighbours' entries. Per band and sweep that is
// two shared loads and two shared stores instead of 2 + 2*RW, and the
// staging boxes are free for the next tile's TMA load from the first sweep
// on. Slots -1 and 2*NW of the exchange rows (above the first band, below
// the last) stay zero; the cells that read them lie outside the region that
// is still exact.
// ---------------------------------------------------------------------------
template <int D, int CH, int RW, int NW>
struct EtbrShape {
    static constexpr int BX = 128 * CH;
    static constexpr int BY = NW * RW;
    static constexpr int HX = (D + 3) / 4 * 4;
    static constexpr int TX = BX - 2 * HX;
    static constexpr int TY = BY - 2 * D;
    static constexpr size_t BOX_BYTES = (size_t)BX * BY * sizeof(float);
    static constexpr int XROWS = 2 * NW + 2;  // exchange slots -1 .. 2*NW
    static constexpr size_t SMEM =
        256 + 2 * BOX_BYTES + 2 * (size_t)XROWS * BX * sizeof(float);
    static_assert(TX >= 4 && TY >= 1, "tile too small for this depth");
    static_assert(BX <= 256 && BY <= 256, "TMA box dimension limit");
    static_assert(SMEM <= 227 * 1024, "shared memory per block");
};

// Update of row j of a band held in registers from its input state u[j]
// and the input states of the rows above (north) and below (south); j must
// be a constant after unrolling. RESID and LAST as in etb_sweep.
template <int D, int CH, int RW, int NW, bool FAST, bool EDGE, bool RESID,
          bool LAST>
__device__ __forceinline__ void etbr_row(int j, float4 (&u)[RW][CH],
                                         const float4 (&b)[RW][CH],
                                         const float4 (&north)[CH],
                                         const float4 (&south)[CH],
                                         float *__restrict__ out, int n,
                                         long long ld, float r, float d,
                                         float y, int bxo, int byo,
                                         const unsigned (&colmask)[CH],
                                         const bool (&in_tile)[CH],
                                         float &rmf) {
    using S = EtbrShape<D, CH, RW, NW>;
    const int lane = threadIdx.x & 31;
    const int band = (threadIdx.x >> 5) * RW;
    const int col = 4 * lane;
    const int left = (lane + 31) & 31, right = (lane + 1) & 31;
    float wv[CH], ev[CH];
#pragma unroll
    for (int c = 0; c < CH; ++c) {
        wv[c] = __shfl_sync(FULL, u[j][c].w, left);
        ev[c] = __shfl_sync(FULL, u[j][c].x, right);
    }
    const int row = band + j;
    const int gy = byo + row;
    const bool row_ok = !EDGE || (gy >= 1 && gy <= n - 2);
#pragma unroll
    for (int c = 0; c < CH; ++c) {
        const float w = (c > 0 && lane == 0) ? wv[c - 1] : wv[c];
        const float e = (c < CH - 1 && lane == 31) ? ev[c + 1] : ev[c];
        const float4 cur = u[j][c];
        float4 nv = update4_we<FAST, false>(north[c], cur, south[c], b[j][c], w, e, r,
                                     d, y);
        if (RESID) {
            const bool tile_row = row >= D && row < D + S::TY;
            if (in_tile[c] && tile_row && row_ok) {
                const unsigned m = colmask[c];
                const float2 d01 = __fadd2_rn(make_float2(nv.x, nv.y),
                                              make_float2(-cur.x, -cur.y));
                const float2 d23 = __fadd2_rn(make_float2(nv.z, nv.w),
                                              make_float2(-cur.z, -cur.w));
                if (m & 1u) rmf = max_nan_abs(rmf, d01.x);
                if (m & 2u) rmf = max_nan_abs(rmf, d01.y);
                if (m & 4u) rmf = max_nan_abs(rmf, d23.x);
                if (m & 8u) rmf = max_nan_abs(rmf, d23.y);
            }
        }
        if (EDGE) nv = hold4(nv, cur, row_ok, colmask[c]);
        if (LAST) {
            const bool tile_row = row >= D && row < D + S::TY;
            if (in_tile[c] && tile_row && row_ok) {
                float *g = out + (long long)gy * ld + (bxo + 128 * c + col);
                if (colmask[c] == 0xfu) {
                    gst4(g, nv);
                } else {
                    if (colmask[c] & 1u) gst1(g + 0, nv.x);
                    if (colmask[c] & 2u) gst1(g + 1, nv.y);
                    if (colmask[c] & 4u) gst1(g + 2, nv.z);
                    if (colmask[c] & 8u) gst1(g + 3, nv.w);
                }
            }
        }
        u[j][c] = nv;
    }
}

// One sweep of a band held in registers, top to bottom. hn / hs: the row
// above / below the band (input state of this sweep).
template <int D, int CH, int RW, int NW, bool FAST, bool EDGE, bool RESID,
          bool LAST>
__device__ __forceinline__ void etbr_band(float4 (&u)[RW][CH],
                                          const float4 (&b)[RW][CH],
                                          const float4 (&hn)[CH],
                                          const float4 (&hs)[CH],
                                          float *__restrict__ out, int n,
                                          long long ld, float r, float d,
                                          float y, int bxo, int byo,
                                          const unsigned (&colmask)[CH],
                                          const bool (&in_tile)[CH],
                                          float &rmf) {
    float4 prev[CH], cur[CH];
#pragma unroll
    for (int c = 0; c < CH; ++c) prev[c] = hn[c];
#pragma unroll
    for (int j = 0; j < RW; ++j) {
#pragma unroll
        for (int c = 0; c < CH; ++c) cur[c] = u[j][c];
        if (j + 1 < RW)
            etbr_row<D, CH, RW, NW, FAST, EDGE, RESID, LAST>(
                j, u, b, prev, u[j + 1 < RW ? j + 1 : j], out, n, ld, r, d, y,
                bxo, byo, colmask, in_tile, rmf);
        else
            etbr_row<D, CH, RW, NW, FAST, EDGE, RESID, LAST>(
                j, u, b, prev, hs, out, n, ld, r, d, y, bxo, byo, colmask,
                in_tile, rmf);
#pragma unroll
        for (int c = 0; c < CH; ++c) prev[c] = cur[c];
    }
}

// D sweeps of one tile with register-resident bands. xb: the exchange rows
// (two parities of XROWS rows of BX floats; slot k of parity q at row
// q * XROWS + k + 1). Consecutive exchanges use alternate parities, counted
// in xpar across tiles as well: a warp may start a tile's first exchange
// while a slower one still reads the previous tile's last, and the two must
// not share a parity (with the same parity at every tile's start, an odd
// number of exchanges per tile would make them collide). On entry u, b, hn,
// hs hold the tile's input, possibly still in flight from the staging
// boxes: thread 0 runs after_first_barrier() once the first sweep's exchange
// barrier has been passed, when every warp has consumed what it read from
// the staging boxes.
template <int D, int CH, int RW, int NW, bool FAST, bool EDGE, bool FUSED,
          class F>
__device__ __forceinline__ void etbr_sweeps(float4 (&u)[RW][CH],
                                            const float4 (&b)[RW][CH],
                                            float4 (&hn)[CH], float4 (&hs)[CH],
                                            float *xb, float *__restrict__ out,
                                            int n, long long ld, float r,
                                            float d, float y, int bxo, int byo,
                                            unsigned &rm, int &xpar,
                                            F after_first_barrier) {
    using S = EtbrShape<D, CH, RW, NW>;
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int band = warp * RW;
    const int col = 4 * lane;
    unsigned colmask[CH];
    bool in_tile[CH];
#pragma unroll
    for (int c = 0; c < CH; ++c) {
        const int bx = 128 * c + col;
        unsigned m = 0;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int gx = bxo + bx + k;
            m |= (gx >= 1 && gx <= n - 2) ? (1u << k) : 0u;
        }
        colmask[c] = EDGE ? m : 0xfu;
        in_tile[c] = bx >= S::HX && bx < S::HX + S::TX;
    }
    float rmf = __uint_as_float(rm);
    // This band's own slots (2*warp: top row, 2*warp + 1: bottom row) and
    // those of the rows next to it, at parity 0; parity 1 is XROWS rows on.
    float *own = xb + (2 * warp + 1) * S::BX + col;
    const float *above = xb + (2 * warp) * S::BX + col;      // slot 2w - 1
    const float *below = xb + (2 * warp + 3) * S::BX + col;  // slot 2w + 2
    constexpr int PAR = S::XROWS * S::BX;

    // Publish the band's edge rows into parity q and, past the barrier, read
    // the rows next to the band for sweep s + 1.
    auto exchange = [&](int s) {
        const int q = xpar;
        xpar ^= 1;
        if (band + RW > s + 1 && band < S::BY - 1 - s) {
#pragma unroll
            for (int c = 0; c < CH; ++c) {
                sts4(own + q * PAR + 128 * c, u[0][c]);
                sts4(own + q * PAR + S::BX + 128 * c, u[RW - 1][c]);
            }
        }
        __syncthreads();
        if (s == 0 && threadIdx.x == 0) after_first_barrier();
        if (band + RW > s + 2 && band < S::BY - 2 - s) {
#pragma unroll
            for (int c = 0; c < CH; ++c) {
                hn[c] = lds4(above + q * PAR + 128 * c);
                hs[c] = lds4(below + q * PAR + 128 * c);
            }
        }
    };

    if (band + RW > 1 && band < S::BY - 1)
        etbr_band<D, CH, RW, NW, FAST, EDGE, FUSED, false>(
            u, b, hn, hs, out, n, ld, r, d, y, bxo, byo, colmask, in_tile, rmf);
    exchange(0);
#pragma unroll 1
    for (int s = 1; s < D - 1; ++s) {
        if (band + RW > s + 1 && band < S::BY - 1 - s)
            etbr_band<D, CH, RW, NW, FAST, EDGE, false, false>(
                u, b, hn, hs, out, n, ld, r, d, y, bxo, byo, colmask, in_tile,
                rmf);
        exchange(s);
    }
    if (band + RW > D && band < S::BY - D)
        etbr_band<D, CH, RW, NW, FAST, EDGE, false, true>(
            u, b, hn, hs, out, n, ld, r, d, y, bxo, byo, colmask, in_tile, rmf);
    rm = __float_as_uint(rmf);
}


// Persistent kernel with register-resident bands: block k handles tiles k,
// k + gridDim.x, ... One staging set: the next tile's boxes are loaded as
// soon as every warp has taken the current tile into registers.
template <int D, int CH, int RW, int NW, int MINB, bool FAST, bool FUSED>
__global__ void __launch_bounds__(32 * NW, MINB)
k_etbr(const __grid_constant__ CUtensorMap map_src,
       const __grid_constant__ CUtensorMap map_b, float *__restrict__ out,
       int n, long long ld, float r, float d, float y, unsigned *err,
       const int *stop, LoopParams lp, int tiles_x, int tiles) {
    using S = EtbrShape<D, CH, RW, NW>;
    using L = EtbShape<D, CH, RW, NW, 1>;  // tile geometry for load_tile
    __shared__ unsigned fin_scratch[33];
    allow_dependents();

    // [barrier | u box | b box | exchange rows], box rows 512 or 1024 bytes.
    extern __shared__ __align__(128) unsigned char smem_raw[];
    bounds_begin(smem_raw, 0, out, nullptr, nullptr, nullptr, n, ld, err);
    const unsigned pad = (128u - (smem_addr(smem_raw) & 127u)) & 127u;
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem_raw + pad);
    float *su = reinterpret_cast<float *>(smem_raw + pad + 128);
    float *sb = su + S::BX * S::BY;
    float *xb = sb + S::BX * S::BY;

    const int tid = threadIdx.x;
    for (int k = tid; k < S::BX; k += 32 * NW)
        for (int q = 0; q < 2; ++q) {
            sts1(xb + q * S::XROWS * S::BX + k, 0.f);  // slot -1
            sts1(xb + (q * S::XROWS + S::XROWS - 1) * S::BX + k, 0.f);  // slot 2 NW
        }
    if (tid == 0) {
        mbar_init(bar);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    grid_dependency_wait();
    if (stop && *stop) return;  // same value for every thread of the launch
    if (tid == 0 && (int)blockIdx.x < tiles)
        load_tile<L>(&map_src, &map_b, bar, su, sb, blockIdx.x, tiles_x, D);
    __syncthreads();

    const int lane = tid & 31;
    const int band = (tid >> 5) * RW;
    unsigned rm = 0u;
    bool failed = false;
    unsigned fail_parity = 0u;
    int i = 0;
    int xpar = 1;  // parity of the next exchange (etbr_sweeps)
    for (int t = blockIdx.x; t < tiles; t += gridDim.x, ++i) {
        const unsigned parity = (unsigned)i & 1u;
        const bool ok = mbar_wait_parity(bar, parity);
        if (__syncthreads_or(!ok)) {
            failed = true;
            fail_parity = parity;
            break;
        }
        float4 u[RW][CH], b[RW][CH], hn[CH], hs[CH];
#pragma unroll
        for (int j = 0; j < RW; ++j)
#pragma unroll
            for (int c = 0; c < CH; ++c) {
                u[j][c] = lds4(su + (band + j) * S::BX + 128 * c + 4 * lane);
                b[j][c] = lds4(sb + (band + j) * S::BX + 128 * c + 4 * lane);
            }
#pragma unroll
        for (int c = 0; c < CH; ++c) {
            hn[c] = band > 0 ? lds4(su + (band - 1) * S::BX + 128 * c + 4 * lane)
                             : make_float4(0.f, 0.f, 0.f, 0.f);
            hs[c] = band + RW < S::BY
                        ? lds4(su + (band + RW) * S::BX + 128 * c + 4 * lane)
                        : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        // The staging boxes are consumed once every warp is past the first
        // sweep's exchange barrier: thread 0 then loads the next tile into
        // them. Until then the reads above overlap the first sweep.
        const int next = t + (int)gridDim.x;
        auto prefetch = [&]() {
            if (next < tiles) {
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                load_tile<L>(&map_src, &map_b, bar, su, sb, next, tiles_x, D);
            }
        };
        const int gx0 = (t % tiles_x) * S::TX, gy0 = (t / tiles_x) * S::TY;
        const int bxo = gx0 - S::HX, byo = gy0 - D;
        const bool edge = bxo < 1 || byo < 1 || bxo + S::BX > n - 1 ||
                          byo + S::BY > n - 1;
        if (edge)
            etbr_sweeps<D, CH, RW, NW, FAST, true, FUSED>(
                u, b, hn, hs, xb, out, n, ld, r, d, y, bxo, byo, rm, xpar,
                prefetch);
        else
            etbr_sweeps<D, CH, RW, NW, FAST, false, FUSED>(
                u, b, hn, hs, xb, out, n, ld, r, d, y, bxo, byo, rm, xpar,
                prefetch);
    }
    if (failed) {
        if (tid == 0) atomicOr(err, (unsigned)ERR_TMA_TIMEOUT);
        // Only the load waited on can be in flight: give it one more bounded
        // wait before shared memory is released.
        mbar_wait_parity(bar, fail_parity);
    }
    if (FUSED) fused_block_finish(rm, lp, fin_scratch);
}

// ---------------------------------------------------------------------------
// Persistent exact temporal blocking (JACOBI_CONTROL_PERSISTENT). One
// cooperative launch runs a whole time step: rounds of D sweeps over all
// tiles, as k_etbr launches would, separated by a grid-wide barrier instead
// of a kernel boundary. Round q reads u (q even) or u_alt (q odd) and writes
// the other. The first round of every check interval also reduces
// max |J(u) - u| of its input; at the barrier after it, the last block to
// arrive applies the stopping rule (loop_decide, the same as the device
// loop's fused launch), and every block reads the outcome once released.
// The answer is then the input of that round, as with the device loop.
//
// The barrier counts arrivals in LoopState::bar_arrive (all rounds) and
// releases by advancing LoopState::bar_epoch; every wait gives up after
// ~1 s and sets ERR_SYNC_TIMEOUT, so a block that cannot be scheduled ends
// the step with an error instead of a hang. The launch is cooperative, so
// all blocks are resident together or the launch fails.
// ---------------------------------------------------------------------------
__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned *p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_release_gpu(unsigned *p, unsigned v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Grid barrier number `round` (0, 1, ...). The last block to arrive runs
// `last` before releasing the others. Returns the step's stop flag as seen
// after the barrier (1 as well when the wait gave up).
template <class F>
__device__ __forceinline__ bool etbp_barrier(LoopState *st, unsigned round,
                                             unsigned *s_flag, F last) {
    __syncthreads();
    if (threadIdx.x == 0) {
        bool ok = true;
        __threadfence();
        const unsigned target = (round + 1u) * gridDim.x;
        if (atomicAdd(&st->bar_arrive, 1u) + 1u == target) {
            __threadfence();  // every block's atomics and stores are visible
            last();
            __threadfence();
            st_release_gpu(&st->bar_epoch, round + 1u);
        } else {
            unsigned spins = 0;
            uint64_t t0 = 0;
            while (ld_acquire_gpu(&st->bar_epoch) < round + 1u) {
                if ((++spins & 255u) == 0u) {
                    const uint64_t t = global_ns();
                    if (t0 == 0) {
                        t0 = t;
                    } else if (t - t0 > 1000000000ull) {
                        ok = false;
                        break;
                    }
                }
            }
            if (!ok) atomicOr(&st->err, (unsigned)ERR_SYNC_TIMEOUT);
        }
        *s_flag = ok ? (unsigned)ld_acquire_gpu(reinterpret_cast<const unsigned *>(&st->stop))
                     : 1u;
        // The next round's TMA loads (async proxy) read what other blocks
        // stored with ordinary stores before the barrier.
        asm volatile("fence.proxy.async.global;" ::: "memory");
    }
    __syncthreads();
    return *s_flag != 0u;
}

template <int D, int CH, int RW, int NW, int MINB, bool FAST>
__global__ void __launch_bounds__(32 * NW, MINB)
k_etbp(const __grid_constant__ CUtensorMap map_u,
       const __grid_constant__ CUtensorMap map_alt,
       const __grid_constant__ CUtensorMap map_b, float *__restrict__ u,
       float *__restrict__ u_alt, int n, long long ld, float r, float d,
       float y, LoopParams lp, int rounds_per_check, int tiles_x, int tiles) {
    using S = EtbrShape<D, CH, RW, NW>;
    using L = EtbShape<D, CH, RW, NW, 1>;
    __shared__ unsigned red[33];
    __shared__ unsigned s_flag;

    extern __shared__ __align__(128) unsigned char smem_raw[];
    bounds_begin(smem_raw, 0, u, u_alt, nullptr, nullptr, n, ld, &lp.state->err);
    const unsigned pad = (128u - (smem_addr(smem_raw) & 127u)) & 127u;
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem_raw + pad);
    float *su = reinterpret_cast<float *>(smem_raw + pad + 128);
    float *sb = su + S::BX * S::BY;
    float *xb = sb + S::BX * S::BY;

    const int tid = threadIdx.x;
    LoopState *st = lp.state;
    for (int k = tid; k < S::BX; k += 32 * NW)
        for (int q = 0; q < 2; ++q) {
            sts1(xb + q * S::XROWS * S::BX + k, 0.f);
            sts1(xb + (q * S::XROWS + S::XROWS - 1) * S::BX + k, 0.f);
        }
    if (tid == 0) {
        mbar_init(bar);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    // A step whose predecessor failed is marked stopped before it starts.
    if (*reinterpret_cast<volatile const int *>(&st->stop)) return;

    const int lane = tid & 31, warp = tid >> 5;
    const int band = warp * RW;
    int i = 0;  // loads so far: load i completes mbarrier phase i
    int xpar = 1;  // parity of the next exchange (etbr_sweeps)
    for (unsigned round = 0;; ++round) {
        const bool from_alt = (round & 1u) != 0u;
        const CUtensorMap *msrc = from_alt ? &map_alt : &map_u;
        float *out = from_alt ? u : u_alt;
        const bool fused = round % (unsigned)rounds_per_check == 0u;
        unsigned rm = 0u;
        bool failed = false;
        if (tid == 0 && (int)blockIdx.x < tiles)
            load_tile<L>(msrc, &map_b, bar, su, sb, blockIdx.x, tiles_x, D);
        for (int t = blockIdx.x; t < tiles; t += gridDim.x, ++i) {
            const unsigned parity = (unsigned)i & 1u;
            const bool ok = mbar_wait_parity(bar, parity);
            if (__syncthreads_or(!ok)) {
                // Let the load land (bounded) before the buffers are reused,
                // report, and skip the rest of the round; the barrier below
                // still sees this block, and the decision stops the step.
                mbar_wait_parity(bar, parity);
                if (tid == 0) atomicOr(&st->err, (unsigned)ERR_TMA_TIMEOUT);
                failed = true;
                ++i;
                break;
            }
            float4 uu[RW][CH], bb[RW][CH], hn[CH], hs[CH];
#pragma unroll
            for (int j = 0; j < RW; ++j)
#pragma unroll
                for (int c = 0; c < CH; ++c) {
                    uu[j][c] = lds4(su + (band + j) * S::BX + 128 * c + 4 * lane);
                    bb[j][c] = lds4(sb + (band + j) * S::BX + 128 * c + 4 * lane);
                }
#pragma unroll
            for (int c = 0; c < CH; ++c) {
                hn[c] = band > 0 ? lds4(su + (band - 1) * S::BX + 128 * c + 4 * lane)
                                 : make_float4(0.f, 0.f, 0.f, 0.f);
                hs[c] = band + RW < S::BY
                            ? lds4(su + (band + RW) * S::BX + 128 * c + 4 * lane)
                            : make_float4(0.f, 0.f, 0.f, 0.f);
            }
            __syncthreads();  // staging consumed
            if (tid == 0 && t + (int)gridDim.x < tiles) {
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                load_tile<L>(msrc, &map_b, bar, su, sb, t + gridDim.x, tiles_x, D);
            }
            const int gx0 = (t % tiles_x) * S::TX, gy0 = (t / tiles_x) * S::TY;
            const int bxo = gx0 - S::HX, byo = gy0 - D;
            const bool edge = bxo < 1 || byo < 1 || bxo + S::BX > n - 1 ||
                              byo + S::BY > n - 1;
            auto none = []() {};  // the next tile's load is already issued
            if (fused) {
                if (edge)
                    etbr_sweeps<D, CH, RW, NW, FAST, true, true>(
                        uu, bb, hn, hs, xb, out, n, ld, r, d, y, bxo, byo, rm, xpar, none);
                else
                    etbr_sweeps<D, CH, RW, NW, FAST, false, true>(
                        uu, bb, hn, hs, xb, out, n, ld, r, d, y, bxo, byo, rm, xpar, none);
            } else {
                if (edge)
                    etbr_sweeps<D, CH, RW, NW, FAST, true, false>(
                        uu, bb, hn, hs, xb, out, n, ld, r, d, y, bxo, byo, rm, xpar, none);
                else
                    etbr_sweeps<D, CH, RW, NW, FAST, false, false>(
                        uu, bb, hn, hs, xb, out, n, ld, r, d, y, bxo, byo, rm, xpar, none);
            }
        }
        (void)failed;
        if (fused) {
            // This block's share of max |J(u) - u| of the round's input.
            rm = warp_max_u(rm);
            __syncthreads();
            if (lane == 0) red[warp] = rm;
            __syncthreads();
            if (tid == 0) {
                unsigned br = 0u;
                for (int w = 0; w < NW; ++w) br = max(br, red[w]);
                if (br) atomicMax(&st->rbits, br);
            }
        }
        const bool stop = etbp_barrier(st, round, &s_flag, [&]() {
            if (fused) {
                LoopParams lq = lp;
                lq.src_is_alt = from_alt ? 1 : 0;
                const unsigned bits = atomicExch(&st->rbits, 0u);
                loop_decide(lq, __fmul_rn(lp.d, __uint_as_float(bits)), st->bmax);
            } else if (st->err) {
                st->status = -2;  // JACOBI_ERR_CUDA
                st->where = from_alt ? 0 : 1;
                st->result_k = st->k;
                st->stop = 1;
            }
        });
        if (stop) break;
    }
}

// Shapes per depth: {KIND, CH, RW, NW, NB}; KIND 0 ping-pongs the box
// through shared memory (k_etb, NB buffer sets), KIND 1 keeps the bands in
// registers (k_etbr, one staging set). Without a tile size the default is
// the register-resident one-block-per-SM shape that leaves each SM the
// fewest box rows to sweep for this grid (etb_default_variant), else the
// first shape of the depth; with one, the shape of that exact tile size, the
// first listed winning. The 12-warp x 9-row boxes exist for their tile
// counts: at N = 2048 a D = 8 launch needs 4 rounds of the 152 SMs with
// 80-row tiles and 3 with 92-row ones (measured on GB300: 14.9 against
// 16.3 ms per ten-step solve; D = 16: 14.1 against 14.8 ms). Taller bands
// in fewer warps lose more per row than their tile count saves (8 warps x 13
// rows: 17.2 ms), and 12 x 12 or 16 x 7 rows spill registers.
struct EtbVariant {
    int depth, kind, ch, rw, nw, nb, minb;
};
constexpr EtbVariant kVariants[] = {
    {2, 0, 1, 3, 32, 2, 1}, {2, 0, 1, 4, 16, 2, 1}, {2, 0, 2, 4, 16, 1, 1},
    {4, 1, 1, 6, 16, 1, 1}, {4, 0, 1, 4, 16, 2, 1}, {4, 0, 2, 4, 16, 1, 1},
    {4, 1, 1, 3, 16, 1, 2},
    {8, 1, 1, 6, 16, 1, 1}, {8, 0, 1, 4, 16, 2, 1}, {8, 0, 1, 4, 32, 1, 1},
    {8, 0, 2, 4, 16, 1, 1},
    {16, 1, 1, 6, 16, 1, 1}, {16, 0, 1, 4, 32, 1, 1}, {16, 0, 2, 3, 32, 1, 1},
    {8, 1, 1, 9, 12, 1, 1}, {16, 1, 1, 9, 12, 1, 1},
};

template <int K, int D, int CH, int RW, int NW, int NB, int MB, bool F,
          bool FU>
constexpr auto etb_kernel() {
    if constexpr (K == 0)
        return k_etb<D, CH, RW, NW, NB, MB, F, FU>;
    else
        return k_etbr<D, CH, RW, NW, MB, F, FU>;
}

template <int K, int D, int CH, int RW, int NW, int NB>
constexpr size_t etb_smem() {
    if constexpr (K == 0)
        return EtbShape<D, CH, RW, NW, NB>::SMEM;
    else
        return EtbrShape<D, CH, RW, NW>::SMEM;
}

template <int K, int D, int CH, int RW, int NW, int NB, int MB>
cudaError_t launch_variant(const GridDesc &g, const TileConf &tc,
                           const CUtensorMap *map_src,
                           const CUtensorMap *map_b, float *out,
                           unsigned *err, const LaunchCtl &ctl,
                           cudaStream_t stream) {
    using S = EtbShape<D, CH, RW, NW, NB>;
    constexpr size_t smem = etb_smem<K, D, CH, RW, NW, NB>();
    const int tiles_x = (g.n - 1 + S::TX - 1) / S::TX;
    const int tiles = tiles_x * ((g.n - 1 + S::TY - 1) / S::TY);
#define TBJ_K(F, FU)                                                          \
    launch_pdl(etb_kernel<K, D, CH, RW, NW, NB, MB, F, FU>(), dim3(tc.ctas),     \
               dim3(32 * NW), smem, stream, *map_src, *map_b, out, g.n,      \
               g.ld, g.r, g.d, g.y, err, ctl.stop, ctl.lp, tiles_x, tiles)
    if (g.fast) return ctl.fused ? TBJ_K(true, true) : TBJ_K(true, false);
    return ctl.fused ? TBJ_K(false, true) : TBJ_K(false, false);
#undef TBJ_K
}

template <int K, int D, int CH, int RW, int NW, int NB, int MB>
cudaError_t prepare_variant(TileConf &tc, int n) {
    using S = EtbShape<D, CH, RW, NW, NB>;
    constexpr size_t smem = etb_smem<K, D, CH, RW, NW, NB>();
    static_assert(smem <= 227 * 1024, "shared memory per block");
    const void *kernels[4] = {
        (const void *)etb_kernel<K, D, CH, RW, NW, NB, MB, true, false>(),
        (const void *)etb_kernel<K, D, CH, RW, NW, NB, MB, false, false>(),
        (const void *)etb_kernel<K, D, CH, RW, NW, NB, MB, true, true>(),
        (const void *)etb_kernel<K, D, CH, RW, NW, NB, MB, false, true>()};
    for (const void *k : kernels) {
        cudaError_t e = cudaFuncSetAttribute(
            k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    // Persistent grid: as many blocks as fit on the GPU at once, at most one
    // per tile.
    int dev = 0, sms = 0, per_sm = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
            &per_sm, etb_kernel<K, D, CH, RW, NW, NB, MB, true, false>(), 32 * NW,
            smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    const int tiles = ((n - 1 + S::TX - 1) / S::TX) * ((n - 1 + S::TY - 1) / S::TY);
    tc.ctas = sms * per_sm < tiles ? sms * per_sm : tiles;
    tc.smem = smem;
    return cudaSuccess;
}

template <int D, int CH, int RW, int NW, int MB>
cudaError_t prepare_persistent(TileConf &tc, int n) {
    using S = EtbrShape<D, CH, RW, NW>;
    const void *kernels[2] = {(const void *)k_etbp<D, CH, RW, NW, MB, true>,
                              (const void *)k_etbp<D, CH, RW, NW, MB, false>};
    for (const void *k : kernels) {
        cudaError_t e = cudaFuncSetAttribute(
            k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)S::SMEM);
        if (e != cudaSuccess) return e;
    }
    // Every block must be resident at once (grid barriers): as many as fit,
    // at most one per tile.
    int dev = 0, sms = 0, per_sm = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
            &per_sm, k_etbp<D, CH, RW, NW, MB, true>, 32 * NW, S::SMEM);
    if (e == cudaSuccess) {
        int per_sm2 = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
            &per_sm2, k_etbp<D, CH, RW, NW, MB, false>, 32 * NW, S::SMEM);
        if (per_sm2 < per_sm) per_sm = per_sm2;
    }
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    const int tiles = ((n - 1 + S::TX - 1) / S::TX) * ((n - 1 + S::TY - 1) / S::TY);
    tc.ctas = sms * per_sm < tiles ? sms * per_sm : tiles;
    tc.smem = S::SMEM;
    return cudaSuccess;
}

template <int D, int CH, int RW, int NW, int MB>
cudaError_t launch_persistent(const GridDesc &g, const TileConf &tc,
                              const CUtensorMap *map_u,
                              const CUtensorMap *map_alt,
                              const CUtensorMap *map_b, float *u, float *u_alt,
                              const LoopParams &lp, int rounds_per_check,
                              cudaStream_t stream) {
    using S = EtbrShape<D, CH, RW, NW>;
    const int tiles_x = (g.n - 1 + S::TX - 1) / S::TX;
    const int tiles = tiles_x * ((g.n - 1 + S::TY - 1) / S::TY);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(tc.ctas);
    cfg.blockDim = dim3(32 * NW);
    cfg.dynamicSmemBytes = S::SMEM;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (g.fast)
        return cudaLaunchKernelEx(&cfg, k_etbp<D, CH, RW, NW, MB, true>, *map_u,
                                  *map_alt, *map_b, u, u_alt, g.n, g.ld, g.r,
                                  g.d, g.y, lp, rounds_per_check, tiles_x, tiles);
    return cudaLaunchKernelEx(&cfg, k_etbp<D, CH, RW, NW, MB, false>, *map_u,
                              *map_alt, *map_b, u, u_alt, g.n, g.ld, g.r, g.d,
                              g.y, lp, rounds_per_check, tiles_x, tiles);
}

// Compiled shapes, one line each: I (index into kVariants), PART (the
// translation unit that instantiates it), KIND, D, CH, RW, NW, NB, MINB.
#define TBJ_ETB_VARIANTS(X)           \
    X(0, 0, 0, 2, 1, 3, 32, 2, 1)     \
    X(1, 0, 0, 2, 1, 4, 16, 2, 1)     \
    X(2, 0, 0, 2, 2, 4, 16, 1, 1)     \
    X(3, 1, 1, 4, 1, 6, 16, 1, 1)     \
    X(4, 0, 0, 4, 1, 4, 16, 2, 1)     \
    X(5, 0, 0, 4, 2, 4, 16, 1, 1)     \
    X(6, 1, 1, 4, 1, 3, 16, 1, 2)     \
    X(7, 2, 1, 8, 1, 6, 16, 1, 1)     \
    X(8, 1, 0, 8, 1, 4, 16, 2, 1)     \
    X(9, 1, 0, 8, 1, 4, 32, 1, 1)     \
    X(10, 1, 0, 8, 2, 4, 16, 1, 1)    \
    X(11, 3, 1, 16, 1, 6, 16, 1, 1)   \
    X(12, 0, 0, 16, 1, 4, 32, 1, 1)   \
    X(13, 0, 0, 16, 2, 3, 32, 1, 1)   \
    X(14, 2, 1, 8, 1, 9, 12, 1, 1)    \
    X(15, 3, 1, 16, 1, 9, 12, 1, 1)

constexpr int kEtbParts = 4;

// Entry points of part P: each handles the variants whose PART is P and
// returns cudaErrorInvalidValue for the others (they are not compiled here).
template <int P>
cudaError_t part_launch(int v, const GridDesc &g, const TileConf &tc,
                        const CUtensorMap *map_src, const CUtensorMap *map_b,
                        float *out, unsigned *err, const LaunchCtl &ctl,
                        cudaStream_t stream) {
    switch (v) {
#define TBJ_LAUNCH(I, PT, K, D, CH, RW, NW, NB, MB)                              \
    case I:                                                                      \
        if constexpr (PT == P)                                                   \
            return launch_variant<K, D, CH, RW, NW, NB, MB>(g, tc, map_src, map_b, \
                                                            out, err, ctl, stream); \
        return cudaErrorInvalidValue;
        TBJ_ETB_VARIANTS(TBJ_LAUNCH)
#undef TBJ_LAUNCH
        default:
            return cudaErrorInvalidValue;
    }
}

template <int P>
cudaError_t part_prepare(int v, TileConf &tc, int n) {
    switch (v) {
#define TBJ_PREP(I, PT, K, D, CH, RW, NW, NB, MB)                   \
    case I:                                                         \
        if constexpr (PT == P)                                      \
            return prepare_variant<K, D, CH, RW, NW, NB, MB>(tc, n); \
        return cudaErrorInvalidValue;
        TBJ_ETB_VARIANTS(TBJ_PREP)
#undef TBJ_PREP
        default:
            return cudaErrorInvalidValue;
    }
}

template <int P>
cudaError_t part_prepare_persistent(int v, TileConf &tc, int n) {
    switch (v) {
#define TBJ_PPREP(I, PT, K, D, CH, RW, NW, NB, MB)                  \
    case I:                                                         \
        if constexpr (PT == P && K == 1)                            \
            return prepare_persistent<D, CH, RW, NW, MB>(tc, n);    \
        return cudaErrorInvalidValue;
        TBJ_ETB_VARIANTS(TBJ_PPREP)
#undef TBJ_PPREP
        default:
            return cudaErrorInvalidValue;
    }
}

template <int P>
cudaError_t part_launch_persistent(int v, const GridDesc &g, const TileConf &tc,
                                   const CUtensorMap *map_u,
                                   const CUtensorMap *map_alt,
                                   const CUtensorMap *map_b, float *u,
                                   float *u_alt, const LoopParams &lp,
                                   long long rounds_per_check,
                                   cudaStream_t stream) {
    switch (v) {
#define TBJ_PLAUNCH(I, PT, K, D, CH, RW, NW, NB, MB)                     \
    case I:                                                              \
        if constexpr (PT == P && K == 1)                                 \
            return launch_persistent<D, CH, RW, NW, MB>(                 \
                g, tc, map_u, map_alt, map_b, u, u_alt, lp,              \
                (int)rounds_per_check, stream);                          \
        return cudaErrorInvalidValue;
        TBJ_ETB_VARIANTS(TBJ_PLAUNCH)
#undef TBJ_PLAUNCH
        default:
            return cudaErrorInvalidValue;
    }
}

// The translation unit of each variant.
constexpr int kVariantPart[] = {
#define TBJ_PART(I, PT, K, D, CH, RW, NW, NB, MB) PT,
    TBJ_ETB_VARIANTS(TBJ_PART)
#undef TBJ_PART
};

}  // namespace

// Non-template entry points of each part, defined by TBJ_ETB_DEFINE_PART in
// kernels_etb_part<P>.cu.
#define TBJ_ETB_PART_DECLS(P)                                                  \
    cudaError_t etb_part##P##_launch(                                          \
        int v, const GridDesc &g, const TileConf &tc,                          \
        const CUtensorMap *map_src, const CUtensorMap *map_b, float *out,      \
        unsigned *err, const LaunchCtl &ctl, cudaStream_t stream);             \
    cudaError_t etb_part##P##_prepare(int v, TileConf &tc, int n);             \
    cudaError_t etb_part##P##_prepare_persistent(int v, TileConf &tc, int n);  \
    cudaError_t etb_part##P##_launch_persistent(                               \
        int v, const GridDesc &g, const TileConf &tc, const CUtensorMap *map_u, \
        const CUtensorMap *map_alt, const CUtensorMap *map_b, float *u,        \
        float *u_alt, const LoopParams &lp, long long rounds_per_check,        \
        cudaStream_t stream);
TBJ_ETB_PART_DECLS(0)
TBJ_ETB_PART_DECLS(1)
TBJ_ETB_PART_DECLS(2)
TBJ_ETB_PART_DECLS(3)

#define TBJ_ETB_DEFINE_PART(P)                                                 \
    cudaError_t etb_part##P##_launch(                                          \
        int v, const GridDesc &g, const TileConf &tc,                          \
        const CUtensorMap *map_src, const CUtensorMap *map_b, float *out,      \
        unsigned *err, const LaunchCtl &ctl, cudaStream_t stream) {            \
        return part_launch<P>(v, g, tc, map_src, map_b, out, err, ctl, stream); \
    }                                                                          \
    cudaError_t etb_part##P##_prepare(int v, TileConf &tc, int n) {            \
        return part_prepare<P>(v, tc, n);                                      \
    }                                                                          \
    cudaError_t etb_part##P##_prepare_persistent(int v, TileConf &tc, int n) { \
        return part_prepare_persistent<P>(v, tc, n);                           \
    }                                                                          \
    cudaError_t etb_part##P##_launch_persistent(                               \
        int v, const GridDesc &g, const TileConf &tc, const CUtensorMap *map_u, \
        const CUtensorMap *map_alt, const CUtensorMap *map_b, float *u,        \
        float *u_alt, const LoopParams &lp, long long rounds_per_check,        \
        cudaStream_t stream) {                                                 \
        return part_launch_persistent<P>(v, g, tc, map_u, map_alt, map_b, u,   \
                                         u_alt, lp, rounds_per_check, stream); \
    }

}  // namespace tbj
