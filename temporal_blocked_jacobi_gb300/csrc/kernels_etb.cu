// Exact temporal blocking ("Synchronous vs block-async Jacobi on one RTX
// 5050", section 02): choice of the compiled shape for a grid and depth, and
// dispatch to the translation unit that instantiates it. The kernels are in
// etb_kernels.cuh.
#include "etb_kernels.cuh"

namespace tbj {

namespace {

// The default shape of a depth for an N x N grid: among the register-resident
// shapes with one block per SM, the fewest box rows per SM,
// ceil(tiles / SMs) x box height (the box is 128 columns wide for all of
// them), the first listed winning ties. -1 when the depth has no such shape
// or the SM count cannot be read.
int etb_default_variant(int n, int depth) {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
            cudaSuccess ||
        sms < 1) {
        cudaGetLastError();
        return -1;
    }
    int pick = -1;
    long long best = 0;
    for (int v = 0; v < (int)(sizeof(kVariants) / sizeof(kVariants[0])); ++v) {
        const EtbVariant &k = kVariants[v];
        if (k.depth != depth || k.kind != 1 || k.minb != 1 || k.ch != 1) continue;
        const int hx = (depth + 3) / 4 * 4;
        const int by = k.nw * k.rw;
        const long long tx = 128 - 2 * hx, ty = by - 2 * depth;
        const long long tiles = ((n - 1 + tx - 1) / tx) * ((n - 1 + ty - 1) / ty);
        const long long rows = (tiles + sms - 1) / sms * by;
        if (pick < 0 || rows < best) {
            pick = v;
            best = rows;
        }
    }
    return pick;
}

}  // namespace

int etb_configure(int n, int depth, int tile_x, int tile_y, TileConf *tc,
                  bool streamed) {
    if (depth != 2 && depth != 4 && depth != 8 && depth != 16) return -1;
    // Whole columns: the column-streamed kernel (kernels_etbs.cu), also the
    // default at D = 8 on grids with enough rows per warp.
    if (tile_y == 0 && tile_x == 128 - 2 * ((depth + 3) / 4 * 4))
        return etbs_configure(n, depth, tc) ? 0 : -5;
    if (streamed && tile_x == 0 && tile_y == 0 && depth == 8) {
        int dev = 0, sms = 0;
        if (cudaGetDevice(&dev) == cudaSuccess &&
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) ==
                cudaSuccess &&
            sms > 0 && etbs_preferred(n, sms))
            return etbs_configure(n, depth, tc) ? 0 : -5;
        cudaGetLastError();
    }
    int pick = tile_x == 0 && tile_y == 0 ? etb_default_variant(n, depth) : -1;
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
    tc->smem = 0;  // set by prepare_sweep_etb
    tc->variant = pick;
    tc->ctas = 0;  // set by prepare_sweep_etb
    tc->stream = tc->ch = tc->sx = tc->sy = tc->grid_x = tc->grid_y = 0;
    tc->work = nullptr;
    tc->bands = 0;
    return 0;
}

namespace {

bool valid_variant(int v) {
    return v >= 0 && v < (int)(sizeof(kVariants) / sizeof(kVariants[0]));
}

}  // namespace

cudaError_t prepare_sweep_etb(TileConf &tc, int n) {
    if (tc.variant == kEtbsVariant) return prepare_sweep_etbs(tc, n);
    if (!valid_variant(tc.variant)) return cudaErrorInvalidValue;
    switch (kVariantPart[tc.variant]) {
        case 0: return etb_part0_prepare(tc.variant, tc, n);
        case 1: return etb_part1_prepare(tc.variant, tc, n);
        case 2: return etb_part2_prepare(tc.variant, tc, n);
        case 3: return etb_part3_prepare(tc.variant, tc, n);
        default: return cudaErrorInvalidValue;
    }
}

bool etb_persistent_ok(const TileConf &tc) {
    return tc.variant >= 0 &&
           tc.variant < (int)(sizeof(kVariants) / sizeof(kVariants[0])) &&
           kVariants[tc.variant].kind == 1;
}

cudaError_t prepare_etb_persistent(TileConf &tc, int n) {
    if (!etb_persistent_ok(tc)) return cudaErrorInvalidValue;
    switch (kVariantPart[tc.variant]) {
        case 0: return etb_part0_prepare_persistent(tc.variant, tc, n);
        case 1: return etb_part1_prepare_persistent(tc.variant, tc, n);
        case 2: return etb_part2_prepare_persistent(tc.variant, tc, n);
        case 3: return etb_part3_prepare_persistent(tc.variant, tc, n);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_etb_persistent(const GridDesc &g, const TileConf &tc,
                                  const CUtensorMap *map_u,
                                  const CUtensorMap *map_alt,
                                  const CUtensorMap *map_b, float *u,
                                  float *u_alt, const LoopParams &lp,
                                  long long rounds_per_check,
                                  cudaStream_t stream) {
    if (!etb_persistent_ok(tc)) return cudaErrorInvalidValue;
#define TBJ_P(P)                                                           \
    case P:                                                                \
        return etb_part##P##_launch_persistent(tc.variant, g, tc, map_u,   \
                                               map_alt, map_b, u, u_alt,   \
                                               lp, rounds_per_check, stream);
    switch (kVariantPart[tc.variant]) {
        TBJ_P(0) TBJ_P(1) TBJ_P(2) TBJ_P(3)
        default: return cudaErrorInvalidValue;
    }
#undef TBJ_P
}

cudaError_t launch_sweep_etb(const GridDesc &g, const TileConf &tc,
                             const CUtensorMap *map_src,
                             const CUtensorMap *map_b, const float *src,
                             const float *b, float *out, ResidualOut *status,
                             const LaunchCtl &ctl, cudaStream_t stream) {
    unsigned *err = ctl.lp.state ? &ctl.lp.state->err : &status->err;
    if (tc.variant == kEtbsVariant)
        return launch_sweep_etbs(g, tc, src, b, out, err, ctl, stream);
    if (!valid_variant(tc.variant)) return cudaErrorInvalidValue;
#define TBJ_P(P)                                                          \
    case P:                                                               \
        return etb_part##P##_launch(tc.variant, g, tc, map_src, map_b, out, \
                                    err, ctl, stream);
    switch (kVariantPart[tc.variant]) {
        TBJ_P(0) TBJ_P(1) TBJ_P(2) TBJ_P(3)
        default: return cudaErrorInvalidValue;
    }
#undef TBJ_P
}

}  // namespace tbj
