// Depth controllers for the block-asynchronous strategy ("Synchronous vs
// block-async Jacobi on one RTX 5050", section 02: D is only a kernel
// argument, so it can change between launches; G-asc, G-desc and the
// feedback controller G-fb). Host code only: the solver calls
// jacobi_adapt_next after each residual check with that check's
// rho = rmax / bmax and the interval's device time.
#include <cmath>
#include <cstring>

#include "../../include/jacobi.h"

namespace {

// rho thresholds at which G-asc / G-desc change D (section 02).
constexpr double kThresholds[3] = {1e-2, 1e-3, 1e-4};
// G-fb: a rate below this fraction of the previous one is a drop.
constexpr double kHoldFraction = 0.9;
// G-fb: measurements skipped after a change of D.
constexpr int kSettle = 1;

bool power_of_two_depth(int d) {
    return d == 2 || d == 4 || d == 8 || d == 16;
}

int log2_int(int d) {
    int k = 0;
    while ((1 << (k + 1)) <= d) ++k;
    return k;
}

bool valid(const jacobi_adapt_state_t *st) {
    if (!st || !power_of_two_depth(st->depth_max)) return false;
    if (st->policy < JACOBI_ADAPT_G_ASC || st->policy > JACOBI_ADAPT_G_FB)
        return false;
    return st->depth >= 1 && st->depth <= st->depth_max &&
           (st->depth & (st->depth - 1)) == 0 && st->level >= 0 &&
           st->level <= 3 && st->settle >= 0;
}

void set_depth(jacobi_adapt_state_t *st, int d) {
    if (d < 1) d = 1;
    if (d > st->depth_max) d = st->depth_max;
    if (d != st->depth) {
        st->depth = d;
        st->changes += 1;
        if (st->policy == JACOBI_ADAPT_G_FB) st->settle = kSettle;
    }
}

}  // namespace

extern "C" {

int jacobi_adapt_init(jacobi_adapt_state_t *st, int policy, int depth_max) {
    if (!st) return JACOBI_ERR_INVALID_ARG;
    if (policy < JACOBI_ADAPT_G_ASC || policy > JACOBI_ADAPT_G_FB ||
        !power_of_two_depth(depth_max))
        return JACOBI_ERR_INVALID_ARG;
    std::memset(st, 0, sizeof *st);
    st->policy = policy;
    st->depth_max = depth_max;
    st->depth = policy == JACOBI_ADAPT_G_DESC ? depth_max : 1;
    return JACOBI_OK;
}

int jacobi_adapt_next(jacobi_adapt_state_t *st, double rho, double ms) {
    if (!valid(st)) return JACOBI_ERR_INVALID_ARG;
    if (st->policy != JACOBI_ADAPT_G_FB) {
        // Thresholds crossed by this rho; the level never goes back down.
        int crossed = 0;
        for (double t : kThresholds) crossed += (rho < t) ? 1 : 0;
        if (crossed > st->level) st->level = crossed;
        const int steps = st->level < log2_int(st->depth_max)
                              ? st->level
                              : log2_int(st->depth_max);
        set_depth(st, st->policy == JACOBI_ADAPT_G_ASC ? (1 << steps)
                                                       : (st->depth_max >> steps));
        return st->depth;
    }
    // G-fb. A rate needs the previous check's rho, both positive, and a
    // positive interval time; otherwise this check only records rho.
    const bool measurable = st->have_prev && st->rho_prev > 0.0 && rho > 0.0 &&
                            ms > 0.0 && std::isfinite(rho) &&
                            std::isfinite(st->rho_prev);
    const double rate = measurable ? -std::log(rho / st->rho_prev) / ms : 0.0;
    st->rho_prev = rho;
    st->have_prev = 1;
    if (!measurable) return st->depth;
    if (st->settle > 0) {
        st->settle -= 1;
        return st->depth;
    }
    const bool holds = !st->have_ref || rate >= kHoldFraction * st->rate_ref;
    st->rate_ref = rate;
    st->have_ref = 1;
    set_depth(st, holds ? 2 * st->depth : st->depth / 2);
    return st->depth;
}

}  // extern "C"
