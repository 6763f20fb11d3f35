// Exhaustive verification of the fixed-divisor division (div_fixed and its
// packed form div2_fixed in jacobi_kernels.cuh) against the IEEE quotient,
// and the exact host-side reciprocal it needs.
#include <cmath>
#include <cstring>

#include "jacobi_kernels.cuh"

namespace tbj {
namespace {

// Each thread checks 2^8 consecutive bit patterns; the grid covers 2^32.
constexpr unsigned kPerThread = 256;
constexpr unsigned kThreads = 256;
constexpr unsigned kBlocks = (unsigned)((1ull << 32) / (kPerThread * kThreads));

__global__ void __launch_bounds__(kThreads)
k_fastdiv_verify(float d, float y, unsigned long long *count) {
    const unsigned base =
        (blockIdx.x * kThreads + threadIdx.x) * kPerThread;
    unsigned bad = 0;
    for (unsigned k = 0; k < kPerThread; ++k) {
        const unsigned bits = base + k;
        if ((bits & 0x7f800000u) == 0x7f800000u) continue;  // Inf / NaN
        const float x = __uint_as_float(bits);
        const float want = __fdiv_rn(x, d);
        const float got = div_fixed(x, d, y);
        bad += (__float_as_uint(want) != __float_as_uint(got)) ? 1u : 0u;
        // The packed form, on x and -x.
        const float2 got2 = div2_fixed(make_float2(x, -x), make_float2(d, d),
                                       make_float2(y, y));
        bad += (__float_as_uint(want) != __float_as_uint(got2.x)) ? 1u : 0u;
        bad += (__float_as_uint(__fdiv_rn(-x, d)) != __float_as_uint(got2.y))
                   ? 1u : 0u;
    }
    for (int o = 16; o > 0; o >>= 1) bad += __shfl_xor_sync(0xffffffffu, bad, o);
    if ((threadIdx.x & 31) == 0 && bad) atomicAdd(count, (unsigned long long)bad);
}

}  // namespace

cudaError_t fastdiv_verify_launch(float d, float y, unsigned long long *count,
                                  cudaStream_t stream) {
    k_fastdiv_verify<<<kBlocks, kThreads, 0, stream>>>(d, y, count);
    return cudaGetLastError();
}

float reciprocal_rn(float d) {
    // The float nearest to 1/d: among the float32 neighbours of the double
    // quotient, take the one whose product with d (exact in double) is
    // closest to 1; ties cannot occur for d > 0 that is not a power of two,
    // and for powers of two the reciprocal is exact.
    const float c = (float)(1.0 / (double)d);
    float best = c;
    double err = std::fabs((double)c * (double)d - 1.0);
    const float cand[2] = {std::nextafter(c, 0.0f), std::nextafter(c, 2.0f * c + 1.0f)};
    for (float v : cand) {
        const double e = std::fabs((double)v * (double)d - 1.0);
        if (e < err) {
            err = e;
            best = v;
        }
    }
    return best;
}

}  // namespace tbj
