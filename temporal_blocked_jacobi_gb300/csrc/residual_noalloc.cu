// Residual norms for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc at the moment they need the norms:
// code that runs while a CUDA stream is being captured into a graph (an
// allocation there is not allowed or breaks the capture), latency-critical
// loops where cudaMalloc/cudaFree would synchronise the whole device, and
// host applications whose device memory is handed out by their own
// allocator. jacobi_residual_noalloc serves them: it computes exactly what
// jacobi_residual computes, but keeps its reduction scratch in a fixed
// array in this file's device memory instead of in memory owned by a
// solver handle, and it allocates nothing.
//
// The scratch array is reserved on every GPU that loads this library and
// stays reserved until the process exits. All calls share it, so calls that
// may overlap on a GPU (different streams, or different host threads) race
// on it and must be serialised by the caller.
#include <cmath>
#include <mutex>

#include "../../include/jacobi.h"
#include "jacobi_kernels.cuh"

namespace tbj {
namespace {

constexpr int kWarps = 4;
constexpr int kRows = 32;
constexpr unsigned FULL = 0xffffffffu;

// Per-block partial maxima (2 words per block) followed by the last-block
// ticket. Zero at load. The last block of every launch sets the ticket back
// to zero, so it is zero again whenever a launch has run to its end; it is
// cleared explicitly only on the first call after a call on the same device
// that failed (a launch that could not be enqueued or completed).
constexpr int kMaxBlocks = JACOBI_RESIDUAL_NOALLOC_MAX_BLOCKS;
constexpr int kTicket = 2 * kMaxBlocks;
static __device__ __align__(256) unsigned g_residual_scratch[2 * kMaxBlocks + 64];

// Device address of g_residual_scratch for each device, looked up once per
// device with that device current (in host code the symbol's name is only a
// stand-in, not a device address).
constexpr int kMaxDevices = 64;
unsigned *g_scratch_ptr[kMaxDevices] = {nullptr};
// Per device: an earlier call failed, so the ticket may not be zero.
bool g_ticket_suspect[kMaxDevices] = {false};
std::mutex g_scratch_mutex;

__device__ __forceinline__ float4 ld4(const float *p) {
    return *reinterpret_cast<const float4 *>(p);
}

__device__ __forceinline__ unsigned fbits(float x) {
    return __float_as_uint(fabsf(x));
}

__device__ __forceinline__ void cell_norms(float c, float west, float east,
                                           float north, float south, float bb,
                                           int i, int x, int n, float r,
                                           float d, unsigned &rm,
                                           unsigned &bm) {
    if (x < 1 || x > n - 2) return;
    const float ju = jacobi_update(west, east, north, south, bb, r, d);
    const float e = __fmul_rn(d, fabsf(__fsub_rn(ju, c)));
    const float qw = (x - 1 == 0) ? west : 0.f;
    const float qe = (x + 1 == n - 1) ? east : 0.f;
    const float qn = (i - 1 == 0) ? north : 0.f;
    const float qs = (i + 1 == n - 1) ? south : 0.f;
    const float q = __fadd_rn(__fadd_rn(qw, qe), __fadd_rn(qn, qs));
    const float bi = __fadd_rn(bb, __fmul_rn(r, q));
    rm = max(rm, fbits(e));
    bm = max(bm, fbits(bi));
}

__device__ __forceinline__ unsigned warp_max(unsigned v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(FULL, v, o));
    return v;
}

// Same traversal and arithmetic as the handle's residual kernel: a warp
// walks a strip 128 floats wide down kRows rows; block maxima go to the
// scratch; the last block to finish writes norms[0] = rmax, norms[1] = bmax
// and re-arms the ticket.
__global__ void __launch_bounds__(32 * kWarps)
k_residual_noalloc(const float *__restrict__ u, const float *__restrict__ b,
                   int n, long long ld, float r, float d,
                   unsigned *__restrict__ scratch, float *__restrict__ norms) {
    const int lane = threadIdx.x;
    const int vx = blockIdx.x * 32 + lane;
    const int x0 = vx * 4;
    const bool active = x0 < n;
    const int i0 = 1 + (blockIdx.y * kWarps + threadIdx.y) * kRows;
    const int i1 = min(i0 + kRows, n - 1);
    unsigned rm = 0u, bm = 0u;
    if (i0 <= n - 2) {
        float4 top = make_float4(0.f, 0.f, 0.f, 0.f), mid = top;
        if (active) {
            top = ld4(u + (long long)(i0 - 1) * ld + x0);
            mid = ld4(u + (long long)i0 * ld + x0);
        }
        for (int i = i0; i < i1; ++i) {
            const long long row = (long long)i * ld;
            float4 bot = make_float4(0.f, 0.f, 0.f, 0.f), bb = bot;
            float edge = 0.f;
            if (active) {
                bot = ld4(u + row + ld + x0);
                bb = ld4(b + row + x0);
                if (lane == 0 && x0 > 0) edge = u[row + x0 - 1];
                if (lane == 31 && x0 + 4 < n) edge = u[row + x0 + 4];
            }
            float west = __shfl_up_sync(FULL, mid.w, 1);
            float east = __shfl_down_sync(FULL, mid.x, 1);
            if (lane == 0) west = edge;
            if (lane == 31) east = edge;
            if (active) {
                cell_norms(mid.x, west, mid.y, top.x, bot.x, bb.x, i, x0 + 0, n, r, d, rm, bm);
                cell_norms(mid.y, mid.x, mid.z, top.y, bot.y, bb.y, i, x0 + 1, n, r, d, rm, bm);
                cell_norms(mid.z, mid.y, mid.w, top.z, bot.z, bb.z, i, x0 + 2, n, r, d, rm, bm);
                cell_norms(mid.w, mid.z, east, top.w, bot.w, bb.w, i, x0 + 3, n, r, d, rm, bm);
            }
            top = mid;
            mid = bot;
        }
    }
    rm = warp_max(rm);
    bm = warp_max(bm);
    __shared__ unsigned s_r[kWarps], s_b[kWarps];
    __shared__ bool s_last;
    if (lane == 0) {
        s_r[threadIdx.y] = rm;
        s_b[threadIdx.y] = bm;
    }
    __syncthreads();
    const unsigned nblocks = gridDim.x * gridDim.y;
    const unsigned bid = blockIdx.y * gridDim.x + blockIdx.x;
    if (threadIdx.y == 0 && lane == 0) {
        unsigned br = 0u, bbm = 0u;
        for (int w = 0; w < kWarps; ++w) {
            br = max(br, s_r[w]);
            bbm = max(bbm, s_b[w]);
        }
        scratch[2 * bid] = br;
        scratch[2 * bid + 1] = bbm;
        __threadfence();
        const unsigned t = atomicAdd(&scratch[kTicket], 1u);
        s_last = (t == nblocks - 1);
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    const int tid = threadIdx.y * 32 + lane;
    rm = 0u;
    bm = 0u;
    const volatile unsigned *vp = scratch;
    for (unsigned k = tid; k < nblocks; k += 32 * kWarps) {
        rm = max(rm, vp[2 * k]);
        bm = max(bm, vp[2 * k + 1]);
    }
    rm = warp_max(rm);
    bm = warp_max(bm);
    __syncthreads();
    if (lane == 0) {
        s_r[threadIdx.y] = rm;
        s_b[threadIdx.y] = bm;
    }
    __syncthreads();
    if (tid == 0) {
        unsigned br = 0u, bbm = 0u;
        for (int w = 0; w < kWarps; ++w) {
            br = max(br, s_r[w]);
            bbm = max(bbm, s_b[w]);
        }
        norms[0] = __uint_as_float(br);
        norms[1] = __uint_as_float(bbm);
        scratch[kTicket] = 0u;
    }
}

// Look up (once per device) the device address of the scratch array.
// *suspect: whether an earlier call on this device failed (cleared here).
cudaError_t scratch_for_current_device(unsigned **out, int *dev_out,
                                       bool *suspect) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_residual_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_ptr[dev] = static_cast<unsigned *>(p);
    }
    *out = g_scratch_ptr[dev];
    *dev_out = dev;
    *suspect = g_ticket_suspect[dev];
    g_ticket_suspect[dev] = false;
    return cudaSuccess;
}

void mark_ticket_suspect(int dev) {
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    g_ticket_suspect[dev] = true;
}

bool aligned16(const void *p) {
    return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

}  // namespace
}  // namespace tbj

extern "C" int jacobi_residual_noalloc(int n, long long ld, float r,
                                       const float *u, const float *b,
                                       float *norms, void *cuda_stream) {
    using namespace tbj;
    if (n < 3 || ld < n || ld % 4 != 0) return JACOBI_ERR_INVALID_ARG;
    if (!std::isfinite(r) || r < 0.f) return JACOBI_ERR_INVALID_ARG;
    if (!u || !b || !norms || !aligned16(u) || !aligned16(b) ||
        (reinterpret_cast<uintptr_t>(norms) & 7u))
        return JACOBI_ERR_INVALID_ARG;
    const int nvec = (n + 3) / 4;
    const long long gx = (nvec + 31) / 32;
    const long long gy = (n - 2 + kWarps * kRows - 1) / (kWarps * kRows);
    if (gx * gy > kMaxBlocks) return JACOBI_ERR_UNSUPPORTED;  // n too large
    unsigned *scratch = nullptr;
    int dev = 0;
    bool suspect = false;
    if (scratch_for_current_device(&scratch, &dev, &suspect) != cudaSuccess)
        return JACOBI_ERR_CUDA;
    cudaStream_t stream = static_cast<cudaStream_t>(cuda_stream);
    // The ticket is zero after every launch that ran to its end; after a
    // failed call it is cleared once more. The per-block partials are always
    // written before they are read.
    if (suspect &&
        cudaMemsetAsync(scratch + kTicket, 0, sizeof(unsigned), stream) !=
            cudaSuccess) {
        mark_ticket_suspect(dev);
        return JACOBI_ERR_CUDA;
    }
    volatile float four_r = 4.0f * r;
    const float d = 1.0f + four_r;
    k_residual_noalloc<<<dim3((unsigned)gx, (unsigned)gy), dim3(32, kWarps), 0,
                         stream>>>(u, b, n, ld, r, d, scratch, norms);
    if (cudaGetLastError() != cudaSuccess) {
        mark_ticket_suspect(dev);
        return JACOBI_ERR_CUDA;
    }
    return JACOBI_OK;
}
