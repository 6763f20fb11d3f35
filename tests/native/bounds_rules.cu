// Host-side check of the bounds-checked build's range rules
// (temporal_blocked_jacobi_gb300/csrc/jacobi_kernels.cuh): prints one line
// per case, "<rule> <arguments> <0|1>", for tests/test_bounds_rules.py to
// compare with the expected answers. Built with nvcc, run on the host.
#include <cstdio>

#include "../../temporal_blocked_jacobi_gb300/csrc/jacobi_kernels.cuh"

int main() {
    using namespace tbj;
    const long long smem[][3] = {{0, 16, 128},  {112, 16, 128}, {116, 16, 128},
                                 {128, 16, 128}, {-16, 16, 128}, {124, 4, 128},
                                 {126, 4, 128}, {128, 4, 128},  {0, 16, 8}};
    for (auto &c : smem)
        std::printf("smem %lld %lld %lld %d\n", c[0], c[1], c[2],
                    (int)smem_access_ok(c[0], (unsigned)c[1],
                                        (unsigned long long)c[2]));
    // n = 6, ld = 8: interior rows and columns 1 .. 4, padding columns 6, 7
    const long long grid[][2] = {{0, 1},  {47, 1}, {48, 1}, {44, 4},
                                 {45, 4}, {-1, 1}, {9, 4},  {10, 4}};
    for (auto &c : grid)
        std::printf("grid %lld %lld %d\n", c[0], c[1],
                    (int)grid_access_ok(c[0], (int)c[1], 6, 8));
    const long long inner[][2] = {{9, 4},  {10, 4}, {10, 3}, {12, 1}, {13, 1},
                                  {8, 1},  {1, 1},  {41, 1}, {33, 4}, {14, 1},
                                  {36, 1}, {33, 1}};
    for (auto &c : inner)
        std::printf("interior %lld %lld %d\n", c[0], c[1],
                    (int)interior_access_ok(c[0], (int)c[1], 6, 8));
    const int xs[] = {0, 4, -4, 2, -3, 1, 120};
    for (int x : xs) std::printf("tma %d %d\n", x, (int)tma_x_ok(x));
    return 0;
}
