// Exact-temporal-blocking kernels of the shapes whose PART is 0 in
// TBJ_ETB_VARIANTS (etb_kernels.cuh); compiled on its own so that the four
// parts build in parallel.
#include "etb_kernels.cuh"

namespace tbj {
TBJ_ETB_DEFINE_PART(0)
}  // namespace tbj
