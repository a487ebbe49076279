// Kernel instances for head dimension 128 with fp8 (e4m3) K/V caches.
#include "gqa_launch_impl.cuh"

namespace gqa {

cudaError_t launch_d128_fp8(const LaunchArgs& a) {
    return a.row_tiles == 1 ? launch_splitkv<128, 1, true>(a) : launch_splitkv<128, 2, true>(a);
}

}  // namespace gqa
