// Kernel instances for head dimension 128.
#include "gqa_launch_impl.cuh"

namespace gqa {

cudaError_t launch_d128(const LaunchArgs& a) {
    return a.row_tiles == 1 ? launch_splitkv<128, 1, false>(a)
                            : launch_splitkv<128, 2, false>(a);
}

}  // namespace gqa
