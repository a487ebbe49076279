// Kernel instances for head dimension 64.
#include "gqa_launch_impl.cuh"

namespace gqa {

cudaError_t launch_d64(const LaunchArgs& a) {
    return a.row_tiles == 1 ? launch_splitkv<64, 1, false>(a)
                            : launch_splitkv<64, 2, false>(a);
}

}  // namespace gqa
