// Prefill kernel instantiations (D = 64, 128) and their launch.
#include <atomic>

#include "gqa_launch.h"
#include "gqa_prefill.cuh"

namespace gqa {

namespace {

template <int D>
cudaError_t launch_prefill_t(const PrefillLaunchArgs& a) {
    using PS = PrefillShape<D>;
    // The shared-memory opt-in is per function and per device.
    static std::atomic<unsigned long long> attr_set_mask{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = 1ull << (dev & 63);
    if (!(attr_set_mask.load() & bit)) {
        e = cudaFuncSetAttribute(gqa_prefill_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 PS::kSmemBytes);
        if (e != cudaSuccess) return e;
        attr_set_mask.fetch_or(bit);
    }
    gqa_prefill_kernel<D><<<a.grid, PS::kThreads, PS::kSmemBytes, a.stream>>>(a.tm_k, a.tm_v, a.p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill(int D, const PrefillLaunchArgs& a) {
    return D == 64 ? launch_prefill_t<64>(a) : launch_prefill_t<128>(a);
}

int prefill_smem_bytes(int D) { return D == 64 ? PrefillShape<64>::kSmemBytes : PrefillShape<128>::kSmemBytes; }

}  // namespace gqa
