// The tensor-core decode kernel's instance and launcher.
#include <atomic>

#include "gqa_launch.h"
#include "gqa_decode_tc.cuh"

namespace gqa {

cudaError_t launch_decode_tc(const LaunchArgs& a) {
    using TS = TcShape<128>;
    // The shared-memory opt-in is per function and per device.
    static std::atomic<unsigned long long> attr_set_mask{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = 1ull << (dev & 63);
    if (!(attr_set_mask.load() & bit)) {
        e = cudaFuncSetAttribute(gqa_decode_tc_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 TS::kSmemBytes);
        if (e != cudaSuccess) return e;
        attr_set_mask.fetch_or(bit);
    }
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.p.ctas);
    cfg.blockDim = dim3(TS::kThreads);
    cfg.dynamicSmemBytes = TS::kSmemBytes;
    cfg.stream = a.stream;
    cfg.attrs = attr;
    cfg.numAttrs = a.pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, gqa_decode_tc_kernel<128>, a.tm_k, a.tm_v, a.p);
}

int decode_tc_smem_bytes() { return TcShape<128>::kSmemBytes; }
int decode_tc_threads() { return TcShape<128>::kThreads; }

}  // namespace gqa
