// Launch code shared by the per-head-dimension translation units.
#pragma once

#include <atomic>

#include "gqa_launch.h"
#include "gqa_splitkv.cuh"

namespace gqa {

template <int D, int MT, bool KV8>
cudaError_t launch_splitkv(const LaunchArgs& a) {
    using KS = KernelShape<D, MT, KV8>;
    // The shared-memory opt-in is per function and per device.
    static std::atomic<unsigned long long> attr_set_mask{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = 1ull << (dev & 63);
    if (!(attr_set_mask.load() & bit)) {
        e = cudaFuncSetAttribute(gqa_splitkv_kernel<D, MT, KV8>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, KS::kSmemBytes);
        if (e != cudaSuccess) return e;
        attr_set_mask.fetch_or(bit);
    }
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.p.ctas);
    cfg.blockDim = dim3(KS::kThreads);
    cfg.dynamicSmemBytes = KS::kSmemBytes;
    cfg.stream = a.stream;
    cfg.attrs = attr;
    cfg.numAttrs = a.pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, gqa_splitkv_kernel<D, MT, KV8>, a.tm_k, a.tm_v, a.p);
}

}  // namespace gqa
