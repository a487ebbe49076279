// Prefill kernel instantiations (D = 64, 128) and their launch.
#include <atomic>

#include "gqa_launch.h"
#include "gqa_prefill.cuh"

namespace gqa {

namespace {

template <int D, bool SPLIT>
cudaError_t launch_prefill_t(const PrefillLaunchArgs& a) {
    using PS = PrefillShape<D>;
    // The shared-memory opt-in is per function and per device.
    static std::atomic<unsigned long long> attr_set_mask{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = 1ull << (dev & 63);
    if (!(attr_set_mask.load() & bit)) {
        e = cudaFuncSetAttribute(gqa_prefill_kernel<D, SPLIT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 PS::kSmemBytes);
        if (e != cudaSuccess) return e;
        attr_set_mask.fetch_or(bit);
    }
    // The combine of a split chunk launches with programmatic dependent launch
    // (a.pdl) and waits (griddepcontrol.wait) for the prefill grid before it
    // reads the partials: the short D = 64 chunk 20.4 -> 17.8 us. The prefill
    // kernel itself launches plainly: moving its set-up ahead of the length
    // read, to overlap it with the grid before, made the 8k-token prefill 12 %
    // slower, and a wait at its top gained nothing measurable.
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.grid);
    cfg.blockDim = dim3(PS::kThreads);
    cfg.dynamicSmemBytes = PS::kSmemBytes;
    cfg.stream = a.stream;
    cfg.attrs = attr;
    cfg.numAttrs = 0;
    e = cudaLaunchKernelEx(&cfg, gqa_prefill_kernel<D, SPLIT>, a.tm_k, a.tm_v, a.p);
    cfg.numAttrs = a.pdl ? 1 : 0;   // the combine
    if (e != cudaSuccess || !SPLIT) return e;
    // One warp per row: (items x 2 tiles) x 16 CTAs of 8 warps.
    cfg.gridDim = dim3(a.grid / a.p.splits * 2 * (kPfRows / 8));
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = 0;
    return cudaLaunchKernelEx(&cfg, gqa_prefill_combine<D>, a.p);
}

}  // namespace

cudaError_t launch_prefill(int D, const PrefillLaunchArgs& a) {
    if (a.p.splits > 1) return D == 64 ? launch_prefill_t<64, true>(a) : launch_prefill_t<128, true>(a);
    return D == 64 ? launch_prefill_t<64, false>(a) : launch_prefill_t<128, false>(a);
}

size_t prefill_workspace_bytes(int D, long long items, int splits) {
    return splits <= 1 ? 0 : sizeof(float) * (size_t)items * splits * 2 * kPfRows * prefill_part_stride(D);
}

int prefill_smem_bytes(int D) { return D == 64 ? PrefillShape<64>::kSmemBytes : PrefillShape<128>::kSmemBytes; }

}  // namespace gqa
