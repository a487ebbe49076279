// Internal interface between the C ABI (api.cu) and the kernel translation
// units (one per head dimension, so that they compile in parallel).
#pragma once

#include <cuda.h>
#include <cuda_runtime_api.h>

#include "gqa_common.h"

namespace gqa {

struct LaunchArgs {
    CUtensorMap tm_k;
    CUtensorMap tm_v;
    DecodeParams p;
    int row_tiles;   // 1 or 2
    bool kv8;        // fp8 e4m3 K/V codes with per-tile scales
    bool pdl;        // launch with programmatic stream serialization
    cudaStream_t stream;
};

// Enqueue the split-KV kernel (one launch per decode step) for D = 64 / D = 128.
cudaError_t launch_d64(const LaunchArgs& a);
cudaError_t launch_d128(const LaunchArgs& a);
cudaError_t launch_d128_fp8(const LaunchArgs& a);

// The prefill kernel: one CTA per 128-row tile of one (sequence, KV head).
struct PrefillLaunchArgs {
    CUtensorMap tm_k;
    CUtensorMap tm_v;
    PrefillParams p;
    unsigned grid;
    cudaStream_t stream;
    bool pdl;        // the combine: launch with programmatic stream serialization
};
cudaError_t launch_prefill(int D, const PrefillLaunchArgs& a);   // + the combine when split
size_t prefill_workspace_bytes(int D, long long items, int splits);
int prefill_smem_bytes(int D);

// Dynamic shared memory and threads per CTA of the split-KV kernel.
int splitkv_smem_bytes(int D, int row_tiles, bool kv8 = false);
int splitkv_threads(int D, int row_tiles, bool kv8 = false);
int splitkv_stages(int D, int row_tiles, bool kv8 = false);

}  // namespace gqa
