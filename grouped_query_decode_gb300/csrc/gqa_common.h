// Types and constants shared by the host launcher and the kernels.
#pragma once

#include <cstddef>
#include <cstdint>

namespace gqa {

constexpr int kTileTokens = 64;   // tokens per pipeline stage (one TMA box of rows)
constexpr int kSlices = 4;        // consumer warps per 16-row tile, 16 tokens each per stage
constexpr int kMaxRowTiles = 2;   // R <= 32 query rows per KV head
constexpr int kBoxCols = 64;      // bf16 elements per 128-byte swizzle box row
constexpr uint64_t kWaitTimeoutNs = 2000000000ull;  // bounded device waits: 2 s

// Status bits of the per-device status word.
constexpr unsigned kStatusTimeout = 1u;

// Workspace: [int64 prefix[B + 1]] padded to 256 B, then per CTA two partial
// slots: O[R][D] (normalised by its own l), m[R], l[R], each slot padded to a
// multiple of 4 floats so that every slot starts on a 16-byte boundary (the
// combine kernel reads O with 16-byte loads).
inline size_t ws_prefix_bytes(int B) {
    size_t b = sizeof(long long) * (size_t)(B + 1);
    return (b + 255) & ~size_t(255);
}
__host__ __device__ inline size_t ws_slot_floats(int R, int D) {
    return (size_t)R * D + (((size_t)2 * R + 3) & ~(size_t)3);
}
inline size_t ws_total_bytes(int B, int R, int D, int ctas) {
    return ws_prefix_bytes(B) + sizeof(float) * ws_slot_floats(R, D) * 2 * (size_t)ctas;
}

struct DecodeParams {
    const uint16_t* q;       // [B, sq, H, D] bf16 bits
    const int32_t* seq_lens; // [B]
    uint16_t* out;           // [B, sq, H, D] bf16 bits
    float* lse;              // [B, sq, H] or nullptr
    long long* ws_prefix;    // [B + 1]
    float* ws_part;          // [ctas][2][R*(D+2)]
    unsigned* status;        // per-device status word (kStatus* bits)
    float scale_log2;        // scale * log2(e)
    int B, sq, H, G, Tmax, R, heads_per_group, ctas;
};

template <int D, int MT>
struct KernelShape {
    static constexpr int kConsumerWarps = kSlices * MT;
    static constexpr int kThreads = (kConsumerWarps + 1) * 32;
    static constexpr int kBoxes = D / kBoxCols;
    static constexpr int kTileBytes = kTileTokens * D * 2;   // K (or V) of one stage
    static constexpr int kStageBytes = 2 * kTileBytes;
    static constexpr int kMergeBytes = MT * (kSlices - 1) * 16 * D * 4;
    static constexpr int kMlBytes = MT * kSlices * 16 * 2 * 4;
    static constexpr int kStages = D == 128 ? (MT == 1 ? 5 : 4) : 8;
    static constexpr int kBarBytes = 8 * (2 * kStages + 2 * MT) + 64;
    // +1024 so the ring can be aligned to the 1 KB swizzle atom at run time.
    static constexpr int kSmemBytes =
        1024 + kStages * kStageBytes + kMergeBytes + kMlBytes + kBarBytes;
};

}  // namespace gqa
