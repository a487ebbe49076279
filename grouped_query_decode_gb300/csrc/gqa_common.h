// Types and constants shared by the host launcher and the kernels.
#pragma once

#include <cstddef>
#include <cstdint>

namespace gqa {

constexpr int kTileTokens = 64;   // tokens per pipeline stage (one TMA box of rows)
constexpr int kSlices = 4;        // consumer warps per 16-row tile, 16 tokens each per stage
constexpr int kMaxRowTiles = 2;   // R <= 32 query rows per KV head
constexpr int kBoxCols = 64;      // bf16 elements per 128-byte swizzle box row
constexpr uint64_t kWaitTimeoutNs = 2000000000ull;  // bounded device waits: 2 s by default
constexpr float kRescaleSlack = 8.0f;   // lazy online-softmax rescale threshold (base 2)
// Most CTAs whose partials one merge can combine (the merge keeps per-
// contributor state in shared memory); the grid never exceeds it.
constexpr int kMaxMergeContrib = 180;
// Units split over at most this many CTAs are merged by each thread in one
// round of loads (the contributors' values held in registers); more
// contributors take the cooperative three-step merge. Kernels with room in
// their register budget take more (KernelShape::kFastMerge).
constexpr int kFastMerge = 8;

// Status bits of the per-device status word.
constexpr unsigned kStatusTimeout = 1u;

// Workspace: one 64-bit arrival counter per (sequence, KV head, 16-row tile),
// padded to 256 B, then per CTA two partial slots: O[R][D] (normalised by its
// own l), m[R], l[R], each slot padded to a multiple of 4 floats so that every
// slot starts on a 16-byte boundary (the merge reads O with 16-byte loads).
// The counters carry the call's epoch, so no part of the workspace needs
// clearing.
inline size_t ws_counter_bytes(int B, int G) {
    size_t b = sizeof(unsigned long long) * (size_t)B * G * kMaxRowTiles;
    return (b + 255) & ~size_t(255);
}
__host__ __device__ inline size_t ws_slot_floats(int R, int D) {
    return (size_t)R * D + (((size_t)2 * R + 3) & ~(size_t)3);
}
inline size_t ws_total_bytes(int B, int G, int R, int D, int ctas) {
    return ws_counter_bytes(B, G) + sizeof(float) * ws_slot_floats(R, D) * 2 * (size_t)ctas;
}

struct DecodeParams {
    const uint16_t* q;       // [B, sq, H, D] bf16 bits
    const int32_t* seq_lens; // [B]
    uint16_t* out;           // [B, sq, H, D] bf16 bits
    float* lse;              // [B, sq, H] or nullptr
    unsigned long long* ws_counters;  // [B*G][kMaxRowTiles] arrival counters
    float* ws_part;          // [ctas][2][slot]
    unsigned long long epoch;  // this call's tag in the counters (48 bits)
    unsigned* status;        // per-device status word (kStatus* bits)
    unsigned long long wait_timeout_ns;  // limit of every device-side wait
    float scale_log2;        // scale * log2(e)
    int B, sq, H, G, Tmax, R, heads_per_group, ctas;
    int even_rule;           // 1: with equal tile counts, even_ctas CTAs share the tiles
    int even_ctas;           // the CTAs of the equal-length rule (host-computed, see api.cu)
    int small_plan;          // 1: B <= 64 and B * G * ceil(Tmax / 64) < 2^31 (32-bit plan)
    int skip_tile;           // fault injection for tests: CTA 0 never loads its tile
                             // number skip_tile (-1: off), so its consumers' wait expires
    // Fused append (all null for a plain decode): the sq new tokens' K/V,
    // [B, sq, G, D] bf16, go to cache positions T_b - sq + s before attending.
    const uint16_t* k_new;
    const uint16_t* v_new;
    uint16_t* k_cache;       // the caches, for writing the new rows
    uint16_t* v_cache;
    // Paged caches (null block_table for a contiguous cache): K/V pages
    // [num_pages, G, page_size, D]; block_table [B, max_pages] maps logical
    // page j of sequence b to its physical page.
    const int32_t* block_table;
    int page_size, max_pages;
    // Pages shorter than a tile: the two extra warps issue the per-page TMA
    // boxes (half of a tile's pages each) instead of the producer alone.
    int page_loader;
    // fp8 caches (KV8 kernels): per (unit, 64-token tile) dequantisation
    // scales, [B*G][scale_tiles] fp32; element value = e4m3 code * scale.
    const float* k_scale;
    const float* v_scale;
    int scale_tiles;
};

// Prefill kernel parameters (one CTA per 128-row tile of one (b, g) unit).
struct PrefillParams {
    const uint16_t* q;        // [B, sq, H, D] bf16
    const int32_t* seq_lens;  // [B]
    uint16_t* out;            // [B, sq, H, D] bf16
    float* lse;               // [B, sq, H] or nullptr
    unsigned* status;         // per-device status word
    unsigned long long wait_timeout_ns;
    float scale_log2;
    int B, sq, H, G, Tmax, R, heads_per_group, row_tiles;
    int skip_tile;            // fault injection for tests (-1: off)
    // Split key ranges (short chunks): each pair of row tiles is shared by
    // `splits` CTAs over consecutive key ranges; with splits > 1 every CTA
    // writes per-row partials (O/l, m, l) to `ws_part` instead of out/lse,
    // and gqa_prefill_combine merges them.
    int splits;
    float* ws_part;           // [B*G][pairs][splits][2 tiles][128 rows][D + 4]: O, m, l, pad
};

// One CTA per SM. Every 16-row tile of the group has four consumer warps
// ("slices"); one more warp issues the TMA copies, (bf16) two more issue the
// boxes of pages shorter than a tile, and one tags the arrival counters. With
// two row tiles (12 warps) a thread gets 168 registers, so those warps keep
// their Q fragments in shared memory rather than in registers.
template <int D, int MT, bool KV8 = false>
struct KernelShape {
    // fp8 with one row tile: two groups of four consumer warps take
    // alternate tiles of each segment (a 16 KB fp8 stage is consumed at the
    // rate of a 32 KB bf16 one otherwise) and merge at the segment's end.
    static constexpr bool kDual = KV8 && MT == 1;
    // bf16 caches: "wide" slices. The four consumer warps of a row tile are
    // two groups that take alternate tiles of each segment, and a warp reads
    // 32 of its tile's 64 tokens (group = slice / 2, half = slice % 2): each Q
    // fragment then serves four n8 token tiles, and the softmax's reductions,
    // the stage wait and the arrival are paid once per 32 tokens. The four
    // warps still merge as four slices at the end of each segment.
    static constexpr bool kWide = !KV8;
    static constexpr int kGroups = (kDual || kWide) ? 2 : 1;
    // Tokens of a stage one consumer warp reads.
    static constexpr int kWarpTokens = kWide ? 32 : 16;
    static constexpr int kConsumerWarps = kSlices * MT * (kDual ? 2 : 1);
    // Consumer warps that read each stage (its "empty" barrier's count).
    static constexpr int kStageReaders = kConsumerWarps / kGroups;
    // bf16 caches: two more warps issue the TMA boxes of pages shorter than a
    // tile (DecodeParams::page_loader); they exit at once otherwise. They
    // cost no registers: the register file is allocated in steps of four
    // warps (5 -> 8 and 9 -> 12 either way).
    static constexpr int kLoaderWarps = KV8 ? 0 : 2;
    // The last warp gives the arrival counters of the CTA's partial units the
    // call's tag before any arrival (see the kernel). Every shape has a free
    // slot for it in its allocation step: 8 -> 8, 11 -> 12, 9 -> 10 of 12.
    static constexpr int kCounterWarp = kConsumerWarps + 1 + kLoaderWarps;
    static constexpr int kThreads = (kCounterWarp + 1) * 32;
    // Registers per thread: the 64K register file for one CTA, with warps
    // counted in the allocation steps of 4, in steps of 8 registers, <= 255.
    static constexpr int kAllocWarps = (kThreads / 32 + 3) / 4 * 4;
    static constexpr int kMaxRegs =
        (65536 / (kAllocWarps * 32)) / 8 * 8 > 255 ? 255 : (65536 / (kAllocWarps * 32)) / 8 * 8;
    static constexpr bool kQInSmem = MT > 1 || kDual;
    // One-round merges for up to 24 contributors where the register budget
    // allows (one row tile, bf16, D = 128: 5 warps, up to 255 registers; long
    // context B = 1 splits units about 19 ways); 8 elsewhere (at D = 64 the
    // larger merge raised the kernel from 167 to 245 registers and measured
    // slower on the tiny workload).
    static constexpr int kFastMerge = (kMaxRegs >= 240 && D == 128) ? 24 : ::gqa::kFastMerge;
    // bf16 at D = 128 with one row tile: with pages shorter than a tile the
    // stage is page-major (one 4-D box per page brings both 64-column blocks
    // of its rows). Two row tiles keep the block-major stage, whose block
    // offset is a constant (a runtime one cost them 3%), and one box per block.
    static constexpr bool kPageMajor = !KV8 && D == 128 && MT == 1;
    static constexpr int kQBytesPerWarp = kQInSmem ? 16 * D * 2 : 0;
    // K/V elements as stored in the cache: bf16, or fp8 e4m3 codes (KV8).
    static constexpr int kElemBytes = KV8 ? 1 : 2;
    static constexpr int kBoxElems = 128 / kElemBytes;        // elements per 128-byte box row
    static constexpr int kBoxes = D / kBoxElems;
    static constexpr int kTileBytes = kTileTokens * D * kElemBytes;   // K (or V) of one stage
    static constexpr int kStageBytes = 2 * kTileBytes;
    // Per row tile: the slice-merge buffer (3 slices x 16 x D floats), which
    // the cross-CTA merge reuses for a slot index, 16 maxima and 16 weights per
    // contributor.
    static constexpr int kMergeFloatsPerTile =
        (kSlices - 1) * 16 * D > kMaxMergeContrib * 33 ? (kSlices - 1) * 16 * D
                                                         : kMaxMergeContrib * 33;
    static constexpr int kMergeBytes = MT * kMergeFloatsPerTile * 4;
    static constexpr int kMlBytes = MT * kSlices * 16 * 2 * 4;
    static constexpr int kQBytes = kConsumerWarps * kQBytesPerWarp;
    // fp8 stages are half as large: twice as many keep the same bytes in flight.
    static constexpr int kStages = KV8 ? 8 : (D == 128 ? 4 : 8);
    // With groups on alternate tiles, a warp waits on tile t having read only
    // every other tile before it. Tile t - kStages, the stage's previous
    // load, must then be its own group's (read, hence landed, by this warp):
    // the copies of different stages land in any order, and a stage whose
    // previous load is still in flight shows the phase two loads back, whose
    // parity equals tile t's, so the wait would pass before tile t landed.
    // An even ring keeps tile t - kStages in the warp's own group (across a
    // segment boundary the segment-end merge barrier has seen every earlier
    // tile land).
    static_assert(kStages % kGroups == 0, "the ring depth must be a multiple of the groups");
    // Dual groups: group 1's per-lane state (m, l partials and the O
    // fragments of each slice) for group 0 to merge.
    static constexpr int kGroupBytes = kDual ? kSlices * 32 * (D / 8 * 4 + 4) * 4 : 0;
    // + 64: plan words, abort and last flags; + 128: the row table (32 rows).
    static constexpr int kBarBytes = 8 * (2 * kStages + 4 * MT + 2) + 64 + 128;
    // +1024 so the ring can be aligned to the 1 KB swizzle atom at run time.
    static constexpr int kSmemBytes =
        1024 + kStages * kStageBytes + kMergeBytes + kMlBytes + kQBytes + kGroupBytes + kBarBytes;
};

}  // namespace gqa
