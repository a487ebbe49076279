// Split-KV grouped-query decode attention kernel for sm_103a.
//
// One persistent CTA per SM. The K/V stream of every (sequence b, KV head g)
// unit is cut into 64-token tiles; the tiles of all units are laid end to end
// (b-major, then g, then position) and each CTA takes an equal contiguous
// share of that list. A CTA therefore walks one or more "segments" (runs of
// tiles of one unit). A segment that covers a whole unit is finished in the
// CTA and written straight to out/lse. A segment that covers part of a unit
// leaves a partial (O, m, l) in the workspace and counts itself on the unit's
// arrival counter; the CTA that arrives last merges the unit's partials with
// the log-sum-exp rescale and writes out/lse. One launch does the whole step.
//
// Inside a CTA one thread streams K and V tiles HBM -> shared memory with TMA
// tensor copies (128-byte swizzle, so the ldmatrix reads below are
// bank-conflict free) into a ring of mbarrier-guarded stages. All R = (H/G)*sq
// query rows of the unit's group sit in registers as the A operand of
// m16n8k16 bf16 tensor-core MMAs (one 16-row tile per group of four consumer
// warps), so each K/V byte is read from HBM once for the whole group -- "GQA
// analysis", section "Grouped broadcast": the group index selects the KV head
// and K/V are never copied per query head. The four consumer warps of a row
// tile split each 64-token stage 16 tokens apiece, run an online softmax in
// fp32 (base 2, running max and sum per row, quad shuffles), and merge their
// states through shared memory at the end of each segment.
#pragma once

#include <cstdint>

#include "gqa_common.h"
#include "gqa_device.cuh"
#include "ptx.cuh"

namespace gqa {

struct Segment {
    int b, g, tb;        // unit and its valid length (clamped)
    int t0;              // first tile of the segment within the unit
    int ntiles;          // tiles in the segment
    long long ub, ue;    // the unit's tile range in the flattened list
    bool complete;       // the segment covers the whole unit
    bool first;          // the CTA's first segment (partial slot 0, else slot 1)
};

// A compile-time int carried by a value (template arguments of generic lambdas).
template <int N>
struct IntC {
    static constexpr int value = N;
};

// Tiles of TT tokens covering tb valid tokens.
template <int TT = kTileTokens>
__device__ __forceinline__ long long tiles_of(int tb) { return (tb + TT - 1) / TT; }

// Walks the CTA's share [lo, hi) of the flattened list of TT-token tiles, one
// segment at a time. Every warp runs its own copy; they all see the same
// sequence.
template <int TT = kTileTokens>
struct SegmentWalkerT {
    const int32_t* seq_lens;
    int G, Tmax;
    long long x, lo, hi, pre_b;
    int b;

    __device__ bool next(Segment& s) {
        while (x < hi) {
            const int tb = clamp_len(__ldg(seq_lens + b), Tmax);
            const long long nt = tiles_of<TT>(tb);
            const long long span = nt * G;
            if (x >= pre_b + span) {
                pre_b += span;
                ++b;
                continue;
            }
            const long long off = x - pre_b;
            // 32-bit division when both fit (every workload here): a far
            // shorter instruction sequence than the 64-bit one.
            const int g = (off < (1ll << 31) && nt < (1ll << 31)) ? (int)off / (int)nt : (int)(off / nt);
            const long long ub = pre_b + (long long)g * nt, ue = ub + nt;
            const long long e = hi < ue ? hi : ue;
            s.b = b;
            s.g = g;
            s.tb = tb;
            s.t0 = (int)(x - ub);
            s.ntiles = (int)(e - x);
            s.ub = ub;
            s.ue = ue;
            s.complete = (x == ub) && (e == ue);
            s.first = (x == lo);
            x = e;
            return true;
        }
        return false;
    }
};
using SegmentWalker = SegmentWalkerT<>;

// Counts one arrival on a unit's counter and returns the arrivals so far in
// this call. The counter holds (epoch << 16) | count. An arrival adds one;
// when the tag it finds is this call's, the count it returns is exact in
// that one atomic. Otherwise the word is another call's (or bytes the
// workspace held before): the arrival then restarts the count under this
// call's tag, or counts itself once the tag is there, with compare-and-swap
// (its add on the old word is overwritten, and so not counted twice). So
// the workspace never needs clearing. A CAS only fails when another CTA
// changed the word, so the loop ends; it is bounded all the same.
__device__ __forceinline__ unsigned arrive_unit(unsigned long long* ctr, unsigned long long epoch,
                                                unsigned* status) {
    const unsigned long long old = atomicAdd(ctr, 1ull);
    if ((old >> 16) == epoch) return (unsigned)(old & 0xffffu) + 1u;
    unsigned long long cur = old + 1ull;
    for (int i = 0; i < (1 << 20); ++i) {
        const unsigned long long next = ((cur >> 16) == epoch) ? cur + 1 : ((epoch << 16) | 1ull);
        const unsigned long long prev = atomicCAS(ctr, cur, next);
        if (prev == cur) return (unsigned)(next & 0xffffu);
        cur = prev;
    }
    atomicOr(status, kStatusTimeout);
    return 0;
}

// Gives a unit's counter this call's tag with a zero count if it holds another
// tag, and leaves a word with this call's tag alone. It is not an arrival:
// an arrival whose add landed on the old word counts itself again under the
// new tag (arrive_unit), so overwriting that add loses nothing. Done early by
// the counter warp, it lets the arrivals at the segments' ends take the one-
// add path instead of contending in compare-and-swap loops. Bounded; if it
// gives up, the arrivals retag as before.
__device__ __forceinline__ void retag_unit(unsigned long long* ctr, unsigned long long epoch) {
    unsigned long long cur = *reinterpret_cast<volatile unsigned long long*>(ctr);
    for (int i = 0; i < 64 && (cur >> 16) != epoch; ++i) {
        const unsigned long long prev = atomicCAS(ctr, cur, epoch << 16);
        if (prev == cur) return;
        cur = prev;
    }
}

// The arrival that completes a unit's count sets the count back to zero
// under the call's tag: a launch replayed from a CUDA graph carries the tag
// of the call that was captured, so the next replay counts from zero, every
// arrival in one atomic. No other CTA of the launch touches the counter
// after the last arrival.
__device__ __forceinline__ void release_unit(unsigned long long* ctr, unsigned long long epoch) {
    atomicExch(ctr, epoch << 16);
}

// a / b for a >= 0, b > 0: the 32-bit unsigned division when both fit (every
// workload here), a far shorter instruction sequence than the 64-bit one.
__device__ __forceinline__ long long div_nonneg(long long a, long long b) {
    if (((unsigned long long)a | (unsigned long long)b) >> 32) return a / b;
    return (long long)((unsigned)a / (unsigned)b);
}

// The CTA holding tile x, and CTA c's share, for the equal partition of W
// tiles over P CTAs.
__device__ __forceinline__ long long cta_of_tile(long long x, long long W, long long P) {
    return div_nonneg((x + 1) * P - 1, W);
}

// CTAs that hold a share of the unit whose tiles are [ub, ue): with at least
// one tile per CTA every CTA from the first to the last holder; otherwise the
// non-empty shares among them are counted.
__device__ __forceinline__ unsigned unit_contributors(long long ub, long long ue, long long W, long long P) {
    const long long cf = cta_of_tile(ub, W, P), cl = cta_of_tile(ue - 1, W, P);
    if (W >= P) return (unsigned)(cl - cf + 1);
    unsigned n = 0;
    for (long long c = cf; c <= cl; ++c) n += div_nonneg(c * W, P) < div_nonneg((c + 1) * W, P) ? 1u : 0u;
    return n;
}

// Counts a unit's arrival for row tile mt; the arrival that completes the
// count resets the counter. Returns true for that (last) arrival.
__device__ __forceinline__ bool arrive_and_release(const DecodeParams& p, const Segment& s, int mt, long long W,
                                                   long long P) {
    unsigned long long* ctr = p.ws_counters + ((size_t)s.b * p.G + s.g) * kMaxRowTiles + mt;
    const unsigned contributors = unit_contributors(s.ub, s.ue, W, P);
    if (arrive_unit(ctr, p.epoch, p.status) != contributors) return false;
    release_unit(ctr, p.epoch);
    return true;
}

// Byte offset of row r (0..63), 64-column block bx, in a stage of a cache
// with P = 2^lp rows per TMA box (P = 64, one box per tile, or the page size
// of a paged cache with shorter pages): boxes of P rows are laid out one
// after the other, each as [block][row][128 B], with the 128-byte swizzle
// applied by the caller on the 16-byte chunk. At lp = 6 this is
// [block][64 rows][128 B].
template <int NB>
__device__ __forceinline__ uint32_t stage_off(int r, int bx, int lp) {
    return (uint32_t)((((r >> lp) * NB + bx) << (lp + 7)) + ((r & ((1 << lp) - 1)) << 7));
}

// The same for a kernel shape: page-major stages (KernelShape::kPageMajor)
// take lp at run time; the others are always [block][64 rows][128 B], with
// the block offset a constant.
template <class KS>
__device__ __forceinline__ uint32_t stage_row_off(int r, int bx, int lp) {
    if constexpr (KS::kPageMajor) return stage_off<KS::kBoxes>(r, bx, lp);
    else return (uint32_t)(bx * (kTileTokens * 128) + r * 128);
}

// One tile of the CTA's share, with where its rows live. For a paged cache a
// 64-token tile covers part of one page (pages of >= 64 tokens) or
// 64 / page_size whole pages; `page` holds their physical numbers (pages that
// start at or past the sequence's length are not looked up and stay -1).
struct TileRef {
    int unit, g, tb, t;      // unit = b*G + g; t = tile index within the unit
    int page[4];
};

// Hands out the CTA's tiles in order and issues their TMA copies into the
// ring: stage it % S, armed on full[it % S] once empty[it % S] shows that the
// consumers are done with the tile S places earlier. The next tile is looked
// up one step ahead, so that its block-table reads (paged caches) are in
// flight while the producer waits for a free stage.
template <int D, int MT, int S, bool KV8>
struct TileIssuer {
    SegmentWalker walk;
    Segment sg;
    int i = 0;
    bool have = false;
    uint32_t issued = 0;  // tiles handed out so far (== index of the next)
    TileRef cur;
    bool have_cur = false;
    int part = 0, nparts = 1;   // short pages: this issuer's pages of a tile are j % nparts == part

    __device__ bool next(const DecodeParams& p, TileRef& r) {
        while (!have || i >= sg.ntiles) {
            if (!walk.next(sg)) return false;
            have = true;
            i = 0;
        }
        r.unit = sg.b * walk.G + sg.g;
        r.g = sg.g;
        r.tb = sg.tb;
        r.t = sg.t0 + i;
        ++i;
        r.page[0] = r.page[1] = r.page[2] = r.page[3] = -1;
        if (p.block_table != nullptr) {
            const int32_t* bt = p.block_table + (size_t)sg.b * p.max_pages;
            const int tok0 = r.t * kTileTokens;
            if (p.page_size >= kTileTokens) {
                r.page[0] = __ldg(bt + tok0 / p.page_size);
            } else {
                const int n = kTileTokens / p.page_size;   // 2 or 4 pages of 32 or 16 tokens
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    if (j < n && tok0 + j * p.page_size < r.tb) r.page[j] = __ldg(bt + tok0 / p.page_size + j);
            }
        }
        return true;
    }

    __device__ void start(const DecodeParams& p) { have_cur = next(p, cur); }

    // Issues the current tile, if any, once its stage is free, and looks up
    // the one after it. Returns false when a wait gave up.
    __device__ bool issue_one(uint32_t ring, uint32_t full_bar, uint32_t empty_bar,
                              const CUtensorMap* tm_k, const CUtensorMap* tm_v, const DecodeParams& p,
                              volatile int* abort_flag, bool& done) {
        if (!have_cur) {
            done = true;
            return true;
        }
        const TileRef r = cur;
        const uint32_t it = issued;
        const int s = it % S;
        if (!wait_phase(empty_bar + 8 * s, ((it / S) & 1) ^ 1, abort_flag, p.status, p.wait_timeout_ns))
            return false;
        issued = it + 1;
        issue_copies(r, s, ring, full_bar, tm_k, tm_v, p, it);
        // Look the next tile up now: its block-table reads are in flight
        // while the producer waits for the next free stage.
        have_cur = next(p, cur);
        return true;
    }

    __device__ void issue_copies(const TileRef& r, int s, uint32_t ring, uint32_t full_bar,
                                 const CUtensorMap* tm_k, const CUtensorMap* tm_v,
                                 const DecodeParams& p, uint32_t it) {
        if (blockIdx.x == 0 && (int)it == p.skip_tile) return;  // injected fault
        using KS = KernelShape<D, MT, KV8>;
        constexpr int kStageBytes = KS::kStageBytes;
        constexpr int kTileBytes = KS::kTileBytes;
        constexpr int NB = KS::kBoxes;
        constexpr int kBoxCols = KS::kBoxElems;
        const uint32_t fb = full_bar + 8 * s;
        // K and V are read once per launch: evict-first in L2, so the
        // lengths, Q, block tables and partials stay (ragged sq = 4 615.6 ->
        // 609.7 us, MQA end 49.1 -> 48.8 us).
        const uint64_t pol = l2_policy_evict_first();
        const uint32_t kdst = ring + s * kStageBytes;
        const uint32_t vdst = kdst + kTileBytes;
        if (p.block_table == nullptr) {
            mbar_arrive_expect_tx(fb, kStageBytes);
            const int y = r.t * kTileTokens;
#pragma unroll
            for (int bx = 0; bx < NB; ++bx) {
                tma_load_3d_hint(kdst + bx * (kTileTokens * 128), tm_k, fb, bx * kBoxCols, y, r.unit, pol);
                tma_load_3d_hint(vdst + bx * (kTileTokens * 128), tm_v, fb, bx * kBoxCols, y, r.unit, pol);
            }
        } else if (p.page_size >= kTileTokens) {
            // One box of 64 rows inside page r.page[0]: tensor map [D, page_size, pages*G].
            mbar_arrive_expect_tx(fb, kStageBytes);
            const int y = (r.t * kTileTokens) % p.page_size;
            const int z = r.page[0] * p.G + r.g;
#pragma unroll
            for (int bx = 0; bx < NB; ++bx) {
                tma_load_3d_hint(kdst + bx * (kTileTokens * 128), tm_k, fb, bx * kBoxCols, y, z, pol);
                tma_load_3d_hint(vdst + bx * (kTileTokens * 128), tm_v, fb, bx * kBoxCols, y, z, pol);
            }
        } else {
            // One box of page_size rows per page that starts before the end of
            // the sequence, at that page's place in the stage (stage_off with
            // P = page_size); rows past the length are never used (masked, and
            // zeroed in V), so the pages after the last one are not read.
            const int ps = p.page_size;
            int npages = 0;
#pragma unroll
            for (int j = 0; j < 4; ++j) npages += (r.page[j] >= 0 && j % nparts == part) ? 1 : 0;
            mbar_arrive_expect_tx(fb, (uint32_t)npages * NB * ps * 128 * 2);  // paged: bf16 only
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                if (r.page[j] < 0 || j % nparts != part) continue;
                const int z = r.page[j] * p.G + r.g;
                // Page j's rows at stage_off(j * ps, 0, lp).
                const uint32_t off = (uint32_t)(j * (KS::kPageMajor ? NB : 1) * ps * 128);
                // Page-major stage (KernelShape::kPageMajor): the tensor map is
                // 4-D and one box brings both 64-column blocks of the page's
                // rows (per-box overhead, not bytes, bounds these short
                // copies); else one box per block.
                if constexpr (KS::kPageMajor) {
                    tma_load_4d_hint(kdst + off, tm_k, fb, 0, 0, 0, z, pol);
                    tma_load_4d_hint(vdst + off, tm_v, fb, 0, 0, 0, z, pol);
                } else {
#pragma unroll
                    for (int bx = 0; bx < NB; ++bx) {
                        tma_load_3d_hint(kdst + off + bx * (kTileTokens * 128), tm_k, fb, bx * kBoxCols, 0, z, pol);
                        tma_load_3d_hint(vdst + off + bx * (kTileTokens * 128), tm_v, fb, bx * kBoxCols, 0, z, pol);
                    }
                }
            }
        }
    }

    // Waits (bounded) until the copies of tiles [consumed, issued) have landed,
    // so that the CTA never exits with a copy into its shared memory in flight.
    __device__ void drain(uint32_t consumed, uint32_t full_bar, const DecodeParams& p) {
        for (uint32_t j = consumed; j < issued; ++j) {
            if (blockIdx.x == 0 && (int)j == p.skip_tile) continue;
            const uint64_t t0 = global_timer_ns();
            while (!mbar_try_wait(full_bar + 8 * (j % S), (j / S) & 1)) {
                if (global_timer_ns() - t0 > p.wait_timeout_ns) {
                    atomicOr(p.status, kStatusTimeout);
                    break;
                }
            }
        }
    }
};

// One warp: total tiles W (of TT tokens), the number of CTAs that share
// them, and where this CTA's share starts, into shared_ll[0..3] = W, first
// sequence, tiles before it, P. Lengths are read once; lane i keeps
// sequences i, i+32, ... of the first 256.
//
// When every unit has the same number of tiles (all lengths equal), the
// tiles are shared by p.even_ctas CTAs (the host's equal-length rule: a
// grid that lines up with the units); the CTAs left over exit.
// plan_share for up to 64 sequences and fewer than 2^31 tiles in all
// (DecodeParams::small_plan, set by the host from B and B * G *
// ceil(Tmax / 64)): lane i holds sequences i and i + 32, and every sum is a
// 32-bit scan. Same result as plan_share; it exists because every kernel
// launch pays for the plan before its first copy, so the plan is kept short.
template <int TT>
__device__ __forceinline__ void plan_share_small(const DecodeParams& p, int lane, long long* shared_ll) {
    const bool has0 = lane < p.B, has1 = lane + 32 < p.B;
    const int n0 = has0 ? (int)tiles_of<TT>(clamp_len(__ldg(p.seq_lens + lane), p.Tmax)) : 0;
    const int n1 = has1 ? (int)tiles_of<TT>(clamp_len(__ldg(p.seq_lens + lane + 32), p.Tmax)) : 0;
    const int v0 = n0 * p.G, v1 = n1 * p.G;
    int s0 = v0, s1 = v1;   // inclusive scans over the lanes
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int u0 = __shfl_up_sync(0xffffffffu, s0, o), u1 = __shfl_up_sync(0xffffffffu, s1, o);
        if (lane >= o) {
            s0 += u0;
            s1 += u1;
        }
    }
    const int tot0 = __shfl_sync(0xffffffffu, s0, 31);
    const int total = tot0 + __shfl_sync(0xffffffffu, s1, 31);
    const unsigned big = 0x7fffffffu;
    const int nt_min = (int)__reduce_min_sync(0xffffffffu, min(has0 ? (unsigned)n0 : big, has1 ? (unsigned)n1 : big));
    const int nt_max = (int)__reduce_max_sync(0xffffffffu, (unsigned)max(n0, n1));
    const int P = (p.even_rule && nt_min == nt_max && nt_max > 0) ? p.even_ctas : p.ctas;
    int bstart = p.B, prestart = total;
    if ((int)blockIdx.x < P) {
        const int lo = (int)div_nonneg((long long)blockIdx.x * total, P);
        const unsigned hit0 = __ballot_sync(0xffffffffu, has0 && s0 > lo);
        const unsigned hit1 = __ballot_sync(0xffffffffu, has1 && tot0 + s1 > lo);
        if (hit0) {
            const int src = __ffs(hit0) - 1;
            bstart = src;
            prestart = __shfl_sync(0xffffffffu, s0 - v0, src);
        } else if (hit1) {
            const int src = __ffs(hit1) - 1;
            bstart = 32 + src;
            prestart = tot0 + __shfl_sync(0xffffffffu, s1 - v1, src);
        }
    }
    if (lane == 0) {
        shared_ll[0] = total;
        shared_ll[1] = bstart;
        shared_ll[2] = prestart;
        shared_ll[3] = P;
    }
}

template <int TT>
__device__ __forceinline__ void plan_share(const DecodeParams& p, int lane, long long* shared_ll) {
    constexpr int kCached = 8;       // sequences 0..255 stay in registers
    long long cached[kCached];
    long long total = 0;
    int nt_min = 0x7fffffff, nt_max = 0;
    auto tiles_times_g = [&](int b) -> long long {
        if (b >= p.B) return 0;
        const int nt = (int)tiles_of<TT>(clamp_len(__ldg(p.seq_lens + b), p.Tmax));
        nt_min = min(nt_min, nt);
        nt_max = max(nt_max, nt);
        return (long long)nt * p.G;
    };
    auto scan_add = [&](long long v) {
        long long incl = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const long long n = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += n;
        }
        return incl;
    };
#pragma unroll
    for (int k = 0; k < kCached; ++k) {
        cached[k] = 0;
        if (k * 32 < p.B) {
            cached[k] = tiles_times_g(k * 32 + lane);
            long long sum = cached[k];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
            total += sum;
        }
    }
    for (int b0 = kCached * 32; b0 < p.B; b0 += 32)
        total += __shfl_sync(0xffffffffu, scan_add(tiles_times_g(b0 + lane)), 31);
    nt_min = __reduce_min_sync(0xffffffffu, nt_min);
    nt_max = __reduce_max_sync(0xffffffffu, nt_max);
    const long long P = (p.even_rule && nt_min == nt_max && nt_max > 0) ? p.even_ctas : p.ctas;
    // First sequence whose tiles reach past lo, and the tiles before it.
    const long long lo = (long long)blockIdx.x * total / P;
    long long pre = 0;
    int bstart = p.B;
    long long prestart = total;
    bool found = (long long)blockIdx.x >= P;
    auto find = [&](int b0, long long v) {
        const long long incl = scan_add(v);
        const unsigned hit = __ballot_sync(0xffffffffu, b0 + lane < p.B && pre + incl > lo);
        if (hit) {
            const int src = __ffs(hit) - 1;
            bstart = b0 + src;
            prestart = pre + __shfl_sync(0xffffffffu, incl - v, src);
            found = true;
        } else {
            pre += __shfl_sync(0xffffffffu, incl, 31);
        }
    };
#pragma unroll
    for (int k = 0; k < kCached; ++k)
        if (!found && k * 32 < p.B) find(k * 32, cached[k]);
    for (int b0 = kCached * 32; !found && b0 < p.B; b0 += 32) find(b0, tiles_times_g(b0 + lane));
    if (lane == 0) {
        shared_ll[0] = total;
        shared_ll[1] = bstart;
        shared_ll[2] = prestart;
        shared_ll[3] = P;
    }
}

template <int D, int MT, bool KV8>
__global__ void __maxnreg__((KernelShape<D, MT, KV8>::kMaxRegs))
    gqa_splitkv_kernel(const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const DecodeParams p) {
    using KS = KernelShape<D, MT, KV8>;
    constexpr int S = KS::kStages;
    constexpr int KSTEPS = D / 16;   // k16 steps of Q.K^T
    constexpr int NTILE_D = D / 8;   // n8 tiles of P.V (columns of O)
    constexpr bool kQs = KS::kQInSmem;

    extern __shared__ __align__(1024) unsigned char smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t ring = (raw + 1023u) & ~1023u;
    unsigned char* ring_ptr = smem_raw + (ring - raw);
    float* merge_buf = reinterpret_cast<float*>(ring_ptr + S * KS::kStageBytes);
    float* ml_buf = merge_buf + KS::kMergeBytes / 4;
    unsigned char* q_smem = reinterpret_cast<unsigned char*>(ml_buf + KS::kMlBytes / 4);
    float* group_buf = reinterpret_cast<float*>(q_smem + KS::kQBytes);   // dual groups only
    uint64_t* bars = reinterpret_cast<uint64_t*>(q_smem + KS::kQBytes + KS::kGroupBytes);
    const uint32_t full_bar = smem_addr(bars);
    const uint32_t empty_bar = full_bar + 8 * S;
    const uint32_t merge_bar = empty_bar + 8 * S;          // [MT][4]: A, B, C, D
    const uint32_t group_bar = merge_bar + 8 * 4 * MT;     // E, F (dual groups)
    long long* shared_ll = reinterpret_cast<long long*>(bars + 2 * S + 4 * MT + 2);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(shared_ll + 4);
    volatile int* last_flag = abort_flag + 1;              // [MT]
    // Row r of a KV head's R rows: (new token s << 16) | head j within the
    // group, r = j * sq + s; written once so that no segment divides by sq.
    int* rowtab = reinterpret_cast<int*>(shared_ll + 8);   // [kMaxRowTiles * 16]

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const bool is_producer = warp == KS::kConsumerWarps;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            // One arrival with the copy's bytes, or one per issuer (page_loader).
            mbar_init(full_bar + 8 * s, p.page_loader ? KS::kLoaderWarps : 1);
            // Each stage is read by the warps of one group.
            mbar_init(empty_bar + 8 * s, KS::kStageReaders);
        }
        for (int m = 0; m < 4 * MT; ++m) mbar_init(merge_bar + 8 * m, kSlices * 32);
        mbar_init(group_bar, KS::kConsumerWarps * 32);
        mbar_init(group_bar + 8, KS::kConsumerWarps * 32);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (threadIdx.x == KS::kConsumerWarps * 32) {
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
    }
    if (threadIdx.x >= 32 && threadIdx.x < 32 + p.R) {
        const int r = threadIdx.x - 32;
        rowtab[r] = ((r % p.sq) << 16) | (r / p.sq);
    }
    // Inputs may be written by the previous grid in the stream.
    pdl_wait_primary();

    // Warp 0: this CTA's share of the tiles (plan_share).
    if (warp == 0) {
        if (p.small_plan)
            plan_share_small<kTileTokens>(p, lane, shared_ll);
        else
            plan_share<kTileTokens>(p, lane, shared_ll);
    }
    __syncthreads();
    pdl_launch_dependents();

    const long long W = shared_ll[0];
    const long long P = shared_ll[3];   // CTAs sharing the tiles (<= gridDim.x)
    SegmentWalker walk;
    walk.seq_lens = p.seq_lens;
    walk.G = p.G;
    walk.Tmax = p.Tmax;
    walk.lo = (long long)blockIdx.x < P ? div_nonneg((long long)blockIdx.x * W, P) : W;
    walk.hi = (long long)blockIdx.x < P ? div_nonneg((long long)(blockIdx.x + 1) * W, P) : W;
    walk.x = walk.lo;
    walk.b = (int)shared_ll[1];
    walk.pre_b = shared_ll[2];

    if (warp == KS::kCounterWarp) {
        // ------------------------------------------ counter warp
        // Before the first segment ends, the counters of every partial unit
        // of this CTA's share (lane mt: row tile mt's) get this call's tag.
        // Without it the first arrivals of a unit each found the previous
        // call's tag and retagged in a compare-and-swap loop: with 16-19
        // CTAs a unit arriving together (long context B = 1) that chain of
        // retries took up to 10 us.
        if (lane < MT) {
            SegmentWalker w = walk;
            Segment sg;
            while (w.next(sg))
                if (!sg.complete)
                    retag_unit(p.ws_counters + ((size_t)sg.b * p.G + sg.g) * kMaxRowTiles + lane, p.epoch);
        }
        return;
    }

    if (warp > KS::kConsumerWarps) {
        // ------------------------------------------ second and third issuers
        // Pages shorter than a tile: the per-page TMA boxes of a tile (up to
        // four pages each of K and V) are issued by these two warps' first
        // lanes, each for half of the pages, and each arrives on the stage's
        // full barrier with its own bytes. One thread issuing them all was the
        // limit at 16-token pages (68.5 -> 63.8 us on the Llama-shaped layer).
        if constexpr (KS::kLoaderWarps > 0) {
            if (!p.page_loader || lane != 0) return;
            TileIssuer<D, MT, S, KV8> issuer;
            issuer.walk = walk;
            issuer.part = warp - KS::kConsumerWarps - 1;
            issuer.nparts = KS::kLoaderWarps;
            issuer.start(p);
            bool done = false;
            while (!done)
                if (!issuer.issue_one(ring, full_bar, empty_bar, &tm_k, &tm_v, p, abort_flag, done)) break;
            issuer.drain(issuer.issued > (uint32_t)S ? issuer.issued - S : 0, full_bar, p);
        }
        return;
    }

    if (is_producer) {
        // ------------------------------------------ dedicated producer warp
        if (lane != 0 || p.page_loader) return;
        TileIssuer<D, MT, S, KV8> issuer;
        issuer.walk = walk;
        issuer.start(p);
        bool done = false;
        while (!done)
            if (!issuer.issue_one(ring, full_bar, empty_bar, &tm_k, &tm_v, p, abort_flag, done)) break;
        // Every tile but the last S was waited on through its stage's empty
        // barrier; leave only once the copies of those last S have landed.
        issuer.drain(issuer.issued > (uint32_t)S ? issuer.issued - S : 0, full_bar, p);
        return;
    }

    // ---------------------------------------------------------- consumers
    const int slice = warp % kSlices;
    const int mt = KS::kDual ? 0 : warp / kSlices;
    // Groups take alternate tiles: the fp8 kernel's dual groups (warps 0-3 and
    // 4-7), or the two halves of a row tile's warps (wide slices).
    const int group = KS::kDual ? warp / kSlices : (KS::kWide ? slice >> 1 : 0);
    const int quad = lane & 3;
    const int grp = lane >> 2;
    const int tid_mt = slice * 32 + lane;                   // 0..127 within the row tile
    const uint32_t mbarA = merge_bar + 8 * (4 * mt);
    const uint32_t mbarB = mbarA + 8;
    const uint32_t mbarC = mbarA + 16;
    const uint32_t mbarD = mbarA + 24;
    float* my_merge = merge_buf + mt * KS::kMergeFloatsPerTile;
    float* my_ml = ml_buf + mt * kSlices * 16 * 2;
    const size_t slot_floats = ws_slot_floats(p.R, D);
    const uint64_t tmo = p.wait_timeout_ns;

    // This warp's tokens of a stage: [tok0, tok0 + kWarpTokens).
    constexpr int WT = KS::kWarpTokens;
    constexpr int NJ = WT / 8;   // n8 token tiles of the warp's S
    const int tok0 = KS::kWide ? (slice & 1) * WT : slice * WT;
    // ldmatrix row addressing inside a stage (bytes from the stage base), for
    // the warp's first 16 tokens (16 * jj more for the jj-th 16).
    // Q.K^T (B operand, non-transposed): matrix m = lane/8 -> n8 tile (m>>1),
    // k half (m&1); row = token.
    const int k_tok = tok0 + ((lane >> 4) << 3) + (lane & 7);
    const int k_half = (lane >> 3) & 1;
    // P.V (B operand, transposed): matrix m -> d tile (m>>1), token half (m&1).
    const int v_tok = tok0 + (((lane >> 3) & 1) << 3) + (lane & 7);
    const int v_dt = lane >> 4;
    // e4m3 K and V (one byte per element, one 128-byte box row per token):
    // matrix m -> tokens 8*(m&1).., 16-byte chunk + (m>>1).
    const int k8_tok = v_tok;
    // Stage layout (stage_row_off): boxes of 2^lp rows -- the page size for a
    // paged cache with pages shorter than a tile, else the whole tile.
    const int lp = (KS::kPageMajor && p.block_table != nullptr && p.page_size < kTileTokens)
                       ? 31 - __clz(p.page_size) : 6;
    // Block 1 of a row sits 2^(lp+7) bytes after block 0 (stage_off).
    uint32_t k_off0[NJ / 2], v_off0[NJ / 2];
#pragma unroll
    for (int jj = 0; jj < NJ / 2; ++jj) {
        k_off0[jj] = stage_row_off<KS>(k_tok + 16 * jj, 0, lp);
        v_off0[jj] = stage_row_off<KS>(v_tok + 16 * jj, 0, lp);
    }
    const uint32_t bx_stride = KS::kPageMajor ? 1u << (lp + 7) : kTileTokens * 128;

    uint32_t it_base = 0;      // tiles of this CTA's earlier segments
    uint32_t e_parity = 0;     // phases of group barriers E and F (dual groups)
    uint32_t seg_parity = 0;   // phases of merge barriers A and B (every segment)
    uint32_t c_parity = 0;     // phases of merge barrier C (partial segments)
    uint32_t d_parity = 0;     // phases of merge barrier D (merges)
    bool failed = false;
    bool arrived_here = false;   // lane 0 of a row tile's slice 0: this segment's arrival counted
    Segment sg;
    while (!failed && walk.next(sg)) {
        arrived_here = false;
        // Rows of this warp's 16-row tile: r = j*sq + s (head j of the group,
        // new token s), the row fold of section 7 of "Same GQA, Different
        // Execution Cost Across Backends".
        const int r_lo = mt * 16 + grp, r_hi = r_lo + 8;
        int lim_lo = sg.tb - 1, lim_hi = sg.tb - 1;
        int out_lo = -1, out_hi = -1;  // flat (b, s, h) row index for output
        uint32_t qa[kQs ? 1 : KSTEPS][4];
        {
            const uint16_t* q_lo = nullptr;
            const uint16_t* q_hi = nullptr;
            if (r_lo < p.R) {
                const int e = rowtab[r_lo], j = e & 0xffff, s = e >> 16;
                out_lo = (sg.b * p.sq + s) * p.H + sg.g * p.heads_per_group + j;
                q_lo = p.q + (size_t)out_lo * D;
                lim_lo = sg.tb - p.sq + s;
            }
            if (r_hi < p.R) {
                const int e = rowtab[r_hi], j = e & 0xffff, s = e >> 16;
                out_hi = (sg.b * p.sq + s) * p.H + sg.g * p.heads_per_group + j;
                q_hi = p.q + (size_t)out_hi * D;
                lim_hi = sg.tb - p.sq + s;
            }
            if constexpr (!kQs) {
#pragma unroll
                for (int kk = 0; kk < KSTEPS; ++kk) {
                    if constexpr (KV8) {
                        // fp16 MMAs (Q converted exactly within fp16's range),
                        // with the k order of the e4m3 K fragments: this thread's
                        // k slots 2q, 2q+1 | 2q+8, 2q+9 hold d = 4q, 4q+1 | 4q+2,
                        // 4q+3 of the step's 16 (the dot product is the same sum
                        // in another order).
                        const int c = kk * 16 + 4 * quad;
                        const uint2 lo = q_lo ? __ldg(reinterpret_cast<const uint2*>(q_lo + c)) : make_uint2(0u, 0u);
                        const uint2 hi = q_hi ? __ldg(reinterpret_cast<const uint2*>(q_hi + c)) : make_uint2(0u, 0u);
                        qa[kk][0] = bf16x2_to_f16x2(lo.x);
                        qa[kk][2] = bf16x2_to_f16x2(lo.y);
                        qa[kk][1] = bf16x2_to_f16x2(hi.x);
                        qa[kk][3] = bf16x2_to_f16x2(hi.y);
                    } else {
                        const int c = kk * 16 + 2 * quad;
                        qa[kk][0] = q_lo ? __ldg(reinterpret_cast<const unsigned*>(q_lo + c)) : 0u;
                        qa[kk][1] = q_hi ? __ldg(reinterpret_cast<const unsigned*>(q_hi + c)) : 0u;
                        qa[kk][2] = q_lo ? __ldg(reinterpret_cast<const unsigned*>(q_lo + c + 8)) : 0u;
                        qa[kk][3] = q_hi ? __ldg(reinterpret_cast<const unsigned*>(q_hi + c + 8)) : 0u;
                    }
                }
            } else {
                // This warp's 16 Q rows into its own shared-memory copy, 16-byte
                // chunks swizzled by row so that ldmatrix reads are conflict free.
                // Every load is issued before the first store: one global round
                // trip per segment, not one per chunk.
                unsigned char* qw = q_smem + warp * KS::kQBytesPerWarp;
                if constexpr (KV8) {
                    // fp16, each 16-wide k step stored as the A fragments of the
                    // e4m3 k order: chunk 2c holds d {0,1,4,5,8,9,12,13} of step
                    // c, chunk 2c+1 d {2,3,6,7,10,11,14,15}.
                    constexpr int kIters = 16 * (D / 16) / 32;
                    uint4 qa4[kIters], qb4[kIters];
#pragma unroll
                    for (int u = 0; u < kIters; ++u) {
                        const int idx = lane + 32 * u;
                        const int row = idx / (D / 16), c16 = idx % (D / 16);
                        const int r = mt * 16 + row;
                        qa4[u] = make_uint4(0u, 0u, 0u, 0u);
                        qb4[u] = qa4[u];
                        if (r < p.R) {
                            const int e = rowtab[r], j = e & 0xffff, sq_i = e >> 16;
                            const int qrow = (sg.b * p.sq + sq_i) * p.H + sg.g * p.heads_per_group + j;
                            const uint4* src = reinterpret_cast<const uint4*>(p.q + (size_t)qrow * D) + 2 * c16;
                            qa4[u] = __ldg(src);
                            qb4[u] = __ldg(src + 1);
                        }
                    }
#pragma unroll
                    for (int u = 0; u < kIters; ++u) {
                        const int idx = lane + 32 * u;
                        const int row = idx / (D / 16), c16 = idx % (D / 16);
                        const uint4 a = qa4[u], b = qb4[u];
                        const uint4 ev = make_uint4(bf16x2_to_f16x2(a.x), bf16x2_to_f16x2(a.z),
                                                    bf16x2_to_f16x2(b.x), bf16x2_to_f16x2(b.z));
                        const uint4 od = make_uint4(bf16x2_to_f16x2(a.y), bf16x2_to_f16x2(a.w),
                                                    bf16x2_to_f16x2(b.y), bf16x2_to_f16x2(b.w));
                        *reinterpret_cast<uint4*>(qw + row * (D * 2) + (((2 * c16) ^ (row & 7)) << 4)) = ev;
                        *reinterpret_cast<uint4*>(qw + row * (D * 2) + (((2 * c16 + 1) ^ (row & 7)) << 4)) = od;
                    }
                } else {
                    constexpr int kIters = 16 * (D / 8) / 32;
                    uint4 v[kIters];
#pragma unroll
                    for (int u = 0; u < kIters; ++u) {
                        const int idx = lane + 32 * u;
                        const int row = idx / (D / 8), chunk = idx % (D / 8);
                        const int r = mt * 16 + row;
                        v[u] = make_uint4(0u, 0u, 0u, 0u);
                        if (r < p.R) {
                            const int e = rowtab[r], j = e & 0xffff, sq_i = e >> 16;
                            const int qrow = (sg.b * p.sq + sq_i) * p.H + sg.g * p.heads_per_group + j;
                            v[u] = __ldg(reinterpret_cast<const uint4*>(p.q + (size_t)qrow * D) + chunk);
                        }
                    }
#pragma unroll
                    for (int u = 0; u < kIters; ++u) {
                        const int idx = lane + 32 * u;
                        const int row = idx / (D / 8), chunk = idx % (D / 8);
                        *reinterpret_cast<uint4*>(qw + row * (D * 2) + ((chunk ^ (row & 7)) << 4)) = v[u];
                    }
                }
                __syncwarp();
            }
        }
        // ldmatrix of the A fragment (rows 0-7 / 8-15, k 0-7 / 8-15) of step kk.
        const int qa_row = (lane & 7) + (((lane >> 3) & 1) << 3);
        const uint32_t qa_base = smem_addr(q_smem) + warp * KS::kQBytesPerWarp + qa_row * (D * 2);
        // Tiles that end at or before every row's last visible key need no mask.
        const int lim_min = __reduce_min_sync(0xffffffffu, min(lim_lo, lim_hi));

        float m_lo = -INFINITY, m_hi = -INFINITY, l_lo = 0.f, l_hi = 0.f;
        float o[NTILE_D][4];
#pragma unroll
        for (int n = 0; n < NTILE_D; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;

        // KV8: the dequantisation scales of this unit's tiles, read one tile
        // ahead of use so that their latency hides behind the current tile.
        const size_t scale_row = ((size_t)sg.b * p.G + sg.g) * p.scale_tiles;
        float ks_next = 1.f, vs_next = 1.f;
        if constexpr (KV8) {
            if (group < sg.ntiles) {
                ks_next = __ldg(p.k_scale + scale_row + sg.t0 + group);
                vs_next = __ldg(p.v_scale + scale_row + sg.t0 + group);
            }
        }

        // Dual groups take alternate tiles of the segment; otherwise every
        // consumer warp reads every tile.
        for (int i = group; i < sg.ntiles; i += KS::kGroups) {
            const uint32_t it = it_base + i;
            const int s = it % S;
            const float ks = ks_next, vs = vs_next;
            if constexpr (KV8) {
                if (i + KS::kGroups < sg.ntiles) {
                    ks_next = __ldg(p.k_scale + scale_row + sg.t0 + i + KS::kGroups);
                    vs_next = __ldg(p.v_scale + scale_row + sg.t0 + i + KS::kGroups);
                }
            }
            if (!wait_phase(full_bar + 8 * s, (it / S) & 1, abort_flag, p.status, tmo)) {
                failed = true;
                break;
            }
            const uint32_t kst = ring + s * KS::kStageBytes;
            const uint32_t vst = kst + KS::kTileBytes;
            const int tbase = (sg.t0 + i) * kTileTokens;

            // Rows past the valid length may hold anything (NaN included);
            // zero them in V so that p = 0 times them stays 0.
            if (tbase + kTileTokens > sg.tb) {
                constexpr int kChunks = D * KS::kElemBytes / 16;   // 16-byte chunks per row
                bool wrote = false;
                for (int idx = lane; idx < WT * kChunks; idx += 32) {
                    const int row = tok0 + idx / kChunks;
                    const int chunk = idx % kChunks;
                    if (tbase + row >= sg.tb) {
                        const int bx = chunk >> 3, cc = chunk & 7;
                        st_shared_zero16(vst + stage_row_off<KS>(row, bx, lp) + ((cc ^ (row & 7)) << 4));
                        wrote = true;
                    }
                }
                if (wrote) fence_proxy_async_smem();
                __syncwarp();
            }

            // Fused append: the new tokens' rows of this warp's slice
            // come from k_new/v_new, not from the cache the TMA just read. The
            // warp patches them into the stage before reading it and (one row
            // tile's warp) stores them to the cache. Each position lies in
            // exactly one tile, which one CTA owns, so no other CTA reads it.
            if (!KV8 && p.k_new != nullptr) {
                const int new_lo = sg.tb - p.sq;
                const int lo = max(new_lo, tbase + tok0);
                const int hi = min(sg.tb, tbase + tok0 + WT);
                if (lo < hi) {
                    const size_t unit_row0 = ((size_t)sg.b * p.G + sg.g) * p.Tmax;
                    for (int idx = lane; idx < (hi - lo) * (D / 8); idx += 32) {
                        const int t = lo + idx / (D / 8);
                        const int chunk = idx % (D / 8);
                        const size_t src = (((size_t)sg.b * p.sq + (t - new_lo)) * p.G + sg.g) * D + chunk * 8;
                        const uint4 kv = __ldg(reinterpret_cast<const uint4*>(p.k_new + src));
                        const uint4 vv = __ldg(reinterpret_cast<const uint4*>(p.v_new + src));
                        const int row = t - tbase;
                        const uint32_t off = stage_row_off<KS>(row, chunk >> 3, lp) + (((chunk & 7) ^ (row & 7)) << 4);
                        st_shared_v4(kst + off, kv);
                        st_shared_v4(vst + off, vv);
                        if (mt == 0) {
                            const size_t dst = (unit_row0 + t) * D + chunk * 8;
                            *reinterpret_cast<uint4*>(p.k_cache + dst) = kv;
                            *reinterpret_cast<uint4*>(p.v_cache + dst) = vv;
                        }
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                }
            }

            // S = Q K^T for this warp's tokens: NJ n8 tiles.
            float sc[NJ][4];
#pragma unroll
            for (int j = 0; j < NJ; ++j) sc[j][0] = sc[j][1] = sc[j][2] = sc[j][3] = 0.f;
            if constexpr (KV8) {
                // e4m3 codes straight from the stage: an 8x8 b16 ldmatrix of K
                // rows gives each thread 4 consecutive codes (d = 4q..4q+3 of a
                // 16-wide k step) of one token, i.e. both B registers of that
                // step in the k order the Q fragments were given. One x4 load
                // covers 2 tokens tiles x 2 k steps. With two row tiles the odd
                // k steps accumulate apart (summed after the loop): half-length
                // MMA chains (one row tile measured slower that way).
                constexpr bool kSplitK = MT > 1;
                float sd[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
                for (int kk = 0; kk < KSTEPS; kk += 2) {
                    const int c8 = kk + (lane >> 4);
                    uint32_t r0, r1, r2, r3;
                    ldsm_x4(kst + k8_tok * 128 + ((c8 ^ (k8_tok & 7)) << 4), r0, r1, r2, r3);
                    uint32_t a0_s[4], a1_s[4];
                    if constexpr (kQs) {
                        const int qc = kk * 2 + (lane >> 4);
                        ldsm_x4(qa_base + ((qc ^ (qa_row & 7)) << 4), a0_s[0], a0_s[1], a0_s[2], a0_s[3]);
                        ldsm_x4(qa_base + (((qc + 2) ^ (qa_row & 7)) << 4), a1_s[0], a1_s[1], a1_s[2], a1_s[3]);
                    }
                    const uint32_t(&a0)[4] = kQs ? a0_s : qa[kQs ? 0 : kk];
                    const uint32_t(&a1)[4] = kQs ? a1_s : qa[kQs ? 0 : kk + 1];
                    mma_f16_16816(sc[0], a0, e4m3x2_to_f16x2((uint16_t)r0), e4m3x2_to_f16x2((uint16_t)(r0 >> 16)));
                    mma_f16_16816(sc[1], a0, e4m3x2_to_f16x2((uint16_t)r1), e4m3x2_to_f16x2((uint16_t)(r1 >> 16)));
                    float(&s1)[2][4] = kSplitK ? sd : sc;
                    mma_f16_16816(s1[0], a1, e4m3x2_to_f16x2((uint16_t)r2), e4m3x2_to_f16x2((uint16_t)(r2 >> 16)));
                    mma_f16_16816(s1[1], a1, e4m3x2_to_f16x2((uint16_t)r3), e4m3x2_to_f16x2((uint16_t)(r3 >> 16)));
                }
                if constexpr (kSplitK) {
#pragma unroll
                    for (int j = 0; j < 2; ++j)
#pragma unroll
                        for (int c = 0; c < 4; ++c) sc[j][c] += sd[j][c];
                }
            } else {
                // Each k step: one Q fragment, NJ/2 ldmatrix of K (16 tokens
                // each), NJ independent MMA chains.
#pragma unroll
                for (int kk = 0; kk < KSTEPS; ++kk) {
                    const int chunk = kk * 2 + k_half;
                    const int bx = chunk >> 3, cc = chunk & 7;
                    uint32_t a_s[4];
                    if constexpr (kQs) {
                        const int qc = kk * 2 + (lane >> 4);
                        ldsm_x4(qa_base + ((qc ^ (qa_row & 7)) << 4), a_s[0], a_s[1], a_s[2], a_s[3]);
                    }
                    const uint32_t(&a)[4] = kQs ? a_s : qa[kQs ? 0 : kk];
#pragma unroll
                    for (int jj = 0; jj < NJ / 2; ++jj) {
                        // (k_tok + 16 jj) & 7 == k_tok & 7: the same swizzle.
                        uint32_t b0, b1, b2, b3;
                        if constexpr (KS::kPageMajor)
                            ldsm_x4(kst + k_off0[jj] + bx * bx_stride + ((cc ^ (k_tok & 7)) << 4), b0, b1, b2, b3);
                        else
                            ldsm_x4(kst + bx * (kTileTokens * 128) + (k_tok + 16 * jj) * 128 +
                                        ((cc ^ (k_tok & 7)) << 4),
                                    b0, b1, b2, b3);
                        mma_bf16_16816(sc[2 * jj], a, b0, b1);
                        mma_bf16_16816(sc[2 * jj + 1], a, b2, b3);
                    }
                }
            }
            const float sscale = KV8 ? p.scale_log2 * ks : p.scale_log2;

            // Scale into the base-2 domain and mask invisible keys.
            float x[NJ][4];
            if (tbase + kTileTokens - 1 <= lim_min) {
#pragma unroll
                for (int j = 0; j < NJ; ++j)
#pragma unroll
                    for (int c = 0; c < 4; ++c) x[j][c] = sc[j][c] * sscale;
            } else {
                const int tok = tbase + tok0 + 2 * quad;
#pragma unroll
                for (int j = 0; j < NJ; ++j) {
                    const int t = tok + 8 * j;
                    x[j][0] = (t <= lim_lo) ? sc[j][0] * sscale : -INFINITY;
                    x[j][1] = (t + 1 <= lim_lo) ? sc[j][1] * sscale : -INFINITY;
                    x[j][2] = (t <= lim_hi) ? sc[j][2] * sscale : -INFINITY;
                    x[j][3] = (t + 1 <= lim_hi) ? sc[j][3] * sscale : -INFINITY;
                }
            }
            float mx_lo = fmaxf(fmaxf(x[0][0], x[0][1]), fmaxf(x[1][0], x[1][1]));
            float mx_hi = fmaxf(fmaxf(x[0][2], x[0][3]), fmaxf(x[1][2], x[1][3]));
#pragma unroll
            for (int j = 2; j < NJ; j += 2) {
                mx_lo = fmaxf(mx_lo, fmaxf(fmaxf(x[j][0], x[j][1]), fmaxf(x[j + 1][0], x[j + 1][1])));
                mx_hi = fmaxf(mx_hi, fmaxf(fmaxf(x[j][2], x[j][3]), fmaxf(x[j + 1][2], x[j + 1][3])));
            }
            mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, 1));
            mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, 2));
            mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, 1));
            mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, 2));
            // The running max moves only when a score exceeds it by more than
            // kRescaleSlack (base 2): until then p = 2^(x - m) stays below
            // 2^kRescaleSlack, safe in fp32 and bf16, and the O/l rescale
            // (a multiply of every accumulator) is skipped. The result is
            // exact either way: O, l and m stay consistent with each other.
            const bool up_lo = mx_lo > m_lo + kRescaleSlack;
            const bool up_hi = mx_hi > m_hi + kRescaleSlack;
            const float mn_lo = up_lo ? mx_lo : m_lo, mn_hi = up_hi ? mx_hi : m_hi;
            const float base_lo = mn_lo == -INFINITY ? 0.f : mn_lo;
            const float base_hi = mn_hi == -INFINITY ? 0.f : mn_hi;

            float pr[NJ][4];
#pragma unroll
            for (int j = 0; j < NJ; ++j) {
                pr[j][0] = fast_exp2(x[j][0] - base_lo);
                pr[j][1] = fast_exp2(x[j][1] - base_lo);
                pr[j][2] = fast_exp2(x[j][2] - base_hi);
                pr[j][3] = fast_exp2(x[j][3] - base_hi);
            }
            if (__any_sync(0xffffffffu, up_lo || up_hi)) {
                const float a_lo = fast_exp2(m_lo - base_lo), a_hi = fast_exp2(m_hi - base_hi);
                l_lo *= a_lo;
                l_hi *= a_hi;
#pragma unroll
                for (int n = 0; n < NTILE_D; ++n) {
                    o[n][0] *= a_lo;
                    o[n][1] *= a_lo;
                    o[n][2] *= a_hi;
                    o[n][3] *= a_hi;
                }
            }
            m_lo = mn_lo;
            m_hi = mn_hi;
#pragma unroll
            for (int j = 0; j < NJ; j += 2) {
                l_lo += (pr[j][0] + pr[j][1]) + (pr[j + 1][0] + pr[j + 1][1]);
                l_hi += (pr[j][2] + pr[j][3]) + (pr[j + 1][2] + pr[j + 1][3]);
            }

            // The S accumulator layout is the A-operand layout of P.V: n8
            // token tiles 2kk and 2kk + 1 are the A fragment of k step kk.
            uint32_t pa[NJ / 2][4];
#pragma unroll
            for (int kk = 0; kk < NJ / 2; ++kk) {
                if constexpr (KV8) {
                    // P times the tile's V scale: O accumulates code-valued V.
                    pa[kk][0] = pack_f16x2(pr[2 * kk][0] * vs, pr[2 * kk][1] * vs);
                    pa[kk][1] = pack_f16x2(pr[2 * kk][2] * vs, pr[2 * kk][3] * vs);
                    pa[kk][2] = pack_f16x2(pr[2 * kk + 1][0] * vs, pr[2 * kk + 1][1] * vs);
                    pa[kk][3] = pack_f16x2(pr[2 * kk + 1][2] * vs, pr[2 * kk + 1][3] * vs);
                } else {
                    pa[kk][0] = pack_bf16x2(pr[2 * kk][0], pr[2 * kk][1]);
                    pa[kk][1] = pack_bf16x2(pr[2 * kk][2], pr[2 * kk][3]);
                    pa[kk][2] = pack_bf16x2(pr[2 * kk + 1][0], pr[2 * kk + 1][1]);
                    pa[kk][3] = pack_bf16x2(pr[2 * kk + 1][2], pr[2 * kk + 1][3]);
                }
            }
            if constexpr (KV8) {
                // e4m3 V: a transposed 8x8 b16 ldmatrix of V rows gives each
                // thread codes d = 2n, 2n+1 (n = lane / 4) of tokens 2q and
                // 2q+1. A byte permute splits them into the B registers of two
                // "virtual" n8 tiles: o[2c] holds the even columns 16c + 2n of
                // 16-wide chunk c, o[2c+1] the odd ones; the writes below put
                // the columns back in order.
#pragma unroll
                for (int blk = 0; blk < D / 16; blk += 2) {
                    const int c8 = blk + (lane >> 4);
                    uint32_t r[4];
                    ldsm_x4_trans(vst + k8_tok * 128 + ((c8 ^ (k8_tok & 7)) << 4), r[0], r[1], r[2], r[3]);
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const uint32_t lo = r[2 * e], hi = r[2 * e + 1];   // tokens 0-7, 8-15
                        mma_f16_16816(o[2 * (blk + e)], pa[0],
                                      e4m3x2_to_f16x2((uint16_t)__byte_perm(lo, 0u, 0x0020)),
                                      e4m3x2_to_f16x2((uint16_t)__byte_perm(hi, 0u, 0x0020)));
                        mma_f16_16816(o[2 * (blk + e) + 1], pa[0],
                                      e4m3x2_to_f16x2((uint16_t)__byte_perm(lo, 0u, 0x0031)),
                                      e4m3x2_to_f16x2((uint16_t)__byte_perm(hi, 0u, 0x0031)));
                    }
                }
            } else {
#pragma unroll
                for (int kk = 0; kk < NJ / 2; ++kk) {
#pragma unroll
                    for (int n = 0; n < NTILE_D; n += 2) {
                        const int chunk = n + v_dt;
                        const int bx = chunk >> 3, cc = chunk & 7;
                        uint32_t b0, b1, b2, b3;
                        if constexpr (KS::kPageMajor)
                            ldsm_x4_trans(vst + v_off0[kk] + bx * bx_stride + ((cc ^ (v_tok & 7)) << 4), b0, b1, b2,
                                          b3);
                        else
                            ldsm_x4_trans(vst + bx * (kTileTokens * 128) + (v_tok + 16 * kk) * 128 +
                                              ((cc ^ (v_tok & 7)) << 4),
                                          b0, b1, b2, b3);
                        mma_bf16_16816(o[n], pa[kk], b0, b1);
                        mma_bf16_16816(o[n + 1], pa[kk], b2, b3);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(empty_bar + 8 * s);
        }
        it_base += sg.ntiles;
        if (failed) break;

        if constexpr (KS::kDual) {
            // ---- group 1 hands each slice's per-lane state (m, partial l,
            // O fragments) to the same slice and lane of group 0, which
            // merges it with the log-sum-exp rescale; group 1 then moves on.
            constexpr int kLaneFloats = NTILE_D * 4 + 4;
            float* gb = group_buf + (size_t)slice * 32 * kLaneFloats;
            if (group == 1) {
                float4* dst = reinterpret_cast<float4*>(gb);
#pragma unroll
                for (int n = 0; n < NTILE_D; ++n) dst[n * 32 + lane] = make_float4(o[n][0], o[n][1], o[n][2], o[n][3]);
                dst[NTILE_D * 32 + lane] = make_float4(m_lo, m_hi, l_lo, l_hi);
            }
            mbar_arrive(group_bar);
            if (!wait_phase(group_bar, e_parity, abort_flag, p.status, tmo)) { failed = true; break; }
            if (group == 0) {
                const float4* src = reinterpret_cast<const float4*>(gb);
                float a_lo, b_lo, a_hi, b_hi;
                {
                    const float4 ml = src[NTILE_D * 32 + lane];
                    const float M_lo = fmaxf(m_lo, ml.x), M_hi = fmaxf(m_hi, ml.y);
                    a_lo = m_lo == -INFINITY ? 0.f : fast_exp2(m_lo - M_lo);
                    b_lo = ml.x == -INFINITY ? 0.f : fast_exp2(ml.x - M_lo);
                    a_hi = m_hi == -INFINITY ? 0.f : fast_exp2(m_hi - M_hi);
                    b_hi = ml.y == -INFINITY ? 0.f : fast_exp2(ml.y - M_hi);
                    l_lo = l_lo * a_lo + ml.z * b_lo;
                    l_hi = l_hi * a_hi + ml.w * b_hi;
                    m_lo = M_lo;
                    m_hi = M_hi;
                }
#pragma unroll
                for (int n = 0; n < NTILE_D; ++n) {
                    const float4 v = src[n * 32 + lane];
                    o[n][0] = fmaf(o[n][0], a_lo, v.x * b_lo);
                    o[n][1] = fmaf(o[n][1], a_lo, v.y * b_lo);
                    o[n][2] = fmaf(o[n][2], a_hi, v.z * b_hi);
                    o[n][3] = fmaf(o[n][3], a_hi, v.w * b_hi);
                }
            }
            // The buffer is free again once group 0 has read it.
            mbar_arrive(group_bar + 8);
            if (!wait_phase(group_bar + 8, e_parity, abort_flag, p.status, tmo)) { failed = true; break; }
            e_parity ^= 1;
            if (group == 1) continue;
        }

        // ---- merge the four slices' (m, l, O) of this row tile
        l_lo += __shfl_xor_sync(0xffffffffu, l_lo, 1);
        l_lo += __shfl_xor_sync(0xffffffffu, l_lo, 2);
        l_hi += __shfl_xor_sync(0xffffffffu, l_hi, 1);
        l_hi += __shfl_xor_sync(0xffffffffu, l_hi, 2);
        if (quad == 0) {
            my_ml[(slice * 16 + grp) * 2 + 0] = m_lo;
            my_ml[(slice * 16 + grp) * 2 + 1] = l_lo;
            my_ml[(slice * 16 + grp + 8) * 2 + 0] = m_hi;
            my_ml[(slice * 16 + grp + 8) * 2 + 1] = l_hi;
        }
        mbar_arrive(mbarA);
        if (!wait_phase(mbarA, seg_parity, abort_flag, p.status, tmo)) { failed = true; break; }
        float M_lo = -INFINITY, M_hi = -INFINITY;
#pragma unroll
        for (int w = 0; w < kSlices; ++w) {
            M_lo = fmaxf(M_lo, my_ml[(w * 16 + grp) * 2]);
            M_hi = fmaxf(M_hi, my_ml[(w * 16 + grp + 8) * 2]);
        }
        float L_lo = 0.f, L_hi = 0.f, f_lo = 0.f, f_hi = 0.f;
#pragma unroll
        for (int w = 0; w < kSlices; ++w) {
            const float mw_lo = my_ml[(w * 16 + grp) * 2], lw_lo = my_ml[(w * 16 + grp) * 2 + 1];
            const float mw_hi = my_ml[(w * 16 + grp + 8) * 2], lw_hi = my_ml[(w * 16 + grp + 8) * 2 + 1];
            const float fl = mw_lo == -INFINITY ? 0.f : fast_exp2(mw_lo - M_lo);
            const float fh = mw_hi == -INFINITY ? 0.f : fast_exp2(mw_hi - M_hi);
            L_lo += lw_lo * fl;
            L_hi += lw_hi * fh;
            if (w == slice) {
                f_lo = fl;
                f_hi = fh;
            }
        }
        if (slice != 0) {
            float4* dst = reinterpret_cast<float4*>(my_merge + (slice - 1) * 16 * D);
#pragma unroll
            for (int n = 0; n < NTILE_D; ++n)
                dst[n * 32 + lane] = make_float4(o[n][0] * f_lo, o[n][1] * f_lo, o[n][2] * f_hi, o[n][3] * f_hi);
        }
        mbar_arrive(mbarB);
        if (!wait_phase(mbarB, seg_parity, abort_flag, p.status, tmo)) { failed = true; break; }
        seg_parity ^= 1;

        const float inv_lo = L_lo > 0.f ? 1.f / L_lo : 0.f;
        const float inv_hi = L_hi > 0.f ? 1.f / L_hi : 0.f;
        if (slice == 0) {
#pragma unroll
            for (int n = 0; n < NTILE_D; ++n) {
                o[n][0] *= f_lo;
                o[n][1] *= f_lo;
                o[n][2] *= f_hi;
                o[n][3] *= f_hi;
#pragma unroll
                for (int w = 0; w < kSlices - 1; ++w) {
                    const float4 v = reinterpret_cast<const float4*>(my_merge + w * 16 * D)[n * 32 + lane];
                    o[n][0] += v.x;
                    o[n][1] += v.y;
                    o[n][2] += v.z;
                    o[n][3] += v.w;
                }
            }
        }
        if (sg.complete) {
            if (slice != 0) continue;
            if (out_lo >= 0) {
                uint16_t* orow = p.out + (size_t)out_lo * D;
                if constexpr (KV8) {
#pragma unroll
                    for (int c = 0; c < D / 16; ++c)
                        *reinterpret_cast<uint2*>(orow + 16 * c + 4 * quad) =
                            make_uint2(pack_bf16x2(o[2 * c][0] * inv_lo, o[2 * c + 1][0] * inv_lo),
                                       pack_bf16x2(o[2 * c][1] * inv_lo, o[2 * c + 1][1] * inv_lo));
                } else {
#pragma unroll
                    for (int n = 0; n < NTILE_D; ++n)
                        *reinterpret_cast<uint32_t*>(orow + n * 8 + 2 * quad) =
                            pack_bf16x2(o[n][0] * inv_lo, o[n][1] * inv_lo);
                }
                if (p.lse && quad == 0)
                    p.lse[out_lo] = L_lo > 0.f ? (M_lo + log2f(L_lo)) * 0.69314718055994531f : -INFINITY;
            }
            if (out_hi >= 0) {
                uint16_t* orow = p.out + (size_t)out_hi * D;
                if constexpr (KV8) {
#pragma unroll
                    for (int c = 0; c < D / 16; ++c)
                        *reinterpret_cast<uint2*>(orow + 16 * c + 4 * quad) =
                            make_uint2(pack_bf16x2(o[2 * c][2] * inv_hi, o[2 * c + 1][2] * inv_hi),
                                       pack_bf16x2(o[2 * c][3] * inv_hi, o[2 * c + 1][3] * inv_hi));
                } else {
#pragma unroll
                    for (int n = 0; n < NTILE_D; ++n)
                        *reinterpret_cast<uint32_t*>(orow + n * 8 + 2 * quad) =
                            pack_bf16x2(o[n][2] * inv_hi, o[n][3] * inv_hi);
                }
                if (p.lse && quad == 0)
                    p.lse[out_hi] = L_hi > 0.f ? (M_hi + log2f(L_hi)) * 0.69314718055994531f : -INFINITY;
            }
            continue;
        }

        // ---- partial segment: O normalised by its own l, plus m and l, in
        // slot 0 (the CTA's first segment) or 1 (its last); then count the
        // arrival. The CTA that completes the count merges the unit.
        const long long cf = cta_of_tile(sg.ub, W, P);
        const long long cl = cta_of_tile(sg.ue - 1, W, P);
        if (slice == 0) {
            float* slot = p.ws_part + ((size_t)blockIdx.x * 2 + (sg.first ? 0 : 1)) * slot_floats;
            float* om = slot + (size_t)p.R * D;
            float* ol = om + p.R;
            if (r_lo < p.R) {
                if constexpr (KV8) {
#pragma unroll
                    for (int c = 0; c < D / 16; ++c)
                        __stcg(reinterpret_cast<float4*>(slot + (size_t)r_lo * D + 16 * c + 4 * quad),
                               make_float4(o[2 * c][0] * inv_lo, o[2 * c + 1][0] * inv_lo,
                                           o[2 * c][1] * inv_lo, o[2 * c + 1][1] * inv_lo));
                } else {
#pragma unroll
                    for (int n = 0; n < NTILE_D; ++n)
                        __stcg(reinterpret_cast<float2*>(slot + (size_t)r_lo * D + n * 8 + 2 * quad),
                               make_float2(o[n][0] * inv_lo, o[n][1] * inv_lo));
                }
                if (quad == 0) {
                    __stcg(om + r_lo, M_lo);
                    __stcg(ol + r_lo, L_lo);
                }
            }
            if (r_hi < p.R) {
                if constexpr (KV8) {
#pragma unroll
                    for (int c = 0; c < D / 16; ++c)
                        __stcg(reinterpret_cast<float4*>(slot + (size_t)r_hi * D + 16 * c + 4 * quad),
                               make_float4(o[2 * c][2] * inv_hi, o[2 * c + 1][2] * inv_hi,
                                           o[2 * c][3] * inv_hi, o[2 * c + 1][3] * inv_hi));
                } else {
#pragma unroll
                    for (int n = 0; n < NTILE_D; ++n)
                        __stcg(reinterpret_cast<float2*>(slot + (size_t)r_hi * D + n * 8 + 2 * quad),
                               make_float2(o[n][2] * inv_hi, o[n][3] * inv_hi));
                }
                if (quad == 0) {
                    __stcg(om + r_hi, M_hi);
                    __stcg(ol + r_hi, L_hi);
                }
            }
            __threadfence();
            __syncwarp();
            if (lane == 0) {
                last_flag[mt] = arrive_and_release(p, sg, mt, W, P) ? 1 : 0;
                arrived_here = true;
            }
        }
        mbar_arrive(mbarC);
        if (!wait_phase(mbarC, c_parity, abort_flag, p.status, tmo)) { failed = true; break; }
        c_parity ^= 1;
        if (!last_flag[mt]) continue;
        __threadfence();   // the other contributors' partials are visible from here on

        if (W >= P && cl - cf < KS::kFastMerge) {
            // ---- few contributors (every CTA from cf to cl has a share): each
            // thread merges four columns of one row in a single round of
            // independent loads. Slot 0 is a CTA's first segment: for every
            // CTA after cf this unit is where its share starts; cf's share
            // starts at the unit's first tile exactly when cf * W / P == ub.
            const int ncand = (int)(cl - cf + 1);
            const int first_slot = (int)(cf * 2 + (div_nonneg(cf * W, P) == sg.ub ? 0 : 1));
            const int rows_here = (p.R - mt * 16) < 16 ? (p.R - mt * 16) : 16;
            // NC candidate slots held per item, NI items of this thread merged
            // from one round of loads: up to four with at most two
            // contributors (the common split of a unit over two CTAs), two
            // with up to 16 where the registers hold them (long context
            // B = 1: 16 CTAs per unit, 86.1 -> 84.4 us), else one.
            auto merge_items = [&](auto nc_c, auto ni_c) {
                constexpr int NC = decltype(nc_c)::value, NI = decltype(ni_c)::value;
                constexpr int C4 = D / 4;
                const int n_items = rows_here * C4;
                for (int item0 = tid_mt; item0 < n_items; item0 += NI * kSlices * 32) {
                    float mk[NI][NC], lk[NI][NC];
                    float4 ok4[NI][NC];
#pragma unroll
                    for (int u = 0; u < NI; ++u) {
                        const int item = item0 + u * kSlices * 32;
                        const int r = mt * 16 + item / C4;
                        const int c4 = (item % C4) * 4;
#pragma unroll
                        for (int k = 0; k < NC; ++k) {
                            mk[u][k] = -INFINITY;
                            lk[u][k] = 0.f;
                            ok4[u][k] = make_float4(0.f, 0.f, 0.f, 0.f);
                            if (k < ncand && item < n_items) {
                                const int sl = k == 0 ? first_slot : (int)((cf + k) * 2);
                                const float* base = p.ws_part + (size_t)sl * slot_floats;
                                mk[u][k] = __ldcg(base + (size_t)p.R * D + r);
                                lk[u][k] = __ldcg(base + (size_t)p.R * D + p.R + r);
                                ok4[u][k] = __ldcg(reinterpret_cast<const float4*>(base + (size_t)r * D + c4));
                            }
                        }
                    }
#pragma unroll
                    for (int u = 0; u < NI; ++u) {
                        const int item = item0 + u * kSlices * 32;
                        if (item >= n_items) break;
                        const int r = mt * 16 + item / C4;
                        const int c4 = (item % C4) * 4;
                        float M = mk[u][0];
#pragma unroll
                        for (int k = 1; k < NC; ++k) M = fmaxf(M, mk[u][k]);
                        float L = 0.f;
                        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                        for (int k = 0; k < NC; ++k) {
                            const float w =
                                (mk[u][k] == -INFINITY || lk[u][k] == 0.f) ? 0.f : lk[u][k] * fast_exp2(mk[u][k] - M);
                            L += w;
                            acc.x += w * ok4[u][k].x;
                            acc.y += w * ok4[u][k].y;
                            acc.z += w * ok4[u][k].z;
                            acc.w += w * ok4[u][k].w;
                        }
                        const float inv = L > 0.f ? 1.f / L : 0.f;
                        const int e = rowtab[r], j = e & 0xffff, s = e >> 16;
                        const int row = (sg.b * p.sq + s) * p.H + sg.g * p.heads_per_group + j;
                        *reinterpret_cast<uint2*>(p.out + (size_t)row * D + c4) =
                            make_uint2(pack_bf16x2(acc.x * inv, acc.y * inv), pack_bf16x2(acc.z * inv, acc.w * inv));
                        if (c4 == 0 && p.lse) p.lse[row] = L > 0.f ? (M + log2f(L)) * 0.69314718055994531f : -INFINITY;
                    }
                }
            };
            if (ncand <= 2)
                merge_items(IntC<2>{}, IntC<4>{});
            else if (KS::kFastMerge >= 16 && ncand <= 16)
                merge_items(IntC<(KS::kFastMerge >= 16 ? 16 : 2)>{}, IntC<2>{});
            else
                merge_items(IntC<KS::kFastMerge>{}, IntC<1>{});
            continue;
        }

        // ---- this CTA arrived last: merge the unit's partials for the rows
        // of this row tile with the log-sum-exp rescale
        //   M = max_c m_c,  L = sum_c l_c 2^(m_c - M),  O = sum_c O_c l_c 2^(m_c - M) / L
        // and write out and lse. The 128 threads of the row tile share the
        // work in steps separated by a (bounded) barrier, each with one round
        // of independent global loads: (1) the contributing slots and all
        // their (m, l) pairs into shared memory, (2) per row the weights
        // w_c = l_c 2^(m_c - M) / L (a warp per row, lanes over contributors),
        // (3) the weighted sums of O.
        {
            int* slot_of = reinterpret_cast<int*>(my_merge);             // [ncand]
            float* mbuf = my_merge + kMaxMergeContrib;                    // [ncand][16]
            float* wts = mbuf + kMaxMergeContrib * 16;                    // [ncand][16]
            const int ncand = (int)(cl - cf + 1);
            const int rows_here = (p.R - mt * 16) < 16 ? (p.R - mt * 16) : 16;
            for (int k = tid_mt; k < ncand; k += kSlices * 32) {
                const long long c = cf + k;
                const long long clo = div_nonneg(c * W, P);
                slot_of[k] = clo < div_nonneg((c + 1) * W, P) ? (int)(c * 2 + (clo >= sg.ub ? 0 : 1)) : -1;
            }
            mbar_arrive(mbarD);
            if (!wait_phase(mbarD, d_parity, abort_flag, p.status, tmo)) { failed = true; break; }
            d_parity ^= 1;
            for (int idx = tid_mt; idx < ncand * 16; idx += kSlices * 32) {
                const int k = idx >> 4, rr = idx & 15;
                const int sl = slot_of[k];
                float m = -INFINITY, l = 0.f;
                if (sl >= 0 && rr < rows_here) {
                    const float* mp = p.ws_part + (size_t)sl * slot_floats + (size_t)p.R * D;
                    m = __ldcg(mp + mt * 16 + rr);
                    l = __ldcg(mp + p.R + mt * 16 + rr);
                }
                mbuf[idx] = m;
                wts[idx] = l;
            }
            mbar_arrive(mbarD);
            if (!wait_phase(mbarD, d_parity, abort_flag, p.status, tmo)) { failed = true; break; }
            d_parity ^= 1;
            for (int rr = slice; rr < rows_here; rr += kSlices) {
                float M = -INFINITY;
                for (int k = lane; k < ncand; k += 32) M = fmaxf(M, mbuf[k * 16 + rr]);
#pragma unroll
                for (int o2 = 16; o2 > 0; o2 >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o2));
                float L = 0.f;
                for (int k = lane; k < ncand; k += 32) {
                    const float m = mbuf[k * 16 + rr], l = wts[k * 16 + rr];
                    const float e = (m == -INFINITY || l == 0.f) ? 0.f : l * fast_exp2(m - M);
                    wts[k * 16 + rr] = e;
                    L += e;
                }
#pragma unroll
                for (int o2 = 16; o2 > 0; o2 >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o2);
                const float inv = L > 0.f ? 1.f / L : 0.f;
                for (int k = lane; k < ncand; k += 32) wts[k * 16 + rr] *= inv;
                if (lane == 0 && p.lse) {
                    const int r = mt * 16 + rr;
                    const int e = rowtab[r], j = e & 0xffff, s = e >> 16;
                    const int row = (sg.b * p.sq + s) * p.H + sg.g * p.heads_per_group + j;
                    p.lse[row] = L > 0.f ? (M + log2f(L)) * 0.69314718055994531f : -INFINITY;
                }
            }
            mbar_arrive(mbarD);
            if (!wait_phase(mbarD, d_parity, abort_flag, p.status, tmo)) { failed = true; break; }
            d_parity ^= 1;
            constexpr int C4 = D / 4;
            for (int item = tid_mt; item < rows_here * C4; item += kSlices * 32) {
                const int rr = item / C4;
                const int r = mt * 16 + rr;
                const int c4 = (item % C4) * 4;
                float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 8
                for (int k = 0; k < ncand; ++k) {
                    const int sl = slot_of[k];
                    const float w = wts[k * 16 + rr];
                    if (sl < 0 || w == 0.f) continue;
                    const float4 v = __ldcg(reinterpret_cast<const float4*>(
                        p.ws_part + (size_t)sl * slot_floats + (size_t)r * D + c4));
                    acc.x += w * v.x;
                    acc.y += w * v.y;
                    acc.z += w * v.z;
                    acc.w += w * v.w;
                }
                const int e = rowtab[r], j = e & 0xffff, s = e >> 16;
                const int row = (sg.b * p.sq + s) * p.H + sg.g * p.heads_per_group + j;
                uint2 packed;
                packed.x = pack_bf16x2(acc.x, acc.y);
                packed.y = pack_bf16x2(acc.z, acc.w);
                *reinterpret_cast<uint2*>(p.out + (size_t)row * D + c4) = packed;
            }
            // The merge area is the slice-merge buffer of the next segment.
            mbar_arrive(mbarD);
            if (!wait_phase(mbarD, d_parity, abort_flag, p.status, tmo)) { failed = true; break; }
            d_parity ^= 1;
        }
    }

    if (failed) {
        // A wait gave up; the status word says so and the outputs are
        // undefined. The counters must still end the launch at zero: a CUDA
        // graph replays this launch with the same epoch, and a count left
        // part-way would let the next replay merge before its partials are
        // written. So the row tile's slice-0 lane 0 counts this CTA's arrival
        // on every partial unit of its share it has not counted yet (the
        // interrupted segment included); the arrival that completes a count
        // resets the counter as usual, and no merge runs here.
        if (slice == 0 && group == 0 && lane == 0) {
            bool have = true;
            bool counted = arrived_here;
            while (have) {
                if (!sg.complete && !counted) arrive_and_release(p, sg, mt, W, P);
                counted = false;
                have = walk.next(sg);
            }
        }
        return;
    }

    // ---- sequences with no valid entry have no tile and no CTA: CTA
    // (b mod grid) writes out = 0 and lse = -inf for all their rows.
    {
        const int nthreads = KS::kConsumerWarps * 32;
        for (int b = blockIdx.x; b < p.B; b += p.ctas) {
            if (clamp_len(__ldg(p.seq_lens + b), p.Tmax) != 0) continue;
            const int rows = p.sq * p.H;
            for (int i = threadIdx.x; i < rows * (D / 8); i += nthreads) {
                const int row = b * rows + i / (D / 8);
                const int c8 = (i % (D / 8)) * 8;
                *reinterpret_cast<uint4*>(p.out + (size_t)row * D + c8) = make_uint4(0u, 0u, 0u, 0u);
                if (p.lse && c8 == 0) p.lse[row] = -INFINITY;
            }
        }
    }
}

}  // namespace gqa
