// Split-KV grouped-query decode attention kernel for sm_103a.
//
// One persistent CTA per SM. The K/V stream of every (sequence b, KV head g)
// unit is cut into 64-token tiles; the tiles of all units are laid end to end
// (b-major, then g, then position) and each CTA takes an equal contiguous
// share of that list. A CTA therefore walks one or more "segments" (runs of
// tiles of one unit). A segment that covers a whole unit is finished in the
// CTA and written straight to out/lse; a segment that covers part of a unit
// leaves a partial (O, m, l) that the combine kernel merges.
//
// Inside a CTA a producer warp streams K and V tiles HBM -> shared memory
// with TMA tensor copies (128-byte swizzle, so the ldmatrix reads below are
// bank-conflict free) into a ring of mbarrier-guarded stages. All R = (H/G)*sq
// query rows of the unit's group sit in registers as the A operand of
// m16n8k16 bf16 tensor-core MMAs (one 16-row tile per consumer warp group),
// so each K/V byte is read from HBM once for the whole group -- "GQA
// analysis", section "Grouped broadcast": the group index selects the KV head,
// K/V are never copied per query head. Four consumer warps per row tile split
// each 64-token stage 16 tokens apiece, run an online softmax in fp32 (base 2,
// running max and sum per row, quad shuffles), and merge their states through
// shared memory at the end of each segment.
#pragma once

#include <cstdint>

#include "gqa_common.h"
#include "ptx.cuh"

namespace gqa {

struct Segment {
    int b, g, tb;        // unit and its valid length (clamped)
    int t0;              // first tile of the segment within the unit
    int ntiles;          // tiles in the segment
    bool complete;       // the segment covers the whole unit
    bool first;          // the CTA's first segment (partial slot 0, else slot 1)
};

__device__ __forceinline__ int clamp_len(int t, int Tmax) { return t < 0 ? 0 : (t > Tmax ? Tmax : t); }

// Walks the CTA's share [lo, hi) of the flattened tile list, one segment at a
// time. Every warp runs its own copy; they all see the same sequence.
struct SegmentWalker {
    const int32_t* seq_lens;
    int G, Tmax;
    long long x, lo, hi, pre_b;
    int b;

    __device__ bool next(Segment& s) {
        while (x < hi) {
            const int tb = clamp_len(__ldg(seq_lens + b), Tmax);
            const long long nt = (tb + kTileTokens - 1) / kTileTokens;
            const long long span = nt * G;
            if (x >= pre_b + span) {
                pre_b += span;
                ++b;
                continue;
            }
            const long long off = x - pre_b;
            const int g = (int)(off / nt);
            const long long ub = pre_b + (long long)g * nt, ue = ub + nt;
            const long long e = hi < ue ? hi : ue;
            s.b = b;
            s.g = g;
            s.tb = tb;
            s.t0 = (int)(x - ub);
            s.ntiles = (int)(e - x);
            s.complete = (x == ub) && (e == ue);
            s.first = (x == lo);
            x = e;
            return true;
        }
        return false;
    }
};

// Bounded wait on an mbarrier phase. On expiry, or when another warp of the
// CTA has already given up, it records the failure and returns false.
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                           unsigned* status) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (global_timer_ns() - t0 > kWaitTimeoutNs) {
            *abort_flag = 1;
            atomicOr(status, kStatusTimeout);
            return false;
        }
    }
}

template <int D, int MT>
__global__ void __launch_bounds__(KernelShape<D, MT>::kThreads, 1)
    gqa_splitkv_kernel(const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const DecodeParams p) {
    using KS = KernelShape<D, MT>;
    constexpr int S = KS::kStages;
    constexpr int NB = KS::kBoxes;
    constexpr int KSTEPS = D / 16;   // k16 steps of Q.K^T
    constexpr int NTILE_D = D / 8;   // n8 tiles of P.V (columns of O)

    extern __shared__ __align__(1024) unsigned char smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t ring = (raw + 1023u) & ~1023u;
    unsigned char* ring_ptr = smem_raw + (ring - raw);
    float* merge_buf = reinterpret_cast<float*>(ring_ptr + S * KS::kStageBytes);
    float* ml_buf = merge_buf + KS::kMergeBytes / 4;
    uint64_t* bars = reinterpret_cast<uint64_t*>(ml_buf + KS::kMlBytes / 4);
    const uint32_t full_bar = smem_addr(bars);
    const uint32_t empty_bar = full_bar + 8 * S;
    const uint32_t merge_bar = empty_bar + 8 * S;          // [MT][2]: A, B
    long long* shared_ll = reinterpret_cast<long long*>(bars + 2 * S + 2 * MT);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(shared_ll + 3);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const bool is_producer = warp == KS::kConsumerWarps;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full_bar + 8 * s, 1);
            mbar_init(empty_bar + 8 * s, KS::kConsumerWarps);
        }
        for (int m = 0; m < 2 * MT; ++m) mbar_init(merge_bar + 8 * m, kSlices * 32);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (is_producer && lane == 0) {
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
    }
    // Inputs may be written by the previous grid in the stream.
    pdl_wait_primary();

    // Warp 0: total tiles W, and where this CTA's share starts.
    if (warp == 0) {
        long long total = 0;
        for (int b0 = 0; b0 < p.B; b0 += 32) {
            const int b = b0 + lane;
            long long v = 0;
            if (b < p.B) {
                const int tb = clamp_len(__ldg(p.seq_lens + b), p.Tmax);
                v = (long long)((tb + kTileTokens - 1) / kTileTokens) * p.G;
            }
            long long incl = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const long long n = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += n;
            }
            if (blockIdx.x == 0 && b < p.B) p.ws_prefix[b] = total + incl - v;
            total += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (blockIdx.x == 0 && lane == 0) p.ws_prefix[p.B] = total;
        const long long lo = (long long)blockIdx.x * total / p.ctas;
        // First sequence whose tiles reach past lo.
        long long pre = 0;
        int bstart = p.B;
        long long prestart = total;
        for (int b0 = 0; b0 < p.B; b0 += 32) {
            const int b = b0 + lane;
            long long v = 0;
            if (b < p.B) {
                const int tb = clamp_len(__ldg(p.seq_lens + b), p.Tmax);
                v = (long long)((tb + kTileTokens - 1) / kTileTokens) * p.G;
            }
            long long incl = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const long long n = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += n;
            }
            const unsigned hit = __ballot_sync(0xffffffffu, b < p.B && pre + incl > lo);
            if (hit) {
                const int src = __ffs(hit) - 1;
                bstart = b0 + src;
                prestart = pre + __shfl_sync(0xffffffffu, incl - v, src);
                break;
            }
            pre += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (lane == 0) {
            shared_ll[0] = total;
            shared_ll[1] = bstart;
            shared_ll[2] = prestart;
        }
    }
    __syncthreads();
    pdl_launch_dependents();

    const long long W = shared_ll[0];
    SegmentWalker walk;
    walk.seq_lens = p.seq_lens;
    walk.G = p.G;
    walk.Tmax = p.Tmax;
    walk.lo = (long long)blockIdx.x * W / p.ctas;
    walk.hi = (long long)(blockIdx.x + 1) * W / p.ctas;
    walk.x = walk.lo;
    walk.b = (int)shared_ll[1];
    walk.pre_b = shared_ll[2];

    if (is_producer) {
        // ------------------------------------------------------ producer
        if (lane != 0) return;
        uint32_t it = 0;
        Segment sg;
        bool ok = true;
        while (ok && walk.next(sg)) {
            const int unit = sg.b * p.G + sg.g;
            for (int i = 0; i < sg.ntiles; ++i, ++it) {
                const int s = it % S;
                if (!wait_phase(empty_bar + 8 * s, ((it / S) & 1) ^ 1, abort_flag, p.status)) {
                    ok = false;
                    break;
                }
                const uint32_t fb = full_bar + 8 * s;
                mbar_arrive_expect_tx(fb, KS::kStageBytes);
                const uint32_t kdst = ring + s * KS::kStageBytes;
                const uint32_t vdst = kdst + KS::kTileBytes;
                const int y = (sg.t0 + i) * kTileTokens;
#pragma unroll
                for (int bx = 0; bx < NB; ++bx) {
                    tma_load_3d(kdst + bx * (kTileTokens * 128), &tm_k, fb, bx * kBoxCols, y, unit);
                    tma_load_3d(vdst + bx * (kTileTokens * 128), &tm_v, fb, bx * kBoxCols, y, unit);
                }
            }
        }
        // Leave only once every copy this warp issued has landed.
        const uint32_t issued = it;
        const uint32_t first = issued > (uint32_t)S ? issued - S : 0;
        for (uint32_t j = first; j < issued; ++j) {
            const uint64_t t0 = global_timer_ns();
            while (!mbar_try_wait(full_bar + 8 * (j % S), (j / S) & 1)) {
                if (global_timer_ns() - t0 > kWaitTimeoutNs) {
                    atomicOr(p.status, kStatusTimeout);
                    break;
                }
            }
        }
        return;
    }

    // ---------------------------------------------------------- consumers
    const int slice = warp % kSlices;
    const int mt = warp / kSlices;
    const int quad = lane & 3;
    const int grp = lane >> 2;
    const uint32_t mbarA = merge_bar + 8 * (2 * mt);
    const uint32_t mbarB = mbarA + 8;
    float* my_merge = merge_buf + mt * (kSlices - 1) * 16 * D;
    float* my_ml = ml_buf + mt * kSlices * 16 * 2;

    // ldmatrix row addressing inside a stage (bytes from the stage base).
    // Q.K^T (B operand, non-transposed): matrix m = lane/8 -> n8 tile (m>>1),
    // k half (m&1); row = token.
    const int k_tok = slice * 16 + ((lane >> 4) << 3) + (lane & 7);
    const int k_half = (lane >> 3) & 1;
    // P.V (B operand, transposed): matrix m -> d tile (m>>1), token half (m&1).
    const int v_tok = slice * 16 + (((lane >> 3) & 1) << 3) + (lane & 7);
    const int v_dt = lane >> 4;

    uint32_t it = 0;
    uint32_t seg_parity = 0;
    Segment sg;
    while (walk.next(sg)) {
        // Rows of this warp's 16-row tile: r = j*sq + s (head j of the group,
        // new token s), the fold of section 7 of the first page.
        const int r_lo = mt * 16 + grp, r_hi = r_lo + 8;
        int lim_lo = sg.tb - 1, lim_hi = sg.tb - 1;
        int out_lo = -1, out_hi = -1;  // flat (b, s, h) row index for output
        uint32_t qa[KSTEPS][4];
        {
            const uint16_t* q_lo = nullptr;
            const uint16_t* q_hi = nullptr;
            if (r_lo < p.R) {
                const int j = r_lo / p.sq, s = r_lo % p.sq;
                out_lo = (sg.b * p.sq + s) * p.H + sg.g * p.heads_per_group + j;
                q_lo = p.q + (size_t)out_lo * D;
                lim_lo = sg.tb - p.sq + s;
            }
            if (r_hi < p.R) {
                const int j = r_hi / p.sq, s = r_hi % p.sq;
                out_hi = (sg.b * p.sq + s) * p.H + sg.g * p.heads_per_group + j;
                q_hi = p.q + (size_t)out_hi * D;
                lim_hi = sg.tb - p.sq + s;
            }
#pragma unroll
            for (int kk = 0; kk < KSTEPS; ++kk) {
                const int c = kk * 16 + 2 * quad;
                qa[kk][0] = q_lo ? __ldg(reinterpret_cast<const unsigned*>(q_lo + c)) : 0u;
                qa[kk][1] = q_hi ? __ldg(reinterpret_cast<const unsigned*>(q_hi + c)) : 0u;
                qa[kk][2] = q_lo ? __ldg(reinterpret_cast<const unsigned*>(q_lo + c + 8)) : 0u;
                qa[kk][3] = q_hi ? __ldg(reinterpret_cast<const unsigned*>(q_hi + c + 8)) : 0u;
            }
        }

        float m_lo = -INFINITY, m_hi = -INFINITY, l_lo = 0.f, l_hi = 0.f;
        float o[NTILE_D][4];
#pragma unroll
        for (int n = 0; n < NTILE_D; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;

        bool ok = true;
        for (int i = 0; i < sg.ntiles; ++i, ++it) {
            const int s = it % S;
            if (!wait_phase(full_bar + 8 * s, (it / S) & 1, abort_flag, p.status)) {
                ok = false;
                break;
            }
            const uint32_t kst = ring + s * KS::kStageBytes;
            const uint32_t vst = kst + KS::kTileBytes;
            const int tbase = (sg.t0 + i) * kTileTokens;

            // Rows past the valid length may hold anything (NaN included);
            // zero them in V so that p = 0 times them stays 0.
            if (tbase + kTileTokens > sg.tb) {
                bool wrote = false;
                for (int idx = lane; idx < 16 * (D / 8); idx += 32) {
                    const int row = slice * 16 + idx / (D / 8);
                    const int chunk = idx % (D / 8);
                    if (tbase + row >= sg.tb) {
                        const int bx = chunk >> 3, cc = chunk & 7;
                        st_shared_zero16(vst + bx * (kTileTokens * 128) + row * 128 +
                                         ((cc ^ (row & 7)) << 4));
                        wrote = true;
                    }
                }
                if (wrote) fence_proxy_async_smem();
                __syncwarp();
            }

            // S = Q K^T for this warp's 16 tokens: two n8 tiles.
            float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
            for (int kk = 0; kk < KSTEPS; ++kk) {
                const int chunk = kk * 2 + k_half;
                const int bx = chunk >> 3, cc = chunk & 7;
                uint32_t b0, b1, b2, b3;
                ldsm_x4(kst + bx * (kTileTokens * 128) + k_tok * 128 + ((cc ^ (k_tok & 7)) << 4), b0,
                        b1, b2, b3);
                mma_bf16_16816(sc[0], qa[kk], b0, b1);
                mma_bf16_16816(sc[1], qa[kk], b2, b3);
            }

            // Scale into the base-2 domain and mask invisible keys.
            const int tok = tbase + slice * 16 + 2 * quad;
            float x[2][4];
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int t = tok + 8 * j;
                x[j][0] = (t <= lim_lo) ? sc[j][0] * p.scale_log2 : -INFINITY;
                x[j][1] = (t + 1 <= lim_lo) ? sc[j][1] * p.scale_log2 : -INFINITY;
                x[j][2] = (t <= lim_hi) ? sc[j][2] * p.scale_log2 : -INFINITY;
                x[j][3] = (t + 1 <= lim_hi) ? sc[j][3] * p.scale_log2 : -INFINITY;
            }
            float mx_lo = fmaxf(fmaxf(x[0][0], x[0][1]), fmaxf(x[1][0], x[1][1]));
            float mx_hi = fmaxf(fmaxf(x[0][2], x[0][3]), fmaxf(x[1][2], x[1][3]));
            mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, 1));
            mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, 2));
            mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, 1));
            mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, 2));
            const float mn_lo = fmaxf(m_lo, mx_lo), mn_hi = fmaxf(m_hi, mx_hi);
            const float base_lo = mn_lo == -INFINITY ? 0.f : mn_lo;
            const float base_hi = mn_hi == -INFINITY ? 0.f : mn_hi;
            const float a_lo = fast_exp2(m_lo - base_lo), a_hi = fast_exp2(m_hi - base_hi);
            m_lo = mn_lo;
            m_hi = mn_hi;

            float pr[2][4];
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                pr[j][0] = fast_exp2(x[j][0] - base_lo);
                pr[j][1] = fast_exp2(x[j][1] - base_lo);
                pr[j][2] = fast_exp2(x[j][2] - base_hi);
                pr[j][3] = fast_exp2(x[j][3] - base_hi);
            }
            l_lo = l_lo * a_lo + (pr[0][0] + pr[0][1] + pr[1][0] + pr[1][1]);
            l_hi = l_hi * a_hi + (pr[0][2] + pr[0][3] + pr[1][2] + pr[1][3]);
#pragma unroll
            for (int n = 0; n < NTILE_D; ++n) {
                o[n][0] *= a_lo;
                o[n][1] *= a_lo;
                o[n][2] *= a_hi;
                o[n][3] *= a_hi;
            }

            // The S accumulator layout is the A-operand layout of P.V.
            uint32_t pa[4];
            pa[0] = pack_bf16x2(pr[0][0], pr[0][1]);
            pa[1] = pack_bf16x2(pr[0][2], pr[0][3]);
            pa[2] = pack_bf16x2(pr[1][0], pr[1][1]);
            pa[3] = pack_bf16x2(pr[1][2], pr[1][3]);
#pragma unroll
            for (int n = 0; n < NTILE_D; n += 2) {
                const int chunk = n + v_dt;
                const int bx = chunk >> 3, cc = chunk & 7;
                uint32_t b0, b1, b2, b3;
                ldsm_x4_trans(vst + bx * (kTileTokens * 128) + v_tok * 128 + ((cc ^ (v_tok & 7)) << 4),
                              b0, b1, b2, b3);
                mma_bf16_16816(o[n], pa, b0, b1);
                mma_bf16_16816(o[n + 1], pa, b2, b3);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(empty_bar + 8 * s);
        }
        if (!ok) return;

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
        if (!wait_phase(mbarA, seg_parity, abort_flag, p.status)) return;
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
        if (!wait_phase(mbarB, seg_parity, abort_flag, p.status)) return;
        seg_parity ^= 1;
        if (slice != 0) continue;

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
        const float inv_lo = L_lo > 0.f ? 1.f / L_lo : 0.f;
        const float inv_hi = L_hi > 0.f ? 1.f / L_hi : 0.f;
        if (sg.complete) {
            if (out_lo >= 0) {
                uint16_t* orow = p.out + (size_t)out_lo * D;
#pragma unroll
                for (int n = 0; n < NTILE_D; ++n)
                    *reinterpret_cast<uint32_t*>(orow + n * 8 + 2 * quad) =
                        pack_bf16x2(o[n][0] * inv_lo, o[n][1] * inv_lo);
                if (p.lse && quad == 0)
                    p.lse[out_lo] = L_lo > 0.f ? (M_lo + log2f(L_lo)) * 0.69314718055994531f : -INFINITY;
            }
            if (out_hi >= 0) {
                uint16_t* orow = p.out + (size_t)out_hi * D;
#pragma unroll
                for (int n = 0; n < NTILE_D; ++n)
                    *reinterpret_cast<uint32_t*>(orow + n * 8 + 2 * quad) =
                        pack_bf16x2(o[n][2] * inv_hi, o[n][3] * inv_hi);
                if (p.lse && quad == 0)
                    p.lse[out_hi] = L_hi > 0.f ? (M_hi + log2f(L_hi)) * 0.69314718055994531f : -INFINITY;
            }
        } else {
            // Partial: O normalised by its own l, plus m and l, in slot 0 (the
            // CTA's first segment) or 1 (its last).
            float* slot = p.ws_part + ((size_t)blockIdx.x * 2 + (sg.first ? 0 : 1)) * ws_slot_floats(p.R, D);
            float* om = slot + (size_t)p.R * D;
            float* ol = om + p.R;
            if (r_lo < p.R) {
#pragma unroll
                for (int n = 0; n < NTILE_D; ++n)
                    *reinterpret_cast<float2*>(slot + (size_t)r_lo * D + n * 8 + 2 * quad) =
                        make_float2(o[n][0] * inv_lo, o[n][1] * inv_lo);
                if (quad == 0) {
                    om[r_lo] = M_lo;
                    ol[r_lo] = L_lo;
                }
            }
            if (r_hi < p.R) {
#pragma unroll
                for (int n = 0; n < NTILE_D; ++n)
                    *reinterpret_cast<float2*>(slot + (size_t)r_hi * D + n * 8 + 2 * quad) =
                        make_float2(o[n][2] * inv_hi, o[n][3] * inv_hi);
                if (quad == 0) {
                    om[r_hi] = M_hi;
                    ol[r_hi] = L_hi;
                }
            }
        }
    }
}

// Merges the partials of every unit whose tiles were split across CTAs.
// One CTA per (b, g) unit; units covered by one CTA were finished by the
// split-KV kernel and are skipped; units with no valid key get out = 0,
// lse = -inf.
template <int D>
__global__ void __launch_bounds__(256)
    gqa_combine_kernel(const DecodeParams p) {
    pdl_wait_primary();
    const int unit = blockIdx.x;
    const int b = unit / p.G, g = unit % p.G;
    const int tb = clamp_len(__ldg(p.seq_lens + b), p.Tmax);
    const long long nt = (tb + kTileTokens - 1) / kTileTokens;
    constexpr int C4 = D / 4;
    const int total = p.R * C4;

    if (nt == 0) {
        for (int i = threadIdx.x; i < total; i += blockDim.x) {
            const int r = i / C4, c = (i % C4) * 4;
            const int j = r / p.sq, s = r % p.sq;
            const int row = (b * p.sq + s) * p.H + g * p.heads_per_group + j;
            *reinterpret_cast<uint2*>(p.out + (size_t)row * D + c) = make_uint2(0u, 0u);
            if (p.lse && c == 0) p.lse[row] = -INFINITY;
        }
        return;
    }
    const long long W = p.ws_prefix[p.B];
    const long long ub = p.ws_prefix[b] + (long long)g * nt, ue = ub + nt;
    const long long P = p.ctas;
    const long long cf = ((ub + 1) * P - 1) / W;
    const long long cl = (ue * P - 1) / W;
    if (cf == cl) return;

    const size_t slot_floats = ws_slot_floats(p.R, D);
    for (int i = threadIdx.x; i < total; i += blockDim.x) {
        const int r = i / C4, c = (i % C4) * 4;
        // CTAs cf..cl cover the unit; when there are fewer tiles than CTAs some
        // of them have an empty share and wrote no partial.
        float M = -INFINITY;
        for (long long cta = cf; cta <= cl; ++cta) {
            const long long clo = cta * W / P, chi = (cta + 1) * W / P;
            if (clo >= chi) continue;
            const float* part = p.ws_part + ((size_t)cta * 2 + (clo >= ub ? 0 : 1)) * slot_floats;
            M = fmaxf(M, part[(size_t)p.R * D + r]);
        }
        float L = 0.f;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        if (M != -INFINITY) {
            for (long long cta = cf; cta <= cl; ++cta) {
                const long long clo = cta * W / P, chi = (cta + 1) * W / P;
                if (clo >= chi) continue;
                const float* part = p.ws_part + ((size_t)cta * 2 + (clo >= ub ? 0 : 1)) * slot_floats;
                const float m = part[(size_t)p.R * D + r];
                const float l = part[(size_t)p.R * D + p.R + r];
                if (m == -INFINITY || l == 0.f) continue;
                const float w = l * fast_exp2(m - M);
                const float4 v = *reinterpret_cast<const float4*>(part + (size_t)r * D + c);
                L += w;
                acc.x += w * v.x;
                acc.y += w * v.y;
                acc.z += w * v.z;
                acc.w += w * v.w;
            }
        }
        const float inv = L > 0.f ? 1.f / L : 0.f;
        const int j = r / p.sq, s = r % p.sq;
        const int row = (b * p.sq + s) * p.H + g * p.heads_per_group + j;
        uint2 packed;
        packed.x = pack_bf16x2(acc.x * inv, acc.y * inv);
        packed.y = pack_bf16x2(acc.z * inv, acc.w * inv);
        *reinterpret_cast<uint2*>(p.out + (size_t)row * D + c) = packed;
        if (p.lse && c == 0)
            p.lse[row] = L > 0.f ? (M + log2f(L)) * 0.69314718055994531f : -INFINITY;
    }
}

}  // namespace gqa
