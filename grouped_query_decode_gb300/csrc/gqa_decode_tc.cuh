// Grouped-query decode on the 5th-generation tensor cores (tcgen05, fp32
// accumulators in tensor memory), for 17..32 query rows per KV head: MQA with
// 32 query heads, and multi-token decode of the larger groups. At these row
// counts the m16n8k16 split-KV kernel is bound by its warps' MMA latency, not
// by HBM; here the products are asynchronous and take a fraction of a tile's
// copy time. Opt-in (GQA_DECODE_TC=1): its steady per-tile rate is higher,
// but segment boundaries, the first tile and the merges cost more than that
// gains on the measured workloads.
//
// The work partition is the split-KV kernel's (an equal share of all units'
// tiles per persistent CTA; whole units finished in place, partial units
// merged by the last CTA to arrive on the unit's counter) with 128-token
// tiles. Tokens sit on the MMA's M axis, so the group's rows need no padding
// to 64 or 128:
//     S^T  = K_j Q^T       M = 128 tokens, N = 32 rows, K = D       (TMEM fp32)
//     O^T += V_j^T P_j^T   M = D,          N = 32 rows, K = 128     (TMEM fp32)
// K_j (K-major) and V_j (MN-major) are A operands straight from the TMA
// stages; Q and P_j^T (bf16) are K-major B operands in shared memory. Query
// row r = j * sq + s is head j of the group at new token s (section 7 of "Same
// GQA, Different Execution Cost Across Backends"), so each K/V byte leaves
// HBM once for the whole group ("GQA analysis", "Grouped broadcast").
//
// Warps 0-3 (thread t = TMEM lane t) run the softmax: thread t owns token t
// of each tile, reads its 32 scores from its lane of S^T and writes its 32
// probabilities into column t of P^T. The running max of each row is common
// to the CTA and moves only when a score exceeds it by more than
// kRescaleSlack (base 2): one vote per tile settles that; only then are the
// tile's row maxima reduced across the four warps and O^T rescaled in tensor
// memory. Each thread keeps partial row sums, reduced once per segment. At a
// segment's end thread d holds row d of O^T, i.e. column d of every output
// row. Warp 4 streams K and V with TMA; warp 5 owns the tensor memory and
// issues the MMAs from one thread, S^T(j+1) ahead of P(j)V(j) within a
// segment. Every wait is bounded; on expiry the CTA records the failure, lets
// its copies and MMAs finish, frees its tensor memory and returns.
#pragma once

#include <cstdint>

#include "gqa_common.h"
#include "gqa_device.cuh"
#include "gqa_splitkv.cuh"
#include "ptx.cuh"
#include "tcgen05.cuh"

namespace gqa {

template <int D>
struct TcShape {
    static_assert(D == 128, "tokens-on-M decode needs M = D = 128 for O^T");
    static constexpr int kBlock = kTcTokens * 128;       // one 64-column block of a tile
    static constexpr int kTileBytes = (D / 64) * kBlock;  // K (or V) of one tile
    static constexpr int kRowBlock = kTcRows * 128;      // one 64-column block of Q or P^T
    static constexpr int kQBytes = (D / 64) * kRowBlock;
    static constexpr int kPBytes = (kTcTokens / 64) * kRowBlock;
    static constexpr int kStages = 3;
    static constexpr int kThreads = 6 * 32;
    // k_full, k_empty, v_full, v_empty rings; s_full[2], s_free[2],
    // p_full[2], p_done[2], q_full, fin, sm_bar.
    static constexpr int kBars = 4 * kStages + 11;
    static constexpr int kGenBytes = 2048;   // scratch, barriers, flags
    static constexpr int kSmemBytes = 1024 + 2 * kStages * kTileBytes + kQBytes + 2 * kPBytes + kGenBytes;
    static constexpr uint32_t kTmemCols = 128;
    static constexpr uint32_t kColS = 0;     // S^T buffers at 0 and 32
    static constexpr uint32_t kColO = 64;
};

// Maximum over the warp (every lane gets it): an integer reduction on an
// order-preserving image of the float bits.
__device__ __forceinline__ float warp_max_f(float v) {
    int k = __float_as_int(v);
    k = k >= 0 ? k : k ^ 0x7fffffff;
    k = __reduce_max_sync(0xffffffffu, k);
    return __int_as_float(k >= 0 ? k : k ^ 0x7fffffff);
}

__device__ __forceinline__ void st_shared_u16(uint32_t addr, uint16_t v) {
    asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
}

template <int D>
__global__ void __launch_bounds__(TcShape<D>::kThreads, 1)
    gqa_decode_tc_kernel(const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v, const DecodeParams p) {
    using TS = TcShape<D>;
    constexpr int S = TS::kStages;
    constexpr int KSTEPS = D / 16;

    extern __shared__ __align__(1024) unsigned char smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    const uint32_t k_s = base;
    const uint32_t v_s = k_s + S * TS::kTileBytes;
    const uint32_t q_s = v_s + S * TS::kTileBytes;
    const uint32_t p_s = q_s + TS::kQBytes;                  // [2] P^T buffers
    unsigned char* gen = smem_raw + (p_s + 2 * TS::kPBytes - raw);
    float* wmax = reinterpret_cast<float*>(gen);              // [4 warps][32 rows]
    float* lsum = wmax + 4 * kTcRows;                         // [4 warps][32 rows]
    int* votes = reinterpret_cast<int*>(lsum + 4 * kTcRows);  // [2 tiles][4 warps]
    // vis_mask[d]: the rows (bits) that see a key d positions past the last
    // key every row sees (d = 0: all R rows; d >= sq: none).
    uint32_t* vis_mask = reinterpret_cast<uint32_t*>(votes + 8);   // [kTcRows + 1]
    uint64_t* bars = reinterpret_cast<uint64_t*>(vis_mask + 40);
    const uint32_t bar0 = smem_addr(bars);
    const uint32_t k_full = bar0, k_empty = bar0 + 8 * S;
    const uint32_t v_full = bar0 + 16 * S, v_empty = bar0 + 24 * S;
    const uint32_t s_full = bar0 + 32 * S;     // [2] S^T(j) written
    const uint32_t s_free = s_full + 16;       // [2] S^T(j) read by the softmax
    const uint32_t p_full = s_free + 16;       // [2] P^T(j) written
    const uint32_t p_done = p_full + 16;       // [2] P(j)V(j) complete
    const uint32_t q_full = p_done + 16;       // one phase per segment
    const uint32_t fin = q_full + 8;
    const uint32_t sm_bar = fin + 8;           // the softmax warps' own barrier
    long long* shared_ll = reinterpret_cast<long long*>(bars + TS::kBars);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(shared_ll + 4);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    volatile int* last_flag = abort_flag + 1;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint64_t tmo = p.wait_timeout_ns;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(k_full + 8 * s, 1);
            mbar_init(k_empty + 8 * s, 1);
            mbar_init(v_full + 8 * s, 1);
            mbar_init(v_empty + 8 * s, 1);
        }
        // The softmax warps arrive once per warp (lane 0, after __syncwarp).
        for (int b = 0; b < 2; ++b) {
            mbar_init(s_full + 8 * b, 1);
            mbar_init(s_free + 8 * b, 4);
            mbar_init(p_full + 8 * b, 4);
            mbar_init(p_done + 8 * b, 1);
        }
        mbar_init(q_full, 4);
        mbar_init(fin, 1);
        mbar_init(sm_bar, 4);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 5) {
        tmem_alloc(smem_addr(tmem_slot), TS::kTmemCols);
        tmem_relinquish();
    }
    if (warp == 4 && lane == 0) {
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
    }
    if (threadIdx.x <= kTcRows) {
        // Row r = j * sq + s sees a key d past that point iff s >= d.
        const int d = threadIdx.x;
        uint32_t msk = 0;
        for (int r = 0; r < p.R && r < kTcRows; ++r)
            if (r % p.sq >= d) msk |= 1u << r;
        vis_mask[d] = msk;
    }
    // Inputs may be written by the previous grid in the stream.
    pdl_wait_primary();
    // Every CTA takes a share: a unit split unevenly costs one cheap merge here.
    if (warp == 0) plan_share<kTcTokens, false>(p, lane, shared_ll);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    pdl_launch_dependents();
    const uint32_t tmem = *tmem_slot;

    const long long W = shared_ll[0];
    const long long P = shared_ll[3];
    SegmentWalkerT<kTcTokens> walk;
    walk.seq_lens = p.seq_lens;
    walk.G = p.G;
    walk.Tmax = p.Tmax;
    walk.lo = (long long)blockIdx.x < P ? (long long)blockIdx.x * W / P : W;
    walk.hi = (long long)blockIdx.x < P ? (long long)(blockIdx.x + 1) * W / P : W;
    walk.x = walk.lo;
    walk.b = (int)shared_ll[1];
    walk.pre_b = shared_ll[2];

    if (warp == 4) {
        // ------------------------------------------------------- TMA producer
        if (lane == 0) {
            uint32_t j = 0, k_issued = 0, v_issued = 0;
            bool ok = true;
            Segment sg;
            while (ok && walk.next(sg)) {
                const int unit = sg.b * p.G + sg.g;
                for (int i = 0; i < sg.ntiles; ++i, ++j) {
                    const int s = (int)(j % S);
                    const uint32_t ph = ((j / S) & 1) ^ 1;
                    const int y = (sg.t0 + i) * kTcTokens;
                    if (!wait_phase(k_empty + 8 * s, ph, abort_flag, p.status, tmo)) { ok = false; break; }
                    if (!(blockIdx.x == 0 && (int)j == p.skip_tile)) {   // injected fault: never loaded
                        mbar_arrive_expect_tx(k_full + 8 * s, TS::kTileBytes);
#pragma unroll
                        for (int bx = 0; bx < D / 64; ++bx)
                            tma_load_3d(k_s + s * TS::kTileBytes + bx * TS::kBlock, &tm_k, k_full + 8 * s, bx * 64,
                                        y, unit);
                        k_issued = j + 1;
                    }
                    if (!wait_phase(v_empty + 8 * s, ph, abort_flag, p.status, tmo)) { ok = false; break; }
                    mbar_arrive_expect_tx(v_full + 8 * s, TS::kTileBytes);
#pragma unroll
                    for (int bx = 0; bx < D / 64; ++bx)
                        tma_load_3d(v_s + s * TS::kTileBytes + bx * TS::kBlock, &tm_v, v_full + 8 * s, bx * 64, y,
                                    unit);
                    v_issued = j + 1;
                }
            }
            // Leave only once the copies of the last tiles have landed (the
            // earlier ones were waited on through their stages' empty barriers).
            for (uint32_t jj = k_issued > (uint32_t)S ? k_issued - S : 0; jj < k_issued; ++jj) {
                if (blockIdx.x == 0 && (int)jj == p.skip_tile) continue;
                const uint64_t t0 = global_timer_ns();
                while (!mbar_try_wait(k_full + 8 * (jj % S), (jj / S) & 1))
                    if (global_timer_ns() - t0 > tmo) break;
            }
            for (uint32_t jj = v_issued > (uint32_t)S ? v_issued - S : 0; jj < v_issued; ++jj) {
                const uint64_t t0 = global_timer_ns();
                while (!mbar_try_wait(v_full + 8 * (jj % S), (jj / S) & 1))
                    if (global_timer_ns() - t0 > tmo) break;
            }
        }
    } else if (warp == 5) {
        // ------------------------------------------------------- MMA issuer
        constexpr uint32_t kIdescS = idesc_bf16_f32(kTcTokens, kTcRows, false, false);
        constexpr uint32_t kIdescO = idesc_bf16_f32(D, kTcRows, true, false);
        auto issue_s = [&](uint32_t j) {
            const uint32_t kst = k_s + (j % S) * TS::kTileBytes;
            const uint32_t s_tm = tmem + TS::kColS + (j & 1) * kTcRows;
#pragma unroll
            for (int kk = 0; kk < KSTEPS; ++kk)
                umma_bf16(s_tm, smem_desc_sw128(kst + (kk >> 2) * TS::kBlock + (kk & 3) * 32, 16, 1024),
                          smem_desc_sw128(q_s + (kk >> 2) * TS::kRowBlock + (kk & 3) * 32, 16, 1024), kIdescS,
                          kk > 0 ? 1u : 0u);
            umma_commit(s_full + 8 * (j & 1));
            umma_commit(k_empty + 8 * (j % S));
        };
        auto issue_pv = [&](uint32_t j, bool first) {
            const uint32_t vst = v_s + (j % S) * TS::kTileBytes;
            const uint32_t pst = p_s + (j & 1) * TS::kPBytes;
#pragma unroll
            for (int kk = 0; kk < kTcTokens / 16; ++kk)
                umma_bf16(tmem + TS::kColO, smem_desc_sw128(vst + kk * 16 * 128, TS::kBlock, 1024),
                          smem_desc_sw128(pst + (kk >> 2) * TS::kRowBlock + (kk & 3) * 32, 16, 1024), kIdescO,
                          (!first || kk > 0) ? 1u : 0u);
            umma_commit(v_empty + 8 * (j % S));
            umma_commit(p_done + 8 * (j & 1));
        };
        // Tile j's V rows at or past the valid length may hold anything (NaN
        // included): zero them so that p = 0 times them stays 0.
        auto zero_v_tail = [&](uint32_t j, const Segment& sg, int i) {
            const int valid = sg.tb - (sg.t0 + i) * kTcTokens;
            if (valid >= kTcTokens) return;
            const uint32_t vst = v_s + (j % S) * TS::kTileBytes;
            const int first = valid > 0 ? valid : 0;
            for (int idx = lane; idx < (kTcTokens - first) * (D / 8); idx += 32) {
                const int row = first + idx / (D / 8);
                const int rest = idx % (D / 8);
                st_shared_zero16(vst + (rest >> 3) * TS::kBlock + row * 128 + ((rest & 7) << 4));
            }
            fence_proxy_async_smem();
            __syncwarp();
        };
        auto wwait = [&](uint32_t bar, uint32_t parity) {
            return warp_wait(bar, parity, abort_flag, p.status, tmo);
        };
        Segment sg;
        bool have = walk.next(sg);
        int i = 0;
        uint32_t j = 0, seg_no = 0;
        bool ok = true, issued_any = false;
        if (have) {
            ok = wwait(q_full, 0) && wwait(k_full, 0);
            if (ok && lane == 0) {
                tc_fence_after();
                issue_s(0);
            }
            issued_any = ok;
            __syncwarp();
        }
        // S^T(j+1) goes before P(j)V(j) within a segment, so the tensor cores
        // have it ready when the softmax is done with tile j. At a segment's
        // end P(j)V(j) goes first: the next segment's Q is written only after
        // the softmax's epilogue, which waits for P(j)V(j).
        auto issue_next_s = [&](uint32_t jn) -> bool {
            // S^T buffer jn & 1 was last read for tile jn - 2.
            if (jn >= 2 && !wwait(s_free + 8 * (jn & 1), ((jn - 2) >> 1) & 1)) return false;
            if (!wwait(k_full + 8 * (jn % S), (jn / S) & 1)) return false;
            if (lane == 0) {
                tc_fence_after();
                issue_s(jn);
            }
            __syncwarp();
            return true;
        };
        while (ok && have) {
            const bool last_in_seg = i + 1 == sg.ntiles;
            Segment nsg = sg;
            const bool nhave = last_in_seg ? walk.next(nsg) : true;
            if (nhave && !last_in_seg && !(ok = issue_next_s(j + 1))) break;
            if (!(ok = wwait(v_full + 8 * (j % S), (j / S) & 1))) break;
            zero_v_tail(j, sg, i);
            if (!(ok = wwait(p_full + 8 * (j & 1), (j >> 1) & 1))) break;
            if (lane == 0) {
                tc_fence_after();
                issue_pv(j, i == 0);
            }
            __syncwarp();
            if (nhave && last_in_seg) {
                ++seg_no;
                if (!(ok = wwait(q_full, seg_no & 1))) break;
                if (!(ok = issue_next_s(j + 1))) break;
            }
            if (last_in_seg) {
                sg = nsg;
                i = 0;
            } else {
                ++i;
            }
            ++j;
            have = nhave;
        }
        // Every MMA this warp issued has completed once `fin` flips.
        if (issued_any && lane == 0) {
            umma_commit(fin);
            const uint64_t t0 = global_timer_ns();
            while (!mbar_try_wait(fin, 0))
                if (global_timer_ns() - t0 > tmo) {
                    atomicOr(p.status, kStatusTimeout);
                    break;
                }
        }
        __syncwarp();
    } else {
        // ------------------------------------------- softmax, epilogue, merge
        const int t = threadIdx.x;                       // token of a tile; row d of O^T
        const uint32_t lane_addr = tmem + ((uint32_t)(warp * 32) << 16);
        const int R = p.R;
        const size_t slot_floats = ws_slot_floats(R, D);
        uint32_t sm_ph = 0;
        // All four softmax warps meet (bounded; a failure anywhere ends it).
        // Lane 0 arrives once the warp's lanes have done their part, and
        // waits for the warp.
        auto sm_sync = [&]() -> bool {
            __syncwarp();
            if (lane == 0) mbar_arrive(sm_bar);
            const bool okk = warp_wait(sm_bar, sm_ph, abort_flag, p.status, tmo);
            sm_ph ^= 1;
            return okk;
        };
        auto warp_arrive = [&](uint32_t bar) {
            __syncwarp();
            if (lane == 0) mbar_arrive(bar);
        };
        auto out_row = [&](int b, int g, int r) -> size_t {
            const int jh = r / p.sq, s = r % p.sq;
            return (size_t)(b * p.sq + s) * p.H + (size_t)g * p.heads_per_group + jh;
        };
        Segment sg;
        uint32_t j = 0;
        bool ok = true;
        float m[kTcRows], l[kTcRows];
        while (ok && walk.next(sg)) {
            // Q rows of the unit -> shared memory, K-major with the 128-byte
            // swizzle; rows past R are zero. Every MMA of the previous
            // segment has read Q: its tiles' S^T were all waited for.
            for (int c = t; c < kTcRows * (D / 8); c += 128) {
                const int r = c / (D / 8), ch = c % (D / 8);
                uint4 v = make_uint4(0u, 0u, 0u, 0u);
                if (r < R) v = __ldg(reinterpret_cast<const uint4*>(p.q + out_row(sg.b, sg.g, r) * D) + ch);
                st_shared_v4(q_s + (ch >> 3) * TS::kRowBlock + r * 128 + (((ch & 7) ^ (r & 7)) << 4), v);
            }
            fence_proxy_async_smem();
            warp_arrive(q_full);
#pragma unroll
            for (int r = 0; r < kTcRows; ++r) {
                m[r] = -INFINITY;
                l[r] = 0.f;
            }
            const int lim0 = sg.tb - p.sq;   // row r sees tokens <= lim0 + r % sq
            for (int i = 0; i < sg.ntiles; ++i, ++j) {
                const int sb = (int)(j & 1);
                const bool good = warp_wait(s_full + 8 * sb, (j >> 1) & 1, abort_flag, p.status, tmo);
                float x[kTcRows];
                bool up = false;
                if (good) {
                    tc_fence_after();
                    uint32_t u[kTcRows];
                    tmem_ld32(lane_addr + TS::kColS + sb * kTcRows, u);
                    tc_fence_before();
                    warp_arrive(s_free + 8 * sb);
                    // Scale into the base-2 domain; rows past R and keys a row
                    // does not see -> -inf.
                    const int dpos = (sg.t0 + i) * kTcTokens + t - lim0;   // > 0: past some rows' limits
                    const uint32_t vis = vis_mask[dpos <= 0 ? 0 : (dpos < p.sq ? dpos : kTcRows)];
#pragma unroll
                    for (int r = 0; r < kTcRows; ++r) {
                        x[r] = ((vis >> r) & 1u) ? __uint_as_float(u[r]) * p.scale_log2 : -INFINITY;
                        up |= x[r] > m[r] + kRescaleSlack;
                    }
                }
                // One vote per tile: a failure, or a row max that moves.
                const int vote = (__any_sync(0xffffffffu, !good) ? 2 : 0) | (__any_sync(0xffffffffu, up) ? 1 : 0);
                if (lane == 0) votes[sb * 4 + warp] = vote;
                if (!sm_sync()) { ok = false; break; }
                const int all = votes[sb * 4] | votes[sb * 4 + 1] | votes[sb * 4 + 2] | votes[sb * 4 + 3];
                if (all & 2) { ok = false; break; }
                if (all & 1) {
                    // New maxima: the tile's row maxima across the CTA, then
                    // O^T and l rescaled where a row's max moved.
                    float mine = -INFINITY;
#pragma unroll
                    for (int r = 0; r < kTcRows; ++r) {
                        const float wm = warp_max_f(x[r]);
                        mine = lane == r ? wm : mine;
                    }
                    wmax[warp * kTcRows + lane] = mine;
                    if (!sm_sync()) { ok = false; break; }
                    float alpha[kTcRows];
                    bool resc = false;
#pragma unroll
                    for (int r = 0; r < kTcRows; ++r) {
                        const float tm = fmaxf(fmaxf(wmax[r], wmax[kTcRows + r]),
                                               fmaxf(wmax[2 * kTcRows + r], wmax[3 * kTcRows + r]));
                        const bool mv = tm > m[r] + kRescaleSlack;
                        const float mn = mv ? tm : m[r];
                        // A row whose max was -inf has O = 0 and l = 0.
                        alpha[r] = (mv && m[r] != -INFINITY) ? fast_exp2(m[r] - mn) : 1.f;
                        resc |= alpha[r] != 1.f;
                        l[r] *= alpha[r];
                        m[r] = mn;
                    }
                    if (resc && i > 0) {
                        // O^T holds P(j-1)V(j-1) and what came before.
                        const uint32_t jp = j - 1;
                        if (!warp_wait(p_done + 8 * (jp & 1), (jp >> 1) & 1, abort_flag, p.status, tmo)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        uint32_t o[kTcRows];
                        tmem_ld32(lane_addr + TS::kColO, o);
#pragma unroll
                        for (int r = 0; r < kTcRows; ++r) o[r] = __float_as_uint(__uint_as_float(o[r]) * alpha[r]);
                        tmem_st32(lane_addr + TS::kColO, o);
                        tmem_st_wait();
                    }
                }
                // P^T buffer sb was last read by P(j-2)V(j-2).
                if (j >= 2) {
                    if (!warp_wait(p_done + 8 * sb, ((j - 2) >> 1) & 1, abort_flag, p.status, tmo)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                }
                // p = 2^(x - m) -> bf16, column t of P^T (K-major, swizzled).
                const uint32_t pcol = p_s + sb * TS::kPBytes + (t >> 6) * TS::kRowBlock + (t & 7) * 2;
                const int chunk = (t & 63) >> 3;
#pragma unroll
                for (int r = 0; r < kTcRows; ++r) {
                    const float bse = m[r] == -INFINITY ? 0.f : m[r];
                    const float pr = fast_exp2(x[r] - bse);
                    l[r] += pr;
                    st_shared_u16(pcol + r * 128 + ((chunk ^ (r & 7)) << 4),
                                  __bfloat16_as_ushort(__float2bfloat16_rn(pr)));
                }
                fence_proxy_async_smem();
                tc_fence_before();
                warp_arrive(p_full + 8 * sb);
            }
            if (!ok) break;

            // ---- segment epilogue: O^T after its last product
            {
                const uint32_t jl = j - 1;
                if (!warp_wait(p_done + 8 * (jl & 1), (jl >> 1) & 1, abort_flag, p.status, tmo)) {
                    ok = false;
                    break;
                }
            }
            tc_fence_after();
            uint32_t ou[kTcRows];
            tmem_ld32(lane_addr + TS::kColO, ou);
            tc_fence_before();
            // Row sums over the 128 threads: a warp reduce-scatter (lane r
            // ends with row r's warp sum), then the four warps' sums.
            {
                float v16[16], v8[8], v4[4], v2[2];
                const bool b16 = lane & 16, b8 = lane & 8, b4 = lane & 4, b2 = lane & 2, b1 = lane & 1;
#pragma unroll
                for (int k = 0; k < 16; ++k)
                    v16[k] = (b16 ? l[k + 16] : l[k]) + __shfl_xor_sync(0xffffffffu, b16 ? l[k] : l[k + 16], 16);
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    v8[k] = (b8 ? v16[k + 8] : v16[k]) + __shfl_xor_sync(0xffffffffu, b8 ? v16[k] : v16[k + 8], 8);
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    v4[k] = (b4 ? v8[k + 4] : v8[k]) + __shfl_xor_sync(0xffffffffu, b4 ? v8[k] : v8[k + 4], 4);
#pragma unroll
                for (int k = 0; k < 2; ++k)
                    v2[k] = (b2 ? v4[k + 2] : v4[k]) + __shfl_xor_sync(0xffffffffu, b2 ? v4[k] : v4[k + 2], 2);
                const float v1 = (b1 ? v2[1] : v2[0]) + __shfl_xor_sync(0xffffffffu, b1 ? v2[0] : v2[1], 1);
                lsum[warp * kTcRows + lane] = v1;
            }
            if (!sm_sync()) { ok = false; break; }
            float L[kTcRows];
#pragma unroll
            for (int r = 0; r < kTcRows; ++r)
                L[r] = (lsum[r] + lsum[kTcRows + r]) + (lsum[2 * kTcRows + r] + lsum[3 * kTcRows + r]);
            // This thread's row of the statistics (t < 32), for lse and the slot.
            float m_t = -INFINITY, L_t = 0.f;
#pragma unroll
            for (int r = 0; r < kTcRows; ++r) {
                m_t = t == r ? m[r] : m_t;
                L_t = t == r ? L[r] : L_t;
            }
            if (sg.complete) {
#pragma unroll
                for (int r = 0; r < kTcRows; ++r) {
                    if (r >= R) break;
                    const float inv = L[r] > 0.f ? 1.f / L[r] : 0.f;
                    p.out[out_row(sg.b, sg.g, r) * D + t] =
                        __bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float(ou[r]) * inv));
                }
                if (p.lse && t < R)
                    p.lse[out_row(sg.b, sg.g, t)] = L_t > 0.f ? (m_t + log2f(L_t)) * 0.69314718055994531f : -INFINITY;
                // lsum is rewritten only after the next segment's first sync.
                continue;
            }

            // ---- partial segment: O normalised by its own l, plus m and l,
            // in slot 0 (the CTA's first segment) or 1 (its last); then count
            // the arrival. The CTA that completes the count merges the unit.
            {
                float* slot = p.ws_part + ((size_t)blockIdx.x * 2 + (sg.first ? 0 : 1)) * slot_floats;
#pragma unroll
                for (int r = 0; r < kTcRows; ++r) {
                    if (r >= R) break;
                    const float inv = L[r] > 0.f ? 1.f / L[r] : 0.f;
                    __stcg(slot + (size_t)r * D + t, __uint_as_float(ou[r]) * inv);
                }
                if (t < R) {
                    __stcg(slot + (size_t)R * D + t, m_t);
                    __stcg(slot + (size_t)R * D + R + t, L_t);
                }
            }
            __threadfence();
            const long long cf = cta_of_tile(sg.ub, W, P);
            const long long cl = cta_of_tile(sg.ue - 1, W, P);
            if (!sm_sync()) { ok = false; break; }
            if (t == 0) {
                // With at least one tile per CTA every CTA from cf to cl has a
                // share of the unit; otherwise count the non-empty ones.
                unsigned contributors = (unsigned)(cl - cf + 1);
                if (W < P) {
                    contributors = 0;
                    for (long long c = cf; c <= cl; ++c) contributors += (c * W / P) < ((c + 1) * W / P) ? 1u : 0u;
                }
                unsigned long long* ctr = p.ws_counters + ((size_t)sg.b * p.G + sg.g) * kMaxRowTiles;
                const unsigned arrived = arrive_unit(ctr, p.epoch, p.status);
                *last_flag = arrived == contributors ? 1 : 0;
                if (arrived == contributors) release_unit(ctr);
            }
            if (!sm_sync()) { ok = false; break; }
            if (!*last_flag) continue;
            __threadfence();   // the other contributors' partials are visible from here on
            // ---- merge: slot 0 is a CTA's first segment; for every CTA after
            // cf this unit is where its share starts, and cf's share starts at
            // the unit's first tile exactly when cf * W / P == ub.
            auto slot_of = [&](long long c) -> const float* {
                const int sl = c == cf ? (int)(c * 2 + ((c * W / P) == sg.ub ? 0 : 1)) : (int)(c * 2);
                return p.ws_part + (size_t)sl * slot_floats;
            };
            auto has_share = [&](long long c) { return (c * W / P) < ((c + 1) * W / P); };
            // (1) Per row r: M = max_c m_c and L = sum_c l_c 2^(m_c - M); thread
            // t takes row t % 32 and every fourth contributor from t / 32.
            const int rr = t & 31, cg = t >> 5;
            const int ncon = (int)(cl - cf + 1);
            float pm = -INFINITY;
            for (int k = cg; k < ncon; k += 4)
                if (rr < R && has_share(cf + k)) pm = fmaxf(pm, __ldcg(slot_of(cf + k) + (size_t)R * D + rr));
            wmax[cg * kTcRows + rr] = pm;
            if (!sm_sync()) { ok = false; break; }
            const float Mr = fmaxf(fmaxf(wmax[rr], wmax[kTcRows + rr]), fmaxf(wmax[2 * kTcRows + rr], wmax[3 * kTcRows + rr]));
            auto weight = [&](long long c) -> float {   // l_c 2^(m_c - M) of row rr
                const float* sl = slot_of(c);
                const float mc = __ldcg(sl + (size_t)R * D + rr), lc = __ldcg(sl + (size_t)R * D + R + rr);
                return (mc == -INFINITY || lc == 0.f) ? 0.f : lc * fast_exp2(mc - Mr);
            };
            float pl = 0.f;
            for (int k = cg; k < ncon; k += 4)
                if (rr < R && has_share(cf + k)) pl += weight(cf + k);
            lsum[cg * kTcRows + rr] = pl;
            if (!sm_sync()) { ok = false; break; }
            const float Lr = (lsum[rr] + lsum[kTcRows + rr]) + (lsum[2 * kTcRows + rr] + lsum[3 * kTcRows + rr]);
            if (p.lse && t < R)   // t < 32: rr = t
                p.lse[out_row(sg.b, sg.g, t)] = Lr > 0.f ? (Mr + log2f(Lr)) * 0.69314718055994531f : -INFINITY;
            const float invL = Lr > 0.f ? 1.f / Lr : 0.f;
            // (2) Normalised weights of up to 128 contributors at a time in the
            // P^T buffers (free: the segment's last P V has completed), then
            // each thread (column t) adds every row of a contributor in one
            // round of independent loads.
            float* wts = reinterpret_cast<float*>(smem_raw + (p_s - raw));   // [128 contributors][32 rows]
            float acc[kTcRows];
#pragma unroll
            for (int r = 0; r < kTcRows; ++r) acc[r] = 0.f;
            bool mok = true;
            for (int k0 = 0; k0 < ncon && mok; k0 += 128) {
                const int kn = ncon - k0 < 128 ? ncon - k0 : 128;
                for (int k = cg; k < kn; k += 4)
                    wts[k * kTcRows + rr] = (rr < R && has_share(cf + k0 + k)) ? weight(cf + k0 + k) * invL : 0.f;
                if (!(mok = sm_sync())) break;
                for (int k = 0; k < kn; ++k) {
                    if (!has_share(cf + k0 + k)) continue;
                    const float* sl = slot_of(cf + k0 + k);
#pragma unroll
                    for (int r = 0; r < kTcRows; ++r)
                        if (r < R) acc[r] += wts[k * kTcRows + r] * __ldcg(sl + (size_t)r * D + t);
                }
                mok = sm_sync();   // before the next chunk's weights
            }
            if (!mok) { ok = false; break; }
#pragma unroll
            for (int r = 0; r < kTcRows; ++r)
                if (r < R) p.out[out_row(sg.b, sg.g, r) * D + t] = __bfloat16_as_ushort(__float2bfloat16_rn(acc[r]));
        }
        // ---- sequences with no valid entry have no tile and no CTA: CTA
        // (b mod grid) writes out = 0 and lse = -inf for all their rows.
        if (ok) {
            for (int b = blockIdx.x; b < p.B; b += p.ctas) {
                if (clamp_len(__ldg(p.seq_lens + b), p.Tmax) != 0) continue;
                const int rows = p.sq * p.H;
                for (int idx = t; idx < rows * (D / 8); idx += 128) {
                    const int row = b * rows + idx / (D / 8);
                    const int c8 = (idx % (D / 8)) * 8;
                    *reinterpret_cast<uint4*>(p.out + (size_t)row * D + c8) = make_uint4(0u, 0u, 0u, 0u);
                    if (p.lse && c8 == 0) p.lse[row] = -INFINITY;
                }
            }
        }
    }

    // Every warp gets here (each wait above is bounded); the tensor memory is
    // freed only once its readers and the MMAs are done.
    tc_fence_before();
    __syncthreads();
    if (warp == 5) {
        tc_fence_after();
        tmem_dealloc(tmem, TS::kTmemCols);
    }
}

}  // namespace gqa
