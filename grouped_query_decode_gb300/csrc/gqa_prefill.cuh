// Grouped-query prefill / chunked-prefill attention kernel for sm_103a on the
// 5th-generation tensor cores (tcgen05, accumulators in tensor memory).
//
// The same operation as the decode kernel -- new token s of sequence b sits at
// position T_b - sq + s and attends to keys t <= T_b - sq + s of KV head
// g(h) = h / (H/G) -- for many new tokens at once. Section 7 of "Same GQA,
// Different Execution Cost Across Backends" folds the group into the row axis
// for prefill ([B, Hkv, G x M, D]): the (H/G) * sq query rows that share KV
// head g form one matrix, so K and V are read once per group and every score
// row keeps its own softmax. Here those rows are taken token-major (row
// r = s * (H/G) + j for head j of the group), which keeps the causal limit of
// a 128-row tile within a narrow band; the order is internal.
//
// One CTA per pair of adjacent 128-row tiles (A, B) of one (b, g) unit; both
// tiles use every 128-token K/V tile the CTA loads. Warpgroup 0 (warps 0-3)
// runs tile A's softmax and epilogue, warpgroup 1 (warps 4-7) tile B's, one
// thread per row (TMEM lane = row). Warp 8 streams K and V tiles with TMA into
// 128-byte-swizzled shared memory; warp 9 allocates tensor memory and one of
// its threads issues the MMAs, alternating between the two tiles so that the
// tensor cores work on one tile while the other tile's softmax runs:
//     S_X(j)  = Q_X K_j^T    M = 128, N = 128, K = D    (TMEM, fp32)
//     O_X    += P_X(j) V_j   M = 128, N = D,   K = 128  (A = P in TMEM)
// P_X(j) (bf16) is written over the first half of S_X(j)'s columns. The MMAs
// of one thread execute in issue order, so S_X(j+1), issued after
// P_X(j) V_j, does not overwrite P_X(j) before that product has read it; and
// the commit that reports S_X(j+1) also reports P_X(j) V_j complete, which is
// what the softmax needs before it rescales O_X. Every wait is bounded; on
// expiry the CTA records the failure, lets its copies and MMAs finish, frees
// its tensor memory and returns.
#pragma once

#include <cstdint>

#include "gqa_common.h"
#include "gqa_device.cuh"
#include "ptx.cuh"
#include "tcgen05.cuh"

namespace gqa {

constexpr int kPfRows = 128;     // query rows per tile (MMA M; one TMEM lane each)
constexpr int kPfTokens = 128;   // keys per K/V tile
constexpr int kPrefetchTiles = 6;  // K/V tiles requested into L2 ahead of their loads
// Floats per row of a split partial: O[D], m, l, padded so that every row
// starts on a 16-byte boundary (the epilogue stores O with 16-byte stores).
__host__ __device__ constexpr int prefill_part_stride(int D) { return D + 4; }

template <int D>
struct PrefillShape {
    static constexpr int kBlockBytes = 128 * 128;        // 128 rows x 128 B, 128-byte swizzle
    static constexpr int kDBlocks = D / 64;              // 64 bf16 columns per block
    static constexpr int kQBytes = kDBlocks * kBlockBytes;      // one Q tile
    static constexpr int kTileBytes = kDBlocks * kBlockBytes;   // one K (or V) tile
    static constexpr int kStages = D == 128 ? 2 : 4;
    static constexpr int kThreads = 11 * 32;
    // k_full, k_empty, v_full, v_empty rings; per tile q_full, s_full,
    // p_full, o_done, fin, tok, s_free.
    static constexpr int kBars = 4 * kStages + 8 + 6;
    static constexpr int kSmemBytes = 1024 + 2 * kQBytes + 2 * kStages * kTileBytes + 8 * kBars + 16;
    static constexpr uint32_t kTmemCols = 512;
    // Columns: S_A | S_B | O_A | O_B.
    // D = 64 leaves room for P beside S (S_A | S_B | P_A | P_B | O_A | O_B),
    // so S(j+1) can be computed once the softmax has read S(j); at D = 128
    // P is written over the first half of S (S_A | S_B | O_A | O_B).
    static constexpr bool kSepP = D == 64;
    static constexpr uint32_t kColS0 = 0, kColS1 = 128;
    static constexpr uint32_t kColP0 = kSepP ? 256 : kColS0, kColP1 = kSepP ? 320 : kColS1;
    static constexpr uint32_t kColO0 = kSepP ? 384 : 256, kColO1 = kColO0 + D;
};

template <int D, bool SPLIT>
__global__ void __launch_bounds__(PrefillShape<D>::kThreads, 1)
    gqa_prefill_kernel(const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const PrefillParams p) {
    using PS = PrefillShape<D>;
    constexpr int S = PS::kStages;
    constexpr uint32_t kBlock = PS::kBlockBytes;

    extern __shared__ __align__(1024) unsigned char smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    const uint32_t q_s = base;                               // [2] Q tiles
    const uint32_t k_s = q_s + 2 * PS::kQBytes;
    const uint32_t v_s = k_s + S * PS::kTileBytes;
    const uint32_t bar0 = v_s + S * PS::kTileBytes;
    const uint32_t k_full = bar0, k_empty = bar0 + 8 * S;
    const uint32_t v_full = bar0 + 16 * S, v_empty = bar0 + 24 * S;
    const uint32_t q_full = bar0 + 32 * S;                   // [2]
    const uint32_t s_full = q_full + 16;                     // [2]
    const uint32_t p_full = s_full + 16;                     // [2]
    const uint32_t o_done = p_full + 16;                     // [2]
    const uint32_t fin = o_done + 16;                        // [2]
    const uint32_t tok = fin + 16;                           // [2] turn tokens of the MMA warps
    const uint32_t s_free = tok + 16;                        // [2] S read by the softmax (kSepP)
    unsigned char* gen = smem_raw + (bar0 + 8 * PS::kBars - raw);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gen);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(gen + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint64_t tmo = p.wait_timeout_ns;

    // Work item: a pair of row tiles (the latest pairs, with the most keys,
    // first) and, for short chunks, one of `splits` key ranges of it.
    const int units = p.B * p.G;
    const int pairs = (p.row_tiles + 1) / 2;
    const int split = SPLIT ? (int)(blockIdx.x % p.splits) : 0;
    const int item = SPLIT ? (int)(blockIdx.x / p.splits) : (int)blockIdx.x;
    const int pr = pairs - 1 - item / units;
    const int unit = item % units;
    const int b = unit / p.G;
    const int tb = clamp_len(__ldg(p.seq_lens + b), p.Tmax);
    const int hpg = p.heads_per_group;
    // Rows and key tiles of tile A (x = 0) and B (x = 1), kept in registers
    // (selected, never indexed at run time).
    auto tile_rows = [&](int x) { return max(0, min(kPfRows, p.R - (2 * pr + x) * kPfRows)); };
    auto tile_nkv = [&](int x) {
        const int rx = tile_rows(x);
        // Token-major rows: a tile's last row has the largest causal limit.
        const int lim_last = rx > 0 ? tb - p.sq + ((2 * pr + x) * kPfRows + rx - 1) / hpg : -1;
        return lim_last < 0 ? 0 : lim_last / kPfTokens + 1;
    };
    const int rows0 = tile_rows(0), rows1 = tile_rows(1);
    // This CTA's key tiles [j0, j0 + n) of the pair; each tile's own count is
    // cut to the keys it sees. Ring stages and phases count from j0.
    const int n_pair = max(tile_nkv(0), tile_nkv(1));
    const int j0 = SPLIT ? (int)((long long)split * n_pair / p.splits) : 0;
    const int j1 = SPLIT ? (int)((long long)(split + 1) * n_pair / p.splits) : n_pair;
    const int nkv0 = SPLIT ? max(0, min(tile_nkv(0), j1) - j0) : tile_nkv(0);
    const int nkv1 = SPLIT ? max(0, min(tile_nkv(1), j1) - j0) : tile_nkv(1);
    const int n_all = max(nkv0, nkv1);

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(k_full + 8 * s, 1);
            mbar_init(k_empty + 8 * s, 2);   // one release per MMA warp
            mbar_init(v_full + 8 * s, 1);
            mbar_init(v_empty + 8 * s, 2);
        }
        for (int x = 0; x < 2; ++x) {
            mbar_init(q_full + 8 * x, kPfRows);
            mbar_init(s_full + 8 * x, 1);
            mbar_init(p_full + 8 * x, kPfRows);
            mbar_init(o_done + 8 * x, 1);
        }
        mbar_init(fin, 1);
        mbar_init(fin + 8, 1);
        mbar_init(tok, 1);
        mbar_init(tok + 8, 1);
        mbar_init(s_free, kPfRows);
        mbar_init(s_free + 8, kPfRows);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 9) {
        tmem_alloc(smem_addr(tmem_slot), PS::kTmemCols);
        tmem_relinquish();
    }
    if (warp == 8 && lane == 0) {
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 8) {
        // ------------------------------------------------------- TMA producer
        if (lane == 0) {
            int k_issued = 0, v_issued = 0;
            // The CTAs of one (b, g) unit read the same K/V tiles at about the
            // same time; asking L2 for tiles a few steps ahead keeps those
            // reads from waiting on DRAM together.
            for (int j = 0; j < kPrefetchTiles && j < n_all; ++j)
#pragma unroll
                for (int bx = 0; bx < PS::kDBlocks; ++bx) {
                    tma_prefetch_l2_3d(&tm_k, bx * 64, (j0 + j) * kPfTokens, unit);
                    tma_prefetch_l2_3d(&tm_v, bx * 64, (j0 + j) * kPfTokens, unit);
                }
            for (int j = 0; j < n_all; ++j) {
                const int s = j % S;
                const uint32_t ph = ((j / S) & 1) ^ 1;
                if (j + kPrefetchTiles < n_all)
#pragma unroll
                    for (int bx = 0; bx < PS::kDBlocks; ++bx) {
                        tma_prefetch_l2_3d(&tm_k, bx * 64, (j0 + j + kPrefetchTiles) * kPfTokens, unit);
                        tma_prefetch_l2_3d(&tm_v, bx * 64, (j0 + j + kPrefetchTiles) * kPfTokens, unit);
                    }
                if (!wait_phase(k_empty + 8 * s, ph, abort_flag, p.status, tmo)) break;
                if (!(blockIdx.x == 0 && j == p.skip_tile)) {   // injected fault: tile never loaded
                    mbar_arrive_expect_tx(k_full + 8 * s, PS::kTileBytes);
#pragma unroll
                    for (int bx = 0; bx < PS::kDBlocks; ++bx)
                        tma_load_3d(k_s + s * PS::kTileBytes + bx * kBlock, &tm_k, k_full + 8 * s, bx * 64,
                                    (j0 + j) * kPfTokens, unit);
                    k_issued = j + 1;
                }
                if (!wait_phase(v_empty + 8 * s, ph, abort_flag, p.status, tmo)) break;
                mbar_arrive_expect_tx(v_full + 8 * s, PS::kTileBytes);
#pragma unroll
                for (int bx = 0; bx < PS::kDBlocks; ++bx)
                    tma_load_3d(v_s + s * PS::kTileBytes + bx * kBlock, &tm_v, v_full + 8 * s, bx * 64,
                                (j0 + j) * kPfTokens, unit);
                v_issued = j + 1;
            }
            // Leave only once the copies of the last tiles have landed (the
            // earlier ones were waited on through their stages' empty barriers).
            for (int j = k_issued > S ? k_issued - S : 0; j < k_issued; ++j) {
                if (blockIdx.x == 0 && j == p.skip_tile) continue;
                const uint64_t t0 = global_timer_ns();
                while (!mbar_try_wait(k_full + 8 * (j % S), (j / S) & 1))
                    if (global_timer_ns() - t0 > tmo) break;
            }
            for (int j = v_issued > S ? v_issued - S : 0; j < v_issued; ++j) {
                const uint64_t t0 = global_timer_ns();
                while (!mbar_try_wait(v_full + 8 * (j % S), (j / S) & 1))
                    if (global_timer_ns() - t0 > tmo) break;
            }
        }
    } else if (warp == 9 || warp == 10) {
        // ------------------------------------- MMA issuers, one warp per tile
        // Warp 9 serves tile A, warp 10 tile B, so that neither tile's
        // products wait behind the other's. Each releases every K/V stage
        // once; a stage is refilled after both have.
        const int x = warp - 9;
        const int nx = x ? nkv1 : nkv0;
        constexpr uint32_t kIdescS = idesc_bf16_f32(kPfRows, kPfTokens, false, false);
        constexpr uint32_t kIdescO = idesc_bf16_f32(kPfRows, D, false, true);
        const uint32_t qst = q_s + x * PS::kQBytes;
        const uint32_t s_tm = tmem + (x ? PS::kColS1 : PS::kColS0);
        const uint32_t o_tm = tmem + (x ? PS::kColO1 : PS::kColO0);
        auto issue_s = [&](int j) {
            const uint32_t kst = k_s + (j % S) * PS::kTileBytes;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t off = (kk >> 2) * kBlock + (kk & 3) * 32;
                umma_bf16(s_tm, smem_desc_sw128(qst + off, 16, 1024), smem_desc_sw128(kst + off, 16, 1024),
                          kIdescS, kk > 0 ? 1u : 0u);
            }
            umma_commit(s_full + 8 * x);
            umma_commit(k_empty + 8 * (j % S));    // K_j has had its last reader from this tile
        };
        const uint32_t p_tm = tmem + (x ? PS::kColP1 : PS::kColP0);
        auto issue_pv = [&](int j) {
            const uint32_t vst = v_s + (j % S) * PS::kTileBytes;
#pragma unroll
            for (int kk = 0; kk < kPfTokens / 16; ++kk)
                umma_bf16_ts(o_tm, p_tm + kk * 8, smem_desc_sw128(vst + kk * 16 * 128, kBlock, 1024), kIdescO,
                             (j > 0 || kk > 0) ? 1u : 0u);
            umma_commit(v_empty + 8 * (j % S));
            if constexpr (PS::kSepP) umma_commit(o_done + 8 * x);   // one phase per product
        };
        auto zero_v_tail = [&](int j) {
            // Keys past the valid length may hold anything (NaN included);
            // zero their V rows so that p = 0 times them stays 0. Both MMA
            // warps may write the same zeros; each does so before its own
            // product reads them.
            const int valid = tb - (j0 + j) * kPfTokens;
            if (valid < kPfTokens) {
                const uint32_t vst = v_s + (j % S) * PS::kTileBytes;
                const int first = valid > 0 ? valid : 0;
                for (int idx = lane; idx < (kPfTokens - first) * PS::kDBlocks * 8; idx += 32) {
                    const int row = first + idx / (PS::kDBlocks * 8);
                    const int rest = idx % (PS::kDBlocks * 8);
                    st_shared_zero16(vst + (rest >> 3) * kBlock + row * 128 + ((rest & 7) << 4));
                }
                fence_proxy_async_smem();
                __syncwarp();
            }
        };
        bool ok = true;
        bool issued_any = false;
        if constexpr (PS::kSepP) {
            // S and P apart: S(j+1) as soon as the softmax has read S(j),
            // P(j) V_j as soon as P(j) is written; the warps need no turns.
            if (nx > 0) ok = warp_wait(q_full + 8 * x, 0, abort_flag, p.status, tmo) &&
                             warp_wait(k_full, 0, abort_flag, p.status, tmo);
            if (ok && nx > 0 && lane == 0) {
                tc_fence_after();
                issue_s(0);
            }
            issued_any = ok && nx > 0;
            __syncwarp();
            for (int j = 0; ok && j < n_all; ++j) {
                const int sv = j % S;
                const uint32_t ph = (j / S) & 1;
                if (j >= nx) {
                    ok = warp_wait(k_full + 8 * sv, ph, abort_flag, p.status, tmo) &&
                         warp_wait(v_full + 8 * sv, ph, abort_flag, p.status, tmo);
                    if (ok && lane == 0) {
                        mbar_arrive(k_empty + 8 * sv);
                        mbar_arrive(v_empty + 8 * sv);
                    }
                    __syncwarp();
                    continue;
                }
                if (j + 1 < nx) {
                    ok = warp_wait(s_free + 8 * x, j & 1, abort_flag, p.status, tmo) &&
                         warp_wait(k_full + 8 * ((j + 1) % S), ((j + 1) / S) & 1, abort_flag, p.status, tmo);
                    if (!ok) break;
                    if (lane == 0) {
                        tc_fence_after();
                        issue_s(j + 1);
                    }
                    __syncwarp();
                }
                ok = warp_wait(v_full + 8 * sv, ph, abort_flag, p.status, tmo);
                if (!ok) break;
                zero_v_tail(j);
                ok = warp_wait(p_full + 8 * x, j & 1, abort_flag, p.status, tmo);
                if (!ok) break;
                if (lane == 0) {
                    tc_fence_after();
                    issue_pv(j);
                }
                __syncwarp();
            }
        } else {
        // The two warps take turns: A issues S_A(0), then B S_B(0), then A
        // its batch {P_A(0) V_0, S_A(1)}, then B its batch, and so on; turn
        // k of warp x is arrival k on tok[x], which the other warp waits for
        // before its own turn. Each tile's softmax then runs while the
        // tensor cores work through the other tile's batch.
        uint32_t turn = 0;                     // turns this warp has taken
        auto my_turn = [&]() {
            // A's turn t follows B's turn t-1; B's turn t follows A's turn t.
            if (x == 0 && turn == 0) return true;
            const uint32_t k = x == 0 ? turn - 1 : turn;
            return warp_wait(tok + 8 * (1 - x), k & 1, abort_flag, p.status, tmo);
        };
        auto end_turn = [&]() {
            __syncwarp();
            if (lane == 0) mbar_arrive(tok + 8 * x);
            ++turn;
        };
        if (nx > 0) ok = warp_wait(q_full + 8 * x, 0, abort_flag, p.status, tmo) &&
                         warp_wait(k_full, 0, abort_flag, p.status, tmo);
        if (ok) ok = my_turn();
        if (ok && nx > 0 && lane == 0) {
            tc_fence_after();
            issue_s(0);
        }
        issued_any = ok && nx > 0;
        if (ok) end_turn();
        for (int j = 0; ok && j < n_all; ++j) {
            const int sv = j % S;
            const uint32_t ph = (j / S) & 1;
            if (j >= nx) {
                // A key tile only the other tile needs: release its stages
                // once their copies have landed, and pass the turn.
                ok = warp_wait(k_full + 8 * sv, ph, abort_flag, p.status, tmo) &&
                     warp_wait(v_full + 8 * sv, ph, abort_flag, p.status, tmo) && my_turn();
                if (ok && lane == 0) {
                    mbar_arrive(k_empty + 8 * sv);
                    mbar_arrive(v_empty + 8 * sv);
                }
                if (ok) end_turn();
                continue;
            }
            ok = warp_wait(v_full + 8 * sv, ph, abort_flag, p.status, tmo);
            if (!ok) break;
            zero_v_tail(j);
            ok = warp_wait(p_full + 8 * x, j & 1, abort_flag, p.status, tmo);
            if (ok && j + 1 < nx)
                ok = warp_wait(k_full + 8 * ((j + 1) % S), ((j + 1) / S) & 1, abort_flag, p.status, tmo);
            if (ok) ok = my_turn();
            if (!ok) break;
            if (lane == 0) {
                tc_fence_after();
                issue_pv(j);
                if (j + 1 < nx)
                    issue_s(j + 1);   // after P(j) V_j, which reads the same columns
                else
                    umma_commit(o_done + 8 * x);
            }
            end_turn();
        }
        }   // kSepP
        // Every MMA this warp issued has completed once `fin` flips.
        if (issued_any && lane == 0) {
            umma_commit(fin + 8 * x);
            const uint64_t t0 = global_timer_ns();
            while (!mbar_try_wait(fin + 8 * x, 0))
                if (global_timer_ns() - t0 > tmo) {
                    atomicOr(p.status, kStatusTimeout);
                    break;
                }
        }
        __syncwarp();
    } else {
        // ------------------------------------------- softmax and epilogue warps
        const int x = warp >> 2;                      // tile A (0) or B (1)
        const int row = threadIdx.x & 127;            // TMEM lane
        const int r = (2 * pr + x) * kPfRows + row;
        const int rows_x = x ? rows1 : rows0;
        const bool valid = row < rows_x;
        const int s_tok = valid ? r / hpg : 0;
        const int lim = valid ? tb - p.sq + s_tok : -1;   // last visible key
        // Global row of (b, s_tok, head g*hpg + j); recomputed where needed
        // from a fresh read of the CTA index so that it is not held in
        // registers through the softmax loop.
        auto out_row = [&](int& unit_o, int& pr_o, int& split_o) -> size_t {
            uint32_t cta;
            asm volatile("mov.u32 %0, %%ctaid.x;" : "=r"(cta));
            split_o = SPLIT ? (int)(cta % p.splits) : 0;
            const int it = SPLIT ? (int)(cta / p.splits) : (int)cta;
            unit_o = it % units;
            pr_o = pairs - 1 - it / units;
            const int rr = (2 * pr_o + x) * kPfRows + row;
            const int bo = unit_o / p.G, go = unit_o % p.G;
            return (size_t)(bo * p.sq + rr / hpg) * p.H + (size_t)go * hpg + rr % hpg;
        };
        const uint32_t lane_addr = tmem + ((uint32_t)((warp & 3) * 32) << 16);
        const uint32_t col_s = x ? PS::kColS1 : PS::kColS0;
        const uint32_t col_o = x ? PS::kColO1 : PS::kColO0;
        const int n = x ? nkv1 : nkv0;

        // Q row -> shared memory, K-major with the 128-byte swizzle.
        if (n > 0) {
            int uo, po, so;
            const uint4* src = reinterpret_cast<const uint4*>(p.q + out_row(uo, po, so) * D);
            const uint32_t qst = q_s + x * PS::kQBytes;
#pragma unroll
            for (int c = 0; c < D / 8; ++c) {
                const uint4 v = valid ? __ldg(src + c) : make_uint4(0u, 0u, 0u, 0u);
                st_shared_v4(qst + (c >> 3) * kBlock + row * 128 + (((c & 7) ^ (row & 7)) << 4), v);
            }
            fence_proxy_async_smem();
            mbar_arrive(q_full + 8 * x);
        }

        float m = -INFINITY, l = 0.f;
        bool ok = true;
        for (int j = 0; j < n; ++j) {
            // S_X(j) is ready, and with it every earlier MMA (P_X(j-1) V_{j-1}).
            ok = wait_phase(s_full + 8 * x, j & 1, abort_flag, p.status, tmo);
            if (!__all_sync(0xffffffffu, ok)) {
                ok = false;
                break;
            }
            tc_fence_after();
            float xs[kPfTokens];
            {
                uint32_t u[kPfTokens];
                tmem_ld128(lane_addr + col_s, u);
#pragma unroll
                for (int i = 0; i < kPfTokens; ++i) xs[i] = __uint_as_float(u[i]);
            }
            if constexpr (PS::kSepP) {
                // S(j) is in registers: its columns may take S(j+1).
                tc_fence_before();
                mbar_arrive(s_free + 8 * x);
            }
            // Invisible keys -> -inf (only tiles that reach past this row's
            // limit). The max is taken on the raw scores (scale > 0) with eight
            // independent partial maxima and sums, so that no dependency chain
            // runs the length of the row.
            const int t0 = (j0 + j) * kPfTokens;
            if (t0 + kPfTokens - 1 > lim) {
#pragma unroll
                for (int i = 0; i < kPfTokens; ++i) xs[i] = (t0 + i <= lim) ? xs[i] : -INFINITY;
            }
            float pm[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) pm[k] = fmaxf(xs[k], xs[k + 8]);
#pragma unroll
            for (int i = 16; i < kPfTokens; i += 16)
#pragma unroll
                for (int k = 0; k < 8; ++k) pm[k] = fmax3(pm[k], xs[i + k], xs[i + 8 + k]);
            const float mx = fmaxf(fmax3(pm[0], pm[1], pm[2]), fmax3(fmax3(pm[3], pm[4], pm[5]), pm[6], pm[7])) *
                             p.scale_log2;
            // The running max moves only when a score exceeds it by more than
            // kRescaleSlack (base 2); until then p <= 2^kRescaleSlack and the
            // O/l rescale is skipped. O, l and m stay consistent either way.
            const bool up = mx > m + kRescaleSlack;
            const float mn = up ? mx : m;
            const float base_m = mn == -INFINITY ? 0.f : mn;
            float ps[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            uint32_t pk[kPfTokens / 2];
#pragma unroll
            for (int i = 0; i < kPfTokens; i += 2) {
                const float e0 = fast_exp2(fmaf(xs[i], p.scale_log2, -base_m));
                const float e1 = fast_exp2(fmaf(xs[i + 1], p.scale_log2, -base_m));
                ps[i & 7] += e0;
                ps[(i + 1) & 7] += e1;
                pk[i / 2] = pack_bf16x2(e0, e1);
            }
            const float sum = ((ps[0] + ps[1]) + (ps[2] + ps[3])) + ((ps[4] + ps[5]) + (ps[6] + ps[7]));
            if constexpr (PS::kSepP) {
                // P_X(j-1) V_{j-1} has completed: P's columns are free and O
                // is settled (with S apart, S(j) no longer implies it).
                if (j > 0) {
                    ok = wait_phase(o_done + 8 * x, (j - 1) & 1, abort_flag, p.status, tmo);
                    if (!__all_sync(0xffffffffu, ok)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                }
            }
            if (j > 0 && __any_sync(0xffffffffu, up)) {
                // O_X holds P_X(j-1) V_{j-1} already: rescale it.
                const float alpha = up ? fast_exp2(m - base_m) : 1.f;
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t u[32];
                    tmem_ld32(lane_addr + col_o + c * 32, u);
#pragma unroll
                    for (int i = 0; i < 32; ++i) u[i] = __float_as_uint(__uint_as_float(u[i]) * alpha);
                    tmem_st32(lane_addr + col_o + c * 32, u);
                }
            }
            if (up) l *= fast_exp2(m - base_m);
            m = mn;
            l += sum;
            // P (bf16 pairs): its own columns at D = 64, the first 64 of S_X at D = 128.
            tmem_st64(lane_addr + (x ? PS::kColP1 : PS::kColP0), pk);
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(p_full + 8 * x);
        }
        if (ok && n > 0) {
            ok = wait_phase(o_done + 8 * x, PS::kSepP ? (n - 1) & 1 : 0, abort_flag, p.status, tmo);
            ok = __all_sync(0xffffffffu, ok);
            if (ok) tc_fence_after();
        }
        if (ok && rows_x > 0) {
            // Epilogue: O / l -> bf16 out and lse = (m + log2 l) ln 2; or, for a
            // split key range, the partial O / l (fp32), m (base 2) and l.
            constexpr bool part = SPLIT;
            const float inv = l > 0.f ? 1.f / l : 0.f;
            int uo, po, so;
            const size_t orow = out_row(uo, po, so);
            uint16_t* dst = p.out + orow * D;
            constexpr int kStride = prefill_part_stride(D);
            float* slot = p.ws_part + ((((size_t)uo * pairs + po) * p.splits + so) * 2 + x) * kPfRows * kStride +
                          (size_t)row * kStride;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint32_t u[32];
                if (n > 0) {
                    tmem_ld32(lane_addr + col_o + c * 32, u);
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) u[i] = 0u;
                }
                if (!valid) continue;
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const float f0 = __uint_as_float(u[4 * k]) * inv, f1 = __uint_as_float(u[4 * k + 1]) * inv;
                    const float f2 = __uint_as_float(u[4 * k + 2]) * inv, f3 = __uint_as_float(u[4 * k + 3]) * inv;
                    if (part)
                        *reinterpret_cast<float4*>(slot + c * 32 + 4 * k) = make_float4(f0, f1, f2, f3);
                    else
                        *reinterpret_cast<uint2*>(dst + c * 32 + 4 * k) =
                            make_uint2(pack_bf16x2(f0, f1), pack_bf16x2(f2, f3));
                }
            }
            if (valid) {
                if (part)
                    *reinterpret_cast<float2*>(slot + D) = make_float2(l > 0.f ? m : -INFINITY, l);
                else if (p.lse)
                    p.lse[orow] = l > 0.f ? (m + log2f(l)) * 0.69314718055994531f : -INFINITY;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 9) {
        tc_fence_after();
        tmem_dealloc(tmem, PS::kTmemCols);
    }
}

// Merges the key-range partials of split prefill CTAs: per row
// M = max_s m_s, L = sum_s l_s 2^(m_s - M), O = sum_s (O/l)_s l_s 2^(m_s - M) / L,
// lse = (M + log2 L) ln 2. One warp per row: lane s holds split s's (m, l)
// (splits <= 32), then the warp sums the O rows, four splits in flight, each
// lane D/32 columns.
template <int D>
__global__ void __launch_bounds__(256) gqa_prefill_combine(const PrefillParams p) {
    // The partials are the previous grid's (programmatic dependent launch).
    pdl_wait_primary();
    pdl_launch_dependents();
    constexpr int kStride = prefill_part_stride(D);
    constexpr int kPer = D / 32;
    const int units = p.B * p.G;
    const int pairs = (p.row_tiles + 1) / 2;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tile = blockIdx.x / (kPfRows / 8);              // (item, x)
    const int row = (blockIdx.x % (kPfRows / 8)) * 8 + warp;
    const int x = tile & 1, item = tile >> 1;
    const int pr = item / units, unit = item % units;
    const int r0 = (2 * pr + x) * kPfRows;
    if (row >= p.R - r0) return;
    const int b = unit / p.G, g = unit % p.G;
    const size_t slot_stride = (size_t)2 * kPfRows * kStride;
    const float* base = p.ws_part + ((((size_t)unit * pairs + pr) * p.splits) * 2 + x) * kPfRows * kStride +
                        (size_t)row * kStride;
    float m = -INFINITY, l = 0.f;
    if (lane < p.splits) {
        const float2 ml = *reinterpret_cast<const float2*>(base + lane * slot_stride + D);
        m = ml.x;
        l = ml.y;
    }
    float M = m;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float w = (l == 0.f || m == -INFINITY) ? 0.f : l * fast_exp2(m - M);
    float L = w;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
    float acc[kPer];
#pragma unroll
    for (int i = 0; i < kPer; ++i) acc[i] = 0.f;
    for (int s0 = 0; s0 < p.splits; s0 += 4) {
        float v[4][kPer];
        float ws[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            ws[u] = __shfl_sync(0xffffffffu, w, (s0 + u) & 31);
            const bool use = s0 + u < p.splits && ws[u] != 0.f;
            const float* src = base + (s0 + u) * slot_stride + lane * kPer;
#pragma unroll
            for (int i = 0; i < kPer; i += 2) {
                const float2 t = use ? *reinterpret_cast<const float2*>(src + i) : make_float2(0.f, 0.f);
                v[u][i] = t.x;
                v[u][i + 1] = t.y;
            }
            if (!use) ws[u] = 0.f;
        }
#pragma unroll
        for (int u = 0; u < 4; ++u)
#pragma unroll
            for (int i = 0; i < kPer; ++i) acc[i] += ws[u] * v[u][i];
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    const int r = r0 + row;
    const size_t orow = (size_t)(b * p.sq + r / p.heads_per_group) * p.H + (size_t)g * p.heads_per_group +
                        r % p.heads_per_group;
    uint16_t* dst = p.out + orow * D + lane * kPer;
#pragma unroll
    for (int i = 0; i < kPer; i += 2)
        *reinterpret_cast<uint32_t*>(dst + i) = pack_bf16x2(acc[i] * inv, acc[i + 1] * inv);
    if (lane == 0 && p.lse) p.lse[orow] = L > 0.f ? (M + log2f(L)) * 0.69314718055994531f : -INFINITY;
}

}  // namespace gqa
