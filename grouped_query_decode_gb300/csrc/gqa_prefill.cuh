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
// One CTA per 128-row tile of one (b, g) unit. Warps 0-3 own one row each per
// thread (TMEM lane = row): they stage Q, turn each 128x128 score tile S into
// probabilities P (base-2 online softmax, lazy rescale of the O accumulator),
// and write the output. Warp 4 streams 128-token K and V tiles with TMA into
// 128-byte-swizzled shared memory. Warp 5 allocates tensor memory and one of
// its threads issues the MMAs:
//     S_j  = Q K_j^T        M = 128, N = 128, K = D   (TMEM, two buffers)
//     O   += P_j V_j        M = 128, N = D,   K = 128 (TMEM)
// S_{j+1} is computed while the softmax warps work on S_j. Every wait is
// bounded; on expiry the CTA records the failure, lets its copies and MMAs
// finish, frees its tensor memory and returns.
#pragma once

#include <cstdint>

#include "gqa_common.h"
#include "gqa_device.cuh"
#include "ptx.cuh"
#include "tcgen05.cuh"

namespace gqa {

constexpr int kPfRows = 128;     // query rows per tile (MMA M; one TMEM lane each)
constexpr int kPfTokens = 128;   // keys per K/V tile

template <int D>
struct PrefillShape {
    static constexpr int kBlockBytes = 128 * 128;        // 128 rows x 128 B, 128-byte swizzle
    static constexpr int kDBlocks = D / 64;              // 64 bf16 columns per block
    static constexpr int kQBytes = kDBlocks * kBlockBytes;
    static constexpr int kPBytes = 2 * kBlockBytes;      // 128 rows x 128 tokens
    static constexpr int kTileBytes = kDBlocks * kBlockBytes;   // one K (or V) tile
    static constexpr int kStages = D == 128 ? 2 : 3;
    static constexpr int kThreads = 6 * 32;
    static constexpr int kBars = 4 * kStages + 6;
    static constexpr int kSmemBytes =
        1024 + kQBytes + kPBytes + 2 * kStages * kTileBytes + 8 * kBars + 16;
    static constexpr uint32_t kTmemCols = 512;           // S0 | S1 | O
    static constexpr uint32_t kColO = 256;
};

// Lane 0 waits (bounded) and the warp agrees on the outcome.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          unsigned* status, uint64_t timeout_ns) {
    bool ok = true;
    if ((threadIdx.x & 31) == 0) ok = wait_phase(bar, parity, abort_flag, status, timeout_ns);
    return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
}

template <int D>
__global__ void __launch_bounds__(PrefillShape<D>::kThreads, 1)
    gqa_prefill_kernel(const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const PrefillParams p) {
    using PS = PrefillShape<D>;
    constexpr int S = PS::kStages;
    constexpr uint32_t kBlock = PS::kBlockBytes;

    extern __shared__ __align__(1024) unsigned char smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    const uint32_t q_s = base;
    const uint32_t p_s = q_s + PS::kQBytes;
    const uint32_t k_s = p_s + PS::kPBytes;
    const uint32_t v_s = k_s + S * PS::kTileBytes;
    const uint32_t bar0 = v_s + S * PS::kTileBytes;
    const uint32_t k_full = bar0, k_empty = bar0 + 8 * S;
    const uint32_t v_full = bar0 + 16 * S, v_empty = bar0 + 24 * S;
    const uint32_t s_full = bar0 + 32 * S;         // [2]
    const uint32_t q_full = s_full + 16, p_full = q_full + 8, o_done = p_full + 8, fin = o_done + 8;
    unsigned char* gen = smem_raw + (bar0 + 8 * PS::kBars - raw);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gen);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(gen + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint64_t tmo = p.wait_timeout_ns;

    // Work item: the latest row tiles (most keys) first.
    const int units = p.B * p.G;
    const int mt = p.row_tiles - 1 - (int)(blockIdx.x / units);
    const int unit = (int)(blockIdx.x % units);
    const int b = unit / p.G, g = unit % p.G;
    const int tb = clamp_len(__ldg(p.seq_lens + b), p.Tmax);
    const int r0 = mt * kPfRows;
    const int rows = min(kPfRows, p.R - r0);
    const int hpg = p.heads_per_group;
    // Token-major rows: the tile's last row has the largest causal limit.
    const int lim_last = tb - p.sq + (r0 + rows - 1) / hpg;
    const int nkv = lim_last < 0 ? 0 : lim_last / kPfTokens + 1;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(k_full + 8 * s, 1);
            mbar_init(k_empty + 8 * s, 1);
            mbar_init(v_full + 8 * s, 1);
            mbar_init(v_empty + 8 * s, 1);
        }
        mbar_init(s_full, 1);
        mbar_init(s_full + 8, 1);
        mbar_init(q_full, kPfRows);
        mbar_init(p_full, kPfRows);
        mbar_init(o_done, 1);
        mbar_init(fin, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 5) {
        tmem_alloc(smem_addr(tmem_slot), PS::kTmemCols);
        tmem_relinquish();
    }
    if (warp == 4 && lane == 0) {
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 4) {
        // ------------------------------------------------------- TMA producer
        if (lane == 0) {
            int k_issued = 0, v_issued = 0;
            for (int j = 0; j < nkv; ++j) {
                const int s = j % S;
                const uint32_t ph = ((j / S) & 1) ^ 1;
                if (!wait_phase(k_empty + 8 * s, ph, abort_flag, p.status, tmo)) break;
                if (!(blockIdx.x == 0 && j == p.skip_tile)) {   // injected fault: tile never loaded
                    mbar_arrive_expect_tx(k_full + 8 * s, PS::kTileBytes);
#pragma unroll
                    for (int bx = 0; bx < PS::kDBlocks; ++bx)
                        tma_load_3d(k_s + s * PS::kTileBytes + bx * kBlock, &tm_k, k_full + 8 * s, bx * 64,
                                    j * kPfTokens, unit);
                    k_issued = j + 1;
                }
                if (!wait_phase(v_empty + 8 * s, ph, abort_flag, p.status, tmo)) break;
                mbar_arrive_expect_tx(v_full + 8 * s, PS::kTileBytes);
#pragma unroll
                for (int bx = 0; bx < PS::kDBlocks; ++bx)
                    tma_load_3d(v_s + s * PS::kTileBytes + bx * kBlock, &tm_v, v_full + 8 * s, bx * 64,
                                j * kPfTokens, unit);
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
    } else if (warp == 5) {
        // ------------------------------------------------------- MMA issuer
        constexpr uint32_t kIdescS = idesc_bf16_f32(kPfRows, kPfTokens, false, false);
        constexpr uint32_t kIdescO = idesc_bf16_f32(kPfRows, D, false, true);
        auto issue_s = [&](int j) {
            const uint32_t kst = k_s + (j % S) * PS::kTileBytes;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t off = (kk >> 2) * kBlock + (kk & 3) * 32;
                umma_bf16(tmem + (j & 1) * kPfTokens, smem_desc_sw128(q_s + off, 16, 1024),
                          smem_desc_sw128(kst + off, 16, 1024), kIdescS, kk > 0 ? 1u : 0u);
            }
        };
        auto issue_pv = [&](int j) {
            const uint32_t vst = v_s + (j % S) * PS::kTileBytes;
#pragma unroll
            for (int kk = 0; kk < kPfTokens / 16; ++kk) {
                const uint32_t a_off = (kk >> 2) * kBlock + (kk & 3) * 32;
                umma_bf16(tmem + PS::kColO, smem_desc_sw128(p_s + a_off, 16, 1024),
                          smem_desc_sw128(vst + kk * 16 * 128, kBlock, 1024), kIdescO,
                          (j > 0 || kk > 0) ? 1u : 0u);
            }
        };
        bool ok = nkv > 0 && warp_wait(q_full, 0, abort_flag, p.status, tmo);
        if (ok) ok = warp_wait(k_full, 0, abort_flag, p.status, tmo);
        const bool issued_any = ok;
        if (ok && lane == 0) {
            tc_fence_after();
            issue_s(0);
            umma_commit(s_full);
            umma_commit(k_empty);
        }
        __syncwarp();
        for (int j = 0; ok && j < nkv; ++j) {
            if (j + 1 < nkv) {
                const int s1 = (j + 1) % S;
                ok = warp_wait(k_full + 8 * s1, ((j + 1) / S) & 1, abort_flag, p.status, tmo);
                if (!ok) break;
                if (lane == 0) {
                    issue_s(j + 1);
                    umma_commit(s_full + 8 * ((j + 1) & 1));
                    umma_commit(k_empty + 8 * s1);
                }
                __syncwarp();
            }
            const int sv = j % S;
            ok = warp_wait(v_full + 8 * sv, (j / S) & 1, abort_flag, p.status, tmo);
            if (!ok) break;
            // Keys past the valid length may hold anything (NaN included);
            // zero their V rows so that p = 0 times them stays 0.
            const int valid = tb - j * kPfTokens;
            if (valid < kPfTokens) {
                const uint32_t vst = v_s + sv * PS::kTileBytes;
                const int first = valid > 0 ? valid : 0;
                for (int idx = lane; idx < (kPfTokens - first) * PS::kDBlocks * 8; idx += 32) {
                    const int row = first + idx / (PS::kDBlocks * 8);
                    const int rest = idx % (PS::kDBlocks * 8);
                    st_shared_zero16(vst + (rest >> 3) * kBlock + row * 128 + ((rest & 7) << 4));
                }
                fence_proxy_async_smem();
                __syncwarp();
            }
            ok = warp_wait(p_full, j & 1, abort_flag, p.status, tmo);
            if (!ok) break;
            if (lane == 0) {
                tc_fence_after();
                issue_pv(j);
                umma_commit(o_done);
                umma_commit(v_empty + 8 * sv);
            }
            __syncwarp();
        }
        // Every MMA this thread issued has completed once `fin` flips.
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
        // ------------------------------------------- softmax and epilogue warps
        const int row = threadIdx.x;                  // 0..127 = TMEM lane
        const int r = r0 + row;
        const bool valid = row < rows;
        const int s_tok = valid ? r / hpg : 0;
        const int jh = valid ? r % hpg : 0;
        const int lim = valid ? tb - p.sq + s_tok : -1;   // last visible key
        const size_t orow = ((size_t)(b * p.sq + s_tok) * p.H + (size_t)g * hpg + jh);
        const uint32_t lane_addr = tmem + ((uint32_t)(warp * 32) << 16);

        // Q row -> shared memory, K-major with the 128-byte swizzle.
        {
            const uint4* src = reinterpret_cast<const uint4*>(p.q + orow * D);
#pragma unroll
            for (int c = 0; c < D / 8; ++c) {
                const uint4 v = valid ? __ldg(src + c) : make_uint4(0u, 0u, 0u, 0u);
                st_shared_v4(q_s + (c >> 3) * kBlock + row * 128 + (((c & 7) ^ (row & 7)) << 4), v);
            }
            fence_proxy_async_smem();
            mbar_arrive(q_full);
        }

        float m = -INFINITY, l = 0.f;
        bool ok = true;
        for (int j = 0; j < nkv; ++j) {
            ok = wait_phase(s_full + 8 * (j & 1), (j >> 1) & 1, abort_flag, p.status, tmo);
            if (!__all_sync(0xffffffffu, ok)) {
                ok = false;
                break;
            }
            tc_fence_after();
            float x[kPfTokens];
            {
                uint32_t u[kPfTokens];
                tmem_ld128(lane_addr + (j & 1) * kPfTokens, u);
#pragma unroll
                for (int i = 0; i < kPfTokens; ++i) x[i] = __uint_as_float(u[i]);
            }
            // Invisible keys -> -inf (only tiles that reach past this row's
            // limit). The max is taken on the raw scores (scale > 0) with eight
            // independent partial maxima and sums, so that no dependency chain
            // runs the length of the row.
            const int t0 = j * kPfTokens;
            if (t0 + kPfTokens - 1 > lim) {
#pragma unroll
                for (int i = 0; i < kPfTokens; ++i) x[i] = (t0 + i <= lim) ? x[i] : -INFINITY;
            }
            float pm[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) pm[k] = x[k];
#pragma unroll
            for (int i = 8; i < kPfTokens; ++i) pm[i & 7] = fmaxf(pm[i & 7], x[i]);
            const float mx = fmaxf(fmaxf(fmaxf(pm[0], pm[1]), fmaxf(pm[2], pm[3])),
                                   fmaxf(fmaxf(pm[4], pm[5]), fmaxf(pm[6], pm[7]))) * p.scale_log2;
            // The running max moves only when a score exceeds it by more than
            // kRescaleSlack (base 2); until then p <= 2^kRescaleSlack and the
            // O/l rescale is skipped. O, l and m stay consistent either way.
            const bool up = mx > m + kRescaleSlack;
            const float mn = up ? mx : m;
            const float base_m = mn == -INFINITY ? 0.f : mn;
            float ps[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int i = 0; i < kPfTokens; ++i) {
                x[i] = fast_exp2(fmaf(x[i], p.scale_log2, -base_m));
                ps[i & 7] += x[i];
            }
            const float sum = ((ps[0] + ps[1]) + (ps[2] + ps[3])) + ((ps[4] + ps[5]) + (ps[6] + ps[7]));
            if (j > 0) {
                // P_{j-1} V_{j-1} has completed: the P buffer is free and O is
                // settled for the rescale.
                ok = wait_phase(o_done, (j - 1) & 1, abort_flag, p.status, tmo);
                if (!__all_sync(0xffffffffu, ok)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (__any_sync(0xffffffffu, up)) {
                    const float alpha = up ? fast_exp2(m - base_m) : 1.f;
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) {
                        uint32_t u[32];
                        tmem_ld32(lane_addr + PS::kColO + c * 32, u);
#pragma unroll
                        for (int i = 0; i < 32; ++i) u[i] = __float_as_uint(__uint_as_float(u[i]) * alpha);
                        tmem_st32(lane_addr + PS::kColO + c * 32, u);
                    }
                    tmem_st_wait();
                }
            }
            if (up) l *= fast_exp2(m - base_m);
            m = mn;
            l += sum;
            // P (bf16) -> shared memory, K-major (tokens) with the 128-byte swizzle.
#pragma unroll
            for (int c = 0; c < kPfTokens / 8; ++c) {
                const uint4 v = make_uint4(pack_bf16x2(x[8 * c], x[8 * c + 1]), pack_bf16x2(x[8 * c + 2], x[8 * c + 3]),
                                           pack_bf16x2(x[8 * c + 4], x[8 * c + 5]),
                                           pack_bf16x2(x[8 * c + 6], x[8 * c + 7]));
                st_shared_v4(p_s + (c >> 3) * kBlock + row * 128 + (((c & 7) ^ (row & 7)) << 4), v);
            }
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(p_full);
        }
        if (ok && nkv > 0) {
            ok = wait_phase(o_done, (nkv - 1) & 1, abort_flag, p.status, tmo);
            ok = __all_sync(0xffffffffu, ok);
            if (ok) tc_fence_after();
        }
        if (ok) {
            // Epilogue: O / l -> bf16 out, lse = (m + log2 l) ln 2.
            const float inv = l > 0.f ? 1.f / l : 0.f;
            uint4* dst = reinterpret_cast<uint4*>(p.out + orow * D);
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint32_t u[32];
                if (nkv > 0) {
                    tmem_ld32(lane_addr + PS::kColO + c * 32, u);
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) u[i] = 0u;
                }
                if (valid) {
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        uint32_t w[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            w[e] = pack_bf16x2(__uint_as_float(u[8 * k + 2 * e]) * inv,
                                               __uint_as_float(u[8 * k + 2 * e + 1]) * inv);
                        dst[c * 4 + k] = make_uint4(w[0], w[1], w[2], w[3]);
                    }
                }
            }
            if (valid && p.lse) p.lse[orow] = l > 0.f ? (m + log2f(l)) * 0.69314718055994531f : -INFINITY;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 5) {
        tc_fence_after();
        tmem_dealloc(tmem, PS::kTmemCols);
    }
}

}  // namespace gqa
