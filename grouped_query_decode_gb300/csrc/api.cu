// C ABI of libgqa_decode.so: argument checks, the work plan, TMA descriptors,
// workspace management and kernel launches. See include/gqa_decode.h for the
// contract of every entry point.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <unistd.h>

#include <atomic>
#include <chrono>
#include <cstdint>
#include <cstdlib>
#include <map>
#include <mutex>
#include <tuple>
#include <utility>

#include "gqa_decode.h"
#include "gqa_launch.h"

namespace {

using namespace gqa;

// Status word the kernels set when a bounded wait expires; one per device.
__device__ unsigned int g_status_word;

thread_local int t_last_cuda_error = 0;

int cuda_fail(cudaError_t e) {
    t_last_cuda_error = (int)e;
    return GQA_ERR_CUDA;
}

struct DeviceInfo {
    int sms = 0;
    unsigned* status = nullptr;
};

std::mutex g_mu;
std::map<int, DeviceInfo> g_devices;
// Library-owned buffers per (device, stream, kind). Kind kDecodeWs holds the
// split-KV arrival counters and partial slots; kind kPrefillWs the prefill's
// split key-range partials, kept apart so that they never land on counters.
constexpr int kDecodeWs = 0, kPrefillWs = 1;
std::map<std::tuple<int, cudaStream_t, int>, std::pair<void*, size_t>> g_workspaces;

int device_info(DeviceInfo* out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    std::lock_guard<std::mutex> lk(g_mu);
    auto it = g_devices.find(dev);
    if (it == g_devices.end()) {
        DeviceInfo info;
        e = cudaDeviceGetAttribute(&info.sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return cuda_fail(e);
        void* sym = nullptr;
        e = cudaGetSymbolAddress(&sym, g_status_word);
        if (e != cudaSuccess) return cuda_fail(e);
        info.status = static_cast<unsigned*>(sym);
        it = g_devices.emplace(dev, info).first;
    }
    *out = it->second;
    return GQA_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// A cache of `slabs` slabs of [rows][D] bf16 -- [B*G units][Tmax][D] for a
// contiguous cache, [pages*G][page_size][D] for a paged one -- viewed as a 3-D
// tensor; boxes of box_rows rows x 64 elements (128 bytes) with the 128-byte
// swizzle (with both_halves, a bf16 D = 128 cache is viewed as 4-D instead and
// a box covers both 64-column halves). Reads past a slab's rows, or of a slab
// out of range, give 0.
int encode_cache_map(CUtensorMap* map, const void* base, long long slabs, int rows, int D,
                     int box_rows, int elem_bytes = 2, bool both_halves = false) {
    PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
    if (!fn) return cuda_fail(cudaErrorNotSupported);
    if (both_halves && elem_bytes == 2 && D == 128) {
        // bf16 rows of 256 bytes as [64 columns][rows][2 halves][slabs]: the
        // halves' stride (128 B) is below the rows' (256 B), so one box of
        // box_rows rows x both halves lands as [half][row][128 B] -- the two
        // 64-column blocks of the stage -- in one copy.
        cuuint64_t dims[4] = {64, (cuuint64_t)rows, 2, (cuuint64_t)slabs};
        cuuint64_t strides[3] = {(cuuint64_t)D * 2, 128, (cuuint64_t)rows * D * 2};
        cuuint32_t box[4] = {64, (cuuint32_t)box_rows, 2, 1};
        cuuint32_t estr[4] = {1, 1, 1, 1};
        CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box,
                        estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return cuda_fail(cudaErrorInvalidValue);
        return GQA_OK;
    }
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)rows, (cuuint64_t)slabs};
    cuuint64_t strides[2] = {(cuuint64_t)D * elem_bytes, (cuuint64_t)rows * D * elem_bytes};
    cuuint32_t box[3] = {(cuuint32_t)(128 / elem_bytes), (cuuint32_t)box_rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(map, elem_bytes == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                    3, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cuda_fail(cudaErrorInvalidValue);
    return GQA_OK;
}

int check_shapes(int B, int sq, int H, int G, int D, int Tmax) {
    if (B <= 0 || sq <= 0 || H <= 0 || G <= 0 || D <= 0 || Tmax <= 0) return GQA_ERR_INVALID_ARG;
    if (H % G != 0) return GQA_ERR_HEAD_RATIO;
    if (D != 64 && D != 128) return GQA_ERR_UNSUPPORTED;
    const long long R = (long long)(H / G) * sq;
    if (R > 16 * kMaxRowTiles) return GQA_ERR_UNSUPPORTED;
    // Index arithmetic in the kernels uses 32-bit row numbers and coordinates.
    if ((long long)B * sq * H >= (1ll << 31) || (long long)B * G >= (1ll << 31))
        return GQA_ERR_UNSUPPORTED;
    return GQA_OK;
}

// Smallest share of tiles worth giving a CTA. The default (16 tiles, 1024
// tokens, a few microseconds of streaming) keeps small problems from being
// cut into partials whose merge costs more than it saves (the 32 x 1024
// tiny workload: 9 us unsplit against 12 us in four-way splits); the
// environment variable exists for sweeps of the plan and for tests that want
// many splits on small inputs.
int min_tiles_per_cta() {
    const char* s = std::getenv("GQA_DECODE_MIN_TILES_PER_CTA");
    const int x = s ? std::atoi(s) : 0;
    return x > 0 ? x : 16;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// A 48-bit tag per call for the workspace's arrival counters. It starts from
// the clock and the process id so that a workspace left over from another
// process or an aborted call is unlikely to hold a matching tag.
unsigned long long next_epoch() {
    static std::atomic<unsigned long long> counter{
        (static_cast<unsigned long long>(std::chrono::steady_clock::now().time_since_epoch().count()) *
             0x9E3779B97F4A7C15ull ^
         (static_cast<unsigned long long>(getpid()) << 20))};
    const unsigned long long e = counter.fetch_add(1) & 0xFFFFFFFFFFFFull;
    return e;
}

// Test hooks, read per call from the environment: GQA_DECODE_DEBUG_TIMEOUT_MS
// shortens the limit of every device-side wait (default 2 s), and
// GQA_DECODE_DEBUG_SKIP_TILE=n makes CTA 0 skip loading its n-th K/V tile, so
// that its consumers' bounded wait expires and the call reports
// GQA_ERR_DEVICE_TIMEOUT -- the failure path, exercised without faulting.
void debug_knobs(unsigned long long* timeout_ns, int* skip_tile) {
    const char* t = std::getenv("GQA_DECODE_DEBUG_TIMEOUT_MS");
    const long long ms = t ? std::atoll(t) : 0;
    *timeout_ns = ms > 0 ? (unsigned long long)ms * 1000000ull : kWaitTimeoutNs;
    const char* k = std::getenv("GQA_DECODE_DEBUG_SKIP_TILE");
    *skip_tile = k ? std::atoi(k) : -1;
}

// Test hook: GQA_DECODE_DEBUG_EPOCH=n gives every call the same counter tag n,
// as the replays of a call captured in a CUDA graph have, so that a test can
// check that a call that timed out leaves the arrival counters clean for the
// next call with the same tag.
unsigned long long call_epoch() {
    const char* s = std::getenv("GQA_DECODE_DEBUG_EPOCH");
    const long long e = s ? std::atoll(s) : 0;
    return e > 0 ? (unsigned long long)e & 0xFFFFFFFFFFFFull : next_epoch();
}

// When every unit has the same number of tiles (all lengths equal; the
// kernel checks that from the lengths), the tiles are shared by fewer CTAs
// if a grid that keeps at least 80% of them busy lines up with the units: a
// whole number of units per CTA (no unit split, nothing to merge), or, with
// fewer units than CTAs, the same whole number of CTAs per unit (every CTA
// one equal partial) on about 85% of the grid. Measured on the long-context
// and MQA-end workloads: about 85% of the SMs, each unit split evenly, beats
// every SM with uneven splits (fewer partials, HBM still saturated). The
// CTAs left over exit. Computed here, once per call, rather than by every
// CTA before its first copy.
int even_split_ctas(long long units, int ctas) {
    long long P = ctas;
    if (units >= P) {
        const long long per = (units + P - 1) / P;
        const long long even = (units + per - 1) / per;
        if (units % per == 0 && 5 * even >= 4 * P) P = even;
    } else {
        const long long even = units * ((P * 85 / 100) / units);
        if (even >= units && 5 * even >= 4 * P) P = even;
    }
    return (int)P;
}

// Grid size override for sweeps of the plan (unset: the heuristic decides).
int forced_ctas() {
    const char* s = std::getenv("GQA_DECODE_CTAS");
    const int x = s ? std::atoi(s) : 0;
    return x > 0 ? x : 0;
}

}  // namespace

extern "C" {

int gqa_decode_plan(int B, int sq, int H, int G, int D, int Tmax, int num_sms,
                    gqa_decode_plan_t* plan) {
    if (!plan || num_sms <= 0) return GQA_ERR_INVALID_ARG;
    int st = check_shapes(B, sq, H, G, D, Tmax);
    if (st != GQA_OK) return st;
    const int R = (H / G) * sq;
    const int mt = (R + 15) / 16;
    const long long tiles_per_unit = (Tmax + kTileTokens - 1) / kTileTokens;
    const long long max_tiles = (long long)B * G * tiles_per_unit;
    long long ctas = (max_tiles + min_tiles_per_cta() - 1) / min_tiles_per_cta();
    if (ctas > num_sms) ctas = num_sms;
    if (forced_ctas() > 0) ctas = forced_ctas();
    if (ctas > kMaxMergeContrib) ctas = kMaxMergeContrib;
    if (ctas < 1) ctas = 1;
    plan->ctas = (int)ctas;
    plan->tile_tokens = kTileTokens;
    plan->row_tiles = mt;
    plan->stages = splitkv_stages(D, mt);
    plan->threads = splitkv_threads(D, mt);
    plan->smem_bytes = splitkv_smem_bytes(D, mt);
    plan->max_tiles = max_tiles;
    return GQA_OK;
}

size_t gqa_decode_workspace_bytes(int B, int sq, int H, int G, int D, int Tmax) {
    DeviceInfo info;
    if (device_info(&info) != GQA_OK) return 0;
    gqa_decode_plan_t plan;
    if (gqa_decode_plan(B, sq, H, G, D, Tmax, info.sms, &plan) != GQA_OK) return 0;
    return ws_total_bytes(B, G, (H / G) * sq, D, plan.ctas);
}

}  // extern "C"

namespace {

// Checks the arguments, builds the TMA descriptors and the kernel parameters,
// and enqueues the one launch of a decode step (with the fused append when
// k_new/v_new are given).
struct Paging {
    const int32_t* block_table = nullptr;  // null: contiguous cache
    int page_size = 0, num_pages = 0, max_pages = 0;
};

struct Fp8Scales {
    const float* k_scale = nullptr;        // null: bf16 cache
    const float* v_scale = nullptr;
};

int enqueue(const void* q, const void* k_cache, const void* v_cache, const int32_t* seq_lens,
            float scale, void* out, float* lse, int B, int sq, int H, int G, int D, int Tmax,
            void* workspace, size_t workspace_bytes, cudaStream_t stream, const void* k_new,
            const void* v_new, const Paging& pg = Paging(), const Fp8Scales& f8 = Fp8Scales()) {
    const bool kv8 = f8.k_scale != nullptr;
    if (!q || !k_cache || !v_cache || !seq_lens || !out) return GQA_ERR_INVALID_ARG;
    int st = check_shapes(B, sq, H, G, D, Tmax);
    if (st != GQA_OK) return st;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(seq_lens) ||
        !aligned16(out) || (lse && !aligned16(lse)) || (k_new && !aligned16(k_new)) ||
        (v_new && !aligned16(v_new)))
        return GQA_ERR_MISALIGNED;
    DeviceInfo info;
    st = device_info(&info);
    if (st != GQA_OK) return st;
    gqa_decode_plan_t plan;
    st = gqa_decode_plan(B, sq, H, G, D, Tmax, info.sms, &plan);
    if (st != GQA_OK) return st;
    const int R = (H / G) * sq;
    const size_t need = ws_total_bytes(B, G, R, D, plan.ctas);
    if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return GQA_ERR_WORKSPACE;

    LaunchArgs a;
    const long long slabs = pg.block_table ? (long long)pg.num_pages * G : (long long)B * G;
    const int rows = pg.block_table ? pg.page_size : Tmax;
    const int box_rows = pg.block_table && pg.page_size < kTileTokens ? pg.page_size : kTileTokens;
    // Pages shorter than a tile, one row tile: the kernel's stage is
    // page-major and one box per page brings both halves of a bf16 D = 128
    // row (the 4-D view); elsewhere one 3-D box per half (measured as fast).
    const bool both_halves = box_rows < kTileTokens && plan.row_tiles == 1;
    st = encode_cache_map(&a.tm_k, k_cache, slabs, rows, D, box_rows, kv8 ? 1 : 2, both_halves);
    if (st != GQA_OK) return st;
    st = encode_cache_map(&a.tm_v, v_cache, slabs, rows, D, box_rows, kv8 ? 1 : 2, both_halves);
    if (st != GQA_OK) return st;
    a.p.q = static_cast<const uint16_t*>(q);
    a.p.seq_lens = seq_lens;
    a.p.out = static_cast<uint16_t*>(out);
    a.p.lse = lse;
    a.p.ws_counters = static_cast<unsigned long long*>(workspace);
    a.p.ws_part = reinterpret_cast<float*>(static_cast<char*>(workspace) + ws_counter_bytes(B, G));
    a.p.epoch = call_epoch();
    a.p.status = info.status;
    a.p.scale_log2 = scale * 1.4426950408889634f;
    a.p.B = B;
    a.p.sq = sq;
    a.p.H = H;
    a.p.G = G;
    a.p.Tmax = Tmax;
    a.p.R = R;
    a.p.heads_per_group = H / G;
    a.p.ctas = plan.ctas;
    a.p.even_rule = forced_ctas() > 0 ? 0 : 1;
    a.p.even_ctas = even_split_ctas((long long)B * G, plan.ctas);
    // Kernels bound per SM rather than by HBM take every SM: pages shorter
    // than a tile (the TMA boxes per tile bound each SM: the MHA end's
    // layer in 16-token pages 122 -> 109 us on all 152 SMs instead of 128),
    // and fp8 caches with fewer units than half the SMs (long context B = 1
    // 63 -> 59 us). With more units, whole units per CTA keep fp8's merges
    // away (the Llama-shaped layer: 28.7 us on 128 CTAs, 32.2 on 152).
    const bool short_pages = pg.block_table && pg.page_size < kTileTokens;
    if (short_pages || (kv8 && 2ll * B * G < plan.ctas)) a.p.even_ctas = plan.ctas;
    a.p.small_plan = (B <= 64 && plan.max_tiles < (1ll << 31)) ? 1 : 0;
    debug_knobs(&a.p.wait_timeout_ns, &a.p.skip_tile);
    a.p.k_new = static_cast<const uint16_t*>(k_new);
    a.p.v_new = static_cast<const uint16_t*>(v_new);
    a.p.k_cache = static_cast<uint16_t*>(const_cast<void*>(k_cache));
    a.p.v_cache = static_cast<uint16_t*>(const_cast<void*>(v_cache));
    a.p.block_table = pg.block_table;
    a.p.page_size = pg.page_size;
    a.p.max_pages = pg.max_pages;
    a.p.page_loader = (pg.block_table && pg.page_size < kTileTokens && !kv8) ? 1 : 0;
    a.p.k_scale = f8.k_scale;
    a.p.v_scale = f8.v_scale;
    a.p.scale_tiles = (Tmax + kTileTokens - 1) / kTileTokens;
    a.kv8 = kv8;
    a.row_tiles = plan.row_tiles;
    a.pdl = true;
    a.stream = stream;
    cudaError_t e = kv8 ? launch_d128_fp8(a) : (D == 64 ? launch_d64(a) : launch_d128(a));
    if (e != cudaSuccess) return cuda_fail(e);
    return GQA_OK;
}

// The library-owned workspace of (current device, stream, kind), grown to
// `need`.
int stream_workspace(cudaStream_t stream, size_t need, void** ws, size_t* have, int kind = kDecodeWs) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    std::lock_guard<std::mutex> lk(g_mu);
    auto& slot = g_workspaces[{dev, stream, kind}];
    if (slot.second < need) {
        if (slot.first) {
            // The old buffer may still be in use by work queued on this stream.
            e = cudaStreamSynchronize(stream);
            if (e != cudaSuccess) return cuda_fail(e);
            cudaFree(slot.first);
            slot = {nullptr, 0};
        }
        void* p = nullptr;
        e = cudaMalloc(&p, need);
        if (e != cudaSuccess) return cuda_fail(e);
        slot = {p, need};
    }
    *ws = slot.first;
    *have = slot.second;
    return GQA_OK;
}

}  // namespace

extern "C" {

int gqa_decode_ex(const void* q, const void* k_cache, const void* v_cache,
                  const int32_t* seq_lens, float scale, void* out, float* lse, int B, int sq,
                  int H, int G, int D, int Tmax, void* workspace, size_t workspace_bytes,
                  cudaStream_t stream) {
    return enqueue(q, k_cache, v_cache, seq_lens, scale, out, lse, B, sq, H, G, D, Tmax, workspace,
                   workspace_bytes, stream, nullptr, nullptr);
}

int gqa_decode(const void* q, const void* k_cache, const void* v_cache, const int32_t* seq_lens,
               float scale, void* out, float* lse, int B, int sq, int H, int G, int D, int Tmax,
               cudaStream_t stream) {
    // More than 32 rows per KV head: the same attention on the prefill kernel.
    if (B > 0 && sq > 0 && H > 0 && G > 0 && H % G == 0 && (long long)(H / G) * sq > 16 * kMaxRowTiles)
        return gqa_prefill(q, k_cache, v_cache, seq_lens, scale, out, lse, B, sq, H, G, D, Tmax, stream);
    int st = check_shapes(B, sq, H, G, D, Tmax);
    if (st != GQA_OK) return st;
    if (!q || !k_cache || !v_cache || !seq_lens || !out) return GQA_ERR_INVALID_ARG;
    const size_t need = gqa_decode_workspace_bytes(B, sq, H, G, D, Tmax);
    if (need == 0) return GQA_ERR_CUDA;
    void* ws = nullptr;
    size_t have = 0;
    st = stream_workspace(stream, need, &ws, &have);
    if (st != GQA_OK) return st;
    return enqueue(q, k_cache, v_cache, seq_lens, scale, out, lse, B, sq, H, G, D, Tmax, ws, have,
                   stream, nullptr, nullptr);
}

int gqa_decode_append(const void* q, const void* k_new, const void* v_new, void* k_cache,
                      void* v_cache, const int32_t* seq_lens, float scale, void* out, float* lse,
                      int B, int sq, int H, int G, int D, int Tmax, cudaStream_t stream) {
    int st = check_shapes(B, sq, H, G, D, Tmax);
    if (st != GQA_OK) return st;
    if (!q || !k_new || !v_new || !k_cache || !v_cache || !seq_lens || !out)
        return GQA_ERR_INVALID_ARG;
    const size_t need = gqa_decode_workspace_bytes(B, sq, H, G, D, Tmax);
    if (need == 0) return GQA_ERR_CUDA;
    void* ws = nullptr;
    size_t have = 0;
    st = stream_workspace(stream, need, &ws, &have);
    if (st != GQA_OK) return st;
    return enqueue(q, k_cache, v_cache, seq_lens, scale, out, lse, B, sq, H, G, D, Tmax, ws, have,
                   stream, k_new, v_new);
}

int gqa_decode_paged(const void* q, const void* k_pages, const void* v_pages,
                     const int32_t* block_table, const int32_t* seq_lens, float scale, void* out,
                     float* lse, int B, int sq, int H, int G, int D, int page_size, int num_pages,
                     int max_pages_per_seq, cudaStream_t stream) {
    if (page_size < 16 || page_size > 65536 || (page_size & (page_size - 1)) || num_pages <= 0 ||
        max_pages_per_seq <= 0)
        return page_size <= 0 || num_pages <= 0 || max_pages_per_seq <= 0 ? GQA_ERR_INVALID_ARG
                                                                           : GQA_ERR_UNSUPPORTED;
    const long long tmax = (long long)max_pages_per_seq * page_size;
    if (tmax >= (1ll << 31) || (long long)num_pages * G >= (1ll << 31)) return GQA_ERR_UNSUPPORTED;
    const int Tmax = (int)tmax;
    int st = check_shapes(B, sq, H, G, D, Tmax);
    if (st != GQA_OK) return st;
    if (!q || !k_pages || !v_pages || !block_table || !seq_lens || !out) return GQA_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(block_table) & 3u) return GQA_ERR_MISALIGNED;
    const size_t need = gqa_decode_workspace_bytes(B, sq, H, G, D, Tmax);
    if (need == 0) return GQA_ERR_CUDA;
    void* ws = nullptr;
    size_t have = 0;
    st = stream_workspace(stream, need, &ws, &have);
    if (st != GQA_OK) return st;
    Paging pg;
    pg.block_table = block_table;
    pg.page_size = page_size;
    pg.num_pages = num_pages;
    pg.max_pages = max_pages_per_seq;
    return enqueue(q, k_pages, v_pages, seq_lens, scale, out, lse, B, sq, H, G, D, Tmax, ws, have,
                   stream, nullptr, nullptr, pg);
}

int gqa_decode_fp8(const void* q, const void* k_codes, const void* v_codes, const float* k_scale,
                   const float* v_scale, const int32_t* seq_lens, float scale, void* out, float* lse,
                   int B, int sq, int H, int G, int D, int Tmax, cudaStream_t stream) {
    int st = check_shapes(B, sq, H, G, D, Tmax);
    if (st != GQA_OK) return st;
    if (D != 128) return GQA_ERR_UNSUPPORTED;
    if (!q || !k_codes || !v_codes || !k_scale || !v_scale || !seq_lens || !out)
        return GQA_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(k_scale) & 3u) || (reinterpret_cast<uintptr_t>(v_scale) & 3u))
        return GQA_ERR_MISALIGNED;
    const size_t need = gqa_decode_workspace_bytes(B, sq, H, G, D, Tmax);
    if (need == 0) return GQA_ERR_CUDA;
    void* ws = nullptr;
    size_t have = 0;
    st = stream_workspace(stream, need, &ws, &have);
    if (st != GQA_OK) return st;
    Fp8Scales f8;
    f8.k_scale = k_scale;
    f8.v_scale = v_scale;
    return enqueue(q, k_codes, v_codes, seq_lens, scale, out, lse, B, sq, H, G, D, Tmax, ws, have,
                   stream, nullptr, nullptr, Paging(), f8);
}

int gqa_prefill(const void* q, const void* k_cache, const void* v_cache, const int32_t* seq_lens,
                float scale, void* out, float* lse, int B, int sq, int H, int G, int D, int Tmax,
                cudaStream_t stream) {
    if (B <= 0 || sq <= 0 || H <= 0 || G <= 0 || D <= 0 || Tmax <= 0) return GQA_ERR_INVALID_ARG;
    if (!(scale > 0.f) || scale > 3.0e38f) return GQA_ERR_INVALID_ARG;   // the row max is taken before scaling
    if (H % G != 0) return GQA_ERR_HEAD_RATIO;
    if (D != 64 && D != 128) return GQA_ERR_UNSUPPORTED;
    if (!q || !k_cache || !v_cache || !seq_lens || !out) return GQA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(seq_lens) ||
        !aligned16(out) || (lse && !aligned16(lse)))
        return GQA_ERR_MISALIGNED;
    const long long R = (long long)(H / G) * sq;
    const long long row_tiles = (R + 127) / 128;
    if ((long long)B * sq * H >= (1ll << 31) || R >= (1ll << 31) ||
        (long long)B * G * row_tiles >= (1ll << 31))
        return GQA_ERR_UNSUPPORTED;
    DeviceInfo info;
    int st = device_info(&info);
    if (st != GQA_OK) return st;
    // Short chunks: when the pairs of row tiles cannot fill the SMs, each
    // pair's key range is shared by several CTAs (at least two key tiles
    // each) and a second kernel merges their partials.
    const long long items = (long long)B * G * ((row_tiles + 1) / 2);
    const long long key_tiles = (Tmax + 127) / 128;
    long long splits = 1;
    if (2 * items <= info.sms) {
        splits = info.sms / items;   // one wave
        if (splits > key_tiles / 2) splits = key_tiles / 2;
        if (splits < 1) splits = 1;
    }
    if (const char* f = std::getenv("GQA_PREFILL_SPLITS")) {   // sweeps and tests
        const long long x = std::atoll(f);
        if (x > 0) splits = x;
    }
    if (splits > 32) splits = 32;   // the combine keeps one split per lane
    if (items * splits >= (1ll << 31)) return GQA_ERR_UNSUPPORTED;
    void* ws = nullptr;
    size_t have = 0;
    const size_t need = prefill_workspace_bytes(D, items, (int)splits);
    if (need > 0) {
        st = stream_workspace(stream, need, &ws, &have, kPrefillWs);
        if (st != GQA_OK) return st;
    }
    PrefillLaunchArgs a{};
    st = encode_cache_map(&a.tm_k, k_cache, (long long)B * G, Tmax, D, 128);
    if (st != GQA_OK) return st;
    st = encode_cache_map(&a.tm_v, v_cache, (long long)B * G, Tmax, D, 128);
    if (st != GQA_OK) return st;
    a.p.q = static_cast<const uint16_t*>(q);
    a.p.seq_lens = seq_lens;
    a.p.out = static_cast<uint16_t*>(out);
    a.p.lse = lse;
    a.p.status = info.status;
    a.p.scale_log2 = scale * 1.4426950408889634f;
    a.p.B = B;
    a.p.sq = sq;
    a.p.H = H;
    a.p.G = G;
    a.p.Tmax = Tmax;
    a.p.R = (int)R;
    a.p.heads_per_group = H / G;
    a.p.row_tiles = (int)row_tiles;
    debug_knobs(&a.p.wait_timeout_ns, &a.p.skip_tile);
    a.p.splits = (int)splits;
    a.p.ws_part = static_cast<float*>(ws);
    a.grid = (unsigned)(items * splits);   // (pair of row tiles, key range)
    // The combine of a split chunk (always one wave of CTAs) launches with
    // programmatic dependent launch.
    a.pdl = a.grid <= (unsigned)info.sms;
    a.stream = stream;
    cudaError_t e = launch_prefill(D, a);
    if (e != cudaSuccess) return cuda_fail(e);
    return GQA_OK;
}

int gqa_decode_check_error(cudaStream_t stream) {
    cudaError_t e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return cuda_fail(e);
    DeviceInfo info;
    int st = device_info(&info);
    if (st != GQA_OK) return st;
    unsigned word = 0;
    e = cudaMemcpy(&word, info.status, sizeof word, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e);
    if (word) {
        const unsigned zero = 0;
        e = cudaMemcpy(info.status, &zero, sizeof zero, cudaMemcpyHostToDevice);
        if (e != cudaSuccess) return cuda_fail(e);
        if (word & kStatusTimeout) return GQA_ERR_DEVICE_TIMEOUT;
    }
    return GQA_OK;
}

int gqa_decode_release_workspace(cudaStream_t stream) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    std::lock_guard<std::mutex> lk(g_mu);
    bool synced = false;
    for (int kind : {kDecodeWs, kPrefillWs}) {
        auto it = g_workspaces.find({dev, stream, kind});
        if (it == g_workspaces.end()) continue;
        // Work already queued on the stream may still use the buffer.
        if (!synced) {
            e = cudaStreamSynchronize(stream);
            if (e != cudaSuccess) return cuda_fail(e);
            synced = true;
        }
        void* buf = it->second.first;
        g_workspaces.erase(it);
        if (buf) {
            e = cudaFree(buf);
            if (e != cudaSuccess) return cuda_fail(e);
        }
    }
    return GQA_OK;
}

int gqa_decode_last_cuda_error(void) { return t_last_cuda_error; }

const char* gqa_decode_strerror(int status) {
    switch (status) {
        case GQA_OK: return "ok";
        case GQA_ERR_INVALID_ARG: return "invalid argument (null pointer or non-positive size)";
        case GQA_ERR_HEAD_RATIO: return "H is not a multiple of G";
        case GQA_ERR_UNSUPPORTED: return "unsupported shape (D must be 64 or 128; (H/G)*sq <= 32 except for gqa_decode and gqa_prefill)";
        case GQA_ERR_MISALIGNED: return "a tensor pointer is not 16-byte aligned";
        case GQA_ERR_WORKSPACE: return "workspace missing, too small or not 256-byte aligned";
        case GQA_ERR_CUDA: return "a CUDA call failed (see gqa_decode_last_cuda_error)";
        case GQA_ERR_DEVICE_TIMEOUT: return "a bounded device-side wait expired";
        default: return "unknown status";
    }
}

}  // extern "C"

namespace gqa {

template <template <int, int, bool> class F>
int shape_query(int D, int mt, bool kv8) {
    if (kv8) return mt == 1 ? F<128, 1, true>::value : F<128, 2, true>::value;
    if (D == 64) return mt == 1 ? F<64, 1, false>::value : F<64, 2, false>::value;
    return mt == 1 ? F<128, 1, false>::value : F<128, 2, false>::value;
}
template <int D, int MT, bool KV8> struct SmemQ { static constexpr int value = KernelShape<D, MT, KV8>::kSmemBytes; };
template <int D, int MT, bool KV8> struct ThrQ { static constexpr int value = KernelShape<D, MT, KV8>::kThreads; };
template <int D, int MT, bool KV8> struct StgQ { static constexpr int value = KernelShape<D, MT, KV8>::kStages; };

int splitkv_smem_bytes(int D, int mt, bool kv8) { return shape_query<SmemQ>(D, mt, kv8); }
int splitkv_threads(int D, int mt, bool kv8) { return shape_query<ThrQ>(D, mt, kv8); }
int splitkv_stages(int D, int mt, bool kv8) { return shape_query<StgQ>(D, mt, kv8); }

}  // namespace gqa
