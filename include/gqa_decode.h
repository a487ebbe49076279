/*
 * gqa_decode.h -- C ABI of the GB300 (sm_103a) grouped-query decode attention
 * library, libgqa_decode.so.
 *
 * The operation ("GQA analysis", section "Grouped broadcast"): with H query
 * heads sharing G key/value heads, query head h reads only KV head
 *     g(h) = floor(h / (H / G)),
 *     score[h] = softmax(Q[h] . K[g(h)]^T * scale),
 *     O[h]     = score[h] . V[g(h)].
 * The page's scale is 1/sqrt(D); here it is an argument. G = H is multi-head
 * attention and G = 1 is multi-query attention ("Fast Transformer Decoding
 * with Multi-Query Attention" digest, section "Multi-Query Attention"); H must
 * be a multiple of G ("keep query heads, cut KV heads", section "three names
 * on one axis").
 *
 * One call is one decode step of one layer: the inner per-head loop of the
 * incremental decode in "GQA analysis", section "Incremental decode", for
 * every sequence of the batch. The sq new tokens' K/V must already be appended
 * to the cache (the page appends before attending), so seq_lens[b] counts them.
 * For sq > 1 the new tokens are causal among themselves, bottom-right aligned
 * (the mask-handling part of section 7 of "Same GQA, Different Execution Cost
 * Across Backends"): new token s sits at absolute position T_b - sq + s and
 * attends to cache positions t <= T_b - sq + s.
 *
 * Layouts (all dense, C-contiguous, device memory, 16-byte aligned):
 *   q        [B, sq, H, D]    bfloat16
 *   k_cache  [B, G, Tmax, D]  bfloat16 (the [batch, kv_heads, seq, head_dim]
 *   v_cache  [B, G, Tmax, D]  bfloat16  cache of "GQA analysis", section 4)
 *   seq_lens [B]              int32, valid entries per sequence (incl. the new
 *                             tokens); values are clamped to [0, Tmax] on the
 *                             device. Entries at t >= seq_lens[b] are never
 *                             used, whatever they hold.
 *   out      [B, sq, H, D]    bfloat16, round-to-nearest-even of the fp32 result
 *   lse      [B, sq, H]       float32, natural log of sum_t exp(scale * q.k_t)
 *                             over the visible keys; may be NULL (not written)
 * Supported: D in {64, 128}. gqa_decode accepts any number of query rows per
 * KV head, R = (H/G)*sq: up to 32 it runs the split-KV decode kernel, above
 * that the prefill kernel (see gqa_prefill, which also needs scale > 0). The
 * other decode entry points (workspace, plan, append, paged, fp8, no-alloc)
 * take R <= 32.
 * A row with no visible key (T_b - sq + s < 0) gets out = 0 and lse = -inf.
 *
 * Device: every pointer is device memory of the current CUDA device (the one
 * cudaGetDevice returns in the calling thread) and `stream` belongs to that
 * device. Like other CUDA libraries, the library does not look up where a
 * pointer lives: a host pointer or another device's memory is undefined
 * behaviour. (The Python binding checks that all tensors share one device and
 * makes it current for the call.)
 *
 * Ownership and ordering: the caller owns every tensor and the stream. All
 * work is enqueued on `stream` (0 = legacy default stream); no call
 * synchronises the host except gqa_decode_check_error. Inputs must not be
 * modified, and outputs not read, until the work on `stream` has completed.
 *
 * Errors: functions return GQA_OK (0) or one of the negative codes below and
 * then enqueue nothing. GQA_ERR_CUDA means a CUDA call failed; the CUDA error
 * is available from gqa_decode_last_cuda_error(). Device-side faults of the
 * kind the kernels can detect (a bounded pipeline wait that expired) are
 * recorded in a per-device status word and reported by
 * gqa_decode_check_error().
 */
#ifndef GQA_DECODE_H
#define GQA_DECODE_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define GQA_OK 0
#define GQA_ERR_INVALID_ARG -1     /* null pointer, a size <= 0, Tmax < sq, ... */
#define GQA_ERR_HEAD_RATIO -2      /* H % G != 0 */
#define GQA_ERR_UNSUPPORTED -3     /* D not in {64,128}, R > 32, sizes out of range */
#define GQA_ERR_MISALIGNED -4      /* a tensor pointer not 16-byte aligned */
#define GQA_ERR_WORKSPACE -5       /* caller workspace NULL or smaller than required */
#define GQA_ERR_CUDA -6            /* a CUDA runtime/driver call failed */
#define GQA_ERR_DEVICE_TIMEOUT -7  /* a bounded device-side wait expired */

/*
 * Decode attention for one step, using a workspace the library owns: one
 * grow-only device buffer per (device, stream), allocated with cudaMalloc on
 * the first call that needs more than the stream's buffer holds. Calls on the
 * same stream are ordered; calls on different streams use different buffers.
 * Make one call per stream before capturing that stream into a CUDA graph, so
 * that no allocation happens during capture. A captured call can be replayed
 * with new contents of the same tensors (values and seq_lens): the plan
 * depends on the shapes only, and the kernels leave the workspace's arrival
 * counters at zero after each merge -- also after a call whose bounded wait
 * expired -- so every replay starts from a clean count.
 *
 * q, k_cache, v_cache, seq_lens, out, lse: device pointers, layouts above.
 * scale: multiplier applied to q.k (1/sqrt(D) for the pages' definition).
 * B, sq, H, G, D, Tmax: sizes; stream: the CUDA stream to enqueue on.
 */
int gqa_decode(const void* q, const void* k_cache, const void* v_cache,
               const int32_t* seq_lens, float scale, void* out, float* lse,
               int B, int sq, int H, int G, int D, int Tmax, cudaStream_t stream);

/*
 * Decode step with the new tokens' K/V appended to the cache in the same
 * launch: the per-layer step of "GQA analysis", section "Incremental decode",
 * which appends k_t and v_t to the caches and then attends over them.
 *
 * k_new, v_new: [B, sq, G, D] bf16, device, 16-byte aligned -- the sq new
 * tokens' keys (already rotated, if the model uses RoPE) and values per KV
 * head. seq_lens counts the cache entries including the new ones, as for
 * gqa_decode: new token s of sequence b is written to
 * k_cache[b, g, T_b - sq + s, :] (T_b clamped to [0, Tmax]; positions below 0
 * are not written) and v_cache likewise; every other cache entry is left as
 * it is. The result is the same as writing those rows first and then calling
 * gqa_decode; the rows are written by the same launch, which reads them from
 * k_new/v_new rather than back from the cache. Library-owned workspace, as for
 * gqa_decode. The caches must not be read or written by other work until the
 * call has completed on `stream`.
 */
int gqa_decode_append(const void* q, const void* k_new, const void* v_new, void* k_cache,
                      void* v_cache, const int32_t* seq_lens, float scale, void* out, float* lse,
                      int B, int sq, int H, int G, int D, int Tmax, cudaStream_t stream);

/*
 * Decode step over a paged KV cache: the same attention as gqa_decode, with
 * each sequence's cache held in fixed-size pages reached through a block table
 * (the PagedAttention placement that "GQA analysis" names as orthogonal to GQA,
 * sections "Tensor parallelism and kernel constraints" and "pros").
 *
 * k_pages, v_pages: [num_pages, G, page_size, D] bf16, device, 16-byte aligned:
 *   page p holds page_size consecutive tokens of one sequence for every KV
 *   head, each head's rows contiguous.
 * block_table: [B, max_pages_per_seq] int32, device: entry (b, j) is the page
 *   holding tokens [j*page_size, (j+1)*page_size) of sequence b. Only entries
 *   for pages that start before seq_lens[b] are read; an entry outside
 *   [0, num_pages) reads as zeros (no fault).
 * page_size: a power of two, 16 <= page_size <= 65536. The cache capacity per
 *   sequence is Tmax = max_pages_per_seq * page_size; seq_lens are clamped to it.
 * Library-owned workspace, as for gqa_decode.
 */
int gqa_decode_paged(const void* q, const void* k_pages, const void* v_pages,
                     const int32_t* block_table, const int32_t* seq_lens, float scale, void* out,
                     float* lse, int B, int sq, int H, int G, int D, int page_size, int num_pages,
                     int max_pages_per_seq, cudaStream_t stream);

/*
 * Decode step over an fp8 KV cache: KV-cache quantisation, which "GQA
 * analysis" names as orthogonal to GQA (element precision, with scale
 * metadata; sections "KV cache" and "pros"). Each element is stored as an
 * e4m3 code (OCP FP8 E4M3: 1 sign, 4 exponent bits with bias 7, 3 mantissa
 * bits, no infinities, S.1111.111 is NaN) and one fp32 scale covers a 64-token
 * block of one (sequence, KV head): value = decode(code) * scale. Same
 * attention and outputs as gqa_decode over the dequantised cache.
 *
 * k_codes, v_codes: [B, G, Tmax, D] uint8 e4m3 codes, device, 16-byte aligned.
 * k_scale, v_scale: [B, G, ceil(Tmax / 64)] fp32, device; entry (b, g, j)
 *   scales tokens [64 j, 64 j + 64) of KV head g of sequence b.
 * D must be 128. The tensor-core products run in fp16 (every e4m3 value and
 * the bf16 queries of ordinary magnitude, |q| < 65504, are exact in fp16).
 * Library-owned workspace, as for gqa_decode.
 */
int gqa_decode_fp8(const void* q, const void* k_codes, const void* v_codes, const float* k_scale,
                   const float* v_scale, const int32_t* seq_lens, float scale, void* out, float* lse,
                   int B, int sq, int H, int G, int D, int Tmax, cudaStream_t stream);

/*
 * Prefill and chunked prefill: the attention of gqa_decode for any number of
 * new tokens per sequence. Section 7 of "Same GQA, Different Execution Cost
 * Across Backends" ("in prefill, merge the group into the sequence axis")
 * folds the H/G query heads that share a KV head into the row axis,
 * [B, Hkv, G x M, D], so each KV head's K and V serve all (H/G) * sq of its
 * rows at once, and each row keeps its own causal limit and softmax. Same
 * arguments, layouts, causal rule (new token s at position T_b - sq + s sees
 * keys t <= T_b - sq + s), outputs and error codes as gqa_decode, with no
 * bound on (H/G) * sq; D in {64, 128}; scale must be finite and > 0
 * (GQA_ERR_INVALID_ARG otherwise). A fresh prefill has T_b = sq; a
 * chunked prefill has the earlier chunks' K/V in the cache as well.
 *
 * The products run on the tcgen05 tensor cores (bf16 inputs, fp32
 * accumulation in tensor memory, probabilities rounded to bf16 for P.V). One
 * CTA computes each pair of 128-row tiles of one (sequence, KV head) over its
 * key range. When those pairs cannot fill the GPU (short chunks), each pair's
 * key range is shared by several CTAs that write partial results to a
 * library-owned workspace (per device and stream, as for gqa_decode; make one
 * call per stream before capturing it into a CUDA graph), and a second kernel
 * merges them. Asynchronous on `stream`; a bounded device-side wait that
 * expires is reported by gqa_decode_check_error().
 */
int gqa_prefill(const void* q, const void* k_cache, const void* v_cache, const int32_t* seq_lens,
                float scale, void* out, float* lse, int B, int sq, int H, int G, int D, int Tmax,
                cudaStream_t stream);

/*
 * Bytes of device workspace gqa_decode_ex needs for these sizes on the current
 * device: one 64-bit arrival counter per (sequence, KV head, 16-row tile),
 * then two partial-result slots (O[R][D] normalised by its own sum, running
 * max m[R], sum l[R]) per split-KV CTA. Returns 0 for unsupported arguments.
 */
size_t gqa_decode_workspace_bytes(int B, int sq, int H, int G, int D, int Tmax);

/*
 * Same as gqa_decode, with a caller-owned device workspace of at least
 * gqa_decode_workspace_bytes(...) bytes, 256-byte aligned. It needs no
 * initialisation. Two calls that are in flight at the same time must not share
 * a workspace.
 */
int gqa_decode_ex(const void* q, const void* k_cache, const void* v_cache,
                  const int32_t* seq_lens, float scale, void* out, float* lse,
                  int B, int sq, int H, int G, int D, int Tmax,
                  void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * The work plan a call would use, for inspection and tests. Host-only; needs
 * no GPU. The KV stream of all (sequence, KV head) units is cut into tiles of
 * `tile_tokens` tokens; the `ctas` persistent CTAs each take an equal,
 * contiguous share of the flattened tile list, so a unit's context is split
 * wherever those shares cut it. `num_sms` is the device's SM count.
 */
typedef struct gqa_decode_plan_t {
    int ctas;              /* grid size of the split-KV kernel */
    int tile_tokens;       /* tokens per pipeline stage */
    int row_tiles;         /* 16-row MMA tiles per KV head: ceil(R / 16) */
    int stages;            /* depth of the shared-memory K/V ring */
    int threads;           /* threads per CTA (consumer, producer, page-loader and counter warps) */
    int smem_bytes;        /* dynamic shared memory per CTA */
    long long max_tiles;   /* B * G * ceil(Tmax / tile_tokens): tiles if every T_b = Tmax */
} gqa_decode_plan_t;

int gqa_decode_plan(int B, int sq, int H, int G, int D, int Tmax, int num_sms,
                    gqa_decode_plan_t* plan);

/*
 * Synchronises `stream`, then reads and clears the current device's status
 * word. Returns GQA_OK, GQA_ERR_DEVICE_TIMEOUT if a kernel gave up on a
 * bounded wait since the last check (its outputs are then undefined), or
 * GQA_ERR_CUDA.
 */
int gqa_decode_check_error(cudaStream_t stream);

/*
 * Allocation-free variant of gqa_decode, for callers that must not allocate
 * device memory while they run: a serving engine that hands all device memory
 * to its own pool at start-up, a plugin inside another framework that gets
 * tensors but no allocator, or a decode loop that cannot afford cudaMalloc's
 * implicit synchronisation. The pages have no counterpart of this; it is a
 * property of this library's interface, not of the attention it computes.
 *
 * Same arguments, layouts and results as gqa_decode for up to 32 query rows
 * per KV head, (H/G)*sq <= 32: the split-KV decode kernel. gqa_decode sends
 * larger row counts to the prefill kernel, whose split key ranges take a
 * library-allocated workspace, so this entry point refuses them with
 * GQA_ERR_UNSUPPORTED and enqueues nothing. The split-KV scratch
 * comes from a fixed array of GQA_NOALLOC_SCRATCH_BYTES in device memory that
 * every GPU which loads the library holds until the process exits; the call
 * makes no cudaMalloc or cudaFree. The first call on a device looks up that
 * array's device address (with the device current), so make that first call
 * before capturing a stream into a CUDA graph.
 *
 * The array is shared by every call on a device and keeps the last call's
 * contents: two calls that overlap on the GPU (different streams, no ordering
 * between them) race on it and give undefined results; order them, or use
 * gqa_decode_ex with one workspace each. A problem whose scratch need,
 * gqa_decode_workspace_bytes(...), exceeds GQA_NOALLOC_SCRATCH_BYTES is
 * rejected with GQA_ERR_WORKSPACE and nothing is enqueued.
 */
#define GQA_NOALLOC_SCRATCH_BYTES (8u << 20) /* 8 MiB per device */

int gqa_decode_noalloc(const void* q, const void* k_cache, const void* v_cache,
                       const int32_t* seq_lens, float scale, void* out, float* lse,
                       int B, int sq, int H, int G, int D, int Tmax, cudaStream_t stream);

/*
 * Frees the workspace the library owns for (current device, `stream`): the
 * buffer gqa_decode, gqa_decode_append, gqa_decode_paged and gqa_decode_fp8
 * grow on that stream, and the separate one of gqa_prefill's split key
 * ranges. Call it before destroying a stream that
 * the library was used on, or to give the memory back; a later call on the
 * stream allocates again. It synchronises `stream` first (work already
 * queued may use the buffer). Returns GQA_OK (also when the library holds
 * nothing for the stream) or GQA_ERR_CUDA. The pages have no counterpart of
 * this; it belongs to this library's memory management ("GQA analysis",
 * section "Incremental decode", leaves the cache to the caller, so the
 * library's own buffers are the only memory it has to give back).
 */
int gqa_decode_release_workspace(cudaStream_t stream);

/* The cudaError_t of the last failed CUDA call in this thread (0 if none). */
int gqa_decode_last_cuda_error(void);

/* A static, human-readable description of a status code. */
const char* gqa_decode_strerror(int status);

#ifdef __cplusplus
}
#endif

#endif /* GQA_DECODE_H */
