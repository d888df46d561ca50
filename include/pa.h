/*
 * pa.h -- C ABI of the GB300 paged-attention decode library (libpa.so).
 *
 * What the library computes comes from three web pages, cited by title and part:
 *   [TALK] "vLLM Project Update" (Bay.Area.AI talk transcript): PagedAttention is an
 *          attention algorithm over blocks of KV cache managed like virtual-memory
 *          pages; the first kernel gave each sequence to one SM, which left SMs
 *          unevenly loaded; the V2 kernel partitions each sequence into pieces spread
 *          over SMs, "similar to flash decoding".
 *   [HN]   "vLLM: Easy, Fast, and Cheap LLM Serving with PagedAttention" (Hacker News
 *          thread): PagedAttention still computes exact attention; the KV cache of one
 *          LLaMA-13B sequence is up to 1.7 GB.
 *   [PR]   "[core] Multi Step Scheduling #7000": the decode metadata slot_mapping,
 *          block_tables and seq_lens, advanced between the steps of a multi-step
 *          decode loop, and the v2 block manager that hands out physical blocks.
 *
 * Conventions shared by every call
 *   Ownership.  The caller owns every buffer.  Device buffers are plain device
 *     pointers (for example from torch); the library never allocates, frees or
 *     retains them.  The decode calls that need scratch take a caller-provided device
 *     workspace sized by the matching *_workspace_size call.
 *   Layouts.  All tensors are dense and row-major, in elements of the call's dtype:
 *       query, out          [num_seqs][num_q_heads][head_size]
 *       key, value (new)    [num_tokens][num_kv_heads][head_size]
 *       key_cache,
 *       value_cache         [num_blocks][num_kv_heads][block_size][head_size]
 *       block_tables        int32 [num_seqs][max_blocks_per_seq]; entry j of row s is
 *                           the physical block holding tokens j*block_size ..
 *                           (j+1)*block_size-1 of sequence s; entries past the
 *                           sequence's last block are never read (pad with -1).
 *       context_lens        int32 [num_seqs], tokens of each sequence INCLUDING the
 *                           token of this step, which reshape_and_cache wrote first.
 *       slot_mapping        int32 [num_tokens], flat slot block*block_size+offset per
 *                           new token; a negative slot marks a padding token.
 *     Query head h attends through kv head h / (num_q_heads / num_kv_heads).
 *     Device pointers must be 16-byte aligned.
 *   Supported shapes.  head_size 64 or 128; block_size 16 or 32; num_q_heads a
 *     multiple of num_kv_heads with a group of at most 16; fp16 or bf16.  Other
 *     combinations return PA_ERR_UNSUPPORTED.
 *   Streams.  Every device call is asynchronous on `stream` (a cudaStream_t; NULL is
 *     the legacy default stream) and never synchronises the host.  The library's kernels
 *     are launched as programmatic dependents (CUDA programmatic dependent launch): each
 *     may start before the kernel ahead of it on the stream has finished, and none writes
 *     global memory before it has waited for that kernel.  A decode kernel lets the kernel
 *     after it launch once its last tiles are being read; a kernel of the caller's that is
 *     launched without the programmatic-serialisation attribute is ordered as usual.
 *   Errors.  Calls return a pa_status; pa_last_error() gives this thread's message
 *     for the last failure.  Host-detectable errors (bad sizes, null pointers) are
 *     reported before any launch.  Errors only the device can see (a slot or block-
 *     table entry outside the pool, a context longer than max_context_len or than
 *     the block-table row, a pipeline wait that exceeded its time limit) never fault:
 *     the offending access is skipped, and if `status_dev` is not NULL the kernel ORs
 *     the matching PA_DEVERR_* bit into that device int32.
 *
 * A typical decode step (one layer, one new token per running sequence)
 *   host    pa_alloc_append_batch        the slot of each sequence's new token (a new
 *                                        block is popped when the last one is full)
 *           pa_alloc_block_tables,       the tables and lengths, copied to the device
 *           pa_alloc_context_lens        with the slots
 *   device  pa_reshape_and_cache         the new K / V rows into the pools by slot
 *           pa_decode_auto               out <- attention of each query over its
 *                                        sequence's pooled tokens (workspace of
 *                                        pa_decode_auto_workspace_size bytes)
 *   pa_decode_step issues both device calls at once; pa_decode_step_host also copies
 *   the step's inputs from host memory and the output back; pa_advance_step moves the
 *   lengths and slots on the device between the steps of a multi-step loop.
 */
#ifndef PA_H_
#define PA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    PA_OK = 0,
    PA_ERR_INVALID_ARG = 1,   /* null pointer, negative size, inconsistent sizes */
    PA_ERR_UNSUPPORTED = 2,   /* dtype / head_size / block_size / group not built */
    PA_ERR_NO_BLOCKS = 3,     /* allocator: not enough free blocks (nothing changed) */
    PA_ERR_CUDA = 4,          /* a CUDA runtime or driver call failed */
    PA_ERR_WORKSPACE = 5      /* workspace NULL or smaller than *_workspace_size */
} pa_status;

/* Element types.  PA_FP8_E4M3 (OCP E4M3FN: 1 sign, 4 exponent bits with bias 7, 3
 * fraction bits, no infinities, largest finite 448) is a cache type only: see
 * pa_reshape_and_cache_fp8 / pa_decode_fp8 / pa_copy_blocks. */
typedef enum { PA_F16 = 0, PA_BF16 = 1, PA_FP8_E4M3 = 2 } pa_dtype;

/* Same type as cudaStream_t, so callers without CUDA headers can still link. */
typedef struct CUstream_st* pa_stream;

/* Bits a kernel ORs into *status_dev. */
#define PA_DEVERR_BAD_SLOT 1   /* slot_mapping entry >= num_blocks * block_size */
#define PA_DEVERR_BAD_BLOCK 2  /* block-table entry outside [0, num_blocks) */
#define PA_DEVERR_BAD_LEN 4    /* context_len > max_context_len or > row capacity; clamped */
#define PA_DEVERR_TIMEOUT 8    /* a shared-memory pipeline wait passed its time limit */

/* Message of this thread's last failed call ("" if none).  Valid until the next call. */
const char* pa_last_error(void);

/* Library version, major * 10000 + minor * 100 + patch. */
int32_t pa_version(void);

/* ------------------------------------------------------------------------------ */
/* reshape_and_cache                                                              */
/* ------------------------------------------------------------------------------ */
/* Scatters the K and V rows of each new token into the paged pools [PR, slot_mapping]:
 *   key_cache[slot / block_size][h][slot % block_size][:] = key[i][h][:]
 * and the same for value, for every token i with slot = slot_mapping[i] >= 0 and every
 * kv head h.  A pure copy: bit-exact.  Slots beyond the pool are skipped and flagged
 * PA_DEVERR_BAD_SLOT.  Two tokens with the same slot in one call race (undefined). */
pa_status pa_reshape_and_cache(const void* key, const void* value, void* key_cache,
                               void* value_cache, const int32_t* slot_mapping,
                               int32_t num_tokens, int32_t num_kv_heads, int32_t head_size,
                               int32_t block_size, int32_t num_blocks, pa_dtype dtype,
                               int32_t* status_dev, pa_stream stream);

/* ------------------------------------------------------------------------------ */
/* Paged decode attention                                                          */
/* ------------------------------------------------------------------------------ */
/* One new query token per sequence attends over its whole context [TALK, HN]:
 *   out[s][h][:] = sum_t softmax_t(scale * q[s][h] . k_t) v_t,   t < context_lens[s],
 * with k_t, v_t row t % block_size of physical block block_tables[s][t / block_size]
 * for kv head h / group.  fp32 accumulation; the output is rounded to `dtype`.
 * A context length of 0 gives a zero row.  max_context_len is an upper bound the
 * host knows (no device read-back); longer contexts are clamped and flagged.
 *
 * pa_decode_v1: one work unit per (sequence, kv head) over the whole context -- the
 *   first kernel of [TALK].  Needs no workspace. */
pa_status pa_decode_v1(void* out, const void* query, const void* key_cache,
                       const void* value_cache, const int32_t* block_tables,
                       int32_t max_blocks_per_seq, const int32_t* context_lens,
                       int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                       int32_t head_size, int32_t block_size, int32_t num_blocks,
                       int32_t max_context_len, float scale, pa_dtype dtype,
                       int32_t* status_dev, pa_stream stream);

/* Bytes of device workspace pa_decode_v2 needs for these sizes. */
size_t pa_decode_v2_workspace_size(int32_t num_seqs, int32_t num_q_heads, int32_t head_size,
                                   int32_t max_context_len, int32_t partition_size);

/* pa_decode_v2: the V2 kernel of [TALK].  Each context is cut into partitions of
 * partition_size tokens (a positive multiple of block_size); each (sequence, kv head,
 * partition) is one work unit, handed to persistent CTAs from a shared counter.  A
 * partition keeps its running max m_p and exp-sum l_p; sequences with more than one
 * partition are merged by log-sum-exp, out = sum_p e^(m_p-M) acc_p / sum_p e^(m_p-M) l_p.
 * `workspace` (device, 256-byte aligned, >= pa_decode_v2_workspace_size bytes) holds the
 * work counter, the partition list and the partial results; its contents need no
 * initialisation and are dead after the call. */
pa_status pa_decode_v2(void* out, const void* query, const void* key_cache,
                       const void* value_cache, const int32_t* block_tables,
                       int32_t max_blocks_per_seq, const int32_t* context_lens,
                       int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                       int32_t head_size, int32_t block_size, int32_t num_blocks,
                       int32_t max_context_len, float scale, pa_dtype dtype,
                       int32_t partition_size, void* workspace, size_t workspace_bytes,
                       int32_t* status_dev, pa_stream stream);

/* Which variant pa_decode_auto runs for these host-known sizes.
 * *variant = 1 (V1) or 2 (V2); for V2, *partition_size is the smallest partition the
 * call may use (0 for V1).  The choice follows [TALK]: whole sequences per unit while
 * every context is short and there are units to fill every SM several times over;
 * otherwise V2 with partitions sized on the device from the actual context lengths --
 * as large as still gives every persistent CTA several units, so that few sequences
 * need a merge -- handed out longest first. */
pa_status pa_decode_auto_plan(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                              int32_t head_size, int32_t block_size, int32_t max_context_len,
                              int32_t* variant, int32_t* partition_size);

/* Workspace bytes pa_decode_auto needs (0 when it picks V1). */
size_t pa_decode_auto_workspace_size(int32_t num_seqs, int32_t num_q_heads,
                                     int32_t num_kv_heads, int32_t head_size,
                                     int32_t block_size, int32_t max_context_len);

/* pa_decode_auto: runs pa_decode_v1 or pa_decode_v2 as pa_decode_auto_plan says. */
pa_status pa_decode_auto(void* out, const void* query, const void* key_cache,
                         const void* value_cache, const int32_t* block_tables,
                         int32_t max_blocks_per_seq, const int32_t* context_lens,
                         int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                         int32_t head_size, int32_t block_size, int32_t num_blocks,
                         int32_t max_context_len, float scale, pa_dtype dtype,
                         void* workspace, size_t workspace_bytes, int32_t* status_dev,
                         pa_stream stream);

/* ------------------------------------------------------------------------------ */
/* fp8 KV cache ([TALK]: fp8 KV cache among the supported quantisation methods)      */
/* ------------------------------------------------------------------------------ */
/* Pools of PA_FP8_E4M3 bytes, [num_blocks][num_kv_heads][block_size][head_size], with
 * one dequantisation scale per pool (k_scale, v_scale > 0): a cached byte c stands for
 * e4m3(c) * scale.
 * pa_reshape_and_cache_fp8: like pa_reshape_and_cache, but key / value (fp16 or bf16,
 * `dtype`) are quantised: each element x becomes e4m3(x * r), r = 1 / scale computed in
 * fp32 (correctly rounded), x * r rounded to fp32, then to E4M3 nearest-even, saturating
 * at +-448 (NaN stays NaN).  Bit-exact with that definition. */
pa_status pa_reshape_and_cache_fp8(const void* key, const void* value, void* key_cache,
                                   void* value_cache, const int32_t* slot_mapping,
                                   int32_t num_tokens, int32_t num_kv_heads, int32_t head_size,
                                   int32_t block_size, int32_t num_blocks, pa_dtype dtype,
                                   float k_scale, float v_scale, int32_t* status_dev,
                                   pa_stream stream);

/* pa_decode_fp8: paged decode over fp8 pools: out = softmax(scale * q . (k_scale * k_t))
 * (v_scale * v_t), query and out fp16 or bf16 (`dtype`), head_size 128.  variant 0 =
 * pa_decode_auto's choice, 1 = V1, 2 = V2 with `partition_size` (a multiple of
 * block_size); workspace as for those (the same *_workspace_size calls apply).
 * Internally the K / V tiles are widened to fp16 (exact); on the tensor-core path (the
 * default, see pa_set_gqa_tensor_cores) the query is rounded to fp16, so queries beyond
 * fp16's range (|q| > 65504) are not supported there.  With 16-token blocks the kernel
 * takes two blocks per step when partitions are multiples of 32 tokens (V1, auto, or
 * such a partition_size), one block otherwise; results meet the same tolerance. */
pa_status pa_decode_fp8(void* out, const void* query, const void* key_cache, const void* value_cache,
                        const int32_t* block_tables, int32_t max_blocks_per_seq,
                        const int32_t* context_lens, int32_t num_seqs, int32_t num_q_heads,
                        int32_t num_kv_heads, int32_t head_size, int32_t block_size,
                        int32_t num_blocks, int32_t max_context_len, float scale, float k_scale,
                        float v_scale, pa_dtype dtype, int32_t variant, int32_t partition_size,
                        void* workspace, size_t workspace_bytes, int32_t* status_dev,
                        pa_stream stream);

/* ------------------------------------------------------------------------------ */
/* Multi-query decode ([TALK], speculative decoding part: attention kernels for several */
/* query tokens per sequence, to verify proposed tokens in one pass)                   */
/* ------------------------------------------------------------------------------ */
/* Every sequence brings q_len >= 1 new tokens, already in the pools (pa_reshape_and_cache
 * with one slot per token), and context_lens[s] = L counts all of them.  New token j
 * (0 <= j < q_len) sits at position L - q_len + j and attends to the tokens before and at
 * it: out[s][j][h] = sum_t softmax_t(scale * q[s][j][h] . k_t) v_t over t < L - q_len + j
 * + 1.  A row with no token to attend to (L < q_len - j) is a zero row.
 *   query, out  [num_seqs][q_len][num_q_heads][head_size], fp16 or bf16 (`dtype`, also
 *               the cache type); other arguments as for pa_decode_v1 / pa_decode_v2.
 * The q_len * group rows of a (sequence, kv head) share one pass over its K/V on the
 * tensor cores, up to 32 rows at a time (more rows re-read the K/V once per 32).  variant 0 =
 * pa_decode_auto's choice (V1 or V2 with adaptive partitions), 1 = V1, 2 = V2 with
 * `partition_size` tokens per partition.  q_len 1 is an ordinary decode.
 * pa_decode_mq_workspace_size: the workspace for variant 2 with `partition_size`, or for
 * variant 0 when partition_size is 0 (V1 needs none); 0 for bad sizes. */
size_t pa_decode_mq_workspace_size(int32_t num_seqs, int32_t q_len, int32_t num_q_heads,
                                   int32_t num_kv_heads, int32_t head_size, int32_t block_size,
                                   int32_t max_context_len, int32_t partition_size);
pa_status pa_decode_mq(void* out, const void* query, const void* key_cache, const void* value_cache,
                       const int32_t* block_tables, int32_t max_blocks_per_seq,
                       const int32_t* context_lens, int32_t num_seqs, int32_t q_len,
                       int32_t num_q_heads, int32_t num_kv_heads, int32_t head_size,
                       int32_t block_size, int32_t num_blocks, int32_t max_context_len,
                       float scale, pa_dtype dtype, int32_t variant, int32_t partition_size,
                       void* workspace, size_t workspace_bytes, int32_t* status_dev,
                       pa_stream stream);

/* Selects the multi-query kernel for head_size 128 with 16-bit caches and more than 8
 * query rows (q_len x group) per kv head: 1 (the default) runs it on the 5th-generation
 * tensor cores (tcgen05, accumulators in tensor memory), 0 on mma.sync.  Other shapes,
 * and fixed V2 partition sizes that are not a multiple of 128 tokens, always take the
 * mma.sync kernel.  The setting belongs to the calling thread: it changes that thread's
 * later calls only (each thread starts at 1).  Returns PA_OK.
 * The tcgen05 kernel's warpgroups divide among themselves the registers each thread is
 * launched with; at its first launch on a device the library checks that the kernel was
 * compiled with the per-thread count that division assumes, and if not, the call fails
 * with PA_ERR_CUDA ("invalid kernel image") instead of launching. */
pa_status pa_set_mq_tcgen05(int32_t enable);

/* One decode step of the hot path on device buffers: pa_reshape_and_cache of the
 * step's new K/V rows, then pa_decode_auto, on the same stream.  Every argument is
 * checked before anything is launched. */
pa_status pa_decode_step(void* out, const void* query, const void* key, const void* value,
                         void* key_cache, void* value_cache, const int32_t* slot_mapping,
                         const int32_t* block_tables, int32_t max_blocks_per_seq,
                         const int32_t* context_lens, int32_t num_seqs, int32_t num_q_heads,
                         int32_t num_kv_heads, int32_t head_size, int32_t block_size,
                         int32_t num_blocks, int32_t max_context_len, float scale,
                         pa_dtype dtype, void* workspace, size_t workspace_bytes,
                         int32_t* status_dev, pa_stream stream);

/* The same step from HOST buffers, for callers whose step inputs live in host memory:
 * copies query [S][Hq][D], key / value [S][Hkv][D], slot_mapping [S], block_tables
 * [S][max_blocks_per_seq] and context_lens [S] from host memory into `staging` (device,
 * 256-byte aligned, >= pa_decode_step_host_staging_size bytes) with one cudaMemcpyAsync
 * each, runs pa_decode_step on the staged copies, and copies out [S][Hq][D] back into
 * out_host.  Everything is enqueued on `stream`; the call does not wait: out_host is valid
 * once the stream has been synchronised.  Host buffers should be page-locked (pinned) for
 * the copies to be asynchronous; pageable buffers work but make the copies synchronous.
 * The pools stay on the device (they are the cache). */
size_t pa_decode_step_host_staging_size(int32_t num_seqs, int32_t num_q_heads,
                                        int32_t num_kv_heads, int32_t head_size,
                                        int32_t max_blocks_per_seq);
pa_status pa_decode_step_host(void* out_host, const void* query_host, const void* key_host,
                              const void* value_host, const int32_t* slot_mapping_host,
                              const int32_t* block_tables_host, const int32_t* context_lens_host,
                              void* key_cache, void* value_cache, int32_t max_blocks_per_seq,
                              int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                              int32_t head_size, int32_t block_size, int32_t num_blocks,
                              int32_t max_context_len, float scale, pa_dtype dtype,
                              void* staging, size_t staging_bytes, void* workspace,
                              size_t workspace_bytes, int32_t* status_dev, pa_stream stream);

/* pa_decode_step_host with the copies on streams of their own, so that a step's copies
 * overlap the kernels of its neighbours.  On `h2d`: the H2D copies, then `staged_event` is
 * recorded; on `compute`: wait for `staged_event`, pa_decode_step, record `done_event`; on
 * `d2h`: wait for `done_event`, the D2H copy of out.  `h2d` and `d2h` must differ from
 * `compute` (they may be one stream, but then a step's input copies queue behind the
 * previous step's output copy, which waits for its kernels).  The events are cudaEvent_t
 * owned by the caller.  A caller that keeps several steps in flight gives each its own
 * staging area, host buffers and events, and reuses them only once that step's D2H has
 * completed (for example an event it records on `d2h` after this call).  Steps must be
 * issued in order: they share the KV pools and the workspace on `compute`.
 * PA_ERR_INVALID_ARG when an event is NULL or a copy stream is `compute`. */
pa_status pa_decode_step_host_overlapped(
    void* out_host, const void* query_host, const void* key_host, const void* value_host,
    const int32_t* slot_mapping_host, const int32_t* block_tables_host,
    const int32_t* context_lens_host, void* key_cache, void* value_cache,
    int32_t max_blocks_per_seq, int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
    int32_t head_size, int32_t block_size, int32_t num_blocks, int32_t max_context_len,
    float scale, pa_dtype dtype, void* staging, size_t staging_bytes, void* workspace,
    size_t workspace_bytes, int32_t* status_dev, pa_stream compute, pa_stream h2d,
    pa_stream d2h, void* staged_event, void* done_event);

/* Compute path for grouped-query attention (group >= 2) and for fp8 caches of any
 * group: 1 (default) contracts the group's query heads with each K/V tile on the tensor
 * cores (mma.sync m16n8k16, fp32 accumulate); 0 uses the CUDA-core path that
 * multi-head attention over 16-bit caches always takes.  Groups above 8 stay on the
 * tensor cores.  Both paths meet the same tolerance.  The setting belongs to the calling
 * thread: it changes that thread's later calls only (each thread starts at 1). */
pa_status pa_set_gqa_tensor_cores(int32_t enable);

/* ------------------------------------------------------------------------------ */
/* V2 decode for callers that cannot allocate device memory                         */
/* ------------------------------------------------------------------------------ */
/* The paper has no counterpart to this call; it exists for callers that are not
 * allowed to allocate device memory and have no workspace handed to them -- for
 * example a plugin's enqueue path inside an inference runtime that owns all device
 * memory, or code that must not call cudaMalloc while a stream is being captured.
 *
 * pa_decode_v2_noalloc computes exactly what pa_decode_v2 computes, but its scratch
 * (work counter, partition list, partial results) lives in one static device array of
 * PA_NOALLOC_SCRATCH_BYTES compiled into the library.  Every GPU that loads the library
 * keeps that array until the process exits.  The caller still passes inputs and outputs.
 *   - It allocates nothing: no cudaMalloc, no cudaFree, no allocating library call.
 *   - It checks its arguments as pa_decode_v2 does and returns the same errors; then,
 *     if pa_decode_v2_workspace_size() for the arguments exceeds
 *     PA_NOALLOC_SCRATCH_BYTES, it returns PA_ERR_WORKSPACE and launches nothing.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call before
 *     any stream capture begins.  The address is kept for the life of the process: after
 *     cudaDeviceReset (or anything else that tears down the device's primary context)
 *     the library's module is loaded again and the cached address is stale, so do not
 *     call this entry point on that device again in the same process.
 *   - All calls share the one array and it keeps the last call's contents (each call
 *     rewrites everything it reads).  Calls whose kernels overlap on the GPU -- on two
 *     streams, or from two threads -- race on it and give wrong results; serialise them. */
#define PA_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)

pa_status pa_decode_v2_noalloc(void* out, const void* query, const void* key_cache,
                               const void* value_cache, const int32_t* block_tables,
                               int32_t max_blocks_per_seq, const int32_t* context_lens,
                               int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                               int32_t head_size, int32_t block_size, int32_t num_blocks,
                               int32_t max_context_len, float scale, pa_dtype dtype,
                               int32_t partition_size, int32_t* status_dev, pa_stream stream);

/* advance_step [PR]: moves every sequence of a multi-step decode loop to its next token
 * on the device, with no host round trip between the steps:
 *   pos = context_lens[s];  context_lens[s] = pos + 1;
 *   slot_mapping[s] = block_tables[s][pos / block_size] * block_size + pos % block_size;
 *   input_positions[s] = pos            (if input_positions is not NULL);
 *   input_tokens[s] = sampled_token_ids[s]  (if both are not NULL).
 * context_lens enters as the lengths BEFORE the step's token and leaves counting it, the
 * convention pa_decode_* expects.  The block holding pos must already be in the table:
 * reserve the loop's blocks with pa_alloc_reserve_batch first.  A missing block gives
 * slot -1 (reshape_and_cache skips it) and sets PA_DEVERR_BAD_BLOCK.  A single small
 * kernel; safe to capture in a CUDA graph with the rest of the loop. */
pa_status pa_advance_step(int32_t* context_lens, int32_t* slot_mapping, const int32_t* block_tables,
                          int32_t max_blocks_per_seq, int32_t num_seqs, int32_t block_size,
                          int32_t num_blocks, int64_t* input_positions, int64_t* input_tokens,
                          const int64_t* sampled_token_ids, int32_t* status_dev, pa_stream stream);

/* Copies whole blocks of both pools on the device, for copy-on-write of shared blocks
 * ([TALK]: blocks shared between requests, prefix caching): for each pair i, block
 * block_pairs[2i+1] of key_cache and value_cache takes the contents of block
 * block_pairs[2i] (every kv head and row; a bit-exact copy).  block_pairs is a device
 * int32 array [num_pairs][2], e.g. the pairs pa_alloc_take_copies returned, copied to
 * the device; run it before reshape_and_cache writes into the new blocks.  Pairs
 * outside the pool are skipped and flagged PA_DEVERR_BAD_BLOCK; a block that is both a
 * source and a destination in one call races.  dtype is the pools' element type
 * (PA_F16, PA_BF16 or PA_FP8_E4M3). */
pa_status pa_copy_blocks(void* key_cache, void* value_cache, const int32_t* block_pairs,
                         int32_t num_pairs, int32_t num_kv_heads, int32_t head_size,
                         int32_t block_size, int32_t num_blocks, pa_dtype dtype,
                         int32_t* status_dev, pa_stream stream);

/* Self-test of the failure path: launches a one-warp kernel that waits on a pipeline
 * barrier nobody arrives on, gives up after limit_us (1 .. 2,000,000) microseconds and
 * ORs PA_DEVERR_TIMEOUT into *status_dev, exactly as the decode kernel does when a copy
 * never completes.  The kernel returns normally; the context stays usable. */
pa_status pa_selftest_wait_timeout(int32_t* status_dev, uint32_t limit_us, pa_stream stream);

/* Profiling hook, for benchmarks and tests; no result depends on it.  When both are
 * non-NULL (cudaEvent_t handles), every later decode call of the calling thread records
 * `start_event` on its stream right before it launches the paged decode kernel and
 * `stop_event` right after, so that the kernel alone can be timed with
 * cudaEventElapsedTime.  NULL, NULL turns the hook off (each thread starts with it off).
 * While it is on, the decode kernel no longer starts early under the kernel before it
 * (the plan or reshape kernel), so a step takes a few microseconds longer. */
pa_status pa_set_kernel_events(void* start_event, void* stop_event);

/* ------------------------------------------------------------------------------ */
/* Host block allocator (the v2 block manager of [PR]; blocks as pages per [TALK])  */
/* ------------------------------------------------------------------------------ */
/* Host memory only; one handle must not be used from two threads at once.
 * Spec: physical ids 0..num_blocks-1 are shuffled by Fisher-Yates (i from
 * num_blocks-1 down to 1, j = r % (i+1), r the next splitmix64 output seeded with
 * `seed`); the result is the free list, popped from its end.  add_seq pops
 * ceil(num_tokens / block_size) blocks in logical order; append pops one block when
 * the new position has no block yet (none reserved ahead), then returns the slot of the
 * new last position; free_seq pushes the blocks back in logical order.  A request that needs
 * more blocks than are free returns PA_ERR_NO_BLOCKS and changes nothing. */
typedef struct pa_alloc pa_alloc;

pa_status pa_alloc_create(int32_t num_blocks, int32_t block_size, uint64_t seed,
                          pa_alloc** out);
void pa_alloc_destroy(pa_alloc* alloc);
int32_t pa_alloc_num_free(const pa_alloc* alloc);
/* Registers sequence seq_id (>= 0, not live) holding num_tokens tokens. */
pa_status pa_alloc_add_seq(pa_alloc* alloc, int32_t seq_id, int32_t num_tokens);
/* Appends one token to seq_id; *slot_out = its slot. */
pa_status pa_alloc_append(pa_alloc* alloc, int32_t seq_id, int32_t* slot_out);
/* Appends one token to each of n sequences (all or nothing); slots_out[i] = slot. */
pa_status pa_alloc_append_batch(pa_alloc* alloc, const int32_t* seq_ids, int32_t n,
                                int32_t* slots_out);
/* Reserves blocks ahead for a multi-step loop: each listed sequence gets blocks until it
 * owns ceil((len + extra_tokens) / block_size) of them, popped in list order; lengths do
 * not change, and later appends use the reserved blocks first.  All or nothing. */
pa_status pa_alloc_reserve_batch(pa_alloc* alloc, const int32_t* seq_ids, int32_t n,
                                 int32_t extra_tokens);
/* Shared prefixes: sequence dst_seq (not live) becomes live with the first num_tokens
 * tokens of src_seq (<= its length), sharing src_seq's first ceil(num_tokens /
 * block_size) blocks; each shared block's reference count goes up by one and nothing
 * is popped.  Before any later append or reserve writes into a block whose count is
 * above one, the allocator gives the writer a private copy: it pops a new block, puts
 * it in the writer's table and records the pair (old, new); take those pairs with
 * pa_alloc_take_copies and copy them with pa_copy_blocks before the step's
 * reshape_and_cache. */
pa_status pa_alloc_fork(pa_alloc* alloc, int32_t src_seq, int32_t dst_seq, int32_t num_tokens);
/* Copy-on-write pairs recorded since the last take. */
int32_t pa_alloc_num_pending_copies(const pa_alloc* alloc);
/* Writes the pending (old, new) pairs, in the order recorded, to pairs_out
 * [max_pairs][2] and clears them; *n_out = their number.  If they do not all fit,
 * nothing is taken and PA_ERR_INVALID_ARG is returned with *n_out set. */
pa_status pa_alloc_take_copies(pa_alloc* alloc, int32_t* pairs_out, int32_t max_pairs,
                               int32_t* n_out);
/* Reference count of a physical block (0 = free), -1 for an id outside the pool. */
int32_t pa_alloc_refcount(const pa_alloc* alloc, int32_t block);
/* Drops seq_id's reference to each of its blocks (blocks no longer referenced return
 * to the free list, in logical order) and forgets the sequence. */
pa_status pa_alloc_free_seq(pa_alloc* alloc, int32_t seq_id);
/* Slots of positions [start, start + n) of seq_id. */
pa_status pa_alloc_slots(const pa_alloc* alloc, int32_t seq_id, int32_t start, int32_t n,
                         int32_t* out);
/* Block-table rows [n][max_blocks_per_seq] of the listed sequences, padded with -1. */
pa_status pa_alloc_block_tables(const pa_alloc* alloc, const int32_t* seq_ids, int32_t n,
                                int32_t max_blocks_per_seq, int32_t* out);
/* Current lengths of the listed sequences. */
pa_status pa_alloc_context_lens(const pa_alloc* alloc, const int32_t* seq_ids, int32_t n,
                                int32_t* out);

#ifdef __cplusplus
}
#endif

#endif /* PA_H_ */
