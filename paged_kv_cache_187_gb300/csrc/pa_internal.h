// pa_internal.h -- interface between the host side of the C ABI (pa_host.cpp) and the
// kernel launchers (pa_decode_*.cu, pa_reshape.cu).  Not part of the public ABI.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "pa_once.h"

namespace pa {

// Head of the V2 workspace.  The plan kernel writes it; the decode kernel's persistent
// CTAs start with the unit of their own index and claim the later ones from `counter`.
struct WsHeader {
    uint32_t counter;         // units claimed so far past the first gridDim.x
    uint32_t total_units;     // partitions * num_kv_heads * row_chunks
    uint32_t total_parts;     // partitions over all sequences
    uint32_t partition_size;  // tokens per partition used by this call
    uint32_t pad[60];
};

struct DecodeParams {
    void* out;                    // [S][q_len][Hq][D] of the dtype
    const void* q;                // [S][q_len][Hq][D]
    const int32_t* block_tables;  // [S][max_blocks_per_seq]
    const int32_t* context_lens;  // [S]
    int32_t max_blocks_per_seq;
    int32_t num_seqs, num_q_heads, num_kv_heads, group;
    int32_t num_blocks;
    int32_t block_size;
    int32_t max_context_len;
    float scale_log2;             // softmax scale (x k_scale for fp8 caches) * log2(e):
                                  // logits live in base-2 units
    float out_scale;              // applied to every output row (v_scale for fp8 caches, else 1)
    int32_t partition_size;       // V2: tokens per partition (the smallest allowed when
                                  // adaptive); 0 = the whole context per unit (V1)
    int32_t adaptive;             // V2: 1 = the plan kernel sizes partitions from the lengths
    int32_t grid_ctas;            // V2: persistent CTAs of the decode launch
    // V2 workspace pieces (null for V1)
    WsHeader* hdr;
    int4* part_list;              // [parts] work order: (sequence, partition, first partition
                                  // slot of the sequence, clamped context length)
    int32_t* arrive;              // [S][Hkv][row_chunks][row_groups] partitions finished so far
    float* part_acc;              // [parts][Hkv][rows][D] unnormalised partial outputs
    float2* part_ml;              // [parts][Hkv][rows] (running max in base-2 units, exp-sum)
    int32_t* status;              // optional device error word
    // Query rows.  A (sequence, kv head) has rows = q_len * group query rows, row
    // j * group + i being query token j of the sequence and query head kv_head * group + i.
    // Ordinary decode: q_len 1, rows = group, row_chunks = row_groups = 1.  Multi-query
    // kernels give a work unit row_groups * heads_cap rows, row group r (heads_cap rows)
    // to its own consumer warps, and split the rows into row_chunks such units.
    int32_t q_len;
    int32_t rows;
    int32_t row_chunks;
    int32_t row_groups;
    int32_t partition_align;      // V2: partitions are multiples of this many tokens (0: block_size)
};

// Multi-query CTAs: each consumer warp holds 8 rows (one mma n-tile).  Up to 8 rows per
// kv head, 2 consumer warps share the tiles (3 CTAs per SM); above that, 4 consumer
// warps (2 CTAs per SM) form up to 4 row groups, so a unit covers up to 32 rows in one
// K/V pass.
constexpr int32_t kMqRowsPerConsumer = 8;

// Decode kernels let the kernels queued after them launch once every CTA has issued the
// copies of its last tile (1), or only when they finish (0).
#ifndef PA_DECODE_TRIGGER
#define PA_DECODE_TRIGGER 1
#endif
constexpr int32_t kMqConsumersNarrow = 2;
constexpr int32_t kMqConsumersWide = 4;

struct WorkspaceLayout {
    size_t hdr, part_list, arrive, part_ml, part_acc, total;
};

WorkspaceLayout v2_workspace_layout(int32_t num_seqs, int32_t num_q_heads, int32_t head_size,
                                    int32_t max_context_len, int32_t partition_size);

// Selects the kernel instantiation.
struct KernelKey {
    int32_t head_size;   // 64 | 128
    int32_t block_size;  // 16 | 32
    bool bf16;           // query / output type
    bool kv8;            // cache in fp8 E4M3
    bool mma;            // tensor-core path (group >= 2) or CUDA-core path
    int32_t heads_cap;   // mma: 8 or 16 (n-tiles * 8); CUDA cores: 1, 2, 4 or 8
    bool mq = false;     // several causal query tokens per sequence (tensor-core path only)
    int32_t mq_consumers = 0;   // multi-query: consumer warps per CTA (2 or 4)
    bool tc = false;            // multi-query on tcgen05 (heads_cap = rows per unit, 16 or 32)
    int32_t tile_blocks = 1;    // pool blocks per consumer tile (2: fp8 with 16-token blocks)
};

// Launchers return cudaSuccess or the launch error.  `persistent` selects the V2
// schedule (grid = resident CTAs, units claimed from the workspace counter).
cudaError_t launch_decode(const KernelKey& key, const CUtensorMap& kmap, const CUtensorMap& vmap,
                          const DecodeParams& p, bool persistent, int32_t num_units,
                          cudaStream_t stream);
cudaError_t launch_plan(const DecodeParams& p, cudaStream_t stream);
cudaError_t launch_reshape_and_cache(const void* key, const void* value, void* key_cache,
                                     void* value_cache, const int32_t* slot_mapping,
                                     int32_t num_tokens, int32_t num_kv_heads,
                                     int32_t head_size, int32_t block_size, int32_t num_blocks,
                                     int32_t* status, cudaStream_t stream);

cudaError_t launch_advance_step(int32_t* context_lens, int32_t* slot_mapping,
                                const int32_t* block_tables, int32_t max_blocks_per_seq,
                                int32_t num_seqs, int32_t block_size, int32_t num_blocks,
                                int64_t* input_positions, int64_t* input_tokens,
                                const int64_t* sampled_token_ids, int32_t* status,
                                cudaStream_t stream);
cudaError_t launch_copy_blocks(void* key_cache, void* value_cache, const int32_t* pairs,
                               int32_t num_pairs, int64_t bytes_per_block, int32_t num_blocks,
                               int32_t* status, cudaStream_t stream);
cudaError_t launch_wait_timeout_probe(int32_t* status, uint64_t limit_ns, cudaStream_t stream);

// The argument checks pa_decode_v2 makes before it looks at its workspace: PA_OK, or the
// status it would return (with this thread's pa_last_error() message set).
int32_t check_decode_v2_args(const void* out, const void* query, const void* key_cache,
                             const void* value_cache, const int32_t* block_tables,
                             int32_t max_blocks_per_seq, const int32_t* context_lens,
                             int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                             int32_t head_size, int32_t block_size, int32_t num_blocks,
                             int32_t max_context_len, int32_t dtype, int32_t partition_size);

// Records `message` as this thread's pa_last_error() text and returns `status`.
int32_t set_last_error(int32_t status, const char* message);

// Resident CTAs per SM of a decode instantiation (0 if it cannot launch).
int32_t decode_ctas_per_sm(const KernelKey& key);

// Per-instantiation family launchers, one per translation unit.
cudaError_t launch_decode_f16_d128(const KernelKey&, const CUtensorMap&, const CUtensorMap&,
                                   const DecodeParams&, bool, int32_t, cudaStream_t, int32_t*);
cudaError_t launch_decode_bf16_d128(const KernelKey&, const CUtensorMap&, const CUtensorMap&,
                                    const DecodeParams&, bool, int32_t, cudaStream_t, int32_t*);
cudaError_t launch_decode_f16_d64(const KernelKey&, const CUtensorMap&, const CUtensorMap&,
                                  const DecodeParams&, bool, int32_t, cudaStream_t, int32_t*);
cudaError_t launch_decode_bf16_d64(const KernelKey&, const CUtensorMap&, const CUtensorMap&,
                                   const DecodeParams&, bool, int32_t, cudaStream_t, int32_t*);
cudaError_t launch_decode_fp8kv_f16q(const KernelKey&, const CUtensorMap&, const CUtensorMap&,
                                     const DecodeParams&, bool, int32_t, cudaStream_t, int32_t*);
cudaError_t launch_decode_fp8kv_bf16q(const KernelKey&, const CUtensorMap&, const CUtensorMap&,
                                      const DecodeParams&, bool, int32_t, cudaStream_t, int32_t*);
cudaError_t launch_decode_mq_f16(const KernelKey&, const CUtensorMap&, const CUtensorMap&,
                                 const DecodeParams&, bool, int32_t, cudaStream_t, int32_t*);
cudaError_t launch_decode_mq_bf16(const KernelKey&, const CUtensorMap&, const CUtensorMap&,
                                  const DecodeParams&, bool, int32_t, cudaStream_t, int32_t*);
cudaError_t launch_decode_mq_tc(const KernelKey&, const CUtensorMap&, const CUtensorMap&,
                                const DecodeParams&, bool, int32_t, cudaStream_t, int32_t*);
// Tokens per tile of the tcgen05 multi-query kernel (its partitions are multiples of it).
constexpr int32_t kTcTileTokens = 128;
cudaError_t launch_reshape_and_cache_fp8(const void* key, const void* value, void* key_cache,
                                         void* value_cache, const int32_t* slot_mapping,
                                         int32_t num_tokens, int32_t num_kv_heads,
                                         int32_t head_size, int32_t block_size, int32_t num_blocks,
                                         bool src_bf16, float k_inv_scale, float v_inv_scale,
                                         int32_t* status, cudaStream_t stream);

}  // namespace pa
