// pa_host.cpp -- host side of the C ABI declared in include/pa.h: argument checks,
// TMA tensor-map encoding, V1 / V2 / auto dispatch, and the host block allocator.
#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <unordered_map>
#include <unordered_set>
#include <vector>

#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/pa.h"
#include "pa_internal.h"

namespace {

thread_local std::string g_last_error;

pa_status fail(pa_status st, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return st;
}

pa_status ok() {
    g_last_error.clear();
    return PA_OK;
}

pa_status cuda_fail(cudaError_t e, const char* what) {
    return fail(PA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// ------------------------------------------------------------------ device facts
struct DeviceInfo {
    int sms = 0;
};

std::mutex g_mu;
std::unordered_map<int, DeviceInfo> g_dev;
std::unordered_map<uint64_t, int32_t> g_occ;   // (device, kernel key) -> CTAs per SM
// Kernel choices and the profiling events belong to the calling thread: one thread's
// setting never changes what another thread's calls launch.
thread_local int32_t g_gqa_mma = 1;
thread_local int32_t g_mq_tc = 1;
thread_local cudaEvent_t g_ev_start = nullptr, g_ev_stop = nullptr;

// Launches the decode kernel, bracketed by the profiling events when they are set.
cudaError_t timed_decode(const pa::KernelKey& k, const CUtensorMap& km, const CUtensorMap& vm,
                         const pa::DecodeParams& p, bool persistent, int32_t units,
                         cudaStream_t st);

pa_status current_device(int* dev, DeviceInfo* info) {
    cudaError_t e = cudaGetDevice(dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    std::lock_guard<std::mutex> lk(g_mu);
    auto it = g_dev.find(*dev);
    if (it == g_dev.end()) {
        DeviceInfo di;
        e = cudaDeviceGetAttribute(&di.sms, cudaDevAttrMultiProcessorCount, *dev);
        if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
        it = g_dev.emplace(*dev, di).first;
    }
    *info = it->second;
    return PA_OK;
}

cudaError_t dispatch_decode(const pa::KernelKey& k, const CUtensorMap& km, const CUtensorMap& vm,
                            const pa::DecodeParams& p, bool persistent, int32_t units,
                            cudaStream_t st, int32_t* occ) {
    if (k.tc) return pa::launch_decode_mq_tc(k, km, vm, p, persistent, units, st, occ);
    if (k.mq)
        return k.bf16 ? pa::launch_decode_mq_bf16(k, km, vm, p, persistent, units, st, occ)
                      : pa::launch_decode_mq_f16(k, km, vm, p, persistent, units, st, occ);
    if (k.kv8)
        return k.bf16 ? pa::launch_decode_fp8kv_bf16q(k, km, vm, p, persistent, units, st, occ)
                      : pa::launch_decode_fp8kv_f16q(k, km, vm, p, persistent, units, st, occ);
    if (k.head_size == 128)
        return k.bf16 ? pa::launch_decode_bf16_d128(k, km, vm, p, persistent, units, st, occ)
                      : pa::launch_decode_f16_d128(k, km, vm, p, persistent, units, st, occ);
    return k.bf16 ? pa::launch_decode_bf16_d64(k, km, vm, p, persistent, units, st, occ)
                  : pa::launch_decode_f16_d64(k, km, vm, p, persistent, units, st, occ);
}

cudaError_t timed_decode(const pa::KernelKey& k, const CUtensorMap& km, const CUtensorMap& vm,
                         const pa::DecodeParams& p, bool persistent, int32_t units,
                         cudaStream_t st) {
    cudaEvent_t a = g_ev_start, b = g_ev_stop;
    if (a && b) {
        cudaError_t e = cudaEventRecord(a, st);
        if (e != cudaSuccess) return e;
    }
    cudaError_t e = dispatch_decode(k, km, vm, p, persistent, units, st, nullptr);
    if (e == cudaSuccess && a && b) e = cudaEventRecord(b, st);
    return e;
}

int32_t ctas_per_sm(int dev, const pa::KernelKey& k) {
    const uint64_t key = (uint64_t)dev << 32 | (uint64_t)k.tile_blocks << 29 | (uint64_t)k.tc << 28 |
                         (uint64_t)k.mq_consumers << 24 |
                         (uint64_t)k.mq << 22 |
                         (uint64_t)k.kv8 << 21 |
                         (uint64_t)(k.head_size == 128) << 20 |
                         (uint64_t)(k.block_size == 32) << 19 | (uint64_t)k.bf16 << 18 |
                         (uint64_t)k.mma << 17 | (uint64_t)k.heads_cap;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        auto it = g_occ.find(key);
        if (it != g_occ.end()) return it->second;
    }
    CUtensorMap dummy;
    std::memset(&dummy, 0, sizeof(dummy));
    pa::DecodeParams p;
    std::memset(&p, 0, sizeof(p));
    int32_t n = 0;
    if (dispatch_decode(k, dummy, dummy, p, true, 0, nullptr, &n) != cudaSuccess) n = 0;
    std::lock_guard<std::mutex> lk(g_mu);
    g_occ[key] = n;
    return n;
}

// ------------------------------------------------------------------ tensor maps
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            p = nullptr;
        return reinterpret_cast<EncodeTiledFn>(p);
    }();
    return fn;
}

// The pool [num_blocks][num_kv_heads][block_size][head_size] viewed as a 2-D matrix of
// rows = num_blocks*num_kv_heads*block_size and head_size columns; a box is 64 columns
// (128 bytes, the swizzle span) by block_size rows, i.e. one half of a (block, head)
// tile when head_size is 128.
pa_status encode_pool_map(CUtensorMap* map, const void* pool, int64_t rows, int32_t head_size,
                          int32_t block_size, bool kv8) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return fail(PA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    const int32_t elem = kv8 ? 1 : 2;
    cuuint64_t dims[2] = {(cuuint64_t)head_size, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)head_size * elem};
    cuuint32_t box[2] = {128u / (cuuint32_t)elem, (cuuint32_t)block_size};   // 128 bytes wide
    cuuint32_t estr[2] = {1u, 1u};
    CUresult r = fn(map, kv8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_UINT16, 2,
                    const_cast<void*>(pool), dims, strides,
                    box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(PA_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    return PA_OK;
}

// ------------------------------------------------------------------ argument checks
struct DecodeArgs {
    void* out;
    const void* query;
    const void* key_cache;
    const void* value_cache;
    const int32_t* block_tables;
    int32_t max_blocks_per_seq;
    const int32_t* context_lens;
    int32_t num_seqs, num_q_heads, num_kv_heads, head_size, block_size, num_blocks;
    int32_t max_context_len;
    float scale;
    pa_dtype dtype;        // query / output type
    int32_t* status;
    cudaStream_t stream;
    bool kv8 = false;      // cache in fp8 E4M3, dequantised by k_scale / v_scale
    float k_scale = 1.f, v_scale = 1.f;
    int32_t q_len = 1;     // query tokens per sequence (> 1: multi-query kernels)
    int32_t partition_size = 0;   // V2 with a fixed partition size (0: none given)
};

// The tcgen05 multi-query kernel takes head_size 128, 16-bit caches, and partitions that
// are multiples of its 128-token tile; it holds 16 or 32 query rows per unit.  It is used
// where it measured faster than the mma.sync kernel, whose three CTAs per SM hide the load
// latency better than its single tile pipeline per SM: above 8 query rows per kv head
// (Llama-3-8B / -70B batches, decode kernel: 8 rows with 16-token blocks 210 vs 205 us;
// 16 rows 203 vs 261 us with 16-token blocks, 617 vs 631 us with 32-token blocks; 32 rows
// 226 vs 379 us and 667 vs 1061 us).
#ifndef PA_MQ_TC_ROWS_BS32
#define PA_MQ_TC_ROWS_BS32 8    // tcgen05 above this many rows per kv head, 32-token blocks
#endif
#ifndef PA_MQ_TC_ROWS_BS16
#define PA_MQ_TC_ROWS_BS16 8    // ... and with 16-token blocks
#endif
bool use_mq_tc(const DecodeArgs& a) {
    const int32_t rows = a.q_len * (a.num_q_heads / std::max(a.num_kv_heads, 1));
    const bool wins = a.block_size == 16 ? rows > PA_MQ_TC_ROWS_BS16 : rows > PA_MQ_TC_ROWS_BS32;
    return g_mq_tc && a.q_len > 1 && wins && a.head_size == 128 && !a.kv8 &&
           (a.partition_size == 0 || a.partition_size % pa::kTcTileTokens == 0);
}
// Rows per unit of the tcgen05 kernel: 16 or 32.
// fp8 caches with 16-token blocks are decoded in tiles of two blocks (32 tokens), which
// needs partitions that are multiples of 32 tokens.
int32_t tile_blocks_for(const DecodeArgs& a) {
#ifndef PA_TILE2_16BIT
#define PA_TILE2_16BIT 0
#endif
    return ((a.kv8 || PA_TILE2_16BIT) && a.block_size == 16 && a.q_len == 1 &&
            (a.partition_size == 0 || a.partition_size % 32 == 0)) ? 2 : 1;
}

int32_t mq_tc_rows(int32_t rows, int32_t) { return rows <= 16 ? 16 : 32; }

// Multi-query kernels: rows per consumer (the head capacity), consumer warps per CTA, row
// groups per unit (a power of two dividing the consumers, so that the consumers of a
// group share its tiles evenly), and the units (chunks) the q_len * group rows of a
// (sequence, kv head) are split into.  Each chunk reads the K/V once.
int32_t mq_heads_cap(int32_t) { return pa::kMqRowsPerConsumer; }
int32_t mq_consumers(int32_t rows) {
    return rows <= pa::kMqRowsPerConsumer ? pa::kMqConsumersNarrow : pa::kMqConsumersWide;
}
int32_t mq_row_groups(int32_t rows) {
    const int32_t need = (rows + pa::kMqRowsPerConsumer - 1) / pa::kMqRowsPerConsumer;
    int32_t g = 1;
    while (g < need && g < mq_consumers(rows)) g *= 2;
    return g;
}
int32_t mq_row_chunks(int32_t rows) {
    const int32_t per = mq_row_groups(rows) * mq_heads_cap(rows);
    return (rows + per - 1) / per;
}

pa_status check_decode(const DecodeArgs& a) {
    if (a.num_seqs < 0 || a.num_q_heads <= 0 || a.num_kv_heads <= 0 || a.num_blocks <= 0 ||
        a.max_blocks_per_seq <= 0 || a.max_context_len < 0)
        return fail(PA_ERR_INVALID_ARG, "decode: sizes must be positive (num_seqs >= 0)");
    if (a.dtype != PA_F16 && a.dtype != PA_BF16) return fail(PA_ERR_UNSUPPORTED, "decode: dtype");
    if (a.head_size != 64 && a.head_size != 128)
        return fail(PA_ERR_UNSUPPORTED, "decode: head_size %d (64 or 128)", a.head_size);
    if (a.kv8 && a.head_size != 128)
        return fail(PA_ERR_UNSUPPORTED, "decode: an fp8 cache needs head_size 128");
    if (a.kv8 && !(a.k_scale > 0.f && a.v_scale > 0.f))
        return fail(PA_ERR_INVALID_ARG, "decode: k_scale and v_scale must be positive");
    if (a.block_size != 16 && a.block_size != 32)
        return fail(PA_ERR_UNSUPPORTED, "decode: block_size %d (16 or 32)", a.block_size);
    if (a.num_q_heads % a.num_kv_heads)
        return fail(PA_ERR_INVALID_ARG, "decode: num_q_heads %% num_kv_heads != 0");
    if (a.num_q_heads / a.num_kv_heads > 16)
        return fail(PA_ERR_UNSUPPORTED, "decode: query group %d > 16",
                    a.num_q_heads / a.num_kv_heads);
    if (a.q_len < 1 || (int64_t)a.q_len * a.num_q_heads > (1 << 20))
        return fail(PA_ERR_INVALID_ARG, "decode: q_len %d (1 .. 2^20 / num_q_heads)", a.q_len);
    if (a.q_len > 1 && a.kv8) return fail(PA_ERR_UNSUPPORTED, "decode: multi-query over an fp8 cache");
    const int64_t rows = (int64_t)a.num_blocks * a.num_kv_heads * a.block_size;
    if (rows + (int64_t)a.num_kv_heads * a.block_size > INT32_MAX)
        return fail(PA_ERR_UNSUPPORTED, "decode: pool has more than 2^31 rows");
    if (a.num_seqs == 0) return PA_OK;
    if (!a.out || !a.query || !a.key_cache || !a.value_cache || !a.block_tables || !a.context_lens)
        return fail(PA_ERR_INVALID_ARG, "decode: null pointer");
    if (!aligned16(a.out) || !aligned16(a.query) || !aligned16(a.key_cache) ||
        !aligned16(a.value_cache))
        return fail(PA_ERR_INVALID_ARG, "decode: device buffers must be 16-byte aligned");
    return PA_OK;
}

pa::KernelKey kernel_key(const DecodeArgs& a) {
    pa::KernelKey k;
    k.head_size = a.head_size;
    k.block_size = a.block_size;
    k.bf16 = a.dtype == PA_BF16;
    k.kv8 = a.kv8;
    const int g = a.num_q_heads / a.num_kv_heads;
    if (a.q_len > 1) {
        k.mq = true;
        k.mma = true;
        if (use_mq_tc(a)) {
            k.tc = true;
            k.heads_cap = mq_tc_rows(a.q_len * g, a.block_size);
            return k;
        }
        k.heads_cap = mq_heads_cap(a.q_len * g);
        k.mq_consumers = mq_consumers(a.q_len * g);
        return k;
    }
    // fp8 caches take the tensor cores for multi-head attention too: widening E4M3 tiles
    // to fp16 fragments is cheaper there than per-element conversion on the CUDA cores
    k.mma = (g >= 2 || a.kv8) && (g > 8 || g_gqa_mma);
    if (k.mma) k.heads_cap = g <= 8 ? 8 : 16;
    else k.heads_cap = g <= 1 ? 1 : g <= 2 ? 2 : g <= 4 ? 4 : 8;
    k.tile_blocks = tile_blocks_for(a);
    return k;
}

pa::DecodeParams base_params(const DecodeArgs& a) {
    pa::DecodeParams p;
    std::memset(&p, 0, sizeof(p));
    p.out = a.out;
    p.q = a.query;
    p.block_tables = a.block_tables;
    p.context_lens = a.context_lens;
    p.max_blocks_per_seq = a.max_blocks_per_seq;
    p.num_seqs = a.num_seqs;
    p.num_q_heads = a.num_q_heads;
    p.num_kv_heads = a.num_kv_heads;
    p.group = a.num_q_heads / a.num_kv_heads;
    p.num_blocks = a.num_blocks;
    p.block_size = a.block_size;
    p.max_context_len = a.max_context_len;
    p.scale_log2 = a.scale * (a.kv8 ? a.k_scale : 1.f) * 1.4426950408889634f;
    p.out_scale = a.kv8 ? a.v_scale : 1.f;
    p.status = a.status;
    p.q_len = a.q_len;
    p.rows = a.q_len * p.group;
    if (use_mq_tc(a)) {
        const int32_t r = mq_tc_rows(p.rows, a.block_size);
        p.row_chunks = (p.rows + r - 1) / r;
        p.row_groups = 1;
        p.partition_align = pa::kTcTileTokens;
    } else {
        p.row_chunks = a.q_len > 1 ? mq_row_chunks(p.rows) : 1;
        p.row_groups = a.q_len > 1 ? mq_row_groups(p.rows) : 1;
        p.partition_align = a.block_size * tile_blocks_for(a);
    }
    return p;
}

pa_status make_maps(const DecodeArgs& a, CUtensorMap* km, CUtensorMap* vm) {
    const int64_t rows = (int64_t)a.num_blocks * a.num_kv_heads * a.block_size;
    pa_status st = encode_pool_map(km, a.key_cache, rows, a.head_size, a.block_size, a.kv8);
    if (st != PA_OK) return st;
    return encode_pool_map(vm, a.value_cache, rows, a.head_size, a.block_size, a.kv8);
}

// The reshape_and_cache of a decode step (pa_decode_step), launched by the decode call
// right before its decode kernel -- after the plan kernel, whose work then overlaps the end
// of the decode kernel before it.
struct StepReshape {
    const void* key;
    const void* value;
    void* key_cache;
    void* value_cache;
    const int32_t* slot_mapping;
    int32_t num_tokens, num_kv_heads, head_size, block_size, num_blocks;
    int32_t* status;
};

pa_status check_reshape(const void* key, const void* value, void* key_cache, void* value_cache,
                        const int32_t* slot_mapping, int32_t num_tokens, int32_t num_kv_heads,
                        int32_t head_size, int32_t block_size, int32_t num_blocks, pa_dtype dtype) {
    if (num_tokens < 0 || num_kv_heads <= 0 || head_size <= 0 || block_size <= 0 || num_blocks <= 0)
        return fail(PA_ERR_INVALID_ARG, "reshape_and_cache: sizes must be positive");
    if (dtype != PA_F16 && dtype != PA_BF16) return fail(PA_ERR_UNSUPPORTED, "reshape_and_cache: dtype");
    if (head_size % 8)
        return fail(PA_ERR_UNSUPPORTED, "reshape_and_cache: head_size must be a multiple of 8");
    if (num_tokens == 0) return PA_OK;
    if (!key || !value || !key_cache || !value_cache || !slot_mapping)
        return fail(PA_ERR_INVALID_ARG, "reshape_and_cache: null pointer");
    if (!aligned16(key) || !aligned16(value) || !aligned16(key_cache) || !aligned16(value_cache))
        return fail(PA_ERR_INVALID_ARG, "reshape_and_cache: buffers must be 16-byte aligned");
    return PA_OK;
}

cudaError_t launch_step_reshape(const StepReshape* rs, cudaStream_t st) {
    if (!rs || rs->num_tokens <= 0) return cudaSuccess;
    return pa::launch_reshape_and_cache(rs->key, rs->value, rs->key_cache, rs->value_cache,
                                        rs->slot_mapping, rs->num_tokens, rs->num_kv_heads,
                                        rs->head_size, rs->block_size, rs->num_blocks, rs->status,
                                        st);
}

pa_status run_v1(const DecodeArgs& a, const StepReshape* rs = nullptr) {
    pa_status st = check_decode(a);
    if (st != PA_OK) return st;
    if (a.num_seqs == 0) {
        cudaError_t e = launch_step_reshape(rs, a.stream);
        return e == cudaSuccess ? ok() : cuda_fail(e, "reshape_and_cache launch");
    }
    CUtensorMap km, vm;
    if ((st = make_maps(a, &km, &vm)) != PA_OK) return st;
    pa::DecodeParams p = base_params(a);
    p.partition_size = 0;
    const int64_t units = (int64_t)a.num_seqs * a.num_kv_heads * p.row_chunks;
    if (units > INT32_MAX) return fail(PA_ERR_UNSUPPORTED, "decode_v1: too many (seq, head) units");
    cudaError_t e = launch_step_reshape(rs, a.stream);
    if (e != cudaSuccess) return cuda_fail(e, "reshape_and_cache launch");
    e = timed_decode(kernel_key(a), km, vm, p, false, (int32_t)units, a.stream);
    if (e != cudaSuccess) return cuda_fail(e, "decode_v1 launch");
    return ok();
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

pa_status run_v2(const DecodeArgs& a_in, int32_t partition_size, void* ws, size_t ws_bytes,
                 bool adaptive = false, const StepReshape* rs = nullptr) {
    DecodeArgs a = a_in;
    a.partition_size = adaptive ? 0 : partition_size;
    pa_status st = check_decode(a);
    if (st != PA_OK) return st;
    if (partition_size <= 0 || partition_size % a.block_size)
        return fail(PA_ERR_INVALID_ARG, "decode_v2: partition_size %d must be a positive multiple "
                    "of block_size %d", partition_size, a.block_size);
    if (a.num_seqs == 0) {
        cudaError_t e = launch_step_reshape(rs, a.stream);
        return e == cudaSuccess ? ok() : cuda_fail(e, "reshape_and_cache launch");
    }
    // partial rows per partition: q_len * num_q_heads
    const pa::WorkspaceLayout L = pa::v2_workspace_layout(a.num_seqs, a.num_q_heads * a.q_len,
                                                          a.head_size, a.max_context_len,
                                                          partition_size);
    if (!ws || ws_bytes < L.total)
        return fail(PA_ERR_WORKSPACE, "decode_v2: workspace of %zu bytes, need %zu", ws_bytes, L.total);
    if (reinterpret_cast<uintptr_t>(ws) & 255u)
        return fail(PA_ERR_INVALID_ARG, "decode_v2: workspace must be 256-byte aligned");
    int dev;
    DeviceInfo di;
    if ((st = current_device(&dev, &di)) != PA_OK) return st;
    CUtensorMap km, vm;
    if ((st = make_maps(a, &km, &vm)) != PA_OK) return st;
    pa::DecodeParams p = base_params(a);
    p.partition_size = partition_size;
    p.adaptive = adaptive ? 1 : 0;
    uint8_t* w = static_cast<uint8_t*>(ws);
    p.hdr = reinterpret_cast<pa::WsHeader*>(w + L.hdr);
    p.part_list = reinterpret_cast<int4*>(w + L.part_list);
    p.arrive = reinterpret_cast<int32_t*>(w + L.arrive);
    p.part_ml = reinterpret_cast<float2*>(w + L.part_ml);
    p.part_acc = reinterpret_cast<float*>(w + L.part_acc);
    const pa::KernelKey k = kernel_key(a);
    const int32_t per_sm = ctas_per_sm(dev, k);
    if (per_sm <= 0) return fail(PA_ERR_CUDA, "decode_v2: kernel cannot be resident on this device");
    const int64_t max_parts_per_seq =
        std::max<int64_t>(1, ((int64_t)a.max_context_len + partition_size - 1) / partition_size);
    const int64_t max_units = (int64_t)a.num_seqs * max_parts_per_seq * a.num_kv_heads * p.row_chunks;
    if (max_units > INT32_MAX) return fail(PA_ERR_UNSUPPORTED, "decode_v2: too many work units");
    const int32_t grid = (int32_t)std::min<int64_t>((int64_t)per_sm * di.sms, max_units);
    p.grid_ctas = grid;
    cudaError_t e = pa::launch_plan(p, a.stream);
    if (e != cudaSuccess) return cuda_fail(e, "decode_v2 plan launch");
    e = launch_step_reshape(rs, a.stream);
    if (e != cudaSuccess) return cuda_fail(e, "reshape_and_cache launch");
    e = timed_decode(k, km, vm, p, true, grid, a.stream);
    if (e != cudaSuccess) return cuda_fail(e, "decode_v2 launch");
    return ok();
}

// pa_decode_auto's choice.  V1 gives a whole context to one work unit, which is fine
// while every context is short and there are many units; otherwise V2 splits contexts
// into partitions that the persistent CTAs share out.
void auto_plan(int32_t num_seqs, int32_t num_kv_heads, int32_t block_size,
               int32_t max_context_len, int32_t* variant, int32_t* psize) {
    int dev = 0;
    DeviceInfo di;
    if (current_device(&dev, &di) != PA_OK || di.sms <= 0) di.sms = 148;
    const int64_t units = (int64_t)num_seqs * num_kv_heads;
    if (max_context_len <= 256 && units >= 4LL * di.sms) {
        *variant = 1;
        *psize = 0;
        return;
    }
    // V2 with adaptive partitions: the plan kernel picks the partition size on the
    // device from the real lengths; 256 tokens is the smallest it may choose, which
    // bounds the workspace.
    *variant = 2;
    *psize = std::max(block_size, (256 / block_size) * block_size);
}

}  // namespace

namespace pa {

int32_t check_decode_v2_args(const void* out, const void* query, const void* key_cache,
                             const void* value_cache, const int32_t* block_tables,
                             int32_t max_blocks_per_seq, const int32_t* context_lens,
                             int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                             int32_t head_size, int32_t block_size, int32_t num_blocks,
                             int32_t max_context_len, int32_t dtype, int32_t partition_size) {
    DecodeArgs a{const_cast<void*>(out), query, key_cache, value_cache, block_tables,
                 max_blocks_per_seq, context_lens, num_seqs, num_q_heads, num_kv_heads,
                 head_size, block_size, num_blocks, max_context_len, 1.f, (pa_dtype)dtype,
                 nullptr, nullptr};
    a.partition_size = partition_size;
    pa_status st = check_decode(a);
    if (st != PA_OK) return st;
    if (partition_size <= 0 || partition_size % block_size)
        return fail(PA_ERR_INVALID_ARG, "decode_v2: partition_size %d must be a positive multiple "
                    "of block_size %d", partition_size, block_size);
    return PA_OK;
}

int32_t set_last_error(int32_t status, const char* message) {
    g_last_error = message ? message : "";
    return status;
}

WorkspaceLayout v2_workspace_layout(int32_t num_seqs, int32_t num_q_heads, int32_t head_size,
                                    int32_t max_context_len, int32_t partition_size) {
    WorkspaceLayout L;
    const int64_t ppseq =
        std::max<int64_t>(1, ((int64_t)std::max(max_context_len, 0) + partition_size - 1) / partition_size);
    const int64_t parts = (int64_t)num_seqs * ppseq;
    size_t off = 0;
    L.hdr = off;
    off = align256(off + sizeof(WsHeader));
    L.part_list = off;
    off = align256(off + sizeof(int4) * (size_t)parts);
    L.arrive = off;   // [num_seqs][num_kv_heads] used; sized by num_q_heads >= num_kv_heads
    off = align256(off + sizeof(int32_t) * (size_t)num_seqs * (size_t)num_q_heads);
    L.part_ml = off;
    off = align256(off + sizeof(float2) * (size_t)parts * (size_t)num_q_heads);
    L.part_acc = off;
    off = align256(off + sizeof(float) * (size_t)parts * (size_t)num_q_heads * (size_t)head_size);
    L.total = off;
    return L;
}

}  // namespace pa

// =====================================================================================
// C ABI
// =====================================================================================
extern "C" {

const char* pa_last_error(void) { return g_last_error.c_str(); }

int32_t pa_version(void) { return 100; }

namespace {

// Device staging of pa_decode_step_host: the step's inputs and its output rows.
struct StagingLayout {
    size_t out, q, k, v, slots, tables, lens, total;
};

StagingLayout staging_layout(int32_t S, int32_t Hq, int32_t Hkv, int32_t D, int32_t maxb) {
    StagingLayout L;
    size_t off = 0;
    L.out = off;
    off = align256(off + (size_t)S * Hq * D * 2);
    L.q = off;
    off = align256(off + (size_t)S * Hq * D * 2);
    L.k = off;
    off = align256(off + (size_t)S * Hkv * D * 2);
    L.v = off;
    off = align256(off + (size_t)S * Hkv * D * 2);
    L.slots = off;
    off = align256(off + (size_t)S * 4);
    L.tables = off;
    off = align256(off + (size_t)S * maxb * 4);
    L.lens = off;
    off = align256(off + (size_t)S * 4);
    L.total = off;
    return L;
}

}  // namespace

size_t pa_decode_step_host_staging_size(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                                        int32_t head_size, int32_t max_blocks_per_seq) {
    if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_size <= 0 ||
        max_blocks_per_seq <= 0)
        return 0;
    return staging_layout(num_seqs, num_q_heads, num_kv_heads, head_size, max_blocks_per_seq).total;
}

namespace {

// pa_decode_step_host and pa_decode_step_host_overlapped: the input copies go on `h2d`,
// the step on `compute`, the output copy on `d2h`; with events the streams are ordered
// through them (see pa.h), with one stream and no events everything is in stream order.
pa_status step_host(void* out_host, const void* query_host, const void* key_host,
                    const void* value_host, const int32_t* slot_mapping_host,
                    const int32_t* block_tables_host, const int32_t* context_lens_host,
                    void* key_cache, void* value_cache, int32_t max_blocks_per_seq,
                    int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_size,
                    int32_t block_size, int32_t num_blocks, int32_t max_context_len, float scale,
                    pa_dtype dtype, void* staging, size_t staging_bytes, void* workspace,
                    size_t workspace_bytes, int32_t* status_dev, cudaStream_t compute,
                    cudaStream_t h2d, cudaStream_t d2h, cudaEvent_t staged, cudaEvent_t done) {
    if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_size <= 0 ||
        max_blocks_per_seq <= 0)
        return fail(PA_ERR_INVALID_ARG, "decode_step_host: sizes must be positive");
    if (num_seqs == 0) return ok();
    if (!out_host || !query_host || !key_host || !value_host || !slot_mapping_host ||
        !block_tables_host || !context_lens_host)
        return fail(PA_ERR_INVALID_ARG, "decode_step_host: null host pointer");
    const StagingLayout L =
        staging_layout(num_seqs, num_q_heads, num_kv_heads, head_size, max_blocks_per_seq);
    if (!staging || staging_bytes < L.total)
        return fail(PA_ERR_WORKSPACE, "decode_step_host: staging of %zu bytes, need %zu",
                    staging_bytes, L.total);
    if (reinterpret_cast<uintptr_t>(staging) & 255u)
        return fail(PA_ERR_INVALID_ARG, "decode_step_host: staging must be 256-byte aligned");
    uint8_t* st = static_cast<uint8_t*>(staging);
    const size_t S = (size_t)num_seqs;
    cudaError_t e;
    struct Copy {
        void* dst;
        const void* src;
        size_t bytes;
    } copies[] = {
        {st + L.q, query_host, S * num_q_heads * head_size * 2},
        {st + L.k, key_host, S * num_kv_heads * head_size * 2},
        {st + L.v, value_host, S * num_kv_heads * head_size * 2},
        {st + L.slots, slot_mapping_host, S * 4},
        {st + L.tables, block_tables_host, S * max_blocks_per_seq * 4},
        {st + L.lens, context_lens_host, S * 4},
    };
    for (const Copy& c : copies) {
        e = cudaMemcpyAsync(c.dst, c.src, c.bytes, cudaMemcpyHostToDevice, h2d);
        if (e != cudaSuccess) return cuda_fail(e, "decode_step_host: H2D copy");
    }
    if (staged) {
        if ((e = cudaEventRecord(staged, h2d)) != cudaSuccess ||
            (e = cudaStreamWaitEvent(compute, staged, 0)) != cudaSuccess)
            return cuda_fail(e, "decode_step_host: staged event");
    }
    pa_status ps = pa_decode_step(
        st + L.out, st + L.q, st + L.k, st + L.v, key_cache, value_cache,
        reinterpret_cast<const int32_t*>(st + L.slots), reinterpret_cast<const int32_t*>(st + L.tables),
        max_blocks_per_seq, reinterpret_cast<const int32_t*>(st + L.lens), num_seqs, num_q_heads,
        num_kv_heads, head_size, block_size, num_blocks, max_context_len, scale, dtype, workspace,
        workspace_bytes, status_dev, (pa_stream)compute);
    if (ps != PA_OK) return ps;
    if (done) {
        if ((e = cudaEventRecord(done, compute)) != cudaSuccess ||
            (e = cudaStreamWaitEvent(d2h, done, 0)) != cudaSuccess)
            return cuda_fail(e, "decode_step_host: done event");
    }
    e = cudaMemcpyAsync(out_host, st + L.out, S * num_q_heads * head_size * 2,
                        cudaMemcpyDeviceToHost, d2h);
    if (e != cudaSuccess) return cuda_fail(e, "decode_step_host: D2H copy");
    return ok();
}

}  // namespace

pa_status pa_decode_step_host(void* out_host, const void* query_host, const void* key_host,
                              const void* value_host, const int32_t* slot_mapping_host,
                              const int32_t* block_tables_host, const int32_t* context_lens_host,
                              void* key_cache, void* value_cache, int32_t max_blocks_per_seq,
                              int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                              int32_t head_size, int32_t block_size, int32_t num_blocks,
                              int32_t max_context_len, float scale, pa_dtype dtype, void* staging,
                              size_t staging_bytes, void* workspace, size_t workspace_bytes,
                              int32_t* status_dev, pa_stream stream) {
    cudaStream_t cs = (cudaStream_t)stream;
    return step_host(out_host, query_host, key_host, value_host, slot_mapping_host,
                     block_tables_host, context_lens_host, key_cache, value_cache,
                     max_blocks_per_seq, num_seqs, num_q_heads, num_kv_heads, head_size,
                     block_size, num_blocks, max_context_len, scale, dtype, staging, staging_bytes,
                     workspace, workspace_bytes, status_dev, cs, cs, cs, nullptr, nullptr);
}

pa_status pa_decode_step_host_overlapped(
    void* out_host, const void* query_host, const void* key_host, const void* value_host,
    const int32_t* slot_mapping_host, const int32_t* block_tables_host,
    const int32_t* context_lens_host, void* key_cache, void* value_cache,
    int32_t max_blocks_per_seq, int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
    int32_t head_size, int32_t block_size, int32_t num_blocks, int32_t max_context_len,
    float scale, pa_dtype dtype, void* staging, size_t staging_bytes, void* workspace,
    size_t workspace_bytes, int32_t* status_dev, pa_stream compute, pa_stream h2d,
    pa_stream d2h, void* staged_event, void* done_event) {
    if (!staged_event || !done_event)
        return fail(PA_ERR_INVALID_ARG, "decode_step_host_overlapped: both events are needed");
    if (compute == h2d || compute == d2h)
        return fail(PA_ERR_INVALID_ARG, "decode_step_host_overlapped: the copies need streams of their own");
    return step_host(out_host, query_host, key_host, value_host, slot_mapping_host,
                     block_tables_host, context_lens_host, key_cache, value_cache,
                     max_blocks_per_seq, num_seqs, num_q_heads, num_kv_heads, head_size,
                     block_size, num_blocks, max_context_len, scale, dtype, staging, staging_bytes,
                     workspace, workspace_bytes, status_dev, (cudaStream_t)compute,
                     (cudaStream_t)h2d, (cudaStream_t)d2h, static_cast<cudaEvent_t>(staged_event),
                     static_cast<cudaEvent_t>(done_event));
}

pa_status pa_advance_step(int32_t* context_lens, int32_t* slot_mapping, const int32_t* block_tables,
                          int32_t max_blocks_per_seq, int32_t num_seqs, int32_t block_size,
                          int32_t num_blocks, int64_t* input_positions, int64_t* input_tokens,
                          const int64_t* sampled_token_ids, int32_t* status_dev, pa_stream stream) {
    if (num_seqs < 0 || max_blocks_per_seq <= 0 || block_size <= 0 || num_blocks <= 0)
        return fail(PA_ERR_INVALID_ARG, "advance_step: sizes must be positive");
    if (num_seqs == 0) return ok();
    if (!context_lens || !slot_mapping || !block_tables)
        return fail(PA_ERR_INVALID_ARG, "advance_step: null pointer");
    if ((input_tokens == nullptr) != (sampled_token_ids == nullptr))
        return fail(PA_ERR_INVALID_ARG, "advance_step: input_tokens and sampled_token_ids go together");
    cudaError_t e = pa::launch_advance_step(context_lens, slot_mapping, block_tables,
                                            max_blocks_per_seq, num_seqs, block_size, num_blocks,
                                            input_positions, input_tokens, sampled_token_ids,
                                            status_dev, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "advance_step launch");
    return ok();
}

pa_status pa_copy_blocks(void* key_cache, void* value_cache, const int32_t* block_pairs,
                         int32_t num_pairs, int32_t num_kv_heads, int32_t head_size,
                         int32_t block_size, int32_t num_blocks, pa_dtype dtype,
                         int32_t* status_dev, pa_stream stream) {
    if (num_pairs < 0 || num_kv_heads <= 0 || head_size <= 0 || block_size <= 0 || num_blocks <= 0)
        return fail(PA_ERR_INVALID_ARG, "copy_blocks: sizes must be positive");
    if (dtype != PA_F16 && dtype != PA_BF16 && dtype != PA_FP8_E4M3)
        return fail(PA_ERR_UNSUPPORTED, "copy_blocks: dtype");
    if (num_pairs == 0) return ok();
    if (!key_cache || !value_cache || !block_pairs)
        return fail(PA_ERR_INVALID_ARG, "copy_blocks: null pointer");
    const int64_t bytes = (int64_t)num_kv_heads * block_size * head_size * (dtype == PA_FP8_E4M3 ? 1 : 2);
    if (!aligned16(key_cache) || !aligned16(value_cache) || bytes % 16)
        return fail(PA_ERR_INVALID_ARG, "copy_blocks: pools must be 16-byte aligned, blocks 16-byte multiples");
    cudaError_t e = pa::launch_copy_blocks(key_cache, value_cache, block_pairs, num_pairs, bytes,
                                           num_blocks, status_dev, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "copy_blocks launch");
    return ok();
}

pa_status pa_selftest_wait_timeout(int32_t* status_dev, uint32_t limit_us, pa_stream stream) {
    if (!status_dev) return fail(PA_ERR_INVALID_ARG, "selftest_wait_timeout: status_dev is NULL");
    if (limit_us == 0 || limit_us > 2000000u)
        return fail(PA_ERR_INVALID_ARG, "selftest_wait_timeout: limit_us must be in 1 .. 2000000");
    cudaError_t e = pa::launch_wait_timeout_probe(status_dev, (uint64_t)limit_us * 1000ull,
                                                  (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "selftest_wait_timeout launch");
    return ok();
}

pa_status pa_set_kernel_events(void* start_event, void* stop_event) {
    if ((start_event == nullptr) != (stop_event == nullptr))
        return fail(PA_ERR_INVALID_ARG, "set_kernel_events: give both events or neither");
    g_ev_start = static_cast<cudaEvent_t>(start_event);
    g_ev_stop = static_cast<cudaEvent_t>(stop_event);
    return ok();
}

pa_status pa_set_gqa_tensor_cores(int32_t enable) {
    g_gqa_mma = enable ? 1 : 0;
    return ok();
}

pa_status pa_set_mq_tcgen05(int32_t enable) {
    g_mq_tc = enable ? 1 : 0;
    return ok();
}

pa_status pa_reshape_and_cache(const void* key, const void* value, void* key_cache,
                               void* value_cache, const int32_t* slot_mapping, int32_t num_tokens,
                               int32_t num_kv_heads, int32_t head_size, int32_t block_size,
                               int32_t num_blocks, pa_dtype dtype, int32_t* status_dev,
                               pa_stream stream) {
    pa_status st = check_reshape(key, value, key_cache, value_cache, slot_mapping, num_tokens,
                                 num_kv_heads, head_size, block_size, num_blocks, dtype);
    if (st != PA_OK || num_tokens == 0) return st == PA_OK ? ok() : st;
    cudaError_t e = pa::launch_reshape_and_cache(key, value, key_cache, value_cache, slot_mapping,
                                                 num_tokens, num_kv_heads, head_size, block_size,
                                                 num_blocks, status_dev, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "reshape_and_cache launch");
    return ok();
}

pa_status pa_decode_v1(void* out, const void* query, const void* key_cache, const void* value_cache,
                       const int32_t* block_tables, int32_t max_blocks_per_seq,
                       const int32_t* context_lens, int32_t num_seqs, int32_t num_q_heads,
                       int32_t num_kv_heads, int32_t head_size, int32_t block_size,
                       int32_t num_blocks, int32_t max_context_len, float scale, pa_dtype dtype,
                       int32_t* status_dev, pa_stream stream) {
    DecodeArgs a{out, query, key_cache, value_cache, block_tables, max_blocks_per_seq,
                 context_lens, num_seqs, num_q_heads, num_kv_heads, head_size, block_size,
                 num_blocks, max_context_len, scale, dtype, status_dev, (cudaStream_t)stream};
    return run_v1(a);
}

size_t pa_decode_v2_workspace_size(int32_t num_seqs, int32_t num_q_heads, int32_t head_size,
                                   int32_t max_context_len, int32_t partition_size) {
    if (num_seqs < 0 || num_q_heads <= 0 || head_size <= 0 || partition_size <= 0) return 0;
    return pa::v2_workspace_layout(num_seqs, num_q_heads, head_size, max_context_len,
                                   partition_size).total;
}

pa_status pa_decode_v2(void* out, const void* query, const void* key_cache, const void* value_cache,
                       const int32_t* block_tables, int32_t max_blocks_per_seq,
                       const int32_t* context_lens, int32_t num_seqs, int32_t num_q_heads,
                       int32_t num_kv_heads, int32_t head_size, int32_t block_size,
                       int32_t num_blocks, int32_t max_context_len, float scale, pa_dtype dtype,
                       int32_t partition_size, void* workspace, size_t workspace_bytes,
                       int32_t* status_dev, pa_stream stream) {
    DecodeArgs a{out, query, key_cache, value_cache, block_tables, max_blocks_per_seq,
                 context_lens, num_seqs, num_q_heads, num_kv_heads, head_size, block_size,
                 num_blocks, max_context_len, scale, dtype, status_dev, (cudaStream_t)stream};
    return run_v2(a, partition_size, workspace, workspace_bytes);
}

pa_status pa_decode_auto_plan(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                              int32_t head_size, int32_t block_size, int32_t max_context_len,
                              int32_t* variant, int32_t* partition_size) {
    (void)num_q_heads;
    (void)head_size;
    if (!variant || !partition_size) return fail(PA_ERR_INVALID_ARG, "auto_plan: null output");
    if (num_seqs < 0 || num_kv_heads <= 0 || block_size <= 0 || max_context_len < 0)
        return fail(PA_ERR_INVALID_ARG, "auto_plan: bad sizes");
    auto_plan(num_seqs, num_kv_heads, block_size, max_context_len, variant, partition_size);
    return ok();
}

size_t pa_decode_auto_workspace_size(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                                     int32_t head_size, int32_t block_size,
                                     int32_t max_context_len) {
    int32_t v = 0, P = 0;
    if (pa_decode_auto_plan(num_seqs, num_q_heads, num_kv_heads, head_size, block_size,
                            max_context_len, &v, &P) != PA_OK)
        return 0;
    if (v == 1) return 0;
    return pa_decode_v2_workspace_size(num_seqs, num_q_heads, head_size, max_context_len, P);
}

pa_status pa_decode_auto(void* out, const void* query, const void* key_cache,
                         const void* value_cache, const int32_t* block_tables,
                         int32_t max_blocks_per_seq, const int32_t* context_lens, int32_t num_seqs,
                         int32_t num_q_heads, int32_t num_kv_heads, int32_t head_size,
                         int32_t block_size, int32_t num_blocks, int32_t max_context_len,
                         float scale, pa_dtype dtype, void* workspace, size_t workspace_bytes,
                         int32_t* status_dev, pa_stream stream) {
    int32_t v = 0, P = 0;
    pa_status st = pa_decode_auto_plan(num_seqs, num_q_heads, num_kv_heads, head_size, block_size,
                                       max_context_len, &v, &P);
    if (st != PA_OK) return st;
    DecodeArgs a{out, query, key_cache, value_cache, block_tables, max_blocks_per_seq,
                 context_lens, num_seqs, num_q_heads, num_kv_heads, head_size, block_size,
                 num_blocks, max_context_len, scale, dtype, status_dev, (cudaStream_t)stream};
    if (v == 1) return run_v1(a);
    return run_v2(a, P, workspace, workspace_bytes, /*adaptive=*/true);
}

pa_status pa_reshape_and_cache_fp8(const void* key, const void* value, void* key_cache,
                                   void* value_cache, const int32_t* slot_mapping,
                                   int32_t num_tokens, int32_t num_kv_heads, int32_t head_size,
                                   int32_t block_size, int32_t num_blocks, pa_dtype dtype,
                                   float k_scale, float v_scale, int32_t* status_dev,
                                   pa_stream stream) {
    if (num_tokens < 0 || num_kv_heads <= 0 || head_size <= 0 || block_size <= 0 || num_blocks <= 0)
        return fail(PA_ERR_INVALID_ARG, "reshape_and_cache_fp8: sizes must be positive");
    if (dtype != PA_F16 && dtype != PA_BF16)
        return fail(PA_ERR_UNSUPPORTED, "reshape_and_cache_fp8: key/value must be fp16 or bf16");
    if (head_size % 8) return fail(PA_ERR_UNSUPPORTED, "reshape_and_cache_fp8: head_size % 8");
    if (!(k_scale > 0.f && v_scale > 0.f))
        return fail(PA_ERR_INVALID_ARG, "reshape_and_cache_fp8: scales must be positive");
    if (num_tokens == 0) return ok();
    if (!key || !value || !key_cache || !value_cache || !slot_mapping)
        return fail(PA_ERR_INVALID_ARG, "reshape_and_cache_fp8: null pointer");
    if (!aligned16(key) || !aligned16(value) || !aligned16(key_cache) || !aligned16(value_cache))
        return fail(PA_ERR_INVALID_ARG, "reshape_and_cache_fp8: buffers must be 16-byte aligned");
    const float k_inv = 1.0f / k_scale, v_inv = 1.0f / v_scale;   // correctly rounded fp32
    cudaError_t e = pa::launch_reshape_and_cache_fp8(key, value, key_cache, value_cache,
                                                     slot_mapping, num_tokens, num_kv_heads,
                                                     head_size, block_size, num_blocks,
                                                     dtype == PA_BF16, k_inv, v_inv, status_dev,
                                                     (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "reshape_and_cache_fp8 launch");
    return ok();
}

pa_status pa_decode_fp8(void* out, const void* query, const void* key_cache, const void* value_cache,
                        const int32_t* block_tables, int32_t max_blocks_per_seq,
                        const int32_t* context_lens, int32_t num_seqs, int32_t num_q_heads,
                        int32_t num_kv_heads, int32_t head_size, int32_t block_size,
                        int32_t num_blocks, int32_t max_context_len, float scale, float k_scale,
                        float v_scale, pa_dtype dtype, int32_t variant, int32_t partition_size,
                        void* workspace, size_t workspace_bytes, int32_t* status_dev,
                        pa_stream stream) {
    DecodeArgs a{out, query, key_cache, value_cache, block_tables, max_blocks_per_seq,
                 context_lens, num_seqs, num_q_heads, num_kv_heads, head_size, block_size,
                 num_blocks, max_context_len, scale, dtype, status_dev, (cudaStream_t)stream};
    a.kv8 = true;
    a.k_scale = k_scale;
    a.v_scale = v_scale;
    if (variant == 1) return run_v1(a);
    if (variant == 2) return run_v2(a, partition_size, workspace, workspace_bytes);
    if (variant != 0) return fail(PA_ERR_INVALID_ARG, "decode_fp8: variant must be 0, 1 or 2");
    int32_t v = 0, P = 0;
    pa_status st = pa_decode_auto_plan(num_seqs, num_q_heads, num_kv_heads, head_size, block_size,
                                       max_context_len, &v, &P);
    if (st != PA_OK) return st;
    if (v == 1) return run_v1(a);
    return run_v2(a, P, workspace, workspace_bytes, /*adaptive=*/true);
}

size_t pa_decode_mq_workspace_size(int32_t num_seqs, int32_t q_len, int32_t num_q_heads,
                                   int32_t num_kv_heads, int32_t head_size, int32_t block_size,
                                   int32_t max_context_len, int32_t partition_size) {
    if (num_seqs < 0 || q_len < 1 || num_q_heads <= 0 || num_kv_heads <= 0 || head_size <= 0 ||
        block_size <= 0 || max_context_len < 0 || partition_size < 0)
        return 0;
    if (partition_size == 0) {
        int32_t v = 0;
        auto_plan(num_seqs * mq_row_chunks(q_len * std::max(num_q_heads / num_kv_heads, 1)),
                  num_kv_heads, block_size, max_context_len, &v, &partition_size);
        if (v == 1) return 0;
    }
    return pa::v2_workspace_layout(num_seqs, num_q_heads * q_len, head_size, max_context_len,
                                   partition_size).total;
}

pa_status pa_decode_mq(void* out, const void* query, const void* key_cache, const void* value_cache,
                       const int32_t* block_tables, int32_t max_blocks_per_seq,
                       const int32_t* context_lens, int32_t num_seqs, int32_t q_len,
                       int32_t num_q_heads, int32_t num_kv_heads, int32_t head_size,
                       int32_t block_size, int32_t num_blocks, int32_t max_context_len,
                       float scale, pa_dtype dtype, int32_t variant, int32_t partition_size,
                       void* workspace, size_t workspace_bytes, int32_t* status_dev,
                       pa_stream stream) {
    DecodeArgs a{out, query, key_cache, value_cache, block_tables, max_blocks_per_seq,
                 context_lens, num_seqs, num_q_heads, num_kv_heads, head_size, block_size,
                 num_blocks, max_context_len, scale, dtype, status_dev, (cudaStream_t)stream};
    a.q_len = q_len;
    if (q_len < 1) return fail(PA_ERR_INVALID_ARG, "decode_mq: q_len %d must be >= 1", q_len);
    if (num_kv_heads <= 0 || num_q_heads <= 0)
        return fail(PA_ERR_INVALID_ARG, "decode_mq: sizes must be positive");
    if (variant == 1) return run_v1(a);
    if (variant == 2) return run_v2(a, partition_size, workspace, workspace_bytes);
    if (variant != 0) return fail(PA_ERR_INVALID_ARG, "decode_mq: variant must be 0, 1 or 2");
    // the auto choice, counting each chunk of query rows as a unit of its own
    int32_t v = 0, P = 0;
    const int32_t chunks = q_len > 1 ? mq_row_chunks(q_len * std::max(num_q_heads / num_kv_heads, 1)) : 1;
    if (num_seqs < 0 || block_size <= 0 || max_context_len < 0)
        return fail(PA_ERR_INVALID_ARG, "decode_mq: bad sizes");
    auto_plan(num_seqs * chunks, num_kv_heads, block_size, max_context_len, &v, &P);
    if (v == 1) return run_v1(a);
    return run_v2(a, P, workspace, workspace_bytes, /*adaptive=*/true);
}

pa_status pa_decode_step(void* out, const void* query, const void* key, const void* value,
                         void* key_cache, void* value_cache, const int32_t* slot_mapping,
                         const int32_t* block_tables, int32_t max_blocks_per_seq,
                         const int32_t* context_lens, int32_t num_seqs, int32_t num_q_heads,
                         int32_t num_kv_heads, int32_t head_size, int32_t block_size,
                         int32_t num_blocks, int32_t max_context_len, float scale, pa_dtype dtype,
                         void* workspace, size_t workspace_bytes, int32_t* status_dev,
                         pa_stream stream) {
    // every argument is checked before anything is launched; the V2 plan goes first so
    // that it may overlap the end of the decode before it (see launch_plan)
    pa_status st = check_reshape(key, value, key_cache, value_cache, slot_mapping, num_seqs,
                                 num_kv_heads, head_size, block_size, num_blocks, dtype);
    if (st != PA_OK) return st;
    int32_t v = 0, P = 0;
    st = pa_decode_auto_plan(num_seqs, num_q_heads, num_kv_heads, head_size, block_size,
                             max_context_len, &v, &P);
    if (st != PA_OK) return st;
    DecodeArgs a{out, query, key_cache, value_cache, block_tables, max_blocks_per_seq,
                 context_lens, num_seqs, num_q_heads, num_kv_heads, head_size, block_size,
                 num_blocks, max_context_len, scale, dtype, status_dev, (cudaStream_t)stream};
    const StepReshape rs{key, value, key_cache, value_cache, slot_mapping, num_seqs, num_kv_heads,
                         head_size, block_size, num_blocks, status_dev};
    if (v == 1) return run_v1(a, &rs);
    return run_v2(a, P, workspace, workspace_bytes, /*adaptive=*/true, &rs);
}

}  // extern "C"
