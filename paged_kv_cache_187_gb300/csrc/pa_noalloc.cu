// pa_noalloc.cu -- pa_decode_v2_noalloc: the V2 decode for callers that may not
// allocate device memory (see include/pa.h).  Its scratch is the file-scope device
// array below; the call itself allocates nothing.
#include <cstdio>
#include <mutex>
#include <unordered_map>

#include <cuda_runtime.h>

#include "../../include/pa.h"
#include "pa_internal.h"

// One array per device that loads the library, held until the process exits.  Host
// code must not use this name as a device address: the address comes from
// cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_pa_noalloc_scratch[PA_NOALLOC_SCRATCH_BYTES];

namespace {

std::mutex g_noalloc_mu;
std::unordered_map<int, void*> g_noalloc_addr;   // device ordinal -> scratch address

// Device address of the scratch array on the current device, looked up once per device.
pa_status scratch_address(void** out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        char msg[256];
        snprintf(msg, sizeof(msg), "decode_v2_noalloc: cudaGetDevice: %s", cudaGetErrorString(e));
        return (pa_status)pa::set_last_error(PA_ERR_CUDA, msg);
    }
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    auto it = g_noalloc_addr.find(dev);
    if (it != g_noalloc_addr.end()) {
        *out = it->second;
        return PA_OK;
    }
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_pa_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) {
        char msg[256];
        snprintf(msg, sizeof(msg), "decode_v2_noalloc: cudaGetSymbolAddress: %s",
                 cudaGetErrorString(e));
        return (pa_status)pa::set_last_error(PA_ERR_CUDA, msg);
    }
    g_noalloc_addr.emplace(dev, p);
    *out = p;
    return PA_OK;
}

}  // namespace

extern "C" pa_status pa_decode_v2_noalloc(
    void* out, const void* query, const void* key_cache, const void* value_cache,
    const int32_t* block_tables, int32_t max_blocks_per_seq, const int32_t* context_lens,
    int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_size,
    int32_t block_size, int32_t num_blocks, int32_t max_context_len, float scale, pa_dtype dtype,
    int32_t partition_size, int32_t* status_dev, pa_stream stream) {
    // the same argument checks (and errors) as pa_decode_v2, before the scratch size
    const int32_t chk = pa::check_decode_v2_args(
        out, query, key_cache, value_cache, block_tables, max_blocks_per_seq, context_lens,
        num_seqs, num_q_heads, num_kv_heads, head_size, block_size, num_blocks, max_context_len,
        (int32_t)dtype, partition_size);
    if (chk != PA_OK) return (pa_status)chk;
    const size_t need = pa_decode_v2_workspace_size(num_seqs, num_q_heads, head_size,
                                                    max_context_len, partition_size);
    if (need > PA_NOALLOC_SCRATCH_BYTES) {
        char msg[256];
        snprintf(msg, sizeof(msg),
                 "decode_v2_noalloc: these sizes need %zu bytes of scratch, more than the "
                 "library's fixed %zu; use pa_decode_v2 with a workspace",
                 need, (size_t)PA_NOALLOC_SCRATCH_BYTES);
        return (pa_status)pa::set_last_error(PA_ERR_WORKSPACE, msg);
    }
    void* scratch = nullptr;
    pa_status st = scratch_address(&scratch);
    if (st != PA_OK) return st;
    return pa_decode_v2(out, query, key_cache, value_cache, block_tables, max_blocks_per_seq,
                        context_lens, num_seqs, num_q_heads, num_kv_heads, head_size, block_size,
                        num_blocks, max_context_len, scale, dtype, partition_size, scratch,
                        PA_NOALLOC_SCRATCH_BYTES, status_dev, stream);
}
