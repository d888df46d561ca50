// pa_aux.cu -- the small kernels around the decode kernel:
//   * reshape_and_cache: scatters each step's new K/V rows into the paged pools through
//     slot_mapping ("[core] Multi Step Scheduling #7000", the slot_mapping / block_tables
//     metadata a decode step carries), as-is or quantised to fp8 E4M3;
//   * plan: lists the V2 partitions of every sequence ("vLLM Project Update" talk, the V2
//     kernel that partitions sequences and spreads them over SMs) in claim order and
//     resets the counters the decode kernel uses.
#include <algorithm>
#include <cstdint>
#include <cuda_runtime.h>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {

namespace {

constexpr int32_t kBadSlot = 1;
constexpr int32_t kBadLen = 4;

__device__ __forceinline__ int32_t clamp_len(const DecodeParams& p, int32_t s, bool report) {
    int32_t L = p.context_lens[s];
    const int64_t row_cap = (int64_t)p.max_blocks_per_seq * p.block_size;
    const int32_t cap = row_cap < p.max_context_len ? (int32_t)row_cap : p.max_context_len;
    if (L < 0 || L > cap) {
        if (report && p.status) atomicOr(p.status, kBadLen);
        L = L < 0 ? 0 : cap;
    }
    return L;
}

// One CTA per new token; 16-byte copies, K then V.
__global__ void __launch_bounds__(128)
    reshape_and_cache_kernel(const uint4* __restrict__ key, const uint4* __restrict__ value,
                             uint4* __restrict__ key_cache, uint4* __restrict__ value_cache,
                             const int32_t* __restrict__ slot_mapping, int32_t num_kv_heads,
                             int32_t head_size, int32_t block_size, int32_t num_blocks,
                             int32_t* status) {
    // The kernel after this one (a decode, or a plan) may launch meanwhile: a decode waits
    // for this kernel before it reads the pools, a plan reads only the context lengths.
    // Nothing is read or written here before the kernel before this one has finished: a
    // decode may still be reading blocks that this step's slots reuse.
    allow_dependent_launch();
    grid_dependency_wait();
    const int32_t i = blockIdx.x;
    const int64_t slot = slot_mapping[i];
    if (slot < 0) return;                                   // padding token
    if (slot >= (int64_t)num_blocks * block_size) {
        if (threadIdx.x == 0 && status) atomicOr(status, kBadSlot);
        return;
    }
    const int64_t block = slot / block_size, offset = slot % block_size;
    const int32_t row_chunks = head_size / 8;               // 16-byte chunks per row
    const int32_t per_tensor = num_kv_heads * row_chunks;
    for (int32_t c = threadIdx.x; c < 2 * per_tensor; c += blockDim.x) {
        const bool is_v = c >= per_tensor;
        const int32_t r = is_v ? c - per_tensor : c;
        const int32_t h = r / row_chunks, dc = r % row_chunks;
        const int64_t src = ((int64_t)i * num_kv_heads + h) * row_chunks + dc;
        const int64_t dst = ((block * num_kv_heads + h) * block_size + offset) * row_chunks + dc;
        if (is_v) value_cache[dst] = __ldg(value + src);
        else key_cache[dst] = __ldg(key + src);
    }
}

// Quantising scatter for an fp8 E4M3 cache: each element stores
// e4m3(x * inv_scale), the fp32 product rounded to E4M3 nearest-even and saturated at
// +-448 (fp8 KV cache, "vLLM Project Update" talk).  One CTA per new token; a thread
// takes 8 elements (16 bytes in, 8 bytes out).
template <bool SRC_BF16>
__global__ void __launch_bounds__(128)
    reshape_and_cache_fp8_kernel(const uint4* __restrict__ key, const uint4* __restrict__ value,
                                 uint2* __restrict__ key_cache, uint2* __restrict__ value_cache,
                                 const int32_t* __restrict__ slot_mapping, int32_t num_kv_heads,
                                 int32_t head_size, int32_t block_size, int32_t num_blocks,
                                 float k_inv, float v_inv, int32_t* status) {
    allow_dependent_launch();   // as in reshape_and_cache_kernel
    grid_dependency_wait();
    const int32_t i = blockIdx.x;
    const int64_t slot = slot_mapping[i];
    if (slot < 0) return;
    if (slot >= (int64_t)num_blocks * block_size) {
        if (threadIdx.x == 0 && status) atomicOr(status, kBadSlot);
        return;
    }
    const int64_t block = slot / block_size, offset = slot % block_size;
    const int32_t row_chunks = head_size / 8;
    const int32_t per_tensor = num_kv_heads * row_chunks;
    for (int32_t c = threadIdx.x; c < 2 * per_tensor; c += blockDim.x) {
        const bool is_v = c >= per_tensor;
        const int32_t r = is_v ? c - per_tensor : c;
        const int32_t h = r / row_chunks, dc = r % row_chunks;
        const int64_t src = ((int64_t)i * num_kv_heads + h) * row_chunks + dc;
        const int64_t dst = ((block * num_kv_heads + h) * block_size + offset) * row_chunks + dc;
        const uint4 x = __ldg((is_v ? value : key) + src);
        const float inv = is_v ? v_inv : k_inv;
        const uint32_t w[4] = {x.x, x.y, x.z, x.w};
        uint32_t q[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            float a, b;
            unpack2<SRC_BF16>(w[j], a, b);
            q[j] = f32x2_to_e4m3x2(__fmul_rn(a, inv), __fmul_rn(b, inv));
        }
        const uint2 out = make_uint2(q[0] | (q[1] << 16), q[2] | (q[3] << 16));
        (is_v ? value_cache : key_cache)[dst] = out;
    }
}

// Block-wide exclusive scan of x over blockDim.x (a multiple of 32) threads; *total
// receives the sum.  `buf` holds 32 ints of shared memory.
__device__ __forceinline__ int32_t block_excl_scan(int32_t x, int32_t* buf, int32_t* total) {
    const int32_t lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    int32_t v = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int32_t y = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += y;
    }
    if (lane == 31) buf[warp] = v;
    __syncthreads();
    if (warp == 0) {
        int32_t w = lane < nw ? buf[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        buf[lane] = w;                       // inclusive over warps
    }
    __syncthreads();
    const int32_t excl = (warp > 0 ? buf[warp - 1] : 0) + v - x;
    *total = buf[31];
    __syncthreads();
    return excl;
}

constexpr int kTailBuckets = 256;
// Batches up to this many sequences keep their (clamped) context lengths in shared
// memory across the plan's passes, so that each is read from global memory once.
constexpr int kPlanLenCache = 4096;

// Adaptive partitioning aims at this many work units per persistent CTA: enough for the
// longest-first order to even out the CTAs' finishing times, few enough that most
// sequences need no merge at all.
#ifndef PA_UNITS_PER_CTA
#define PA_UNITS_PER_CTA 2
#endif

// Single CTA.  Lists the V2 partitions of every sequence in the order the persistent
// decode CTAs will claim them -- all full partitions first, then the partial ones from
// the longest to the shortest, so that the last units handed out are the cheapest
// (longest-processing-time-first) -- and resets the work counter and the per
// (sequence, kv head) arrival counters.  Entry: (sequence, partition, first partition
// slot of the sequence, clamped context length).  Partition slots (where partial
// results go) are numbered sequence by sequence, independent of the claim order.
//
// Launched as a programmatic dependent, it may start while the kernel ahead of it on the
// stream (a decode finishing its last units, a reshape_and_cache) still runs.  Until that
// kernel has finished it only reads -- the context lengths, which nothing between the two
// kernels can have rewritten -- and counts; it writes nothing to global memory before
// grid_dependency_wait(), so that memory the kernel ahead still uses is never touched
// (a stream-ordered allocator may have handed it out again).
__global__ void __launch_bounds__(1024) plan_kernel(const DecodeParams p) {
    __shared__ int32_t scan_buf[32];
    __shared__ int32_t hist[kTailBuckets];    // tail partitions per size bucket
    __shared__ int32_t bstart[kTailBuckets];
    __shared__ unsigned long long total_tokens;
    __shared__ int32_t P_s;
    __shared__ int32_t bad_len_s;
    __shared__ int32_t len_s[kPlanLenCache];
    allow_dependent_launch();   // the decode kernel may set up meanwhile (it waits for us)
    const int32_t tid = threadIdx.x;
    const int32_t bs = p.block_size;
    for (int32_t i = tid; i < kTailBuckets; i += blockDim.x) hist[i] = 0;
    if (tid == 0) {
        total_tokens = 0ull;
        bad_len_s = 0;
    }
    __syncthreads();
    // pass 0: every context length (clamped, errors reported), and the partition size.
    // Fixed (pa_decode_v2), or adaptive: the largest multiple of block_size, not below
    // the given minimum, that still yields about PA_UNITS_PER_CTA units per CTA.
    const bool cached = p.num_seqs <= kPlanLenCache;
    auto len_of = [&](int32_t s) { return cached ? len_s[s] : clamp_len(p, s, false); };
    {
        unsigned long long mine = 0;
        int32_t bad = 0;
        for (int32_t s = tid; s < p.num_seqs; s += blockDim.x) {
            const int32_t L = clamp_len(p, s, false);
            bad |= L != p.context_lens[s];        // clamped: reported after the wait
            if (cached) len_s[s] = L;
            mine += (unsigned)L;
        }
        if (bad) bad_len_s = 1;
        if (p.adaptive) {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) mine += __shfl_xor_sync(0xffffffffu, mine, o);
            if ((tid & 31) == 0) atomicAdd(&total_tokens, mine);   // one shared atomic per warp
        }
        __syncthreads();
    }
    if (p.adaptive) {
        if (tid == 0) {
            const unsigned long long work =
                total_tokens * (unsigned long long)p.num_kv_heads * (unsigned long long)p.row_chunks;
            const unsigned long long want = (unsigned long long)max(p.grid_ctas, 1) * PA_UNITS_PER_CTA;
            const unsigned align = (unsigned)max(bs, p.partition_align);
            unsigned long long Pa = (work / want / align) * align;
            if (Pa > (1ull << 30)) Pa = 1ull << 30;
            P_s = max(p.partition_size, (int32_t)Pa);
        }
    } else if (tid == 0) {
        P_s = p.partition_size;
    }
    __syncthreads();
    const int32_t P = P_s;
    // pass 1: counts
    int32_t parts = 0, full_parts = 0;
    for (int32_t base = 0; base < p.num_seqs; base += blockDim.x) {
        const int32_t s = base + tid;
        int32_t np = 0, nf = 0;
        if (s < p.num_seqs) {
            const int32_t L = len_of(s);
            nf = L / P;
            const int32_t tail = L - nf * P;
            np = nf + ((tail > 0 || L == 0) ? 1 : 0);
            if (tail > 0 || L == 0) {
                const int32_t b = min((tail + bs - 1) / bs, kTailBuckets - 1);
                atomicAdd(&hist[b], 1);
            }
        }
        int32_t tp, tf;
        block_excl_scan(np, scan_buf, &tp);
        block_excl_scan(nf, scan_buf, &tf);
        parts += tp;
        full_parts += tf;
    }
    __syncthreads();
    // Everything below writes global memory: only once the kernel ahead has finished.
    grid_dependency_wait();
    if (tid == 0 && bad_len_s && p.status) atomicOr(p.status, kBadLen);
    {   // first list position of each tail bucket: longer tails first
        const int32_t b = kTailBuckets - 1 - tid;
        int32_t tb;
        const int32_t ex = block_excl_scan(tid < kTailBuckets ? hist[b] : 0, scan_buf, &tb);
        if (tid < kTailBuckets) bstart[b] = full_parts + ex;
        __syncthreads();
        if (tid < kTailBuckets) hist[tid] = 0;              // reused as fill counters
        __syncthreads();
    }
    // pass 2: positions
    int32_t carry_np = 0, carry_nf = 0;
    for (int32_t base = 0; base < p.num_seqs; base += blockDim.x) {
        const int32_t s = base + tid;
        int32_t np = 0, nf = 0, L = 0, tail = 0;
        if (s < p.num_seqs) {
            L = len_of(s);
            nf = L / P;
            tail = L - nf * P;
            np = nf + ((tail > 0 || L == 0) ? 1 : 0);
        }
        int32_t tp, tf;
        const int32_t slot0 = carry_np + block_excl_scan(np, scan_buf, &tp);
        const int32_t full0 = carry_nf + block_excl_scan(nf, scan_buf, &tf);
        if (s < p.num_seqs) {
            for (int32_t j = 0; j < nf; ++j) p.part_list[full0 + j] = make_int4(s, j, slot0, L);
            if (tail > 0 || L == 0) {
                const int32_t b = min((tail + bs - 1) / bs, kTailBuckets - 1);
                const int32_t pos = bstart[b] + atomicAdd(&hist[b], 1);
                p.part_list[pos] = make_int4(s, nf, slot0, L);
            }
        }
        carry_np += tp;
        carry_nf += tf;
    }
    const int32_t pairs = p.num_seqs * p.num_kv_heads * p.row_chunks * p.row_groups;
    for (int32_t i = tid; i < pairs; i += blockDim.x) p.arrive[i] = 0;
    if (tid == 0) {
        p.hdr->total_parts = (uint32_t)parts;
        p.hdr->total_units = (uint32_t)parts * (uint32_t)p.num_kv_heads * (uint32_t)p.row_chunks;
        p.hdr->partition_size = (uint32_t)P;
        p.hdr->counter = 0;
    }
}

// Moves every sequence to its next token on the device, between the steps of a
// multi-step decode loop ("[core] Multi Step Scheduling #7000": the advance_step op that
// updates seq_lens, slot_mapping and block_tables in place, with input tokens and
// positions).  The new token's block must already be in the table: the host reserves
// the loop's blocks up front.  A missing block leaves the slot at -1 (a padding token:
// reshape_and_cache then skips it) and flags PA_DEVERR_BAD_BLOCK.
__global__ void __launch_bounds__(256)
    advance_step_kernel(int32_t* __restrict__ context_lens, int32_t* __restrict__ slot_mapping,
                        const int32_t* __restrict__ block_tables, int32_t max_blocks_per_seq,
                        int32_t num_seqs, int32_t block_size, int32_t num_blocks,
                        int64_t* __restrict__ input_positions, int64_t* __restrict__ input_tokens,
                        const int64_t* __restrict__ sampled_token_ids, int32_t* status) {
    const int32_t s = blockIdx.x * blockDim.x + threadIdx.x;
    if (s >= num_seqs) return;
    const int32_t pos = context_lens[s];          // position of the sequence's next token
    context_lens[s] = pos + 1;
    if (input_positions) input_positions[s] = pos;
    if (input_tokens) input_tokens[s] = sampled_token_ids[s];
    const int32_t logical = pos / block_size;
    int32_t slot = -1;
    if (pos >= 0 && logical < max_blocks_per_seq) {
        const int32_t phys = block_tables[(size_t)s * max_blocks_per_seq + logical];
        if (phys >= 0 && phys < num_blocks) slot = phys * block_size + pos % block_size;
    }
    if (slot < 0 && status) atomicOr(status, 2 /* PA_DEVERR_BAD_BLOCK */);
    slot_mapping[s] = slot;
}

// Copy-on-write of shared blocks ("vLLM Project Update" talk: blocks shared between
// requests, prefix caching): for each (old, new) pair, block `new` of both pools takes
// the contents of block `old` -- every kv head and row, 16 bytes per thread-step.
// Pairs outside the pool are skipped and flagged PA_DEVERR_BAD_BLOCK.
__global__ void __launch_bounds__(256)
    copy_blocks_kernel(uint4* __restrict__ key_cache, uint4* __restrict__ value_cache,
                       const int32_t* __restrict__ pairs, int64_t vecs_per_block, int32_t num_blocks,
                       int32_t* status) {
    const int32_t i = blockIdx.x;
    const int32_t from = pairs[2 * i], to = pairs[2 * i + 1];
    if (from < 0 || from >= num_blocks || to < 0 || to >= num_blocks) {
        if (threadIdx.x == 0 && status) atomicOr(status, 2 /* PA_DEVERR_BAD_BLOCK */);
        return;
    }
    const uint4* ks = key_cache + (int64_t)from * vecs_per_block;
    const uint4* vs = value_cache + (int64_t)from * vecs_per_block;
    uint4* kd = key_cache + (int64_t)to * vecs_per_block;
    uint4* vd = value_cache + (int64_t)to * vecs_per_block;
    for (int64_t e = threadIdx.x + (int64_t)blockIdx.y * blockDim.x; e < vecs_per_block;
         e += (int64_t)gridDim.y * blockDim.x) {
        kd[e] = ks[e];
        vd[e] = vs[e];
    }
}

// Exercises the bounded pipeline wait: waits on a shared-memory barrier that nothing
// will ever arrive on, gives up after limit_ns, and reports PA_DEVERR_TIMEOUT exactly as
// the decode kernel does when a TMA completion never comes.
__global__ void __launch_bounds__(32) wait_timeout_probe_kernel(int32_t* status, uint64_t limit_ns) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_barrier_init();
    }
    __syncwarp();
    const bool ok = mbar_wait_for(&bar, 0, limit_ns);   // phase 0 never completes
    if (threadIdx.x == 0 && !ok && status) atomicOr(status, 8 /* PA_DEVERR_TIMEOUT */);
}

// Launches `kern` as a programmatic dependent of the kernel before it on `stream`: it may
// start while that kernel still runs and waits for it (griddepcontrol.wait) before it
// touches memory.
template <class... KArgs, class... Args>
cudaError_t launch_pdl(dim3 grid, dim3 block, cudaStream_t stream, void (*kern)(KArgs...),
                       Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

}  // namespace

cudaError_t launch_advance_step(int32_t* context_lens, int32_t* slot_mapping,
                                const int32_t* block_tables, int32_t max_blocks_per_seq,
                                int32_t num_seqs, int32_t block_size, int32_t num_blocks,
                                int64_t* input_positions, int64_t* input_tokens,
                                const int64_t* sampled_token_ids, int32_t* status,
                                cudaStream_t stream) {
    // An ordinary launch: it rewrites the lengths, which the plan kernel after it reads
    // before it waits for its predecessor, so it must have finished when that one starts.
    const int32_t threads = 256;
    advance_step_kernel<<<(num_seqs + threads - 1) / threads, threads, 0, stream>>>(
        context_lens, slot_mapping, block_tables, max_blocks_per_seq, num_seqs, block_size,
        num_blocks, input_positions, input_tokens, sampled_token_ids, status);
    return cudaGetLastError();
}

cudaError_t launch_copy_blocks(void* key_cache, void* value_cache, const int32_t* pairs,
                               int32_t num_pairs, int64_t bytes_per_block, int32_t num_blocks,
                               int32_t* status, cudaStream_t stream) {
    if (num_pairs <= 0) return cudaSuccess;
    const int64_t vecs = bytes_per_block / 16;
    const int32_t ys = (int32_t)std::min<int64_t>(8, (vecs + 255) / 256);
    copy_blocks_kernel<<<dim3(num_pairs, ys), 256, 0, stream>>>(
        static_cast<uint4*>(key_cache), static_cast<uint4*>(value_cache), pairs, vecs, num_blocks,
        status);
    return cudaGetLastError();
}

cudaError_t launch_wait_timeout_probe(int32_t* status, uint64_t limit_ns, cudaStream_t stream) {
    wait_timeout_probe_kernel<<<1, 32, 0, stream>>>(status, limit_ns);
    return cudaGetLastError();
}

cudaError_t launch_reshape_and_cache(const void* key, const void* value, void* key_cache,
                                     void* value_cache, const int32_t* slot_mapping,
                                     int32_t num_tokens, int32_t num_kv_heads,
                                     int32_t head_size, int32_t block_size, int32_t num_blocks,
                                     int32_t* status, cudaStream_t stream) {
    if (num_tokens <= 0) return cudaSuccess;
    return launch_pdl(dim3((unsigned)num_tokens), dim3(128), stream, reshape_and_cache_kernel,
                      static_cast<const uint4*>(key), static_cast<const uint4*>(value),
                      static_cast<uint4*>(key_cache), static_cast<uint4*>(value_cache),
                      slot_mapping, num_kv_heads, head_size, block_size, num_blocks, status);
}

cudaError_t launch_reshape_and_cache_fp8(const void* key, const void* value, void* key_cache,
                                         void* value_cache, const int32_t* slot_mapping,
                                         int32_t num_tokens, int32_t num_kv_heads,
                                         int32_t head_size, int32_t block_size, int32_t num_blocks,
                                         bool src_bf16, float k_inv_scale, float v_inv_scale,
                                         int32_t* status, cudaStream_t stream) {
    if (num_tokens <= 0) return cudaSuccess;
    auto kern = src_bf16 ? reshape_and_cache_fp8_kernel<true> : reshape_and_cache_fp8_kernel<false>;
    return launch_pdl(dim3((unsigned)num_tokens), dim3(128), stream, kern,
                      static_cast<const uint4*>(key), static_cast<const uint4*>(value),
                      static_cast<uint2*>(key_cache), static_cast<uint2*>(value_cache),
                      slot_mapping, num_kv_heads, head_size, block_size, num_blocks, k_inv_scale,
                      v_inv_scale, status);
}

cudaError_t launch_plan(const DecodeParams& p, cudaStream_t stream) {
    // Programmatic dependent launch: may start while a preceding reshape_and_cache or
    // decode kernel still runs; it reads the context lengths meanwhile and writes nothing
    // before that kernel has finished (see plan_kernel).
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1);
    // one thread per sequence, between kTailBuckets (the bucket scan takes one thread per
    // bucket) and 1024
#ifndef PA_PLAN_MIN_THREADS
#define PA_PLAN_MIN_THREADS kTailBuckets
#endif
    const int32_t want = (p.num_seqs + 31) / 32 * 32;
    cfg.blockDim = dim3((unsigned)std::min(1024, std::max((int32_t)PA_PLAN_MIN_THREADS, want)));
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, plan_kernel, p);
}

}  // namespace pa
