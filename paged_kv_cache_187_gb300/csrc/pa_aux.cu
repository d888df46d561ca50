// pa_aux.cu -- the small kernels around the decode kernel:
//   * reshape_and_cache: scatters each step's new K/V rows into the paged pools through
//     slot_mapping ("[core] Multi Step Scheduling #7000", the slot_mapping / block_tables
//     metadata a decode step carries);
//   * plan: lists the V2 partitions of every sequence and resets the work counter;
//   * reduce: merges the partitions of a sequence by log-sum-exp ("vLLM Project Update"
//     talk, the V2 kernel "similar to flash decoding").
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

// Single CTA: per-sequence partition counts, exclusive scan, the (sequence, partition)
// list, and the work counter reset.
__global__ void __launch_bounds__(1024) plan_kernel(const DecodeParams p) {
    __shared__ int32_t warp_sums[32];
    __shared__ int32_t carry_s;
    const int32_t tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int32_t P = p.partition_size;
    if (tid == 0) carry_s = 0;
    __syncthreads();
    for (int32_t base = 0; base < p.num_seqs; base += 1024) {
        const int32_t s = base + tid;
        int32_t np = 0;
        if (s < p.num_seqs) {
            const int32_t L = clamp_len(p, s, true);
            np = L > 0 ? (L + P - 1) / P : 1;      // an empty context is one empty unit
        }
        // block-wide exclusive scan of np
        int32_t x = np;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) warp_sums[warp] = x;
        __syncthreads();
        if (warp == 0) {
            int32_t w = warp_sums[lane];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int32_t y = __shfl_up_sync(0xffffffffu, w, o);
                if (lane >= o) w += y;
            }
            warp_sums[lane] = w;                   // inclusive over warps
        }
        __syncthreads();
        const int32_t carry = carry_s;
        const int32_t excl = carry + (warp > 0 ? warp_sums[warp - 1] : 0) + x - np;
        if (s < p.num_seqs) {
            p.part_offset[s] = excl;
            for (int32_t j = 0; j < np; ++j) p.part_list[excl + j] = make_int2(s, j);
        }
        __syncthreads();
        if (tid == 0) carry_s = carry + warp_sums[31];
        __syncthreads();
    }
    if (tid == 0) {
        const int32_t total = carry_s;
        p.part_offset[p.num_seqs] = total;
        p.hdr->total_parts = (uint32_t)total;
        p.hdr->total_units = (uint32_t)total * (uint32_t)p.num_kv_heads;
        p.hdr->counter = 0;
    }
}

// One CTA per (sequence, kv head) with more than one partition; a thread per
// (query head of the group, 4 head dims).  Partials hold unnormalised sums acc_p,
// the running max m_p (base-2 units) and the exp-sum l_p:
//   out = sum_p 2^(m_p - M) acc_p / sum_p 2^(m_p - M) l_p,   M = max_p m_p.
template <int D, bool BF16>
__global__ void __launch_bounds__(128) reduce_kernel(const DecodeParams p) {
    const int32_t s = blockIdx.x, kvh = blockIdx.y;
    const int32_t L = clamp_len(p, s, false);
    if (L <= p.partition_size) return;                      // written by the decode kernel
    const int32_t np = (L + p.partition_size - 1) / p.partition_size;
    const int32_t base = p.part_offset[s];
    const int32_t g = p.group;
    for (int32_t idx = threadIdx.x; idx < g * (D / 4); idx += blockDim.x) {
        const int32_t h = kvh * g + idx / (D / 4);
        const int32_t d = (idx % (D / 4)) * 4;
        float M = -INFINITY;
        for (int32_t j = 0; j < np; ++j)
            M = fmaxf(M, p.part_ml[(size_t)(base + j) * p.num_q_heads + h].x);
        float den = 0.f;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int32_t j = 0; j < np; ++j) {
            const float2 ml = p.part_ml[(size_t)(base + j) * p.num_q_heads + h];
            float w;
            asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(w) : "f"(ml.x - M));
            den += w * ml.y;
            const float4 a = *reinterpret_cast<const float4*>(
                p.part_acc + ((size_t)(base + j) * p.num_q_heads + h) * D + d);
            acc.x += w * a.x;
            acc.y += w * a.y;
            acc.z += w * a.z;
            acc.w += w * a.w;
        }
        const float inv = den > 0.f ? 1.f / den : 0.f;
        uint2 o;
        o.x = pack2<BF16>(acc.x * inv, acc.y * inv);
        o.y = pack2<BF16>(acc.z * inv, acc.w * inv);
        *reinterpret_cast<uint2*>(reinterpret_cast<uint16_t*>(p.out) +
                                  ((size_t)s * p.num_q_heads + h) * D + d) = o;
    }
}

}  // namespace

cudaError_t launch_reshape_and_cache(const void* key, const void* value, void* key_cache,
                                     void* value_cache, const int32_t* slot_mapping,
                                     int32_t num_tokens, int32_t num_kv_heads,
                                     int32_t head_size, int32_t block_size, int32_t num_blocks,
                                     int32_t* status, cudaStream_t stream) {
    if (num_tokens <= 0) return cudaSuccess;
    reshape_and_cache_kernel<<<num_tokens, 128, 0, stream>>>(
        static_cast<const uint4*>(key), static_cast<const uint4*>(value),
        static_cast<uint4*>(key_cache), static_cast<uint4*>(value_cache), slot_mapping,
        num_kv_heads, head_size, block_size, num_blocks, status);
    return cudaGetLastError();
}

cudaError_t launch_plan(const DecodeParams& p, cudaStream_t stream) {
    plan_kernel<<<1, 1024, 0, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_reduce(const DecodeParams& p, int32_t head_size, bool bf16,
                          cudaStream_t stream) {
    dim3 grid(p.num_seqs, p.num_kv_heads);
    if (p.num_seqs <= 0) return cudaSuccess;
    if (head_size == 128) {
        if (bf16) reduce_kernel<128, true><<<grid, 128, 0, stream>>>(p);
        else reduce_kernel<128, false><<<grid, 128, 0, stream>>>(p);
    } else {
        if (bf16) reduce_kernel<64, true><<<grid, 128, 0, stream>>>(p);
        else reduce_kernel<64, false><<<grid, 128, 0, stream>>>(p);
    }
    return cudaGetLastError();
}

}  // namespace pa
