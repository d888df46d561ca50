// pa_decode_family.cuh -- instantiates the decode kernel for one (dtype, head_size)
// family and dispatches on block size and head capacity.  Each pa_decode_*.cu
// translation unit includes this once with PA_FAMILY_BF16 / PA_FAMILY_D defined, so
// the families compile in parallel.
#pragma once

#include "pa_decode.cuh"

// Tensor-core path: two consumer warps for 16-token blocks (short tiles, more of them);
// one for 32-token blocks, whose tiles already carry twice the work per wait.
#ifndef PA_MMA_CONSUMERS
#define PA_MMA_CONSUMERS(BS) ((BS) == 16 ? 2 : 1)
#endif
#ifndef PA_CORE_CONSUMERS
#define PA_CORE_CONSUMERS 2
#endif

namespace pa {

// Ring depth: about 48 KB of K+V stages per CTA, 2..8 stages, rounded up to a multiple
// of the consumer warps (see DecodeCfg).
template <int D, int BS, int NCONS>
constexpr int stages_for() {
    constexpr int per = 2 * D * BS * 2;
    constexpr int n0 = 49152 / per;
    constexpr int n = n0 < 2 ? 2 : (n0 > 8 ? 8 : n0);
    return ((n + NCONS - 1) / NCONS) * NCONS;
}

// Consumer warps per CTA: the CUDA-core path needs more warps to keep up with HBM than
// the tensor-core path does.
#ifndef PA_FP8_MMA_CONSUMERS
#define PA_FP8_MMA_CONSUMERS(BS) ((BS) == 16 ? 2 : 3)
#endif
#ifndef PA_FP8_CORE_CONSUMERS
#define PA_FP8_CORE_CONSUMERS 3
#endif


// Register budget.  The register file of an SM is four 16K-register quarters, one per
// scheduler, and a warp's registers come from one quarter: n CTAs of W warps leave a
// thread 16384 / (32 * ceil(n W / 4)) registers.  Left to itself (no minimum CTA count
// in the launch bounds) the compiler keeps the tensor-core decode kernels compact enough
// for the CTAs their shared memory admits (144 registers for the GQA and fp8 kernels); a
// minimum given explicitly makes it spend registers up to that bound.  Two kinds carry
// one, each measured faster:
//   * CUDA-core kernels with one head per unit (MHA): a minimum of 1 lets the compiler
//     keep more K / V rows in flight per lane (about 100 registers instead of 72), 1-3 %
//     on the MHA workloads; their shared memory still sets the CTAs per SM.  (With more
//     heads the same bound would cost those kernels a CTA.)
//   * 4-consumer multi-query kernels (5 warps): sized for the 2 CTAs their shared memory
//     admits (168 registers instead of the compiler's 128 with spills).
// Two-block tiles for 16-bit caches with 16-token blocks too (off: measured slower).
#ifndef PA_TILE2_16BIT
#define PA_TILE2_16BIT 0
#endif

#ifndef PA_CORE_MIN_CTAS
#define PA_CORE_MIN_CTAS 1
#endif
#ifndef PA_MQ_WIDE_MIN_CTAS
#define PA_MQ_WIDE_MIN_CTAS 2
#endif

template <class C0>
constexpr int decode_min_ctas() {
    constexpr int by_smem = (int)((228 * 1024) / (decode_smem_bytes<C0>() + 1024));
    if (!C0::kMma) return C0::HCAP == 1 ? PA_CORE_MIN_CTAS : 0;
    if (C0::kMq && C0::NCONS >= 4)
        return by_smem >= PA_MQ_WIDE_MIN_CTAS ? PA_MQ_WIDE_MIN_CTAS : 0;
    return 0;
}

// MQC: consumer warps of a multi-query kernel (kMqConsumersNarrow or kMqConsumersWide).
template <bool MMA, int BS, bool KV8, int MQC = 0>
constexpr int consumers_for() {
    // fp8 tiles carry twice the tokens per byte, so their consumers do more work per byte
    // than those of a 16-bit tile.  Measured on the Llama-3-8B / -70B batches, the
    // tensor-core path does best with 3 consumer warps for 32-token tiles (32-token
    // blocks, or two 16-token blocks; 2 and 4 were slower) and 2 for single 16-token
    // blocks (partitions that are not a multiple of 32 tokens); the CUDA-core path with 3.
    // BS here is the tile's token count.
    if (KV8) return MMA ? PA_FP8_MMA_CONSUMERS(BS) : PA_FP8_CORE_CONSUMERS;
    if (MQC) return MQC;
    return MMA ? PA_MMA_CONSUMERS(BS) : PA_CORE_CONSUMERS;
}

// BS: the pool's block size; TB: blocks per tile (a consumer step takes BS * TB tokens).
template <int D, int BS, bool BF16, bool MMA, int HCAP, bool KV8 = false, int MQC = 0, int TB = 1>
cudaError_t launch_one(const CUtensorMap& kmap, const CUtensorMap& vmap, const DecodeParams& p,
                       bool persistent, int32_t num_units, cudaStream_t stream,
                       int32_t* ctas_per_sm_out) {
    constexpr bool MQ = MQC > 0;
    constexpr int kTile = BS * TB;
    constexpr int kCons = consumers_for<MMA, kTile, KV8, MQC>();
    constexpr int kStages = stages_for<D * (KV8 ? 1 : 2) / 2, kTile, kCons>();
    using C0 = DecodeCfg<D, kTile, BF16, MMA, HCAP, kStages, 2, kCons, KV8, MQ, 0, BS>;
    using C = DecodeCfg<D, kTile, BF16, MMA, HCAP, kStages, 2, kCons, KV8, MQ,
                        decode_min_ctas<C0>(), BS>;
    constexpr size_t smem = decode_smem_bytes<C>();
    auto kern = paged_decode_kernel<C>;
    // the shared-memory limit is a per-device attribute: set once on each device
    static PerDeviceOnce configured;
    int dev = 0;
    cudaError_t e0 = cudaGetDevice(&dev);
    if (e0 != cudaSuccess) return e0;
    e0 = static_cast<cudaError_t>(configured.run(dev, [&] {
        return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    }));
    if (e0 != cudaSuccess) return e0;
    if (ctas_per_sm_out) {
        int n = 0;
        cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, C::THREADS, smem);
        *ctas_per_sm_out = (e == cudaSuccess) ? n : 0;
        return e;
    }
    if (num_units <= 0) return cudaSuccess;
    // Programmatic dependent launch: the CTAs may become resident and initialise while the
    // preceding plan / reshape kernel still runs; the kernel waits for it before reading.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)num_units);
    cfg.blockDim = dim3(C::THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, kmap, vmap, p, (int32_t)(persistent ? 1 : 0), num_units);
}

template <int D, bool BF16, bool KV8 = false>
cudaError_t launch_family(const KernelKey& k, const CUtensorMap& kmap, const CUtensorMap& vmap,
                          const DecodeParams& p, bool persistent, int32_t num_units,
                          cudaStream_t stream, int32_t* occ) {
    // fp8 caches with 16-token blocks take two blocks per tile: a consumer step then has
    // 32 tokens to amortise its softmax over, as with 32-token blocks
    if constexpr (KV8 || PA_TILE2_16BIT) {
        if (k.tile_blocks == 2) {
#define PA_CASE2(MMA_, H_)                                                                   \
    if (k.block_size == 16 && k.mma == MMA_ && k.heads_cap == H_)                            \
        return launch_one<D, 16, BF16, MMA_, H_, KV8, 0, 2>(kmap, vmap, p, persistent,       \
                                                           num_units, stream, occ);
            PA_CASE2(true, 8)
            PA_CASE2(true, 16)
            PA_CASE2(false, 1)
            PA_CASE2(false, 2)
            PA_CASE2(false, 4)
            PA_CASE2(false, 8)
#undef PA_CASE2
            return cudaErrorInvalidValue;
        }
    }
#define PA_CASE(BS_, MMA_, H_)                                                            \
    if (k.block_size == BS_ && k.mma == MMA_ && k.heads_cap == H_)                        \
        return launch_one<D, BS_, BF16, MMA_, H_, KV8>(kmap, vmap, p, persistent, num_units, \
                                                       stream, occ);
    PA_CASE(16, true, 8)
    PA_CASE(16, true, 16)
    PA_CASE(16, false, 1)
    PA_CASE(16, false, 2)
    PA_CASE(16, false, 4)
    PA_CASE(16, false, 8)
    PA_CASE(32, true, 8)
    PA_CASE(32, true, 16)
    PA_CASE(32, false, 1)
    PA_CASE(32, false, 2)
    PA_CASE(32, false, 4)
    PA_CASE(32, false, 8)
#undef PA_CASE
    return cudaErrorInvalidValue;
}

// Multi-query kernels of one dtype: both head sizes and block sizes, 8 rows per consumer,
// 2 or 4 consumer warps.
template <bool BF16>
cudaError_t launch_mq_family(const KernelKey& k, const CUtensorMap& kmap, const CUtensorMap& vmap,
                             const DecodeParams& p, bool persistent, int32_t num_units,
                             cudaStream_t stream, int32_t* occ) {
#define PA_CASE(D_, BS_, NC_)                                                                 \
    if (k.head_size == D_ && k.block_size == BS_ && k.heads_cap == kMqRowsPerConsumer &&      \
        k.mq_consumers == NC_)                                                                \
        return launch_one<D_, BS_, BF16, true, kMqRowsPerConsumer, false, NC_>(               \
            kmap, vmap, p, persistent, num_units, stream, occ);
    PA_CASE(128, 16, kMqConsumersNarrow)
    PA_CASE(128, 32, kMqConsumersNarrow)
    PA_CASE(64, 16, kMqConsumersNarrow)
    PA_CASE(64, 32, kMqConsumersNarrow)
    PA_CASE(128, 16, kMqConsumersWide)
    PA_CASE(128, 32, kMqConsumersWide)
    PA_CASE(64, 16, kMqConsumersWide)
    PA_CASE(64, 32, kMqConsumersWide)
#undef PA_CASE
    return cudaErrorInvalidValue;
}

}  // namespace pa
