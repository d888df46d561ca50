// Multi-query decode kernels on tcgen05 (head_size 128): fp16 / bf16, 16- or 32-token
// blocks, 16 or 32 query rows per unit.
#include "pa_decode_tc.cuh"

namespace pa {
namespace {

template <bool BF16, int BS, int RPAD>
cudaError_t launch_tc(const CUtensorMap& kmap, const CUtensorMap& vmap, const DecodeParams& p,
                      bool persistent, int32_t num_units, cudaStream_t stream, int32_t* occ) {
    using C = tc::TcCfg<BF16, BS, RPAD>;
    constexpr size_t smem = tc::tc_smem_bytes<C>();
    static_assert(smem <= 227 * 1024, "shared memory");
    auto kern = tc::paged_decode_tc_kernel<C>;
    // the shared-memory limit is a per-device attribute: set once on each device
    static PerDeviceOnce configured;
    int dev = 0;
    cudaError_t e0 = cudaGetDevice(&dev);
    if (e0 != cudaSuccess) return e0;
    e0 = static_cast<cudaError_t>(configured.run(dev, [&] {
        // The warpgroups re-divide the registers each thread is launched with (setmaxnreg);
        // the division is written for REG_LAUNCH per thread and an increase that the
        // decreases do not cover would wait forever, so any other count is refused here.
        cudaFuncAttributes fa;
        cudaError_t e = cudaFuncGetAttributes(&fa, kern);
        if (e != cudaSuccess) return e;
        if (fa.numRegs != C::REG_LAUNCH) return cudaErrorInvalidKernelImage;
        return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    }));
    if (e0 != cudaSuccess) return e0;
    if (occ) {
        int n = 0;
        cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, C::THREADS, smem);
        *occ = (e == cudaSuccess) ? n : 0;
        return e;
    }
    if (num_units <= 0) return cudaSuccess;
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

}  // namespace

cudaError_t launch_decode_mq_tc(const KernelKey& k, const CUtensorMap& kmap, const CUtensorMap& vmap,
                                const DecodeParams& p, bool persistent, int32_t num_units,
                                cudaStream_t stream, int32_t* occ) {
#define PA_CASE(BF16_, BS_, R_)                                                              \
    if (k.bf16 == BF16_ && k.block_size == BS_ && k.heads_cap == R_)                         \
        return launch_tc<BF16_, BS_, R_>(kmap, vmap, p, persistent, num_units, stream, occ);
    PA_CASE(true, 16, 16)
    PA_CASE(true, 16, 32)
    PA_CASE(true, 32, 16)
    PA_CASE(true, 32, 32)
    PA_CASE(false, 16, 16)
    PA_CASE(false, 16, 32)
    PA_CASE(false, 32, 16)
    PA_CASE(false, 32, 32)
#undef PA_CASE
    return cudaErrorInvalidValue;
}

}  // namespace pa
