// pa_decode_family.cuh -- instantiates the decode kernel for one (dtype, head_size)
// family and dispatches on block size and head capacity.  Each pa_decode_*.cu
// translation unit includes this once with PA_FAMILY_BF16 / PA_FAMILY_D defined, so
// the families compile in parallel.
#pragma once

#include "pa_decode.cuh"

namespace pa {

// Ring depth: about 48 KB of K+V stages per CTA, 2..8 stages.
template <int D, int BS>
constexpr int stages_for() {
    constexpr int per = 2 * D * BS * 2;
    constexpr int n = 49152 / per;
    return n < 2 ? 2 : (n > 8 ? 8 : n);
}

template <int D, int BS, bool BF16, bool MMA, int HCAP>
cudaError_t launch_one(const CUtensorMap& kmap, const CUtensorMap& vmap, const DecodeParams& p,
                       bool persistent, int32_t num_units, cudaStream_t stream,
                       int32_t* ctas_per_sm_out) {
    using C = DecodeCfg<D, BS, BF16, MMA, HCAP, stages_for<D, BS>(), 2>;
    constexpr size_t smem = decode_smem_bytes<C>();
    auto kern = paged_decode_kernel<C>;
    static bool configured = false;   // per instantiation; attribute setting is idempotent
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    if (ctas_per_sm_out) {
        int n = 0;
        cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, C::THREADS, smem);
        *ctas_per_sm_out = (e == cudaSuccess) ? n : 0;
        return e;
    }
    if (num_units <= 0) return cudaSuccess;
    kern<<<num_units, C::THREADS, smem, stream>>>(kmap, vmap, p, persistent ? 1 : 0, num_units);
    return cudaGetLastError();
}

template <int D, bool BF16>
cudaError_t launch_family(const KernelKey& k, const CUtensorMap& kmap, const CUtensorMap& vmap,
                          const DecodeParams& p, bool persistent, int32_t num_units,
                          cudaStream_t stream, int32_t* occ) {
#define PA_CASE(BS_, MMA_, H_)                                                            \
    if (k.block_size == BS_ && k.mma == MMA_ && k.heads_cap == H_)                        \
        return launch_one<D, BS_, BF16, MMA_, H_>(kmap, vmap, p, persistent, num_units,   \
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

}  // namespace pa
