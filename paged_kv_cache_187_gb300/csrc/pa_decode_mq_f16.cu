// Multi-query decode kernels (several causal query tokens per sequence), f16 queries and cache.
#include "pa_decode_family.cuh"

namespace pa {
cudaError_t launch_decode_mq_f16(const KernelKey& k, const CUtensorMap& kmap, const CUtensorMap& vmap,
                                const DecodeParams& p, bool persistent, int32_t num_units,
                                cudaStream_t stream, int32_t* occ) {
    return launch_mq_family<false>(k, kmap, vmap, p, persistent, num_units, stream, occ);
}
}  // namespace pa
