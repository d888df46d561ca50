// Decode kernels for an fp8 E4M3 K/V cache (head_size 128) with fp16 or bf16 queries.
#include "pa_decode_family.cuh"

namespace pa {
cudaError_t launch_decode_fp8kv_f16q(const KernelKey& k, const CUtensorMap& kmap,
                                     const CUtensorMap& vmap, const DecodeParams& p,
                                     bool persistent, int32_t num_units, cudaStream_t stream,
                                     int32_t* occ) {
    return launch_family<128, false, true>(k, kmap, vmap, p, persistent, num_units, stream, occ);
}
cudaError_t launch_decode_fp8kv_bf16q(const KernelKey& k, const CUtensorMap& kmap,
                                      const CUtensorMap& vmap, const DecodeParams& p,
                                      bool persistent, int32_t num_units, cudaStream_t stream,
                                      int32_t* occ) {
    return launch_family<128, true, true>(k, kmap, vmap, p, persistent, num_units, stream, occ);
}
}  // namespace pa
