// Decode kernels for bf16 K/V with head_size 128.
#include "pa_decode_family.cuh"

namespace pa {
cudaError_t launch_decode_bf16_d128(const KernelKey& k, const CUtensorMap& kmap,
                                  const CUtensorMap& vmap, const DecodeParams& p,
                                  bool persistent, int32_t num_units, cudaStream_t stream,
                                  int32_t* occ) {
    return launch_family<128, true>(k, kmap, vmap, p, persistent, num_units, stream, occ);
}
}  // namespace pa
