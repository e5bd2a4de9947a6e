// Prefill on the tcgen05 tensor cores at head_dim 64 (its own translation
// unit, so the two head dims compile in parallel).
#include "paged_prefill_umma.cuh"

namespace pgd {

cudaError_t launch_prefill_umma_d64(const DecodeParams& p, const CUtensorMap& k_map,
                                    const CUtensorMap& v_map, const CUtensorMap& q_map,
                                    int sm_count, bool prepared, int parts, cudaStream_t stream) {
  return launch_prefill_umma<64, 8, 8>(p, k_map, v_map, q_map, sm_count, prepared, parts, stream);
}

}  // namespace pgd
