// Prefill on the tcgen05 tensor cores: the one-tile kernel at head_dim 128,
// the two-tile kernel (paged_prefill_umma_d64.cu) at head_dim 64.
#include "paged_prefill_umma.cuh"

namespace pgd {

// paged_prefill_umma_d64.cu
cudaError_t launch_prefill_umma_d64(const DecodeParams& p, const CUtensorMap& k_map,
                                    const CUtensorMap& v_map, int sm_count, cudaStream_t stream);

cudaError_t launch_prefill_umma(const DecodeParams& p, const CUtensorMap& k_map,
                                const CUtensorMap& v_map, int head_dim, int sm_count,
                                cudaStream_t stream) {
  return head_dim == 64 ? launch_prefill_umma_d64(p, k_map, v_map, sm_count, stream)
                        : launch_prefill_umma<128, 5, 5>(p, k_map, v_map, sm_count, stream);
}

}  // namespace pgd
