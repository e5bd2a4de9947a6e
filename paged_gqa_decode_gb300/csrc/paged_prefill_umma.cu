// Prefill kernels on the tcgen05 tensor cores for head_dim 64 and 128.
#include "paged_prefill_umma.cuh"

namespace pgd {

cudaError_t launch_prefill_umma(const DecodeParams& p, const CUtensorMap& k_map,
                                const CUtensorMap& v_map, int head_dim, int sm_count,
                                cudaStream_t stream) {
  return head_dim == 64 ? launch_prefill_umma<64, 8, 8>(p, k_map, v_map, sm_count, stream)
                        : launch_prefill_umma<128, 5, 5>(p, k_map, v_map, sm_count, stream);
}

}  // namespace pgd
