// Prefill on pairs of SMs (cta_group::2 tcgen05 products), head_dim 128.
#include "paged_prefill_pair.cuh"

namespace pgd {

cudaError_t launch_prefill_pair(const DecodeParams& p, const CUtensorMap& k_map,
                                const CUtensorMap& v_map, const CUtensorMap& q_map, int sm_count,
                                bool prepared, cudaStream_t stream) {
  return launch_prefill_pair<4, 4, 3>(p, k_map, v_map, q_map, sm_count, prepared, stream);
}

}  // namespace pgd
