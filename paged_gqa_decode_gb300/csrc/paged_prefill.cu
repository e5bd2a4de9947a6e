// Tiled prefill kernels for head_dim 64 and 128.
#include "paged_prefill.cuh"

namespace pgd {

cudaError_t launch_prefill_tiled(const DecodeParams& p, const CUtensorMap& k_map,
                                 const CUtensorMap& v_map, int head_dim, int padded,
                                 cudaStream_t stream) {
  return head_dim == 64 ? launch_prefill_for_dim<64>(p, k_map, v_map, padded, stream)
                        : launch_prefill_for_dim<128>(p, k_map, v_map, padded, stream);
}

int prefill_block_tokens(int padded) { return 64 / padded; }

}  // namespace pgd
