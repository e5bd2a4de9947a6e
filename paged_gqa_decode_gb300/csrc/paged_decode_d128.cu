// Decode kernels for head_dim 128 (Mistral / Llama shapes).
#include "paged_decode.cuh"

namespace pgd {

cudaError_t launch_decode_d128(const DecodeParams& p, const CUtensorMap& k_map,
                               const CUtensorMap& v_map, int padded, int grid_splits,
                               cudaStream_t stream) {
  switch (padded) {
    case 1: return launch_decode<128, 1>(p, k_map, v_map, grid_splits, stream);
    case 2: return launch_decode<128, 2>(p, k_map, v_map, grid_splits, stream);
    case 4: return launch_decode<128, 4>(p, k_map, v_map, grid_splits, stream);
    case 8: return launch_decode<128, 8>(p, k_map, v_map, grid_splits, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace pgd
