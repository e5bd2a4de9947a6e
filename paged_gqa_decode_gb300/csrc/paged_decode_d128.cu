// Decode kernels for head_dim 128 (Mistral / Llama shapes).
#include "paged_decode.cuh"

namespace pgd {

cudaError_t launch_decode_d128(const DecodeParams& p, const CUtensorMap& k_map,
                              const CUtensorMap& v_map, int padded, int kernel, int grid_splits,
                              int pages_per_cta, bool short_rows, cudaStream_t stream) {
  return launch_decode_for_dim<128>(p, k_map, v_map, padded, kernel, grid_splits, pages_per_cta,
                                    short_rows, stream);
}

}  // namespace pgd
