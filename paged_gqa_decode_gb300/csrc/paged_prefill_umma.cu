// Prefill on the tcgen05 tensor cores: head_dim 128 here, head_dim 64 in
// paged_prefill_umma_d64.cu.
#include "paged_prefill_umma.cuh"

namespace pgd {

// paged_prefill_umma_d64.cu
cudaError_t launch_prefill_umma_d64(const DecodeParams& p, const CUtensorMap& k_map,
                                    const CUtensorMap& v_map, const CUtensorMap& q_map,
                                    int sm_count, bool prepared, int parts, cudaStream_t stream);

cudaError_t launch_prefill_umma(const DecodeParams& p, const CUtensorMap& k_map,
                                const CUtensorMap& v_map, const CUtensorMap& q_map, int head_dim,
                                int sm_count, bool prepared, int parts, cudaStream_t stream) {
  return head_dim == 64
             ? launch_prefill_umma_d64(p, k_map, v_map, q_map, sm_count, prepared, parts, stream)
             : launch_prefill_umma<128, 4, 4>(p, k_map, v_map, q_map, sm_count, prepared, parts,
                                              stream);
}

cudaError_t launch_prefill_write(const DecodeParams& p, int head_dim, bool umma,
                                 cudaStream_t stream) {
  if (p.rows == 0) return cudaSuccess;
  using C = UmmaPrefillCfg<128, 4, 4>;  // the block geometry is the same at head_dim 64
  const int tokens = C::kTiles * (C::kRows / p.group);
  const int n_blocks = (p.rows + tokens - 1) / tokens;
  int* counter = umma ? reinterpret_cast<int*>(p.ws_acc) : nullptr;
  int* order = umma && p.window == 0 && n_blocks <= kMaxSortedBlocks ? counter + 4 : nullptr;
  const int write_ctas = (p.rows + 31) / 32 < 1024 ? (p.rows + 31) / 32 : 1024;  // a warp a token
  const dim3 grid(1 + write_ctas);
  return head_dim == 64
             ? launch_pdl(prefill_write_kernel<64>, grid, dim3(1024), 0, stream, p, tokens,
                          n_blocks, counter, order)
             : launch_pdl(prefill_write_kernel<128>, grid, dim3(1024), 0, stream, p, tokens,
                          n_blocks, counter, order);
}

int prefill_umma_launches(int rows, int group, int window, int parts) {
  if (rows <= 0) return 0;
  using C = UmmaPrefillCfg<128, 4, 4>;  // the block geometry is the same at head_dim 64
  const int tokens = C::kTiles * (C::kRows / group);
  const int n_blocks = (rows + tokens - 1) / tokens;
  return (window <= 0 && n_blocks <= kMaxSortedBlocks ? 2 : 1) + (parts > 1 ? 1 : 0);
}

}  // namespace pgd
