// KV append: page_slots + write_tokens (Mistral 7B Instruct v0.3 model files,
// src/attention.linnet, GroupedQueryAttention.decode_paged).  Row b's new key
// and value go to position n % 64 of page table[b][n / 64], for every kv head.
// One CTA per row; each thread moves 16-byte chunks of the row's
// 2 x Hkv x D bf16 values.
#include "pgd_device.cuh"
#include "pgd_internal.h"

namespace pgd {

__global__ void __launch_bounds__(256) kv_append_kernel(const AppendParams p) {
  const int b = blockIdx.x;
  const int n = p.positions[b];
  if (n < 0) return;  // inactive row
  const int page_index = n / kPage;
  if (page_index >= p.maxp) {
    if (threadIdx.x == 0) record_error(p.err, PGD_EDEVICE_BOUNDS);
    return;
  }
  const int page = p.table[(size_t)b * p.maxp + page_index];
  if (page < 0 || page >= p.num_pages) {
    if (threadIdx.x == 0) record_error(p.err, PGD_EDEVICE_BOUNDS);
    return;
  }
  const int in_page = n % kPage;
  const int chunks = p.head_dim / 8;  // 16-byte chunks per head
  const int per_tensor = p.hkv * chunks;
  for (int c = threadIdx.x; c < 2 * per_tensor; c += blockDim.x) {
    const int which = c / per_tensor;
    const int h = (c % per_tensor) / chunks;
    const int ch = c % chunks;
    const uint16_t* src = (which ? p.v_new : p.k_new) + ((size_t)b * p.hkv + h) * p.head_dim + ch * 8;
    const size_t tile = p.layout == PGD_PAGE_MAJOR ? (size_t)page * p.hkv + h
                                                   : (size_t)h * p.num_pages + page;
    uint16_t* dst = (which ? p.v_pool : p.k_pool) + (tile * kPage + in_page) * p.head_dim + ch * 8;
    *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(src);
  }
}

cudaError_t launch_kv_append(const AppendParams& p, cudaStream_t stream) {
  if (p.rows == 0) return cudaSuccess;
  const int work = 2 * p.hkv * (p.head_dim / 8);
  int threads = work < 256 ? ((work + 31) / 32) * 32 : 256;
  kv_append_kernel<<<p.rows, threads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace pgd
