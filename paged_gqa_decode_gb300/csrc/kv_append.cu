// KV append: page_slots + write_tokens (Mistral 7B Instruct v0.3 model files,
// src/attention.linnet, GroupedQueryAttention.decode_paged).  Row b's new key
// and value go to position n % 64 of page table[b][n / 64], for every kv head;
// for prefill (prefill_paged in the same file) token b's go to the caller's
// pool position slots[b] instead.
// One CTA per row; each thread moves 16-byte chunks of the row's
// 2 x Hkv x D bf16 values.
#include "pgd_device.cuh"
#include "pgd_internal.h"

namespace pgd {

__global__ void __launch_bounds__(256) kv_append_kernel(const AppendParams p) {
  const int b = blockIdx.x;
  int page, in_page;
  if (p.slots) {  // explicit pool position (prefill's write at the caller's slots)
    const int slot = p.slots[b];
    if (slot < 0) return;  // padding token
    if (slot / kPage >= p.num_pages) {  // (maxp is only used by PGD_ROW_MAJOR)
      if (threadIdx.x == 0) record_error(p.err, PGD_EDEVICE_BOUNDS);
      return;
    }
    page = slot / kPage;
    in_page = slot % kPage;
  } else {
    const int n = p.positions[b];
    if (n < 0) return;  // inactive row
    const int page_index = n / kPage;
    if (page_index >= p.maxp) {
      if (threadIdx.x == 0) record_error(p.err, PGD_EDEVICE_BOUNDS);
      return;
    }
    page = page_of(p.table, b, page_index, p.maxp);
    if (page < 0 || page >= p.num_pages) {
      if (threadIdx.x == 0) record_error(p.err, PGD_EDEVICE_BOUNDS);
      return;
    }
    in_page = n % kPage;
  }
  const int chunks = p.head_dim / 8;  // 16-byte chunks per head
  const int per_tensor = p.hkv * chunks;
  for (int c = threadIdx.x; c < 2 * per_tensor; c += blockDim.x) {
    const int which = c / per_tensor;
    const int h = (c % per_tensor) / chunks;
    const int ch = c % chunks;
    const uint16_t* src = (which ? p.v_new : p.k_new) + ((size_t)b * p.hkv + h) * p.head_dim + ch * 8;
    const int64_t row0 = tile_first_row(p.layout, page, h, p.hkv, p.num_pages, p.maxp);
    uint16_t* dst = (which ? p.v_pool : p.k_pool) + ((size_t)row0 + in_page) * p.head_dim + ch * 8;
    *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(src);
  }
}

// page_slots for P tokens: one thread per token.
__global__ void __launch_bounds__(256) page_slots_kernel(const SlotParams p) {
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= p.tokens) return;
  const int n = p.positions[t];
  if (n < 0) {
    p.slots[t] = -1;
    return;
  }
  const int r = p.row_of ? p.row_of[t] : t;
  const int page_index = n / kPage;
  int slot = -1;
  if (r >= 0 && r < p.table_rows && page_index < p.maxp) {
    const int page = p.table[(size_t)r * p.maxp + page_index];
    if (page >= 0 && page < p.num_pages) slot = page * kPage + n % kPage;
  }
  if (slot < 0) record_error(p.err, PGD_EDEVICE_BOUNDS);
  p.slots[t] = slot;
}

cudaError_t launch_page_slots(const SlotParams& p, cudaStream_t stream) {
  if (p.tokens == 0) return cudaSuccess;
  page_slots_kernel<<<(p.tokens + 255) / 256, 256, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_kv_append(const AppendParams& p, cudaStream_t stream) {
  if (p.rows == 0) return cudaSuccess;
  const int work = 2 * p.hkv * (p.head_dim / 8);
  int threads = work < 256 ? ((work + 31) / 32) * 32 : 256;
  kv_append_kernel<<<p.rows, threads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace pgd
