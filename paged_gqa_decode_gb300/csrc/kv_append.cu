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
  pdl_wait();
  pdl_allow_dependents();
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

// rope_rows + append in one pass (Mistral 7B Instruct v0.3 model files,
// src/attention.linnet, decode_paged: rope_rows at positions[b] on q and k,
// then write_tokens; src/rope.linnet, tables).  The tables follow the pages'
// precision: inverse frequencies (precomputed once on the host) and angles
// in f32; cos/sin of the f32 angle evaluated in fp64 and rounded to f32,
// then to bf16, so every table entry is the correctly rounded one.
// Dimension i pairs with i + D/2; each rotated value is one fp32 rounding of
// the exact result (the products of bf16 values are exact in fp32), then
// rounded to bf16.  One CTA per row: q is rotated in place, k is rotated on
// its way into the pool, v is copied.
__global__ void __launch_bounds__(256) rope_append_kernel(const RopeAppendParams p) {
  pdl_wait();
  pdl_allow_dependents();
  const int b = blockIdx.x;
  const int n = p.positions[b];
  if (n < 0) return;  // inactive row: nothing rotated or written
  int page, in_page;
  if (p.slots) {
    const int slot = p.slots[b];
    if (slot < 0) return;
    if (slot / kPage >= p.num_pages) {
      if (threadIdx.x == 0) record_error(p.err, PGD_EDEVICE_BOUNDS);
      return;
    }
    page = slot / kPage;
    in_page = slot % kPage;
  } else {
    const int page_index = n / kPage;
    page = page_index < p.maxp ? page_of(p.table, b, page_index, p.maxp) : -1;
    if (page < 0 || page >= p.num_pages) {
      if (threadIdx.x == 0) record_error(p.err, PGD_EDEVICE_BOUNDS);
      return;
    }
    in_page = n % kPage;
  }
  const int half = p.head_dim / 2;
  __shared__ float cos_t[64], sin_t[64];
  if ((int)threadIdx.x < half) {
    const int i = threadIdx.x;
    const float angle = (float)n * p.inv_freq[i];
    cos_t[i] = __bfloat162float(__float2bfloat16_rn((float)cos((double)angle)));
    sin_t[i] = __bfloat162float(__float2bfloat16_rn((float)sin((double)angle)));
  }
  __syncthreads();
  const int heads = p.hkv + (p.q ? p.hq : 0);
  for (int e = threadIdx.x; e < heads * half; e += blockDim.x) {
    const int head = e / half, i = e % half;
    const bool is_k = head < p.hkv;
    const uint16_t* src = is_k ? p.k_new + ((size_t)b * p.hkv + head) * p.head_dim
                               : p.q + ((size_t)b * p.hq + head - p.hkv) * p.head_dim;
    const float x = __uint_as_float((uint32_t)src[i] << 16);
    const float y = __uint_as_float((uint32_t)src[i + half] << 16);
    const float c = cos_t[i], s = sin_t[i];
    const uint16_t o1 = __bfloat16_as_ushort(__float2bfloat16_rn(fmaf(x, c, -(y * s))));
    const uint16_t o2 = __bfloat16_as_ushort(__float2bfloat16_rn(fmaf(y, c, x * s)));
    uint16_t* dst;
    if (is_k) {
      const int64_t row0 = tile_first_row(p.layout, page, head, p.hkv, p.num_pages, p.maxp);
      dst = p.k_pool + ((size_t)row0 + in_page) * p.head_dim;
    } else {
      dst = p.q + ((size_t)b * p.hq + head - p.hkv) * p.head_dim;
    }
    dst[i] = o1;
    dst[i + half] = o2;
  }
  const int chunks = p.head_dim / 8;
  for (int c = threadIdx.x; c < p.hkv * chunks; c += blockDim.x) {
    const int h = c / chunks, ch = c % chunks;
    const int64_t row0 = tile_first_row(p.layout, page, h, p.hkv, p.num_pages, p.maxp);
    *reinterpret_cast<uint4*>(p.v_pool + ((size_t)row0 + in_page) * p.head_dim + ch * 8) =
        *reinterpret_cast<const uint4*>(p.v_new + ((size_t)b * p.hkv + h) * p.head_dim + ch * 8);
  }
}

cudaError_t launch_rope_append(const RopeAppendParams& p, cudaStream_t stream) {
  if (p.rows == 0) return cudaSuccess;
  return launch_pdl(rope_append_kernel, dim3(p.rows), dim3(256), 0, stream, p);
}

// page_slots for P tokens: one thread per token.
__global__ void __launch_bounds__(256) page_slots_kernel(const SlotParams p) {
  pdl_wait();
  pdl_allow_dependents();
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
  return launch_pdl(page_slots_kernel, dim3((p.tokens + 255) / 256), dim3(256), 0, stream, p);
}

cudaError_t launch_kv_append(const AppendParams& p, cudaStream_t stream) {
  if (p.rows == 0) return cudaSuccess;
  const int work = 2 * p.hkv * (p.head_dim / 8);
  int threads = work < 256 ? ((work + 31) / 32) * 32 : 256;
  return launch_pdl(kv_append_kernel, dim3(p.rows), dim3(threads), 0, stream, p);
}

}  // namespace pgd
