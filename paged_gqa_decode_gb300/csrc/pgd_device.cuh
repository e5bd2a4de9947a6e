// Device-side building blocks for the sm_103a kernels: shared-memory
// mbarriers, TMA tile loads, bounded waits and the sticky error word.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "pgd.h"

namespace pgd {

constexpr int kPage = 64;  // positions per page

// Records `code` in the sticky device error word `err` (the first error
// wins); the host reads and clears it with pgd_get_device_error.
__device__ __forceinline__ void record_error(unsigned int* err, unsigned int code) {
  atomicCAS(err, 0u, code);
}

// A pipeline wait gives up after this long and reports PGD_EDEVICE_TIMEOUT.
constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void mbar_init_fence() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar))
               : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(
                   smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

// Whether the phase with the given parity has completed, without waiting
// (try_wait may suspend the thread for a while before it answers no).
__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

// Waits for the phase with the given parity to complete.  Returns false (and
// records PGD_EDEVICE_TIMEOUT) if it has not completed within kWaitLimitNs.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  unsigned int* err) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 255u) == 0u && global_ns() - t0 > kWaitLimitNs) {
      record_error(err, PGD_EDEVICE_TIMEOUT);
      return false;
    }
  }
}

// Waits until the shared word *seq equals `want` (written by another warp of
// the CTA).  Returns false (and records PGD_EDEVICE_TIMEOUT) after
// kWaitLimitNs.
__device__ __forceinline__ bool wait_seq_bounded(const volatile int* seq, int want,
                                                 unsigned int* err) {
  if (*seq == want) return true;
  const unsigned long long t0 = global_ns();
  for (uint32_t it = 1;; ++it) {
    __nanosleep(20);
    if (*seq == want) return true;
    if ((it & 255u) == 0u && global_ns() - t0 > kWaitLimitNs) {
      record_error(err, PGD_EDEVICE_TIMEOUT);
      return false;
    }
  }
}

// 2-D tiled TMA load of one box into shared memory, completing on `bar`.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int32_t x,
                                            int32_t y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar))
      : "memory");
}

// 3-D tiled TMA load of one box into shared memory, completing on `bar`.
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int32_t x,
                                            int32_t y, int32_t z, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_addr(bar))
      : "memory");
}

// Brings one box of a 3-D tensor into L2 (no shared memory, no completion).
__device__ __forceinline__ void tma_prefetch_l2_3d(const CUtensorMap* map, int32_t x, int32_t y,
                                                   int32_t z) {
  asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y), "r"(z)
               : "memory");
}

// Brings one box of a 2-D tensor into L2 (no shared memory, no completion).
__device__ __forceinline__ void tma_prefetch_l2_2d(const CUtensorMap* map, int32_t x, int32_t y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y)
               : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Programmatic dependent launch: every kernel of the library is launched
// allowed to start before its predecessor in the stream has finished, and
// calls pdl_wait() before it reads or writes anything another kernel may
// touch (its inputs can come from whatever kernel ran before it).  Without a
// programmatic dependency both are no-ops.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_allow_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Named barrier among the first `threads` threads of the CTA.
__device__ __forceinline__ void named_sync(uint32_t id, uint32_t threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// 2^x on the MUFU unit (flushes denormals; 2^-inf = +0).
__device__ __forceinline__ float exp2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// max(a, b, c) in one instruction.
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// The two bf16 halves of a 32-bit word, widened exactly to fp32.
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// First row of the (page, kv head) tile in the pool seen as a 2-D tensor of
// head_dim-wide rows (`maxp` is the pages per row of PGD_ROW_MAJOR).
__device__ __forceinline__ int64_t tile_first_row(int layout, int64_t page, int kvh, int hkv,
                                                  int num_pages, int maxp) {
  if (layout == PGD_PAGE_MAJOR) return (page * hkv + kvh) * kPage;
  if (layout == PGD_HEAD_MAJOR) return ((int64_t)kvh * num_pages + page) * kPage;
  return (((page / maxp) * hkv + kvh) * maxp + page % maxp) * kPage;  // PGD_ROW_MAJOR
}

// Pool page holding page index j of table row r; with no table (dense rows)
// row r's pages are r * maxp + j.
__device__ __forceinline__ int page_of(const int32_t* table, int r, int j, int maxp) {
  return table ? table[(size_t)r * maxp + j] : r * maxp + j;
}

// Row attention geometry shared by the decode and combine kernels.
struct RowSpan {
  int n;           // position of the new token (< 0: inactive)
  int lo;          // first attended position
  int first_page;  // page index (within the row) of lo
  int pages;       // attended pages
};

__device__ __forceinline__ RowSpan row_span(int n, int window) {
  RowSpan r;
  r.n = n;
  if (n < 0) {
    r.lo = 0;
    r.first_page = 0;
    r.pages = 0;
    return r;
  }
  r.lo = (window > 0 && n - window + 1 > 0) ? n - window + 1 : 0;
  r.first_page = r.lo / kPage;
  r.pages = n / kPage - r.first_page + 1;
  return r;
}

}  // namespace pgd
