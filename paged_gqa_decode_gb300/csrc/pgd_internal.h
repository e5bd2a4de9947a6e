// Launch parameters and launcher declarations shared by the host API
// (pgd_api.cu) and the kernel translation units.  Not part of the C ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "pgd.h"

namespace pgd {

// Launches `kernel` with programmatic stream serialization (see pdl_wait).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

struct AppendParams {
  const uint16_t* k_new;  // [R][Hkv][D] bf16
  const uint16_t* v_new;
  const int32_t* table;  // [R][maxp]
  const int32_t* positions;
  const int32_t* slots;  // prefill: explicit pool positions (table unused); else nullptr
  uint16_t* k_pool;
  uint16_t* v_pool;
  unsigned int* err;  // sticky device error word
  int rows, hkv, head_dim, maxp, num_pages, layout;
};

struct DecodeParams {
  const uint16_t* q;  // [R][Hq][D] bf16
  const int32_t* table;
  const int32_t* positions;
  const int32_t* row_of;  // prefill: table row of each token (nullptr: row b)
  int table_rows;         // rows of the table when row_of is given
  const float* sinks;  // [Hq] or nullptr
  uint16_t* out;       // [R][Hq][D] bf16
  float* ws_acc;       // [R][Hq][max_splits][D]
  float* ws_ml;        // [R][Hq][max_splits][2]: (m, l), m in log2 units
  unsigned int* err;
  int rows, hq, hkv, group, maxp, num_pages, layout, window;
  int pages_per_split;  // pages one split CTA streams
  int max_splits;       // split stride of the workspace
  float q_scale_log2;   // scale * log2(e): scores are kept in log2 units
  // decode step (append fused in): each row's new K/V [R][Hkv][D], written
  // into the pools at its slot by the split holding the row's last page
  // before that page is loaded; nullptr: no append
  const uint16_t* k_new;
  const uint16_t* v_new;
  uint16_t* k_pool;
  uint16_t* v_pool;
  // the pools for plain loads (the window kernel reads rows, not page tiles)
  const uint16_t* k_read;
  const uint16_t* v_read;
};

// With PGD_KERNEL_AUTO, decode windows of 1 .. kMaxWindowKernel positions go
// to the window kernel (a unit of warps per row and kv head, no splits).
constexpr int kMaxWindowKernel = 128;

// Tiles of the window kernel for full attention over a table of max_pages
// pages, its window the whole table: 64 positions a tile, TILES in {1, 2, 4}
// (and 10 at head_dim 64), so that a unit's rows fit its shared memory.
// 0: the table is too wide.
inline int short_row_tiles(int head_dim, int max_pages) {
  if (max_pages <= 1) return 1;
  if (max_pages <= 2) return 2;
  if (max_pages <= 4) return 4;
  if (head_dim == 64 && max_pages <= 10) return 10;
  return 0;
}

// Padded query-group sizes that have a decode kernel instantiation.
int padded_group(int group);  // 0 if unsupported

cudaError_t launch_kv_append(const AppendParams& p, cudaStream_t stream);

struct RopeAppendParams {
  uint16_t* q;  // [R][Hq][D] rotated in place, or nullptr
  const uint16_t* k_new;
  const uint16_t* v_new;
  const int32_t* table;
  const int32_t* positions;
  const int32_t* slots;  // explicit pool positions, or nullptr (table + positions)
  uint16_t* k_pool;
  uint16_t* v_pool;
  unsigned int* err;
  int rows, hq, hkv, head_dim, maxp, num_pages, layout;
  float inv_freq[64];  // theta^(-2i/D) for i < D/2, computed in f32 on the host
};
cudaError_t launch_rope_append(const RopeAppendParams& p, cudaStream_t stream);

struct SlotParams {
  const int32_t* table;
  const int32_t* row_of;  // nullptr: token p uses table row p
  const int32_t* positions;
  int32_t* slots;
  unsigned int* err;
  int tokens, table_rows, maxp, num_pages;
};
cudaError_t launch_page_slots(const SlotParams& p, cudaStream_t stream);
cudaError_t launch_bounded_wait_selftest(unsigned int* err, int* outcome, cudaStream_t stream);

// Decode kernels for one head_dim: the window kernel (AUTO, windows of at
// most kMaxWindowKernel positions; with `short_rows`, full attention over a
// table of short_row_tiles pages or fewer) or the split kernel + combine
// kernel; `padded` is the padded group size, `kernel` a PGD_KERNEL_* choice.
// `pages_per_cta` bounds the pages one split streams (it picks the ring depth).
cudaError_t launch_decode_d64(const DecodeParams& p, const CUtensorMap& k_map,
                              const CUtensorMap& v_map, int padded, int kernel, int grid_splits,
                              int pages_per_cta, bool short_rows, cudaStream_t stream);
cudaError_t launch_decode_d128(const DecodeParams& p, const CUtensorMap& k_map,
                               const CUtensorMap& v_map, int padded, int kernel, int grid_splits,
                               int pages_per_cta, bool short_rows, cudaStream_t stream);

// Tiled prefill (tokens of a block share each page load); no key splits.
cudaError_t launch_prefill_tiled(const DecodeParams& p, const CUtensorMap& k_map,
                                 const CUtensorMap& v_map, int head_dim, int padded,
                                 cudaStream_t stream);
int prefill_block_tokens(int padded);

// Prefill on the tcgen05 tensor cores: persistent, one CTA per SM, blocks of
// 2 x 128 / group tokens; the first word of p.ws_acc is its work counter, the
// block order (when one is computed) starts at the fifth.
// q_map: q as (64 values, heads, tokens) with boxes of 64 x group x
// (128 / group), 128-byte swizzle: the kernel copies each item's Q with it.
// `prepared`: launch_prefill_write (with umma) has already prepared the
// work counter and block order in p.ws_acc, so only the kernel is launched.
// `parts` > 1: each item's pages are cut into that many key parts (work
// units of their own) whose partials (at most p.max_splits - 1 a token and
// head fit the workspace) a combine launch then merges.
cudaError_t launch_prefill_umma(const DecodeParams& p, const CUtensorMap& k_map,
                                const CUtensorMap& v_map, const CUtensorMap& q_map, int head_dim,
                                int sm_count, bool prepared, int parts, cudaStream_t stream);
// Prefill at head_dim 128 on pairs of SMs (clusters of two CTAs sharing
// cta_group::2 tcgen05 products); the same work items, counter, block order
// and `prepared` convention as launch_prefill_umma.  k_map: the K pool in
// whole page tiles (3-D boxes); v_map: the V pool in 64 x 64 boxes.
cudaError_t launch_prefill_pair(const DecodeParams& p, const CUtensorMap& k_map,
                                const CUtensorMap& v_map, const CUtensorMap& q_map, int sm_count,
                                bool prepared, cudaStream_t stream);
// Kernels that launch issues for `rows` tokens (the block-order pass and the
// kernel, or the kernel alone; then the combine when there are key parts).
int prefill_umma_launches(int rows, int group, int window, int parts);
// The prefill step's write launch: each token's p.k_new / p.v_new at its slot
// in p.k_pool / p.v_pool (table row p.row_of[t], position p.positions[t]);
// with `umma`, its first CTA also prepares the tcgen05 kernel's work counter
// and block order in p.ws_acc.  One kernel launch.
cudaError_t launch_prefill_write(const DecodeParams& p, int head_dim, bool umma,
                                 cudaStream_t stream);

}  // namespace pgd
