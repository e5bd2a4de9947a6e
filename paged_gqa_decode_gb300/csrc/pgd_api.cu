// Host side of the C ABI declared in include/pgd.h: argument validation,
// launch planning (pages per split), TMA descriptor encoding and launches.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "pgd.h"
#include "pgd_internal.h"

namespace pgd {

// The sticky device error word of each device that loads the library.
__device__ unsigned int g_device_error = 0;

namespace {

constexpr int kMaxDevices = 64;
constexpr int kPageSize = 64;
constexpr int kMinPagesPerSplit = 24;
constexpr int kMaxPagesPerSplit = 64;

struct DeviceInfo {
  std::once_flag once;
  cudaError_t status = cudaSuccess;
  int sm_count = 0;
  unsigned int* err = nullptr;  // device address of g_device_error
};
DeviceInfo g_devices[kMaxDevices];

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

int current_device(DeviceInfo** info) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PGD_ECUDA;
  DeviceInfo& d = g_devices[dev];
  std::call_once(d.once, [&] {
    d.status = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev);
    if (d.status == cudaSuccess)
      d.status = cudaGetSymbolAddress(reinterpret_cast<void**>(&d.err), g_device_error);
  });
  if (d.status != cudaSuccess) return PGD_ECUDA;
  *info = &d;
  return PGD_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_dims(const pgd_dims* d) {
  if (!d) return PGD_EINVAL;
  if (d->rows < 0 || d->num_q_heads <= 0 || d->num_kv_heads <= 0 || d->head_dim <= 0 ||
      d->num_pages <= 0 || d->max_pages_per_row <= 0)
    return PGD_EINVAL;
  if (d->num_q_heads % d->num_kv_heads != 0) return PGD_EINVAL;
  if (d->layout != PGD_PAGE_MAJOR && d->layout != PGD_HEAD_MAJOR && d->layout != PGD_ROW_MAJOR)
    return PGD_EINVAL;
  if (d->layout == PGD_ROW_MAJOR && d->num_pages % d->max_pages_per_row != 0) return PGD_EINVAL;
  if (d->page_size != kPageSize) return PGD_EUNSUPPORTED;
  if (d->head_dim != 64 && d->head_dim != 128) return PGD_EUNSUPPORTED;
  if (padded_group(d->num_q_heads / d->num_kv_heads) == 0) return PGD_EUNSUPPORTED;
  // Pool rows are addressed with 32-bit TMA coordinates; positions are int32.
  if ((int64_t)d->num_pages * d->num_kv_heads * kPageSize >= (int64_t)INT32_MAX)
    return PGD_EUNSUPPORTED;
  if ((int64_t)d->max_pages_per_row * kPageSize > (int64_t)INT32_MAX) return PGD_EUNSUPPORTED;
  return PGD_OK;
}

struct Plan {
  int pages_per_split;
  int max_splits;
};

// Key parts of the one-SM tcgen05 prefill (AUTO only) for a call of these
// dims: with at most half as many work items (blocks of 2 x 128 / group
// tokens, times the kv heads) as SMs, each item's pages are cut into parts,
// each a work unit of its own, so that the units fill the SMs.  At most 8,
// and at least 8 pages a part on the longest item the table allows (a
// window bounds it): parts of a few pages cost more in partials and the
// combine than they gain.  1: no parts.
constexpr int kMaxKeyParts = 8;
constexpr int kMinPartPages = 8;
int prefill_key_parts(const pgd_dims* d, int sm_count, int32_t window) {
  const int64_t block = 2 * (128 / (d->num_q_heads / d->num_kv_heads));
  const int64_t items = (d->rows + block - 1) / block * d->num_kv_heads;
  if (sm_count <= 0 || items <= 0 || items * 2 > sm_count) return 1;
  int64_t pages = d->max_pages_per_row;
  if (window > 0) {
    const int64_t span = ((int64_t)window + block - 2) / kPageSize + 2;  // window + block - 1 keys
    if (span < pages) pages = span;
  }
  int64_t parts = sm_count / items;
  if (parts > kMaxKeyParts) parts = kMaxKeyParts;
  if (parts > pages / kMinPartPages) parts = pages / kMinPartPages;
  return parts >= 2 ? (int)parts : 1;
}

// Pages per split: enough CTAs for several waves of 2 CTAs per SM when rows
// are about half full, but at least 24 pages (sweeps over 1..64 on GB300
// found every workload fastest at 24 or more: a split's fixed costs --
// setup, merge, partials and the combine -- outweigh the parallelism that
// shorter splits add) and at most 64.
Plan make_plan(const pgd_dims* d, const pgd_decode_options* opts, int sm_count) {
  Plan pl;
  int pps = opts ? opts->pages_per_split : 0;
  if (pps <= 0) {
    const int64_t target = 4ll * 2 * (sm_count > 0 ? sm_count : 1);
    const int64_t expected = (int64_t)d->rows * d->num_kv_heads *
                             (d->max_pages_per_row > 1 ? d->max_pages_per_row / 2 : 1);
    int64_t v = (expected + target - 1) / target;
    pps = (int)(v < kMinPagesPerSplit ? kMinPagesPerSplit
                                      : (v > kMaxPagesPerSplit ? kMaxPagesPerSplit : v));
  }
  if (pps > d->max_pages_per_row) pps = d->max_pages_per_row;
  pl.pages_per_split = pps;
  pl.max_splits = (d->max_pages_per_row + pps - 1) / pps;
  // the same workspace serves a prefill call of these dims: its key parts'
  // partials take one split's room each, beside the work counter
  const int parts = prefill_key_parts(d, sm_count, 0);  // the most any window allows
  if (parts > 1 && parts + 1 > pl.max_splits) pl.max_splits = parts + 1;
  return pl;
}

size_t workspace_bytes(const pgd_dims* d, const Plan& pl) {
  return (size_t)d->rows * d->num_q_heads * pl.max_splits * (d->head_dim + 2) * sizeof(float);
}

// The kernel a call runs: opts->kernel, or for AUTO the per-token split
// kernel, except that prefill with tokens in runs goes to a tcgen05 kernel:
// the one-SM kernel, with key parts (`key_parts` > 1) when its work items
// are at most half the SMs (`sm_count`; 0 = unknown) and long enough to
// cut, else for such calls at head_dim 128 the paired one, which puts two
// SMs on each item.  `window` bounds the items' length.
int resolve_kernel(const pgd_dims* dims, int32_t table_rows, bool prefill,
                   const pgd_decode_options* opts, int* kernel, int sm_count = 0,
                   int* key_parts = nullptr, int32_t window = 0) {
  int k = opts ? opts->kernel : PGD_KERNEL_AUTO;
  if (k < PGD_KERNEL_AUTO || k > PGD_KERNEL_PREFILL_PAIR) return PGD_EINVAL;
  if ((k == PGD_KERNEL_PREFILL_TILED || k == PGD_KERNEL_PREFILL_UMMA ||
       k == PGD_KERNEL_PREFILL_PAIR) &&
      !prefill)
    return PGD_EINVAL;
  if (k == PGD_KERNEL_PREFILL_PAIR && dims->head_dim != 128) return PGD_EINVAL;
  // Prefill: the tcgen05 kernel shares each page load among the tokens of a
  // block, which pays when they come in runs (prompt chunks); tokens that are
  // mostly one per table row (decode steps) go to the per-token split kernel.
  // Calls with at most half as many work items as SMs: key parts on one SM
  // per unit when the items are long enough to cut, else at head_dim 128 a
  // pair of SMs per item (measured on GB300: key parts 41-99 us against
  // 43-109 us for pairs on one Mistral-shaped chunk of 256-512 tokens; with
  // 128 items, pairs 102 us against 96-98 us for one SM per item).
  int parts = 1;
  if (prefill && k == PGD_KERNEL_AUTO && dims->rows >= 8ll * table_rows) {
    k = PGD_KERNEL_PREFILL_UMMA;
    const int group = dims->num_q_heads / dims->num_kv_heads;
    const int64_t block = 2 * (128 / group);  // tokens per work item
    const int64_t items = (dims->rows + block - 1) / block * dims->num_kv_heads;
    parts = prefill_key_parts(dims, sm_count, window);
    if (parts == 1 && dims->head_dim == 128 && sm_count > 0 && items * 2 <= sm_count)
      k = PGD_KERNEL_PREFILL_PAIR;
  }
  *kernel = k;
  if (key_parts) *key_parts = parts;
  return PGD_OK;
}

// AUTO decode with full attention over a table of a few pages runs the
// window kernel, the whole table its window (every row's rows copied at
// once, one warp per 32 positions, no splits), when the split size is the
// library's choice and the batch has between half as many and as many
// (row, kv head) units as SMs: one round of units, each on an SM of its own.
// Outside that range the split kernel measured faster (GB300, per step
// between L2 flushes: Qwen2.5 shapes, 64 rows (128 units) 12.4 against 13.0
// us with the window kernel, 4 rows (8 units) 10.8 against 10.3 us; 64
// dense gpt-oss rows of 640 positions (512 units) 35.3 against 24.3 us).
bool short_row_kernel(const pgd_dims* d, int32_t window, const pgd_decode_options* opts,
                      int kernel, int sm_count) {
  const int64_t units = (int64_t)d->rows * d->num_kv_heads;
  return kernel == PGD_KERNEL_AUTO && window <= 0 && !(opts && opts->pages_per_split > 0) &&
         sm_count > 0 && units * 2 >= sm_count && units <= sm_count &&
         short_row_tiles(d->head_dim, d->max_pages_per_row) > 0;
}

// Pages the split grid must cover per row: the table width, or with a
// window at most ceil((window - 1) / 64) + 1 pages.
int span_pages(const pgd_dims* dims, int32_t window) {
  int grid_pages = dims->max_pages_per_row;
  if (window > 0) {
    const int64_t wp = ((int64_t)window + kPageSize - 2) / kPageSize + 1;
    if (wp < grid_pages) grid_pages = (int)wp;
  }
  return grid_pages;
}

int encode_pool_map_uncached(CUtensorMap* map, const void* pool, const pgd_dims* d, int kind);

// Encoded pool descriptors are reused while the same pool is passed again: a
// small per-process cache keyed by (device, address, pages, kv heads, dim).
struct MapEntry {
  int dev;
  const void* pool;
  int32_t num_pages, kv_heads, head_dim;
  int kind;
  CUtensorMap map;
};
constexpr int kMapCache = 16;
MapEntry g_maps[kMapCache];
int g_map_count = 0, g_map_next = 0;
std::mutex g_map_mutex;

// Box shapes of a pool's tensor map.
enum MapKind {
  kMapBoxes = 0,      // 64 rows x 64 values: a page tile, or a 64-wide half of one
  kMapWholeTile = 1,  // head_dim 128: a page tile's two 64-wide boxes in one copy
};

int encode_pool_map(CUtensorMap* map, const void* pool, const pgd_dims* d,
                    int kind = kMapBoxes) {
  if (d->head_dim != 128) kind = kMapBoxes;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PGD_ECUDA;
  {
    std::lock_guard<std::mutex> lock(g_map_mutex);
    for (int i = 0; i < g_map_count; ++i) {
      const MapEntry& m = g_maps[i];
      if (m.dev == dev && m.pool == pool && m.num_pages == d->num_pages &&
          m.kv_heads == d->num_kv_heads && m.head_dim == d->head_dim && m.kind == kind) {
        *map = m.map;
        return PGD_OK;
      }
    }
  }
  const int rc = encode_pool_map_uncached(map, pool, d, kind);
  if (rc != PGD_OK) return rc;
  std::lock_guard<std::mutex> lock(g_map_mutex);
  MapEntry& slot = g_maps[g_map_next];
  slot = MapEntry{dev, pool, d->num_pages, d->num_kv_heads, d->head_dim, kind, *map};
  g_map_next = (g_map_next + 1) % kMapCache;
  if (g_map_count < kMapCache) ++g_map_count;
  return PGD_OK;
}

bool load_encode() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode != nullptr;
}

// q of a packed prefill, [tokens][Hq][D] bf16, as (64 values, heads,
// tokens) with boxes of 64 x group x (128 / group): one box is one half of a
// query tile's rows (token-major, head-minor), 128-byte swizzled -- the
// layout the tcgen05 prefill's S products read.  Tokens past the end read
// as zeros.
int encode_q_map(CUtensorMap* map, const void* q, const pgd_dims* d) {
  if (!load_encode()) return PGD_ECUDA;
  const int group = d->num_q_heads / d->num_kv_heads;
  const cuuint64_t dims3[3] = {(cuuint64_t)d->head_dim, (cuuint64_t)d->num_q_heads,
                               (cuuint64_t)d->rows};
  const cuuint64_t strides3[2] = {(cuuint64_t)d->head_dim * 2,
                                  (cuuint64_t)d->num_q_heads * d->head_dim * 2};
  const cuuint32_t box3[3] = {64, (cuuint32_t)group, (cuuint32_t)(128 / group)};
  const cuuint32_t elem3[3] = {1, 1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q), dims3,
                        strides3, box3, elem3, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? PGD_OK : PGD_ECUDA;
}

int encode_pool_map_uncached(CUtensorMap* map, const void* pool, const pgd_dims* d, int kind) {
  if (!load_encode()) return PGD_ECUDA;
  // The pool as a 2-D tensor: rows of head_dim bf16 values, one row per
  // (page, kv head, position) in either layout.  A box is 64 rows x 64
  // values (128 bytes): one page tile, or half of one when head_dim is 128.
  const cuuint64_t rows = (cuuint64_t)d->num_pages * d->num_kv_heads * kPageSize;
  if (kind != kMapBoxes) {
    // head_dim 128 as (64 values, rows, 2 halves): strides 256 bytes (a row)
    // and 128 bytes (a half), box 64 x 64 x 2 -- one copy lands a page tile as
    // the two consecutive 128-byte-swizzled 64-wide boxes the 2-D map gives.
    const cuuint64_t dims3[3] = {64, rows, 2};
    const cuuint64_t strides3[2] = {256, 128};
    const cuuint32_t box3[3] = {64, (cuuint32_t)kPageSize, 2};
    const cuuint32_t elem3[3] = {1, 1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(pool),
                          dims3, strides3, box3, elem3, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? PGD_OK : PGD_ECUDA;
  }
  const cuuint64_t dims[2] = {(cuuint64_t)d->head_dim, rows};
  const cuuint64_t strides[1] = {(cuuint64_t)d->head_dim * 2};
  const cuuint32_t box[2] = {64, (cuuint32_t)kPageSize};
  const cuuint32_t elem[2] = {1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(pool), dims,
                        strides, box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? PGD_OK : PGD_ECUDA;
}

}  // namespace

int padded_group(int group) {
  if (group == 1) return 1;
  if (group == 2) return 2;
  if (group >= 3 && group <= 4) return 4;
  if (group >= 5 && group <= 8) return 8;
  return 0;
}

}  // namespace pgd

using namespace pgd;

extern "C" {

static int append_impl(const pgd_dims* dims, const void* k_new, const void* v_new,
                       const int32_t* table, const int32_t* positions, const int32_t* slots,
                       void* k_pool, void* v_pool, pgd_stream_t stream) {
  int rc = check_dims(dims);
  if (rc != PGD_OK) return rc;
  if (dims->rows == 0) return PGD_OK;
  if (!k_new || !v_new || !k_pool || !v_pool) return PGD_EINVAL;
  if (slots == nullptr && (!positions || (!table && dims->layout != PGD_ROW_MAJOR)))
    return PGD_EINVAL;
  if (slots == nullptr && !table &&
      (int64_t)dims->rows * dims->max_pages_per_row > dims->num_pages)
    return PGD_EINVAL;  // dense rows: every row needs its own P pages
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_pool) || !aligned16(v_pool))
    return PGD_EINVAL;
  DeviceInfo* dev = nullptr;
  if ((rc = current_device(&dev)) != PGD_OK) return rc;
  AppendParams p;
  p.k_new = static_cast<const uint16_t*>(k_new);
  p.v_new = static_cast<const uint16_t*>(v_new);
  p.table = table;
  p.positions = positions;
  p.slots = slots;
  p.k_pool = static_cast<uint16_t*>(k_pool);
  p.v_pool = static_cast<uint16_t*>(v_pool);
  p.err = dev->err;
  p.rows = dims->rows;
  p.hkv = dims->num_kv_heads;
  p.head_dim = dims->head_dim;
  p.maxp = dims->max_pages_per_row;
  p.num_pages = dims->num_pages;
  p.layout = dims->layout;
  return launch_kv_append(p, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? PGD_OK
                                                                                     : PGD_ECUDA;
}

int pgd_kv_append_paged(const pgd_dims* dims, const void* k_new, const void* v_new,
                        const int32_t* table, const int32_t* positions, void* k_pool,
                        void* v_pool, pgd_stream_t stream) {
  return append_impl(dims, k_new, v_new, table, positions, nullptr, k_pool, v_pool, stream);
}

int pgd_rope_append_paged(const pgd_dims* dims, float theta, void* q, const void* k_new,
                          const void* v_new, const int32_t* table, const int32_t* positions,
                          const int32_t* slots, void* k_pool, void* v_pool, pgd_stream_t stream) {
  int rc = check_dims(dims);
  if (rc != PGD_OK) return rc;
  if (dims->rows == 0) return PGD_OK;
  if (!(theta > 0.f) || !std::isfinite(theta)) return PGD_EINVAL;
  if (!k_new || !v_new || !positions || !k_pool || !v_pool) return PGD_EINVAL;
  if (!slots && !table && dims->layout != PGD_ROW_MAJOR) return PGD_EINVAL;
  if (!slots && !table && (int64_t)dims->rows * dims->max_pages_per_row > dims->num_pages)
    return PGD_EINVAL;
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_pool) || !aligned16(v_pool) ||
      (q && !aligned16(q)))
    return PGD_EINVAL;
  DeviceInfo* dev = nullptr;
  if ((rc = current_device(&dev)) != PGD_OK) return rc;
  RopeAppendParams p;
  p.q = static_cast<uint16_t*>(q);
  p.k_new = static_cast<const uint16_t*>(k_new);
  p.v_new = static_cast<const uint16_t*>(v_new);
  p.table = table;
  p.positions = positions;
  p.slots = slots;
  p.k_pool = static_cast<uint16_t*>(k_pool);
  p.v_pool = static_cast<uint16_t*>(v_pool);
  p.err = dev->err;
  p.rows = dims->rows;
  p.hq = dims->num_q_heads;
  p.hkv = dims->num_kv_heads;
  p.head_dim = dims->head_dim;
  p.maxp = dims->max_pages_per_row;
  p.num_pages = dims->num_pages;
  p.layout = dims->layout;
  if (dims->head_dim / 2 > 64) return PGD_EUNSUPPORTED;
  // inv_freq[i] = exp(-(i * 2 / D) * log(theta)), in f32 as the tables are written
  const float log_theta = logf(theta);
  for (int i = 0; i < dims->head_dim / 2; ++i) {
    const float scaled = ((float)i * 2.0f) / (float)dims->head_dim;
    p.inv_freq[i] = expf(-scaled * log_theta);
  }
  return launch_rope_append(p, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? PGD_OK
             : PGD_ECUDA;
}

int pgd_page_slots(const pgd_dims* dims, int32_t table_rows, const int32_t* table,
                   const int32_t* rows, const int32_t* positions, int32_t* slots,
                   pgd_stream_t stream) {
  int rc = check_dims(dims);
  if (rc != PGD_OK) return rc;
  if (dims->rows == 0) return PGD_OK;
  if (!table || !positions || !slots) return PGD_EINVAL;
  if (rows != nullptr && table_rows <= 0) return PGD_EINVAL;
  if ((int64_t)dims->num_pages * kPageSize > (int64_t)INT32_MAX) return PGD_EUNSUPPORTED;
  DeviceInfo* dev = nullptr;
  if ((rc = current_device(&dev)) != PGD_OK) return rc;
  SlotParams p;
  p.table = table;
  p.row_of = rows;
  p.positions = positions;
  p.slots = slots;
  p.err = dev->err;
  p.tokens = dims->rows;
  p.table_rows = rows ? table_rows : dims->rows;
  p.maxp = dims->max_pages_per_row;
  p.num_pages = dims->num_pages;
  return launch_page_slots(p, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? PGD_OK
                                                                                     : PGD_ECUDA;
}

int pgd_kv_write_slots(const pgd_dims* dims, const void* k_new, const void* v_new,
                       const int32_t* slots, void* k_pool, void* v_pool, pgd_stream_t stream) {
  const int rc = check_dims(dims);
  if (rc != PGD_OK) return rc;
  if (dims->rows > 0 && !slots) return PGD_EINVAL;
  return append_impl(dims, k_new, v_new, nullptr, nullptr, slots, k_pool, v_pool, stream);
}

size_t pgd_paged_decode_workspace_bytes(const pgd_dims* dims, const pgd_decode_options* opts) {
  if (check_dims(dims) != PGD_OK) return 0;
  DeviceInfo* dev = nullptr;
  if (current_device(&dev) != PGD_OK) return 0;
  return workspace_bytes(dims, make_plan(dims, opts, dev->sm_count));
}

int pgd_attention_kernel_count(const pgd_dims* dims, int32_t table_rows, int32_t window,
                               const pgd_decode_options* opts, int32_t* count) {
  if (!count) return PGD_EINVAL;
  int rc = check_dims(dims);
  if (rc != PGD_OK) return rc;
  if (table_rows < 0) return PGD_EINVAL;
  // The arguments are checked before the device is; AUTO's prefill choice
  // then depends on the SM count, as the split size does.
  int kernel = 0;
  if ((rc = resolve_kernel(dims, table_rows, table_rows > 0, opts, &kernel)) != PGD_OK) return rc;
  DeviceInfo* dev = nullptr;
  if ((rc = current_device(&dev)) != PGD_OK) return rc;
  int parts = 1;
  if ((rc = resolve_kernel(dims, table_rows, table_rows > 0, opts, &kernel, dev->sm_count,
                           &parts, window)) != PGD_OK)
    return rc;
  const Plan pl = make_plan(dims, opts, dev->sm_count);
  if (dims->rows == 0) {
    *count = 0;
  } else if (kernel == PGD_KERNEL_PREFILL_UMMA || kernel == PGD_KERNEL_PREFILL_PAIR) {
    *count = prefill_umma_launches(dims->rows, dims->num_q_heads / dims->num_kv_heads, window,
                                   parts);
  } else if (kernel == PGD_KERNEL_PREFILL_TILED) {
    *count = 1;
  } else if ((kernel == PGD_KERNEL_AUTO && window > 0 && window <= kMaxWindowKernel) ||
             short_row_kernel(dims, window, opts, kernel, dev->sm_count)) {
    *count = 1;  // the window kernel
  } else {
    const int pages = span_pages(dims, window > 0 ? window : 0);
    *count = (pages + pl.pages_per_split - 1) / pl.pages_per_split > 1 ? 2 : 1;
  }
  return PGD_OK;
}

static int decode_impl(const pgd_dims* dims, int32_t table_rows, const int32_t* row_of,
                       const void* q, const void* k_pool, const void* v_pool,
                       const int32_t* table, const int32_t* positions, const float* sinks,
                       int32_t window, float scale, void* out, void* workspace,
                       size_t workspace_size, const pgd_decode_options* opts,
                       pgd_stream_t stream, const void* k_new = nullptr,
                       const void* v_new = nullptr) {
  int rc = check_dims(dims);
  if (rc != PGD_OK) return rc;
  if (dims->rows == 0) return PGD_OK;
  if (!q || !k_pool || !v_pool || !positions || !out) return PGD_EINVAL;
  if (!table && dims->layout != PGD_ROW_MAJOR) return PGD_EINVAL;
  if (row_of != nullptr && table_rows <= 0) return PGD_EINVAL;
  if (!table && (int64_t)(row_of ? table_rows : dims->rows) * dims->max_pages_per_row >
                    dims->num_pages)
    return PGD_EINVAL;  // dense rows: every row needs its own P pages
  if (!aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool) || !aligned16(out))
    return PGD_EINVAL;
  if ((k_new == nullptr) != (v_new == nullptr) ||
      (k_new && (!aligned16(k_new) || !aligned16(v_new))))
    return PGD_EINVAL;
  if (!std::isfinite(scale)) return PGD_EINVAL;
  DeviceInfo* dev = nullptr;
  if ((rc = current_device(&dev)) != PGD_OK) return rc;
  const Plan pl = make_plan(dims, opts, dev->sm_count);
  const size_t need = workspace_bytes(dims, pl);
  if (workspace_size < need) return PGD_EWORKSPACE;
  if (!workspace || !aligned16(workspace)) return PGD_EINVAL;

  int kernel = 0, parts = 1;
  if ((rc = resolve_kernel(dims, table_rows, row_of != nullptr, opts, &kernel, dev->sm_count,
                           &parts, window)) != PGD_OK)
    return rc;
  const int padded = padded_group(dims->num_q_heads / dims->num_kv_heads);
  // the tcgen05 prefills copy a head_dim-128 K page tile with one 3-D box;
  // each CTA of the paired prefill copies one 64-wide half of a V tile
  const bool tcgen05 = kernel == PGD_KERNEL_PREFILL_UMMA || kernel == PGD_KERNEL_PREFILL_PAIR;
  const int k_kind = tcgen05 ? kMapWholeTile : kMapBoxes;
  const int v_kind = kernel == PGD_KERNEL_PREFILL_UMMA ? kMapWholeTile : kMapBoxes;
  CUtensorMap k_map, v_map;
  if ((rc = encode_pool_map(&k_map, k_pool, dims, k_kind)) != PGD_OK) return rc;
  if ((rc = encode_pool_map(&v_map, v_pool, dims, v_kind)) != PGD_OK) return rc;

  DecodeParams p;
  p.q = static_cast<const uint16_t*>(q);
  p.table = table;
  p.positions = positions;
  p.row_of = row_of;
  p.table_rows = table_rows;
  p.sinks = sinks;
  p.out = static_cast<uint16_t*>(out);
  const size_t acc_floats =
      (size_t)dims->rows * dims->num_q_heads * pl.max_splits * dims->head_dim;
  p.ws_acc = static_cast<float*>(workspace);
  p.ws_ml = p.ws_acc + acc_floats;
  p.err = dev->err;
  p.rows = dims->rows;
  p.hq = dims->num_q_heads;
  p.hkv = dims->num_kv_heads;
  p.group = dims->num_q_heads / dims->num_kv_heads;
  p.maxp = dims->max_pages_per_row;
  p.num_pages = dims->num_pages;
  p.layout = dims->layout;
  p.window = window > 0 ? window : 0;
  p.pages_per_split = pl.pages_per_split;
  p.max_splits = pl.max_splits;
  p.q_scale_log2 = (float)((double)scale * 1.4426950408889634);
  p.k_new = static_cast<const uint16_t*>(k_new);
  p.v_new = static_cast<const uint16_t*>(v_new);
  p.k_pool = k_new ? static_cast<uint16_t*>(const_cast<void*>(k_pool)) : nullptr;
  p.v_pool = k_new ? static_cast<uint16_t*>(const_cast<void*>(v_pool)) : nullptr;
  p.k_read = static_cast<const uint16_t*>(k_pool);
  p.v_read = static_cast<const uint16_t*>(v_pool);

  const int grid_pages = span_pages(dims, p.window);
  const int grid_splits = (grid_pages + pl.pages_per_split - 1) / pl.pages_per_split;
  const int pages_per_cta = grid_pages < pl.pages_per_split ? grid_pages : pl.pages_per_split;
  const bool short_rows = short_row_kernel(dims, window, opts, kernel, dev->sm_count);

  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  // prefill step: the tokens' K and V are written by a launch of their own
  // first (a token's keys are read by the other tokens of its row), which
  // also prepares the tcgen05 kernel's work counter and block order
  const bool prefill_write = k_new != nullptr && row_of != nullptr;
  CUtensorMap q_map;
  if (tcgen05 && (rc = encode_q_map(&q_map, q, dims)) != PGD_OK) return rc;
  if (prefill_write) {
    if (launch_prefill_write(p, dims->head_dim, tcgen05, st) != cudaSuccess)
      return PGD_ECUDA;
    p.k_new = p.v_new = nullptr;
    p.k_pool = p.v_pool = nullptr;
  }
  if (kernel == PGD_KERNEL_PREFILL_PAIR)
    return launch_prefill_pair(p, k_map, v_map, q_map, dev->sm_count, prefill_write, st) ==
                   cudaSuccess
               ? PGD_OK
               : PGD_ECUDA;
  if (kernel == PGD_KERNEL_PREFILL_UMMA)
    return launch_prefill_umma(p, k_map, v_map, q_map, dims->head_dim, dev->sm_count,
                               prefill_write, parts, st) == cudaSuccess
               ? PGD_OK
               : PGD_ECUDA;
  if (kernel == PGD_KERNEL_PREFILL_TILED)
    return launch_prefill_tiled(p, k_map, v_map, dims->head_dim, padded, st) == cudaSuccess
               ? PGD_OK
               : PGD_ECUDA;
  cudaError_t e =
      dims->head_dim == 64
          ? launch_decode_d64(p, k_map, v_map, padded, kernel, grid_splits, pages_per_cta,
                              short_rows, st)
          : launch_decode_d128(p, k_map, v_map, padded, kernel, grid_splits, pages_per_cta,
                               short_rows, st);
  return e == cudaSuccess ? PGD_OK : PGD_ECUDA;
}

int pgd_paged_decode_attention(const pgd_dims* dims, const void* q, const void* k_pool,
                               const void* v_pool, const int32_t* table,
                               const int32_t* positions, const float* sinks, int32_t window,
                               float scale, void* out, void* workspace, size_t workspace_size,
                               const pgd_decode_options* opts, pgd_stream_t stream) {
  return decode_impl(dims, dims ? dims->rows : 0, nullptr, q, k_pool, v_pool, table, positions,
                     sinks, window, scale, out, workspace, workspace_size, opts, stream);
}

int pgd_paged_decode_step(const pgd_dims* dims, const void* q, const void* k_new,
                          const void* v_new, void* k_pool, void* v_pool, const int32_t* table,
                          const int32_t* positions, const float* sinks, int32_t window,
                          float scale, void* out, void* workspace, size_t workspace_size,
                          const pgd_decode_options* opts, pgd_stream_t stream) {
  const int rc = check_dims(dims);
  if (rc != PGD_OK) return rc;
  if (dims->rows > 0 && (!k_new || !v_new)) return PGD_EINVAL;
  return decode_impl(dims, dims->rows, nullptr, q, k_pool, v_pool, table, positions,
                     sinks, window, scale, out, workspace, workspace_size, opts, stream, k_new,
                     v_new);
}

int pgd_paged_prefill_attention(const pgd_dims* dims, int32_t table_rows, const void* q,
                                const void* k_pool, const void* v_pool, const int32_t* table,
                                const int32_t* rows, const int32_t* positions,
                                const float* sinks, int32_t window, float scale, void* out,
                                void* workspace, size_t workspace_size,
                                const pgd_decode_options* opts, pgd_stream_t stream) {
  const int rc = check_dims(dims);
  if (rc != PGD_OK) return rc;
  if (dims->rows > 0 && !rows) return PGD_EINVAL;
  return decode_impl(dims, table_rows, rows, q, k_pool, v_pool, table, positions, sinks, window,
                     scale, out, workspace, workspace_size, opts, stream);
}

int pgd_paged_prefill_step(const pgd_dims* dims, int32_t table_rows, const void* q,
                           const void* k_new, const void* v_new, void* k_pool, void* v_pool,
                           const int32_t* table, const int32_t* rows, const int32_t* positions,
                           const float* sinks, int32_t window, float scale, void* out,
                           void* workspace, size_t workspace_size,
                           const pgd_decode_options* opts, pgd_stream_t stream) {
  const int rc = check_dims(dims);
  if (rc != PGD_OK) return rc;
  if (dims->rows > 0 && (!rows || !k_new || !v_new)) return PGD_EINVAL;
  return decode_impl(dims, table_rows, rows, q, k_pool, v_pool, table, positions, sinks, window,
                     scale, out, workspace, workspace_size, opts, stream, k_new, v_new);
}

int pgd_prefill_step_kernel_count(const pgd_dims* dims, int32_t table_rows, int32_t window,
                                  const pgd_decode_options* opts, int32_t* count) {
  if (!count) return PGD_EINVAL;
  if (table_rows <= 0) return PGD_EINVAL;
  int32_t attention = 0;
  int rc = pgd_attention_kernel_count(dims, table_rows, window, opts, &attention);
  if (rc != PGD_OK) return rc;
  if (dims->rows == 0) {
    *count = 0;
    return PGD_OK;
  }
  DeviceInfo* dev = nullptr;
  if ((rc = current_device(&dev)) != PGD_OK) return rc;
  int kernel = 0, parts = 1;
  if ((rc = resolve_kernel(dims, table_rows, true, opts, &kernel, dev->sm_count, &parts,
                           window)) != PGD_OK)
    return rc;
  // the write launch, then the attention kernels (the tcgen05 kernel alone:
  // the write launch prepared its counter and order; then the combine when
  // there are key parts)
  *count = 1 + (kernel == PGD_KERNEL_PREFILL_UMMA || kernel == PGD_KERNEL_PREFILL_PAIR
                    ? 1 + (parts > 1 ? 1 : 0)
                    : attention);
  return PGD_OK;
}

int pgd_get_device_error(pgd_stream_t stream) {
  DeviceInfo* dev = nullptr;
  int rc = current_device(&dev);
  if (rc != PGD_OK) return rc;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return PGD_ECUDA;
  unsigned int word = 0;
  if (cudaMemcpyFromSymbol(&word, g_device_error, sizeof word) != cudaSuccess) return PGD_ECUDA;
  const unsigned int zero = 0;
  if (cudaMemcpyToSymbol(g_device_error, &zero, sizeof zero) != cudaSuccess) return PGD_ECUDA;
  return (int)word;
}

int pgd_selftest_bounded_wait(int32_t* outcome, pgd_stream_t stream) {
  if (!outcome) return PGD_EINVAL;
  DeviceInfo* dev = nullptr;
  const int rc = current_device(&dev);
  if (rc != PGD_OK) return rc;
  return launch_bounded_wait_selftest(dev->err, outcome, reinterpret_cast<cudaStream_t>(stream)) ==
                 cudaSuccess
             ? PGD_OK
             : PGD_ECUDA;
}

const char* pgd_status_string(int status) {
  switch (status) {
    case PGD_OK: return "ok";
    case PGD_EINVAL: return "invalid argument";
    case PGD_EUNSUPPORTED: return "unsupported shape";
    case PGD_ECUDA: return "CUDA error";
    case PGD_EDEVICE_BOUNDS: return "device: table entry or position out of range";
    case PGD_EDEVICE_TIMEOUT: return "device: pipeline wait timed out";
    case PGD_EWORKSPACE: return "workspace too small";
    case PGD_ESCRATCH_LIMIT: return "problem needs more than the library's static scratch";
    default: return "unknown status";
  }
}

int pgd_version(void) { return 200; }

}  // extern "C"

// ---------------------------------------------------------------------------
// Decode without caller-provided workspace, for callers that cannot allocate
// device memory.  The split partials live in this file-scope array (one per
// device that loads the library, held until exit); the host needs its device
// address, looked up once per device.

namespace pgd {
namespace {

static __device__ __align__(256) unsigned char g_static_scratch[PGD_STATIC_SCRATCH_BYTES];

struct StaticScratch {
  std::once_flag once;
  cudaError_t status = cudaSuccess;
  void* ptr = nullptr;
};
StaticScratch g_static[kMaxDevices];

}  // namespace
}  // namespace pgd

extern "C" int pgd_paged_decode_attention_static(const pgd_dims* dims, const void* q,
                                                 const void* k_pool, const void* v_pool,
                                                 const int32_t* table, const int32_t* positions,
                                                 const float* sinks, int32_t window, float scale,
                                                 void* out, const pgd_decode_options* opts,
                                                 pgd_stream_t stream) {
  int rc = check_dims(dims);
  if (rc != PGD_OK) return rc;
  if (dims->rows == 0) return PGD_OK;
  const size_t need = pgd_paged_decode_workspace_bytes(dims, opts);
  if (need == 0) return PGD_ECUDA;
  if (need > PGD_STATIC_SCRATCH_BYTES) return PGD_ESCRATCH_LIMIT;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PGD_ECUDA;
  StaticScratch& sc = g_static[dev];
  std::call_once(sc.once, [&] {
    sc.status = cudaGetSymbolAddress(&sc.ptr, g_static_scratch);
  });
  if (sc.status != cudaSuccess || sc.ptr == nullptr) return PGD_ECUDA;
  return pgd_paged_decode_attention(dims, q, k_pool, v_pool, table, positions, sinks, window,
                                    scale, out, sc.ptr, PGD_STATIC_SCRATCH_BYTES, opts, stream);
}
