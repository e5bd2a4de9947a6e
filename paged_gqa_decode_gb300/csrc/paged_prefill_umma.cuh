// Paged prefill attention on the 5th-generation tensor cores (tcgen05 UMMA
// with TMEM accumulators), sm_103a: a persistent kernel with two query tiles
// per work item.
//
// What it computes is the same as the tiled prefill kernel (Mistral 7B
// Instruct v0.3 model files, src/attention.linnet, prefill_paged; window and
// sinks as GPT-OSS 20B src/attention.linnet, prefill_packed): packed token p at
// position positions[p] of table row rows[p] attends, with each query head of
// its group, over that row's keys at positions (positions[p] - window,
// positions[p]], the head's sink logit in the denominator only.
//
// Work items are (block of 2 x 128 / G consecutive packed tokens, kv head):
// two query tiles of 128 rows, tile t holding tokens t * 128 / G ..
// (t + 1) * 128 / G - 1 of the block, row m = token * G + head, one per TMEM
// lane.  Both tiles share every K and V page the item loads (half the page
// traffic of one tile per item).  One CTA per SM takes items from a counter,
// longest first (without a window a one-CTA pass before the kernel sorts the
// token blocks by the key span of their first and last tokens; with one the
// spans are bounded by it and blocks go in token order, last first).  Within an item the
// tokens split into runs (same table row, consecutive positions); each run
// is one pass over the pages of the union of its tokens' key ranges.  The
// pages of all of a CTA's items form one sequence, and every role walks it:
//   warp 16     K producer: per item, reads its tokens, builds the runs,
//               checks the table and zeroes uncovered outputs (whole warp);
//               then streams each page's K tile (64 x D bf16, 128-byte
//               swizzle) into a ring of shared slots with TMA, pulling pages
//               into L2 ahead of their loads.
//   warp 19     V producer: the same pages' V tiles into a second ring.
//   warp 17     S issuer (one thread) and TMEM owner.  Per item it copies
//               the item's Q rows into shared memory with TMA (q as 64
//               values x heads x tokens, boxes of 64 x G x 128 / G: half a
//               tile's rows, token-major, in the swizzled K-major layout the
//               products read) once the previous item's S products are done;
//               then per page i and tile t:
//                 S_t  = Q_t K_i^T    M 128, N 64, K D   (Q and K shared)
//               into tile t's S buffer i % 2 once P_t V_{i-2} (which reads
//               the same columns) is done.
//   warp 18     P V issuer (one thread), per page i and tile t:
//                 O_t += P_t V_i      M 128, N D,  K 64  (P from TMEM, V shared)
//   warps 0-15  softmax: tile t has two warpgroups (warps 4t .. 4t + 3 and
//               8 + 4t .. 11 + 4t), one thread per query row in each; the
//               first takes keys 0-31 of every page, the second keys 32-63
//               (and half of the O columns each for the rescale and the
//               store).  Per page its scores from TMEM, causal and window
//               mask, its half's max, the row's max over the page through
//               shared memory at the tile's named barrier (which also ORs
//               the threads' failed-wait flags, so the two warpgroups stop
//               together after a timeout), online softmax in
//               log2 units with a lazy running max (raised only when a score
//               exceeds it by more than 2^8, which then rescales that row of
//               O_t in TMEM); P is written over S as a bf16 head and residual
//               (two MMAs, so P V keeps fp32 accuracy).  At the end of a run
//               the halves add their row sums and normalise and store their
//               halves of the O_t row with the sink.  Warpgroup 0 also
//               zeroes the V rows outside the run's key range on boundary
//               pages before the products read them.
// TMEM (512 columns): O_t at [t D, (t + 1) D), then two S / P buffers per
// tile, 64 columns each (S of the next page is computed while the softmax
// works on this one; P per chunk of 32 keys: the bf16 head in the chunk's
// first 16 columns, the residual in the next 16, as packed pairs).  At
// head_dim 128 that is all 512 columns.
// Key parts (a separate build, for calls with few items): each item's runs
// are cut into `parts` consecutive page ranges, one work unit each; a unit
// ends each run by writing the row's partial -- lazy maximum, row sum and
// the O row, unnormalised, fp32 -- to the workspace, and a combine launch
// merges the parts with the sink (the split softmax, as the decode combine).
// Every wait is bounded; a timeout records PGD_EDEVICE_TIMEOUT, stops all
// roles, drains in-flight copies and MMAs and frees TMEM before the CTA exits.
#pragma once

#include "paged_decode.cuh"
#include "pgd_umma.cuh"

namespace pgd {

template <int D, int RK, int RV>
struct UmmaPrefillCfg {
  static constexpr int kRows = 128;  // query rows per tile (TMEM lanes)
  static constexpr int kTiles = 2;   // query tiles per item
  // two warpgroups per tile, each taking half of every page's keys
  static constexpr int kSoftmaxThreads = 512;
  static constexpr int kProducerWarp = 16;
  static constexpr int kMmaWarp = 17;  // S issuer, TMEM owner
  static constexpr int kPvWarp = 18;
  static constexpr int kVWarp = 19;
  static constexpr int kThreads = 640;
  static constexpr int kBoxes = D / 64;
  static constexpr int kTileBytes = kPage * D * 2;  // one K or V slot (one page)
  static constexpr int kVOff = RK * kTileBytes;
  // Q sits in shared memory (K-major, 128-byte swizzle: the layout the MMA
  // reads), copied in per item by the S issuer with TMA; at head_dim 128 the
  // two O accumulators and the S buffers take all 512 TMEM columns
  static constexpr int kQBoxes = D / 64;  // 64-value boxes of a Q row
  static constexpr int kQOff = (RK + RV) * kTileBytes;
  static constexpr int kQBoxBytes = kRows * 128;  // 128 rows x 64 values
  static constexpr int kQTileBytes = kRows * D * 2;
  static constexpr int kBarOff = kQOff + kTiles * kQTileBytes;
  // S / P buffers per tile: two where TMEM has room (head_dim 64), so S of
  // the next page is computed while the softmax works on this one
  static constexpr int kSBufs = 2;
  static constexpr int kNumBars = 2 * RK + 2 * RV + 3 * kTiles * kSBufs + 6 + 2;
  static constexpr int kSmemBytes = 1024 + kBarOff + kNumBars * 8;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kOCol = 0, kSCol = kTiles * D;
  static constexpr uint32_t kIdescS = umma_idesc_bf16(128, kPage, 0, 0);
  static constexpr uint32_t kIdescPV = umma_idesc_bf16(128, D, 0, 1);
  static_assert(D == 64 || D == 128, "head_dim");
  static_assert(kSCol + kTiles * kSBufs * kPage <= kTmemCols, "TMEM columns");
  static_assert(RK == RV, "the K and V rings are streamed by one helper");
  static_assert(kSBufs <= RV, "a V slot is freed when S of the page kSBufs later is issued");
  static_assert(kSmemBytes + 20 * 1024 <= 227 * 1024, "shared memory (dynamic + static)");
};

// Slack of the lazy running max, in log2 units: P values stay below 2^8.
constexpr float kLazyRescaleLog2 = 8.0f;

// How far ahead of its load the producer pulls a page into L2.
constexpr int kL2PrefetchPages = 16;

// mbarrier wait that also gives up when another role of the CTA has set
// *abort (after its own wait timed out).
__device__ __forceinline__ bool mbar_wait_abortable(uint64_t* bar, uint32_t parity,
                                                    unsigned int* err, volatile int* abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 0u) {
      if (*abort) return false;
      if (global_ns() - t0 > kWaitLimitNs) {
        record_error(err, PGD_EDEVICE_TIMEOUT);
        *abort = 1;
        return false;
      }
    }
  }
}

// Named barrier `id` among `count` threads that also ORs `pred` over them:
// every participating thread gets the same answer.
__device__ __forceinline__ bool named_sync_or(uint32_t id, uint32_t count, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, %2, %3, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)pred), "r"(id), "r"(count)
      : "memory");
  return r != 0;
}

// One work item as the producer laid it out for the other roles.
struct PrefillItem {
  int valid;  // 0: no more items
  int t_begin, t_end, kvh, runs;
  // key part `part` of `parts`: each run's pages are cut into `parts`
  // consecutive ranges and this unit takes range `part` (parts 1: all),
  // pages run_pg[r] .. run_last[r] of run r (written for key-part kernels)
  int part, parts;
  int run_end[257];
  int tok_row[256], tok_pos[256], run_bad[256];
  int run_pg[256], run_last[256];
};

// Page sequence of one item: run by run (inactive and bad runs skipped),
// pages first..last of each.
struct ItemCursor {
  int r, pg, last, row, rs, re;
};

// The item's key part of a run's pages first..last (in place): range `part`
// of `parts` near-equal consecutive ranges; false when it is empty.
__device__ __forceinline__ bool part_pages(const PrefillItem& it, int& first, int& last) {
  const int64_t n = last - first + 1;
  const int lo = first + (int)(n * it.part / it.parts);
  const int hi = first + (int)(n * (it.part + 1) / it.parts) - 1;
  first = lo;
  last = hi;
  return lo <= hi;
}

// kParts: the item is one key part of its pages (kernels built for key
// parts: each run's range as the producer wrote it in the descriptor);
// otherwise every page of every run.
template <bool kParts = false>
__device__ __forceinline__ bool item_next_run(const PrefillItem& it, int window, ItemCursor& c) {
  for (++c.r; c.r < it.runs; ++c.r) {
    c.rs = c.r == 0 ? 0 : it.run_end[c.r - 1];
    c.re = it.run_end[c.r];
    c.row = it.tok_row[c.rs];
    if (c.row < 0 || it.run_bad[c.r]) continue;
    if constexpr (kParts) {
      c.pg = it.run_pg[c.r];
      c.last = it.run_last[c.r];
      if (c.pg > c.last) continue;  // no page of this run in the part
    } else {
      const int lo = window > 0 ? max(it.tok_pos[c.rs] - window + 1, 0) : 0;
      c.pg = lo / kPage;
      c.last = it.tok_pos[c.re - 1] / kPage;
    }
    return true;
  }
  return false;
}

// Next page of the item; false at its end.
template <bool kParts = false>
__device__ __forceinline__ bool item_advance(const PrefillItem& it, int window, ItemCursor& c) {
  if (++c.pg <= c.last) return true;
  return item_next_run<kParts>(it, window, c);
}

// kParts: built for key parts (`parts` units per item, partials to
// part_acc / part_ml for the combine launch); otherwise parts is 1 and each
// item's outputs are written directly.  Two builds, so that the direct one
// carries none of the key-part code.
template <int D, int RK, int RV, bool kParts>
__global__ void __launch_bounds__(UmmaPrefillCfg<D, RK, RV>::kThreads, 1)
    paged_prefill_umma_kernel(const __grid_constant__ CUtensorMap k_map,
                              const __grid_constant__ CUtensorMap v_map,
                              const __grid_constant__ CUtensorMap q_map, const DecodeParams p,
                              int* item_counter, const int* block_order, int parts,
                              float* part_acc, float* part_ml) {
  using C = UmmaPrefillCfg<D, RK, RV>;
  const int G = p.group;
  const int T = C::kRows / G;  // tokens per tile
  const int tokens = C::kTiles * T;
  const int n_blocks = (p.rows + tokens - 1) / tokens;
  const int n_items = n_blocks * p.hkv;
  const int n_units = kParts ? n_items * parts : n_items;  // work units: (item, key part)
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

  extern __shared__ unsigned char smem_raw[];
  unsigned char* base = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  unsigned char* k_slots = base;
  unsigned char* v_slots = base + C::kVOff;
  unsigned char* q_smem = base + C::kQOff;  // [tile] Q rows (head_dim 128)
  uint64_t* k_full = reinterpret_cast<uint64_t*>(base + C::kBarOff);  // TMA landed
  uint64_t* k_empty = k_full + RK;         // S of the page read (P V issuer, on the last P)
  uint64_t* v_full = k_empty + RK;
  uint64_t* v_empty = v_full + RV;         // P V of the page done (S issuer, on o_done)
  // per (tile t, buffer b = page % kSBufs) at t * kSBufs + b:
  uint64_t* s_full = v_empty + RV;         // S of the page in TMEM (MMA commit)
  uint64_t* p_full = s_full + C::kTiles * C::kSBufs;  // P in TMEM (and boundary V rows zeroed)
  uint64_t* o_done = p_full + C::kTiles * C::kSBufs;  // P V of the page done (MMA commit)
  uint64_t* item_ready = o_done + C::kTiles * C::kSBufs;  // [item % 2] descriptor written
  uint64_t* item_free = item_ready + 2;       // [item % 2] consumed (softmax, issuers, V producer)
  uint64_t* fin = item_free + 2;              // [issuer] every MMA it issued done
  uint64_t* q_full = fin + 2;                 // the item's Q rows landed (TMA)
  uint64_t* q_free = q_full + 1;              // the item's S products done: Q may be replaced
  __shared__ PrefillItem items[2];
  __shared__ int y_ring[2][64];  // [K, V producer] tile rows of upcoming pages, by page % 64
  // [tile][slot][half][row]: the values the tile's two warpgroups exchange
  // (row maximum of a page, row sum of a run) at the tile's named barrier
  __shared__ float xval[C::kTiles][2][2][C::kRows];
  __shared__ volatile int abort_flag;
  __shared__ uint32_t tmem_slot;

  if (tid == 0) {
    for (int s = 0; s < RK; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
    }
    for (int s = 0; s < RV; ++s) {
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    for (int tb = 0; tb < C::kTiles * C::kSBufs; ++tb) {
      mbar_init(&s_full[tb], 1);
      mbar_init(&p_full[tb], 2 * C::kRows);  // the tile's two warpgroups
      mbar_init(&o_done[tb], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&item_ready[b], 1);
      mbar_init(&item_free[b], C::kSoftmaxThreads + 3);
    }
    mbar_init(&fin[0], 1);
    mbar_init(&fin[1], 1);
    mbar_init(q_full, 1);
    mbar_init(q_free, 1);
    mbar_init_fence();
    abort_flag = 0;
  }
  {
    // rows past T * G of each Q tile hold no token: zero them once (the
    // per-item copies fill rows 0 .. T * G - 1 only)
    const int filled = (C::kRows / G) * G;
    for (int e = tid; e < C::kTiles * C::kQBoxes * (C::kRows - filled) * 8; e += C::kThreads) {
      const int ch = e & 7, r = filled + (e >> 3) % (C::kRows - filled);
      const int tb = (e >> 3) / (C::kRows - filled);  // tile * kQBoxes + box
      *reinterpret_cast<uint4*>(q_smem + (tb / C::kQBoxes) * C::kQTileBytes +
                                (tb % C::kQBoxes) * C::kQBoxBytes + r * 128 + ch * 16) =
          make_uint4(0u, 0u, 0u, 0u);
    }
    fence_proxy_async_shared();
  }
  if (warp == C::kMmaWarp) tmem_alloc(&tmem_slot, C::kTmemCols);
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = tmem_slot;
  // the set-up above touches only this CTA's shared memory and TMEM, so it
  // overlaps the kernel before; everything from here may read its writes
  pdl_wait();
  pdl_allow_dependents();
  auto wait = [&](uint64_t* bar, uint32_t parity) {
    return mbar_wait_abortable(bar, parity, p.err, &abort_flag);
  };

  // One page tile (64 rows x D): head_dim 128 comes through its 3-D map as
  // both 64-wide boxes in one copy.
  auto load_tile = [&](unsigned char* dst, const CUtensorMap* map, int y, uint64_t* bar) {
    if constexpr (D == 128)
      tma_load_3d(dst, map, 0, y, 0, bar);
    else
      tma_load_2d(dst, map, 0, y, bar);
  };

  auto all_ok = [&](bool v) { return __all_sync(0xffffffffu, v); };
  // Streams the pages of item `it` into one ring with the whole warp, page
  // number i onwards: tile rows are looked up 32 at a time (one table load per
  // lane) into `ring` (by page number % 64); lane 0 waits for each slot and
  // issues its copy, and with `prefetch` pulls K and V pages into L2 ahead (the
  // token blocks of a request reach each page together).
  auto stream_item = [&](const PrefillItem& it, int kvh, const CUtensorMap* map,
                         unsigned char* slots, uint64_t* full, uint64_t* empty, int* ring, int& i,
                         bool prefetch) -> bool {
    int n_pages = 0;
    {
      ItemCursor cc{-1, 0, -1, -1, 0, 0};
      for (bool more = item_next_run<kParts>(it, p.window, cc); more;
           more = item_next_run<kParts>(it, p.window, cc))
        n_pages += cc.last - cc.pg + 1;
    }
    const int i_end = i + n_pages;
    ItemCursor fc{-1, 0, -1, -1, 0, 0};
    bool f_more = item_next_run<kParts>(it, p.window, fc);
    int i_fetch = i, ip = i;
    for (; i < i_end; ++i) {
      while (f_more && i_fetch < i + 16) {
        const int n = min(32, fc.last - fc.pg + 1);
        if (lane < n) {
          const int page = page_of(p.table, fc.row, fc.pg + lane, p.maxp);
          ring[(i_fetch + lane) & 63] =
              (int)tile_first_row(p.layout, page, kvh, p.hkv, p.num_pages, p.maxp);
        }
        __syncwarp();
        i_fetch += n;
        fc.pg += n - 1;
        f_more = item_advance<kParts>(it, p.window, fc);
      }
      if (prefetch && lane == 0) {
        for (; ip < min(i + kL2PrefetchPages, i_fetch); ++ip) {
          const int y = ring[ip & 63];
          if constexpr (D == 128) {
            tma_prefetch_l2_3d(&k_map, 0, y, 0);
            tma_prefetch_l2_3d(&v_map, 0, y, 0);
          } else {
            tma_prefetch_l2_2d(&k_map, 0, y);
            tma_prefetch_l2_2d(&v_map, 0, y);
          }
        }
      }
      const int s = i % RK;
      if (i >= RK && !all_ok(wait(&empty[s], ((i / RK) - 1) & 1))) return false;
      if (lane == 0) {
        mbar_arrive_expect_tx(&full[s], C::kTileBytes);
        load_tile(slots + s * C::kTileBytes, map, ring[i & 63], &full[s]);
      }
    }
    return true;
  };

  if (warp == C::kProducerWarp) {
    // ------------------------------------------------------------ K producer
    if (lane == 0) {
      prefetch_tensormap(&k_map);
      prefetch_tensormap(&v_map);
    }
    int ik = 0;  // K loads issued (all items)
    bool ok = true;
    for (int seq = 0; ok; ++seq) {
      const int d = seq & 1;
      PrefillItem& it = items[d];
      int j = 0;
      if (lane == 0) j = atomicAdd(item_counter, 1);
      j = __shfl_sync(0xffffffffu, j, 0);
      // the descriptor slot holds item seq - 2 until both consumers are done
      if (seq >= 2 && !__all_sync(0xffffffffu, wait(&item_free[d], ((seq >> 1) - 1) & 1))) break;
      if (j >= n_units) {
        if (lane == 0) {
          it.valid = 0;
          mbar_arrive(&item_ready[d]);
        }
        break;
      }
      // a unit's key parts are taken one after another, so an item's parts
      // run side by side on different SMs
      const int item = kParts ? j / parts : j;
      const int blk = block_order ? block_order[item / p.hkv] : n_blocks - 1 - item / p.hkv;
      const int kvh = item % p.hkv;
      const int t_begin = blk * tokens, t_end = min(t_begin + tokens, p.rows);
      const int h0 = kvh * G;
      // tokens of the item: rows and positions; bad ones are reported and
      // left out of every run (their outputs are zeroed below)
      for (int k = lane; k < tokens; k += 32) {
        const int t = t_begin + k;
        int row = -1, pos = -1;
        if (t < t_end) {
          row = p.row_of ? p.row_of[t] : t;
          pos = p.positions[t];
          const bool bad = row < 0 || row >= p.table_rows || (pos >= 0 && pos / kPage >= p.maxp);
          if (bad) record_error(p.err, PGD_EDEVICE_BOUNDS);
          if (bad || pos < 0) row = -1;
        }
        it.tok_row[k] = row;
        it.tok_pos[k] = pos;
      }
      __syncwarp();
      // runs: token k ends one when k + 1 starts another (or is past the end)
      {
        int r = 0;
        for (int k0 = 0; k0 < tokens; k0 += 32) {
          const int k = k0 + lane;
          bool brk = false;
          if (k < tokens)
            brk = k + 1 == tokens || it.tok_row[k + 1] != it.tok_row[k] ||
                  it.tok_pos[k + 1] != it.tok_pos[k] + 1 || it.tok_row[k + 1] < 0 ||
                  it.tok_row[k] < 0;
          const unsigned bal = __ballot_sync(0xffffffffu, brk);
          if (brk) it.run_end[r + __popc(bal & ((1u << lane) - 1u))] = k + 1;
          r += __popc(bal);
        }
        if (lane == 0) it.runs = r;
      }
      if (lane == 0) {
        it.valid = 1;
        it.t_begin = t_begin;
        it.t_end = t_end;
        it.kvh = kvh;
        it.part = kParts ? j % parts : 0;
        it.parts = kParts ? parts : 1;
      }
      __syncwarp();
      // a table entry outside the pool marks its run bad (zero outputs,
      // PGD_EDEVICE_BOUNDS); checked before any copy is issued
      for (int r = 0; r < it.runs; ++r) {
        const int rs = r == 0 ? 0 : it.run_end[r - 1], re = it.run_end[r];
        const int row = it.tok_row[rs];
        int bad = 0;
        if (row >= 0) {
          const int lo = p.window > 0 ? max(it.tok_pos[rs] - p.window + 1, 0) : 0;
          const int first = lo / kPage, last = it.tok_pos[re - 1] / kPage;
          for (int pg = first + lane; pg <= last; pg += 32) {
            const int page = page_of(p.table, row, pg, p.maxp);
            if (page < 0 || page >= p.num_pages) bad = 1;
          }
        }
        bad = __any_sync(0xffffffffu, bad);
        if (lane == 0) {
          it.run_bad[r] = bad;
          if (bad) record_error(p.err, PGD_EDEVICE_BOUNDS);
        }
      }
      if constexpr (kParts) {
        // each run's pages in this unit's key part, for every role's walk
        for (int r = lane; r < it.runs; r += 32) {
          const int rs = r == 0 ? 0 : it.run_end[r - 1], re = it.run_end[r];
          const int lo = p.window > 0 ? max(it.tok_pos[rs] - p.window + 1, 0) : 0;
          int first = lo / kPage, last = max(it.tok_pos[re - 1], 0) / kPage;
          part_pages(it, first, last);
          it.run_pg[r] = first;
          it.run_last[r] = last;
        }
      }
      __syncwarp();
      // outputs of tokens that no pass covers (inactive or bad run)
      for (int r = 0; r < it.runs; ++r) {
        const int rs = r == 0 ? 0 : it.run_end[r - 1], re = it.run_end[r];
        if (it.tok_row[rs] >= 0 && !it.run_bad[r]) continue;
        for (int e = lane; e < (re - rs) * G * (D / 8); e += 32) {
          const int tl = rs + e / (G * (D / 8));
          if (t_begin + tl >= t_end) continue;
          const int g = (e / (D / 8)) % G, c = e % (D / 8);
          reinterpret_cast<uint4*>(p.out + ((size_t)(t_begin + tl) * p.hq + h0 + g) * D)[c] =
              make_uint4(0u, 0u, 0u, 0u);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&item_ready[d]);
      ok = stream_item(it, kvh, &k_map, k_slots, k_full, k_empty, y_ring[0], ik, true);
    }
    // drain: the copies still in flight land before the CTA exits
    if (lane == 0)
      for (int j = max(0, ik - RK); j < ik; ++j)
        mbar_wait_bounded(&k_full[j % RK], (j / RK) & 1, p.err);
  } else if (warp == C::kVWarp) {
    // ------------------------------------------------------------ V producer
    int iv = 0;  // V loads issued (all items)
    for (int seq = 0;; ++seq) {
      const int d = seq & 1;
      if (!all_ok(wait(&item_ready[d], (seq >> 1) & 1))) break;
      const PrefillItem& it = items[d];
      if (!it.valid) break;
      if (!stream_item(it, it.kvh, &v_map, v_slots, v_full, v_empty, y_ring[1], iv, false)) break;
      if (lane == 0) mbar_arrive(&item_free[d]);
    }
    if (lane == 0)
      for (int j = max(0, iv - RV); j < iv; ++j)
        mbar_wait_bounded(&v_full[j % RV], (j / RV) & 1, p.err);
  } else if (warp == C::kMmaWarp) {
    // ------------------------------------------------------------ S issuer
    if (lane == 0) {
      const uint32_t k_addr = smem_addr(k_slots);
      int i = 0;  // page index over all items
      bool issued = false, ok = true;
      bool q_pending = false;  // a Q copy issued and not yet seen landed
      int q_phase = 0;
      for (int seq = 0; ok; ++seq) {
        const int d = seq & 1;
        if (!wait(&item_ready[d], (seq >> 1) & 1)) break;
        const PrefillItem& it = items[d];
        if (!it.valid) break;
        {
          // the item's Q rows by TMA ([token][head] rows of 64 values: the
          // swizzled K-major layout the products read), once the previous
          // item's S products, which read the same shared memory, are done;
          // the softmax warps meanwhile finish the previous item
          if (seq > 0 && !wait(q_free, (seq - 1) & 1)) break;
          mbar_arrive_expect_tx(q_full, C::kTiles * C::kQBoxes * T * G * 128);
          for (int t = 0; t < C::kTiles; ++t)
            for (int bx = 0; bx < C::kQBoxes; ++bx)
              tma_load_3d(q_smem + t * C::kQTileBytes + bx * C::kQBoxBytes, &q_map, 64 * bx,
                          it.kvh * G, it.t_begin + t * T, q_full);
          q_pending = true;
          q_phase = seq;
          if (!wait(q_full, seq & 1)) break;
          q_pending = false;
        }
        ItemCursor cur{-1, 0, -1, -1, 0, 0};
        for (bool more = item_next_run<kParts>(it, p.window, cur); more && ok;
             more = item_advance<kParts>(it, p.window, cur), ++i) {
          if (!wait(&k_full[i % RK], (i / RK) & 1)) {
            ok = false;
            break;
          }
          const uint64_t kd = umma_desc_sw128(k_addr + (i % RK) * C::kTileBytes, 16, 1024);
          const int b = i % C::kSBufs;
          for (int t = 0; t < C::kTiles; ++t) {
            // the buffer holds P_t of page i - kSBufs until P V has read it
            const int tb = t * C::kSBufs + b;
            if (i >= C::kSBufs) {
              if (!wait(&o_done[tb], ((i / C::kSBufs) - 1) & 1)) {
                ok = false;
                break;
              }
              // the last tile's P V of page i - kSBufs done (its commit
              // covers every product issued before it): that page's V slot
              // is free -- one thread arrival in place of a commit a page
              if (t == C::kTiles - 1) mbar_arrive(&v_empty[(i - C::kSBufs) % RV]);
            }
            tc_fence_after_sync();
            const uint32_t sb = tmem + C::kSCol + tb * kPage;
            const uint64_t qd = umma_desc_sw128(smem_addr(q_smem) + t * C::kQTileBytes, 16, 1024);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk)
              umma_bf16(sb, umma_desc_advance(qd, (kk >> 2) * C::kQBoxBytes + (kk & 3) * 32),
                        umma_desc_advance(kd, (kk >> 2) * kBoxBytes + (kk & 3) * 32), C::kIdescS,
                        kk > 0);
            umma_commit(&s_full[tb]);
          }
          if (!ok) break;
          issued = true;
        }
        if (ok) umma_commit(q_free);  // this item's S products done: Q may be replaced
        if (ok) mbar_arrive(&item_free[d]);
      }
      // drain: every MMA this thread issued completes before TMEM is freed,
      // and a Q copy still in flight lands before the CTA exits
      if (issued) {
        umma_commit(fin);
        mbar_wait_bounded(fin, 0, p.err);
      }
      if (q_pending) mbar_wait_bounded(q_full, q_phase & 1, p.err);
    }
  } else if (warp == C::kPvWarp) {
    // ------------------------------------------------------------ P V issuer
    if (lane == 0) {
      const uint32_t v_addr = smem_addr(v_slots);
      int i = 0;  // page index over all items
      bool issued = false, ok = true;
      for (int seq = 0; ok; ++seq) {
        const int d = seq & 1;
        if (!wait(&item_ready[d], (seq >> 1) & 1)) break;
        const PrefillItem& it = items[d];
        if (!it.valid) break;
        ItemCursor cur{-1, 0, -1, -1, 0, 0};
        bool first = true;  // O restarts with each item
        for (bool more = item_next_run<kParts>(it, p.window, cur); more && ok;
             more = item_advance<kParts>(it, p.window, cur), ++i) {
          if (!wait(&v_full[i % RV], (i / RV) & 1)) {
            ok = false;
            break;
          }
          const uint64_t vd = umma_desc_sw128(v_addr + (i % RV) * C::kTileBytes, kBoxBytes, 1024);
          const int b = i % C::kSBufs;
          for (int t = 0; t < C::kTiles; ++t) {
            const int tb = t * C::kSBufs + b;
            if (!wait(&p_full[tb], (i / C::kSBufs) & 1)) {
              ok = false;
              break;
            }
            // the last tile's softmax has read its S, whose commit covers
            // both tiles' S products: page i's K slot is free
            if (t == C::kTiles - 1) mbar_arrive(&k_empty[i % RK]);
            tc_fence_after_sync();
            const uint32_t pb = tmem + C::kSCol + tb * kPage;
            const uint32_t od = tmem + C::kOCol + t * D;
            // keys 16 kk .. 16 kk + 15: chunk kk / 2 of the P columns, half
            // kk % 2 of its 16 head (then residual) columns
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              umma_bf16_tmem_a(od, pb + 32 * (kk >> 1) + 8 * (kk & 1),
                               umma_desc_advance(vd, kk * 2048), C::kIdescPV, !(first && kk == 0));
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              umma_bf16_tmem_a(od, pb + 32 * (kk >> 1) + 16 + 8 * (kk & 1),
                               umma_desc_advance(vd, kk * 2048), C::kIdescPV, true);
            umma_commit(&o_done[tb]);
          }
          if (!ok) break;
          first = false;
          issued = true;
        }
        if (ok) mbar_arrive(&item_free[d]);
      }
      if (issued) {
        umma_commit(fin + 1);
        mbar_wait_bounded(fin + 1, 0, p.err);
      }
    }
  } else {
    // ------------------------------------------------------------ softmax
    // row; tile; half h of every page's keys (and of the O columns) this
    // thread takes -- the tile's other warpgroup takes the other half
    const int m = tid & 127, t = (tid >> 7) & 1, h = tid >> 8;
    constexpr int kHalf = kPage / 2;
    int xn = 0;  // exchanges with the other half so far
    const uint32_t lane_base = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
    const float c = p.q_scale_log2;
    const float cc = c > 0.f ? c : 1.f;
    int i = 0;  // page index over all items
    // The tile's two warpgroups exchange values at a named barrier (id 1 +
    // t) that also ORs a failure flag over them, so they leave their loops
    // together: a thread whose wait gave up (`mine` false) carries on to the
    // next exchange, and every thread of the tile stops there (`ok` false).
    bool ok = true, mine = true;
    const uint32_t xid = 1 + t, xcount = 2 * C::kRows;
    const int tl = t * T + m / G, g = m % G;  // token of the block, head of the group
    const bool in_tile = m / G < T;           // rows past T * G hold no token
    // Waits for the descriptor of item seq (its Q is copied in by the S
    // issuer); false when there is no item seq.
    auto next_item = [&](int seq) -> bool {
      const int d = seq & 1;
      if (!all_ok(wait(&item_ready[d], (seq >> 1) & 1))) {
        mine = false;
        return false;
      }
      return items[d].valid != 0;
    };
    bool have = next_item(0);
    ok = !named_sync_or(xid, xcount, !mine);
    for (int seq = 0; ok && have; ++seq) {
      const int d = seq & 1;
      const PrefillItem& it = items[d];
      const int t_begin = it.t_begin, t_end = it.t_end, h0 = it.kvh * G;
      const bool row_ok = in_tile && t_begin + tl < t_end;
      int rs = 0;
      for (int r = 0; r < it.runs && ok; ++r) {
        const int re = it.run_end[r];
        const int row = it.tok_row[rs];
        // with key parts, a row's partial of this part: (m, l) and its O
        // columns, at [token][head][part] (from the descriptor in shared
        // memory where it is written, so that no part of it is held in
        // registers through the page loop)
        auto unit_of = [&]() {
          return ((size_t)(it.t_begin + tl) * p.hq + it.kvh * G + g) * it.parts + it.part;
        };
        if (row < 0 || it.run_bad[r]) {
          // no pass covers these tokens (their outputs are zeroed): the
          // combine leaves them as they are
          if constexpr (kParts) {
            if (h == 0 && row_ok && tl >= rs && tl < re) {
              const size_t u = unit_of();
              part_ml[2 * u] = -INFINITY;
              part_ml[2 * u + 1] = -1.f;
            }
          }
          rs = re;
          continue;
        }
        const bool live = row_ok && tl >= rs && tl < re;
        const int pos = live ? it.tok_pos[tl] : -1;
        const int lo = p.window > 0 ? pos - p.window + 1 : 0;
        const int lo_run = p.window > 0 ? max(it.tok_pos[rs] - p.window + 1, 0) : 0;
        const int pos_last = it.tok_pos[re - 1];
        int first = lo_run / kPage, last = pos_last / kPage;
        if constexpr (kParts) {
          // a key part without pages of this run: the rows' partials are
          // empty (the same for every thread of the tile)
          first = it.run_pg[r];
          last = it.run_last[r];
          if (first > last) {
            if (h == 0 && live) {
              const size_t u = unit_of();
              part_ml[2 * u] = -INFINITY;
              part_ml[2 * u + 1] = 0.f;
            }
            rs = re;
            continue;
          }
        }
        float m_run = -INFINITY;  // running (lazy) max of the row, log2 units
        float l = 0.f;            // row sum relative to m_run
        for (int pg = first; pg <= last; ++pg, ++i) {
          const int tb = t * C::kSBufs + i % C::kSBufs;
          const uint32_t scol = C::kSCol + tb * kPage;
          if (!all_ok(wait(&s_full[tb], (i / C::kSBufs) & 1))) mine = false;
          tc_fence_after_sync();
          float sv[kHalf];
#pragma unroll
          for (int q = 0; q < kHalf / 16; ++q)
            tmem_ld16(lane_base + scol + kHalf * h + 16 * q,
                      *reinterpret_cast<float(*)[16]>(&sv[16 * q]));
          tmem_wait_ld();
          // scores stay raw: the scale is folded into the exponent's FMA (for
          // a positive scale; otherwise it is applied here)
          if (!(c > 0.f)) {
#pragma unroll
            for (int k = 0; k < kHalf; ++k) sv[k] *= c;
          }
          const int pos0 = pg * kPage;
          const int pos0h = pos0 + kHalf * h;  // this half's first key
          if (!(live && pos0h >= lo && pos0h + kHalf - 1 <= pos)) {
#pragma unroll
            for (int k = 0; k < kHalf; ++k)
              if (!(live && pos0h + k >= lo && pos0h + k <= pos)) sv[k] = -INFINITY;
          }
          // eight partial maxima: the first 8 scores, then 24 more two at a
          // time (a block of 16 and a last block of 8)
          float part[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) part[j] = sv[j];
#pragma unroll
          for (int k = 8; k + 16 <= kHalf; k += 16)
#pragma unroll
            for (int j = 0; j < 8; ++j)
              part[j] = fmax3(part[j], sv[k + 2 * j], sv[k + 2 * j + 1]);
          static_assert((kHalf - 8) % 16 == 8, "the last block holds 8 scores");
#pragma unroll
          for (int j = 0; j < 4; ++j)
            part[j] = fmax3(part[j], sv[kHalf - 8 + 2 * j], sv[kHalf - 7 + 2 * j]);
          const float mxh = fmax3(fmax3(part[0], part[1], part[2]),
                                  fmax3(part[3], part[4], part[5]), fmaxf(part[6], part[7])) *
                            cc;
          // the row's max over the whole page: the other half's through
          // shared memory (both halves then take the same lazy decisions)
          float mx;
          {
            const int sl = xn & 1;
            xval[t][sl][h][m] = mxh;
            if (named_sync_or(xid, xcount, !mine)) {
              ok = false;
              break;
            }
            mx = fmaxf(mxh, xval[t][sl][1 - h][m]);
            ++xn;
          }
          float alpha = 1.f;
          bool rose = false;
          if (mx > m_run + kLazyRescaleLog2) {
            if (m_run != -INFINITY) {
              alpha = exp2_approx(m_run - mx);
              rose = true;
            }
            l = m_run == -INFINITY ? 0.f : l * alpha;
            m_run = mx;
          }
          const float nml = m_run == -INFINITY ? 0.f : -m_run;
          // P = 2^(s - m_run) as a bf16 head and residual over the S columns
          // (per chunk of 32 keys: head at +0, residual at +16, column j of a
          // half holding keys 2j, 2j + 1); pairs through the packed fp32 pipe
          const float2 cc2 = make_float2(cc, cc), nml2 = make_float2(nml, nml);
          const float2 minus1 = make_float2(-1.f, -1.f);
          float2 sum2[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) sum2[j] = make_float2(0.f, 0.f);
#pragma unroll
          for (int q = 0; q < kHalf / 32; ++q) {
            uint32_t hw[16], lw[16];
#pragma unroll
            for (int w = 0; w < 16; ++w) {
              const float2 y = __ffma2_rn(make_float2(sv[32 * q + 2 * w], sv[32 * q + 2 * w + 1]),
                                          cc2, nml2);
              const float2 x = make_float2(exp2_approx(y.x), exp2_approx(y.y));
              sum2[w & 3] = __fadd2_rn(sum2[w & 3], x);
              hw[w] = pack_bf16x2(x.x, x.y);
              const float2 rr =
                  __ffma2_rn(make_float2(bf16_lo(hw[w]), bf16_hi(hw[w])), minus1, x);
              lw[w] = pack_bf16x2(rr.x, rr.y);
            }
            tmem_st16(lane_base + scol + kHalf * h + 32 * q, hw);
            tmem_st16(lane_base + scol + kHalf * h + 32 * q + 16, lw);
          }
          const float2 s4 =
              __fadd2_rn(__fadd2_rn(sum2[0], sum2[1]), __fadd2_rn(sum2[2], sum2[3]));
          l += s4.x + s4.y;
          if (__any_sync(0xffffffffu, rose)) {
            // O_t holds P V up to page i - 1, which must be done (with one
            // buffer it was, before S_t of this page was issued)
            bool done = true;
            if (C::kSBufs > 1) {
              const int tp = t * C::kSBufs + (i - 1) % C::kSBufs;
              done = all_ok(wait(&o_done[tp], ((i - 1) / C::kSBufs) & 1));
              if (done) tc_fence_after_sync();
              else mine = false;
            }
            if (done) {
#pragma unroll
              for (int j = 0; j < D / 32; ++j) {  // this half's O columns
                const int q16 = h * (D / 32) + j;
                float ov[16];
                tmem_ld16(lane_base + C::kOCol + t * D + 16 * q16, ov);
                tmem_wait_ld();
#pragma unroll
                for (int k = 0; k < 16; ++k) ov[k] *= alpha;
                tmem_st16(lane_base + C::kOCol + t * D + 16 * q16, ov);
              }
            }
          }
          // V rows outside the run's key range on a boundary page -> zero
          // (warpgroup 0; both tiles' products read them after its P)
          const int rlo = max(lo_run - pos0, 0), rhi = min(pos_last - pos0, kPage - 1);
          bool zero = t == 0 && h == 0 && (rlo > 0 || rhi < kPage - 1);
          if (zero && !all_ok(wait(&v_full[i % RV], (i / RV) & 1))) {
            mine = false;
            zero = false;
          }
          if (zero) {
            const int s = i % RV;
            unsigned char* vt = v_slots + s * C::kTileBytes;
            for (int e = m; e < kPage * (D / 8); e += C::kRows) {
              const int k = e / (D / 8), ch = e % (D / 8);
              if (k < rlo || k > rhi)
                *reinterpret_cast<uint4*>(vt + (ch >> 3) * kBoxBytes + k * 128 + (ch & 7) * 16) =
                    make_uint4(0u, 0u, 0u, 0u);
            }
            fence_proxy_async_shared();  // the zeros are read by the tensor core
          }
          tmem_wait_st();
          tc_fence_before_sync();
          mbar_arrive(&p_full[tb]);
        }
        if (!ok) break;

        // end of run: the O_t row once P V of the last page is done
        const int il = i - 1;
        if (all_ok(wait(&o_done[t * C::kSBufs + il % C::kSBufs], (il / C::kSBufs) & 1)))
          tc_fence_after_sync();
        else
          mine = false;
        {  // the row sum: this half's plus the other half's
          const int sl = xn & 1;
          xval[t][sl][h][m] = l;
          if (named_sync_or(xid, xcount, !mine)) {
            ok = false;
            break;
          }
          l += xval[t][sl][1 - h][m];
          ++xn;
        }
        const int hh = h0 + g;
        if constexpr (kParts) {
          // the row's partial over this part's keys, unnormalised (the sink
          // and the other parts are merged by the combine launch)
          const size_t u = unit_of();
          if (h == 0 && live) {
            part_ml[2 * u] = m_run;
            part_ml[2 * u + 1] = l;
          }
          float* arow = part_acc + u * D;
#pragma unroll
          for (int j = 0; j < D / 32; ++j) {  // this half's O columns
            const int q16 = h * (D / 32) + j;
            float ov[16];
            tmem_ld16(lane_base + C::kOCol + t * D + 16 * q16, ov);
            tmem_wait_ld();
            if (live) {
              float4* dst = reinterpret_cast<float4*>(arow + 16 * q16);
#pragma unroll
              for (int k = 0; k < 4; ++k)
                dst[k] = make_float4(ov[4 * k], ov[4 * k + 1], ov[4 * k + 2], ov[4 * k + 3]);
            }
          }
          tc_fence_before_sync();
          rs = re;
          continue;
        }
        float inv = 0.f;
        if (live) {
          const float sk = p.sinks ? p.sinks[hh] * kLog2e : -INFINITY;
          const float mf = fmaxf(m_run, sk);
          const float scl = exp2_approx(m_run - mf);
          const float total = fmaf(l, scl, exp2_approx(sk - mf));
          inv = total > 0.f ? scl / total : 0.f;
        }
        uint16_t* orow = p.out + ((size_t)(t_begin + (live ? tl : 0)) * p.hq + hh) * D;
#pragma unroll
        for (int j = 0; j < D / 32; ++j) {  // this half's output columns
          const int q16 = h * (D / 32) + j;
          float ov[16];
          tmem_ld16(lane_base + C::kOCol + t * D + 16 * q16, ov);
          tmem_wait_ld();
          if (live) {
            uint32_t w[8];
#pragma unroll
            for (int k = 0; k < 8; ++k)
              w[k] = pack_bf16x2(ov[2 * k] * inv, ov[2 * k + 1] * inv);
            uint4* dst = reinterpret_cast<uint4*>(orow + 16 * q16);
            dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
            dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
          }
        }
        tc_fence_before_sync();
        rs = re;
      }
      if (!ok) break;
      // this item's descriptor is no longer read: free its slot before
      // waiting for the next item
      mbar_arrive(&item_free[d]);
      have = next_item(seq + 1);
      ok = !named_sync_or(xid, xcount, !mine);
    }
  }

  // ---------------------------------------------------------------- teardown
  tc_fence_before_sync();
  __syncthreads();
  if (warp == C::kMmaWarp) {
    __syncwarp();
    tc_fence_after_sync();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

// Token blocks sorted by this many at most; larger calls, and calls with a
// window (whose blocks' spans it bounds: the sort pass measured slower than
// it gained on the gpt-oss sliding-window prefill, 0.0675 against 0.0653
// ms), take them in token order, last block first.
constexpr int kMaxSortedBlocks = 4096;

// Threads of the block-order pass: one per key of the padded sort, so that
// each thread makes one round trip for its block's tokens, and no more (the
// sort's steps meet at a CTA barrier, which costs more the more warps wait
// at it); at least a warp and at most 1024.
inline int block_order_threads(int n_blocks) {
  int n2 = 32;
  while (n2 < n_blocks && n2 < 1024) n2 <<= 1;
  return n2;
}

// Before the prefill kernel (one CTA): zeroes its item counter and writes
// order[0 .. n_blocks) = the token blocks, longest key span first, so that
// the persistent CTAs take the long items first and finish together.  A
// block's span in pages is estimated from its first and last tokens (the
// last token's key range, plus the first token's when the block starts in
// another table row); equal spans keep the later block first.  A bitonic
// sort of (span, block) keys in shared memory.  (Templated on the head_dim
// only to give each translation unit its own instance.)
// The block order, by one CTA (blockDim threads, `key` in its shared memory:
// kMaxSortedBlocks entries).
__device__ __forceinline__ void order_blocks(const DecodeParams& p, int block_tokens,
                                             int n_blocks, int* counter, int* order,
                                             unsigned long long* key) {
  if (threadIdx.x == 0) *counter = 0;
  int n2 = 1;
  while (n2 < n_blocks) n2 <<= 1;
  auto pages = [&](int pos) -> unsigned int {
    if (pos < 0) return 0u;
    const int lo = p.window > 0 ? max(pos - p.window + 1, 0) : 0;
    return (unsigned int)(pos / kPage - lo / kPage + 1);
  };
  for (int b = threadIdx.x; b < n2; b += blockDim.x) {
    unsigned long long k = ~0ull;  // padding sorts last
    if (b < n_blocks) {
      const int t0 = b * block_tokens, t1 = min(t0 + block_tokens, p.rows) - 1;
      const int r0 = p.row_of ? p.row_of[t0] : t0, r1 = p.row_of ? p.row_of[t1] : t1;
      const unsigned int span = pages(p.positions[t1]) + (r0 != r1 ? pages(p.positions[t0]) : 0u);
      k = ((unsigned long long)(~span) << 32) | (unsigned int)(n_blocks - 1 - b);
    }
    key[b] = k;
  }
  __syncthreads();
  for (int size = 2; size <= n2; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = threadIdx.x; i < n2; i += blockDim.x) {
        const int j = i ^ stride;
        if (j > i) {
          const unsigned long long a = key[i], c = key[j];
          const bool up = (i & size) == 0;
          if ((a > c) == up) {
            key[i] = c;
            key[j] = a;
          }
        }
      }
      __syncthreads();
    }
  }
  for (int b = threadIdx.x; b < n_blocks; b += blockDim.x)
    order[b] = n_blocks - 1 - (int)(key[b] & 0xffffffffu);
}

template <int D>
__global__ void __launch_bounds__(1024) prefill_block_order_kernel(const DecodeParams p,
                                                                   int block_tokens, int n_blocks,
                                                                   int* counter, int* order) {
  pdl_wait();
  pdl_allow_dependents();
  __shared__ unsigned long long key[kMaxSortedBlocks];
  order_blocks(p, block_tokens, n_blocks, counter, order, key);
}

// The prefill step's first launch (prefill_paged: page_slots + write_tokens,
// then the attention): CTA 0 prepares the tcgen05 kernel's work counter (and,
// when `order` is given, the longest-first block order); the other CTAs
// write each packed token's K and V at its slot, table[rows[t]][n / 64] * 64
// + n % 64 for its position n, one warp per token.  Inactive tokens (n < 0)
// are skipped; a token whose row, page index or page is out of range is
// reported (PGD_EDEVICE_BOUNDS) and not written, as page_slots and the write
// at slots would leave it.
template <int D>
__global__ void __launch_bounds__(1024) prefill_write_kernel(const DecodeParams p,
                                                             int block_tokens, int n_blocks,
                                                             int* counter, int* order) {
  pdl_wait();
  pdl_allow_dependents();
  __shared__ unsigned long long key[kMaxSortedBlocks];
  if (blockIdx.x == 0) {
    if (order)
      order_blocks(p, block_tokens, n_blocks, counter, order, key);
    else if (counter && threadIdx.x == 0)
      *counter = 0;
    return;
  }
  constexpr int kChunks = D / 8;  // 16-byte chunks of a head's row
  const int lane = threadIdx.x & 31;
  const int warps = (gridDim.x - 1) * (blockDim.x >> 5);
  for (int t = (blockIdx.x - 1) * (blockDim.x >> 5) + (threadIdx.x >> 5); t < p.rows;
       t += warps) {
    int page = -1, in_page = 0;
    if (lane == 0) {
      const int n = p.positions[t];
      const int row = p.row_of ? p.row_of[t] : t;
      if (n >= 0) {
        const bool bad_row = p.row_of && (row < 0 || row >= p.table_rows);
        const int pg = (!bad_row && n / kPage < p.maxp) ? page_of(p.table, row, n / kPage, p.maxp)
                                                        : -1;
        if (pg < 0 || pg >= p.num_pages)
          record_error(p.err, PGD_EDEVICE_BOUNDS);
        else
          page = pg;
        in_page = n % kPage;
      }
    }
    page = __shfl_sync(0xffffffffu, page, 0);
    in_page = __shfl_sync(0xffffffffu, in_page, 0);
    if (page < 0) continue;
    for (int c = lane; c < 2 * p.hkv * kChunks; c += 32) {
      const int which = c / (p.hkv * kChunks);
      const int h = (c / kChunks) % p.hkv, ch = c % kChunks;
      const uint16_t* src = (which ? p.v_new : p.k_new) + ((size_t)t * p.hkv + h) * D + ch * 8;
      const int64_t row0 = tile_first_row(p.layout, page, h, p.hkv, p.num_pages, p.maxp);
      uint16_t* dst = (which ? p.v_pool : p.k_pool) + ((size_t)row0 + in_page) * D + ch * 8;
      *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(src);
    }
  }
}

// Merge of the key parts of the tcgen05 prefill (a call split into `parts`
// units per item): for token t and query head h, with the partials (m_s, l_s,
// O_s) of parts s (m in log2 units, O unnormalised) and the sink logit
// sigma (log2 units here, or none),
//   M = max(max_s m_s, sigma),  L = sum_s l_s 2^(m_s - M) + 2^(sigma - M),
//   out = sum_s O_s 2^(m_s - M) / L,
// the split softmax of the attention step over all of the token's keys, the
// sink in the denominator only (GPT-OSS 20B model files, src/attention.linnet,
// SinkAttention).  A part without keys (m = -inf) adds nothing; a token whose
// partial carries l < 0 was covered by no pass, and its output, already
// zeroed, is left.  One warp per (token, query head), 32 lanes over D.
template <int D>
__global__ void __launch_bounds__(128) prefill_part_combine_kernel(const DecodeParams p,
                                                                   int parts,
                                                                   const float* part_acc,
                                                                   const float* part_ml) {
  constexpr int kDims = D / 32;  // dims of a lane: 2 or 4
  static_assert(kDims == 2 || kDims == 4, "head_dim");
  const int t = blockIdx.y;
  const int h = blockIdx.x * 4 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  // the sinks are an input of the attention kernel as well, which reads them
  // after its own dependency wait; this grid starts once every CTA of it
  // has passed that wait, so they are final here
  const float sk = (p.sinks && h < p.hq) ? p.sinks[h] * kLog2e : -INFINITY;
  pdl_wait();
  pdl_allow_dependents();
  if (h >= p.hq) return;
  const size_t u0 = ((size_t)t * p.hq + h) * parts;
  float mx = sk;
  bool covered = true;
  for (int s = 0; s < parts; ++s) {
    const float ms = part_ml[2 * (u0 + s)], ls = part_ml[2 * (u0 + s) + 1];
    covered = covered && ls >= 0.f;
    mx = fmaxf(mx, ms);
  }
  if (!covered) return;
  uint16_t* o = p.out + ((size_t)t * p.hq + h) * D + lane * kDims;
  float acc[kDims];
#pragma unroll
  for (int j = 0; j < kDims; ++j) acc[j] = 0.f;
  float total = 0.f;
  if (mx != -INFINITY) {
    if (sk != -INFINITY) total = exp2_approx(sk - mx);
    for (int s = 0; s < parts; ++s) {
      const float ms = part_ml[2 * (u0 + s)];
      if (ms == -INFINITY) continue;
      const float w = exp2_approx(ms - mx);
      total = fmaf(part_ml[2 * (u0 + s) + 1], w, total);
      const float* a = part_acc + (u0 + s) * D + lane * kDims;
#pragma unroll
      for (int j = 0; j < kDims; j += 2) {
        const float2 v = *reinterpret_cast<const float2*>(a + j);
        acc[j] = fmaf(v.x, w, acc[j]);
        acc[j + 1] = fmaf(v.y, w, acc[j + 1]);
      }
    }
  }
  const float inv = total > 0.f ? 1.f / total : 0.f;
  uint32_t w2[kDims / 2];
#pragma unroll
  for (int j = 0; j < kDims / 2; ++j) w2[j] = pack_bf16x2(acc[2 * j] * inv, acc[2 * j + 1] * inv);
  if constexpr (kDims == 4) {
    *reinterpret_cast<uint2*>(o) = make_uint2(w2[0], w2[1]);  // 4 values
  } else {
    *reinterpret_cast<uint32_t*>(o) = w2[0];  // 2 values
  }
}

// Where the key parts' partials live in the caller's workspace: after the
// work counter and the block order in p.ws_acc, the O partials
// [token][head][part][D]; the (m, l) pairs [token][head][part][2] in p.ws_ml.
// The workspace holds p.max_splits partials a token and head, so up to
// p.max_splits - 1 parts fit beside the counter and the order.
inline float* prefill_part_acc(const DecodeParams& p, int n_blocks) {
  return p.ws_acc + ((4 + n_blocks + 3) / 4) * 4;
}

// `prepared`: the step's write launch has already zeroed the work counter and
// written the block order (prefill_write_kernel).  `parts` > 1: each item's
// pages are cut into that many key parts, one work unit each, and a combine
// launch merges their partials.
template <int D, int RK, int RV, bool kParts>
cudaError_t configure_prefill_umma() {
  using C = UmmaPrefillCfg<D, RK, RV>;
  static std::atomic<bool> configured[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !configured[dev].load(std::memory_order_acquire)) {
    e = cudaFuncSetAttribute(paged_prefill_umma_kernel<D, RK, RV, kParts>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) configured[dev].store(true, std::memory_order_release);
  }
  return cudaSuccess;
}

template <int D, int RK, int RV>
cudaError_t launch_prefill_umma(const DecodeParams& p, const CUtensorMap& k_map,
                                const CUtensorMap& v_map, const CUtensorMap& q_map, int sm_count,
                                bool prepared, int parts, cudaStream_t stream) {
  using C = UmmaPrefillCfg<D, RK, RV>;
  // the partials' room in the workspace; the combine grid has a row of CTAs
  // per token
  if (parts < 1 || (parts > 1 && (parts > p.max_splits - 1 || p.rows > 65535)))
    return cudaErrorInvalidValue;
  cudaError_t e = parts > 1 ? configure_prefill_umma<D, RK, RV, true>()
                            : configure_prefill_umma<D, RK, RV, false>();
  if (e != cudaSuccess) return e;
  if (p.rows == 0) return cudaSuccess;
  const int tokens = C::kTiles * (C::kRows / p.group);
  const int items = ((p.rows + tokens - 1) / tokens) * p.hkv;
  // the item counter lives in the first word of the caller's workspace, the
  // block order from the fifth (the workspace holds at least
  // rows x (head_dim + 2) floats, and there are at most rows blocks)
  int* counter = reinterpret_cast<int*>(p.ws_acc);
  const int n_blocks = (p.rows + tokens - 1) / tokens;
  int* order = p.window == 0 && n_blocks <= kMaxSortedBlocks ? counter + 4 : nullptr;
  if (prepared)
    e = cudaSuccess;
  else if (order)
    e = launch_pdl(prefill_block_order_kernel<D>, dim3(1), dim3(block_order_threads(n_blocks)), 0,
                   stream, p, tokens, n_blocks, counter, order);
  else
    e = cudaMemsetAsync(counter, 0, sizeof(int), stream);
  if (e != cudaSuccess) return e;
  float* part_acc = parts > 1 ? prefill_part_acc(p, n_blocks) : nullptr;
  float* part_ml = parts > 1 ? p.ws_ml : nullptr;
  const int units = items * parts;
  const int ctas = units < sm_count ? units : sm_count;
  if (parts == 1)
    return launch_pdl(paged_prefill_umma_kernel<D, RK, RV, false>, dim3(ctas), dim3(C::kThreads),
                      C::kSmemBytes, stream, k_map, v_map, q_map, p, counter,
                      static_cast<const int*>(order), 1, part_acc, part_ml);
  e = launch_pdl(paged_prefill_umma_kernel<D, RK, RV, true>, dim3(ctas), dim3(C::kThreads),
                 C::kSmemBytes, stream, k_map, v_map, q_map, p, counter,
                 static_cast<const int*>(order), parts, part_acc, part_ml);
  if (e != cudaSuccess) return e;
  return launch_pdl(prefill_part_combine_kernel<D>, dim3((p.hq + 3) / 4, p.rows), dim3(128), 0,
                    stream, p, parts, static_cast<const float*>(part_acc),
                    static_cast<const float*>(part_ml));
}

}  // namespace pgd
