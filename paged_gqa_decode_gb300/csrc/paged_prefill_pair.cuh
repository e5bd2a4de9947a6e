// Paged prefill attention at head_dim 128 on pairs of SMs (sm_103a): the
// tcgen05 products of a work item run as cta_group::2 operations over the two
// CTAs of a cluster, and every product spans two pages, 128 keys.
//
// What it computes is the same as the one-SM tcgen05 kernel (Mistral 7B
// Instruct v0.3 model files, src/attention.linnet, prefill_paged; window and
// sinks as GPT-OSS 20B src/attention.linnet, prefill_packed): packed token p
// at position positions[p] of table row rows[p] attends, with each query head
// of its group, over that row's keys at positions
// (positions[p] - window, positions[p]], the head's sink logit in the
// denominator only.
//
// Why pairs: a tcgen05 product of M 128 rows and K 16 runs at two thirds of
// the tensor pipe's rate at N 64 (the one-SM kernel's S products, one 64-key
// page each) and at full rate from N 128 on.  A product over the CTA pair
// takes B split along N between the two CTAs; if each CTA holds one whole
// page, one S product covers two pages (N 128) without any rearrangement of
// the page tiles, and each SM copies every other page.  Each work item then
// has two SMs, which is what pays when a call has at most half as many
// items as SMs and they are too short for the one-SM kernel's key parts.
//
// Work items are the one-SM kernel's: (block of 2 x 128 / G consecutive
// packed tokens, kv head), two query tiles of 128 rows (token, head).  A pair
// of CTAs takes one item at a time: tile t lives in the CTA of cluster rank
// t, one TMEM lane per row.  The pages of each run are taken two at a time;
// for the page pair (2j, 2j + 1) of a run:
//   S = Q K^T   M 256, N 128, K 128: A = each CTA's Q tile (shared memory),
//               B = K split by pages: rank r holds page 2j + r whole
//   O += P V    M 256, N 128, K 128 (64 when the run's last pair has one
//               page): A = each CTA's P (TMEM), B = V split by dims: rank r
//               holds dims 64r .. 64r + 63 of both pages
// both issued by one thread of rank 0; the accumulators land in each CTA's
// own TMEM.  A missing second page's keys are masked (their S columns are
// never used) and its P V steps are not issued.
// Warps of each CTA:
//   0-15  softmax of the CTA's tile: four warpgroups, one thread per query
//         row in each; warpgroup q takes keys 32q .. 32q + 31 of every pair
//         (half q % 2 of page 2j + q / 2) and O columns 32q .. 32q + 31 for
//         the rescale and the store.  Per pair: its scores from TMEM, causal
//         / window mask, its max, the row's max over the pair through shared
//         memory, online softmax in log2 units with a lazy running max
//         (raised only when a score exceeds it by more than 2^8, which then
//         rescales that row of O in TMEM); P written over S as a bf16 head
//         and residual (two products, so P V keeps fp32 accuracy).
//         Warpgroups 0 and 2 also wait for their page's V half and zero its
//         rows outside the run's key range on boundary pages.
//   16    K producer: rank 0 takes items from the counter and hands each
//         index to rank 1 through its shared memory; both build the item's
//         runs (checking the table), zero their own tile's uncovered
//         outputs, and stream their page of each pair into a ring (L2
//         prefetch of their K page and V halves ahead).
//   17    TMEM owner in both; each CTA copies its Q tile per item; rank 0
//         issues the S products, rank 1 forwards its Q tile's landing.
//   18    rank 0: P V issuer; rank 1: forwards each K page's landing and its
//         softmax warps' P signal (one stream each, in pair order, polled
//         in turn) to rank 0's barriers.
//   19    V producer: the CTA's V halves of both pages of each pair.
// Signals between the CTAs are single remote arrivals by that forwarding
// thread (a cluster-scope arrival costs about a thousand cycles, too much
// for the softmax warps' own path).  Completions of pair products are
// committed to the barriers of both CTAs at once (multicast).  Every wait is
// bounded; a CTA that gives up tells the other, both drain their copies and
// products, and the pair frees its TMEM together.
#pragma once

#include "paged_prefill_umma.cuh"

namespace pgd {

template <int RK, int RV, int SB>
struct PairPrefillCfg {
  static constexpr int D = 128;
  static constexpr int kRows = 128;  // query rows of the CTA's tile (TMEM lanes)
  static constexpr int kSoftmaxThreads = 512;
  static constexpr int kKWarp = 16;
  static constexpr int kSWarp = 17;
  static constexpr int kPvWarp = 18;
  static constexpr int kVWarp = 19;
  static constexpr int kThreads = 640;
  static constexpr int kKBytes = kPage * D * 2;       // one page: two 8 KB boxes
  static constexpr int kVHalfBytes = kPage * 64 * 2;  // 64 keys x 64 dims: one box
  static constexpr int kVBytes = 2 * kVHalfBytes;     // both pages of a pair
  static constexpr int kVOff = RK * kKBytes;
  static constexpr int kQOff = kVOff + RV * kVBytes;
  static constexpr int kQBoxBytes = kRows * 128;  // 128 rows x 64 values
  static constexpr int kQTileBytes = kRows * D * 2;
  static constexpr int kBarOff = kQOff + kQTileBytes;
  static constexpr int kSCols = 2 * kPage;  // S / P columns of a pair
  static constexpr int kNumBars = 2 * RK + 2 * RV + 4 * SB + 14;
  static constexpr int kSmemBytes = 1024 + kBarOff + kNumBars * 8;
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kOCol = 0, kSCol = D;
  static constexpr uint32_t kIdescS = umma_idesc_bf16(256, kSCols, 0, 0);
  static constexpr uint32_t kIdescPV = umma_idesc_bf16(256, D, 0, 1);
  static_assert(kSCol + SB * kSCols <= kTmemCols, "TMEM columns");
  static_assert(kSmemBytes + 20 * 1024 <= 227 * 1024, "shared memory (dynamic + static)");
};

// Pair walk of an item's runs: c.pg is the first page of the current pair.
__device__ __forceinline__ bool item_advance_pair(const PrefillItem& it, int window,
                                                  ItemCursor& c) {
  c.pg += 2;
  if (c.pg <= c.last) return true;
  return item_next_run(it, window, c);
}

__device__ __forceinline__ int item_pairs(const PrefillItem& it, int window) {
  int n = 0;
  ItemCursor cc{-1, 0, -1, -1, 0, 0};
  for (bool more = item_next_run(it, window, cc); more; more = item_next_run(it, window, cc))
    n += (cc.last - cc.pg + 2) / 2;
  return n;
}

template <int RK, int RV, int SB>
__global__ void __cluster_dims__(2, 1, 1)
    __launch_bounds__(PairPrefillCfg<RK, RV, SB>::kThreads, 1)
        paged_prefill_pair_kernel(const __grid_constant__ CUtensorMap k_map,
                                  const __grid_constant__ CUtensorMap v_map,
                                  const __grid_constant__ CUtensorMap q_map, const DecodeParams p,
                                  int* item_counter, const int* block_order) {
  using C = PairPrefillCfg<RK, RV, SB>;
  constexpr int D = C::D;
  const int G = p.group;
  const int T = C::kRows / G;  // tokens per tile
  const int tokens = 2 * T;
  const int n_blocks = (p.rows + tokens - 1) / tokens;
  const int n_items = n_blocks * p.hkv;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const uint32_t rank = cluster_ctarank();
  const bool lead = rank == 0;

  extern __shared__ unsigned char smem_raw[];
  unsigned char* base = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  unsigned char* k_slots = base;
  unsigned char* v_slots = base + C::kVOff;
  unsigned char* q_smem = base + C::kQOff;
  uint64_t* k_full = reinterpret_cast<uint64_t*>(base + C::kBarOff);  // rank 0: both pages
  uint64_t* k_empty = k_full + RK;      // S of the pair done (multicast commit)
  uint64_t* v_full = k_empty + RK;      // this CTA's V halves of the pair landed
  uint64_t* v_empty = v_full + RV;      // P V of the pair done (multicast commit)
  uint64_t* s_full = v_empty + RV;      // [buffer] S in TMEM (multicast commit)
  uint64_t* p_full = s_full + SB;       // [buffer] rank 0: both CTAs' P (and V) ready
  uint64_t* p_peer = p_full + SB;       // [buffer] rank 1: its softmax warps' P ready
  uint64_t* o_done = p_peer + SB;       // [buffer] P V of the pair done (multicast commit)
  uint64_t* item_ready = o_done + SB;   // [item % 2] descriptor written
  uint64_t* item_free = item_ready + 2; // [item % 2] descriptor consumed by every role
  uint64_t* fin = item_free + 2;        // rank 0: [issuer] every product it issued done
  uint64_t* q_full = fin + 2;           // rank 0: both Q tiles landed; rank 1: its own
  uint64_t* q_free = q_full + 1;        // the item's S products done (multicast commit)
  uint64_t* j_ready = q_free + 1;       // rank 1: [item % 2] the item index written
  uint64_t* j_free = j_ready + 2;       // rank 0: [item % 2] rank 1 has read the index
  __shared__ PrefillItem items[2];
  __shared__ int y_ring[2][2][64];       // [K, V producer][page of the pair] tile rows
  __shared__ float xval[2][4][C::kRows];  // [slot][quarter][row]: values exchanged at the named barrier
  __shared__ volatile int abort_flag;
  __shared__ uint32_t tmem_slot;
  __shared__ volatile int j_slot[2];
  __shared__ volatile int pairs_total;  // rank 1: pairs streamed in all (-1: not yet known)

  if (tid == 0) {
    for (int s = 0; s < RK; ++s) {
      mbar_init(&k_full[s], lead ? 2 : 1);  // rank 0: its copy + rank 1's forwarded landing
      mbar_init(&k_empty[s], 1);
    }
    for (int s = 0; s < RV; ++s) {
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    for (int b = 0; b < SB; ++b) {
      mbar_init(&s_full[b], 1);
      mbar_init(&p_full[b], 16 + 1);  // rank 0's softmax warps + rank 1's forwarded signal
      mbar_init(&p_peer[b], 16);
      mbar_init(&o_done[b], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&item_ready[b], 1);
      // softmax threads + S issuer, P V issuer, V producer (rank 0); + Q copier,
      // V producer (rank 1)
      mbar_init(&item_free[b], C::kSoftmaxThreads + (lead ? 3 : 2));
      mbar_init(&j_ready[b], 1);
      mbar_init(&j_free[b], 1);
    }
    mbar_init(&fin[0], 1);
    mbar_init(&fin[1], 1);
    mbar_init(q_full, lead ? 2 : 1);
    mbar_init(q_free, 1);
    mbar_init_fence();
    abort_flag = 0;
    pairs_total = -1;
  }
  {
    // rows past T * G of the Q tile hold no token: zero them once (the
    // per-item copies fill rows 0 .. T * G - 1 only)
    const int filled = T * G;
    for (int e = tid; e < 2 * (C::kRows - filled) * 8; e += C::kThreads) {
      const int ch = e & 7, r = filled + (e >> 3) % (C::kRows - filled);
      const int bx = (e >> 3) / (C::kRows - filled);
      *reinterpret_cast<uint4*>(q_smem + bx * C::kQBoxBytes + r * 128 + ch * 16) =
          make_uint4(0u, 0u, 0u, 0u);
    }
    fence_proxy_async_shared();
  }
  if (warp == C::kSWarp) tmem_alloc_pair(&tmem_slot, C::kTmemCols);
  tc_fence_before_sync();
  // both CTAs' barriers are initialised and the pair's TMEM allocated before
  // either CTA signals the other
  cluster_sync_all();
  tc_fence_after_sync();
  const uint32_t tmem = tmem_slot;
  // the set-up above touches only this CTA's shared memory and TMEM, so it
  // overlaps the kernel before; everything from here may read its writes
  pdl_wait();
  pdl_allow_dependents();
  const uint32_t peer_abort = cluster_map(smem_addr(const_cast<int*>(&abort_flag)), rank ^ 1u);
  // Bounded wait that also gives up when either CTA has; a CTA that gives up
  // tells the other.  `remote`: the phase is completed by an arrival from
  // the other CTA, so the acquire covers the cluster.
  auto wait_impl = [&](uint64_t* bar, uint32_t parity, bool remote) {
    auto test = [&]() {
      return remote ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity);
    };
    if (test()) return true;
    const unsigned long long t0 = global_ns();
    for (uint32_t it = 1;; ++it) {
      if (test()) return true;
      if ((it & 63u) == 0u) {
        if (abort_flag) return false;
        if (global_ns() - t0 > kWaitLimitNs) {
          record_error(p.err, PGD_EDEVICE_TIMEOUT);
          abort_flag = 1;
          st_cluster_u32(peer_abort, 1u);
          return false;
        }
      }
    }
  };
  auto wait = [&](uint64_t* bar, uint32_t parity) { return wait_impl(bar, parity, false); };
  auto wait_remote = [&](uint64_t* bar, uint32_t parity) { return wait_impl(bar, parity, true); };
  auto all_ok = [&](bool v) { return __all_sync(0xffffffffu, v); };
  auto to_lead = [&](uint64_t* bar) { return cluster_map(smem_addr(bar), 0); };

  // Streams this CTA's share of the page pairs of item `it` into one ring,
  // pair number i onwards (whole warp): the tile rows of both pages of the
  // next pairs are looked up by the lanes into `ring`; lane 0 waits for each
  // slot and issues the copies -- K: page 2j + rank whole (none for a pair
  // without that page: the slot's barrier is then arrived without bytes);
  // V: the CTA's 64-wide half of each page.  With `prefetch` the K page and
  // V halves are pulled into L2 ahead.
  auto stream_item = [&](const PrefillItem& it, int kvh, int (*ring)[64], int& i,
                         bool is_k) -> bool {
    const int i_end = i + item_pairs(it, p.window);
    ItemCursor fc{-1, 0, -1, -1, 0, 0};
    bool f_more = item_next_run(it, p.window, fc);
    int i_fetch = i, ip = i;
    for (; i < i_end; ++i) {
      while (f_more && i_fetch < i + 16) {
        const int n = min(32, (fc.last - fc.pg + 2) / 2);  // pairs left in this run
        if (lane < n) {
          const int pg0 = fc.pg + 2 * lane;
          const int page0 = page_of(p.table, fc.row, pg0, p.maxp);
          ring[0][(i_fetch + lane) & 63] =
              (int)tile_first_row(p.layout, page0, kvh, p.hkv, p.num_pages, p.maxp);
          int y1 = -1;
          if (pg0 + 1 <= fc.last) {
            const int page1 = page_of(p.table, fc.row, pg0 + 1, p.maxp);
            y1 = (int)tile_first_row(p.layout, page1, kvh, p.hkv, p.num_pages, p.maxp);
          }
          ring[1][(i_fetch + lane) & 63] = y1;
        }
        __syncwarp();
        i_fetch += n;
        fc.pg += 2 * (n - 1);
        f_more = item_advance_pair(it, p.window, fc);
      }
      if (is_k && lane == 0) {
        for (; ip < min(i + kL2PrefetchPages / 2, i_fetch); ++ip) {
          const int ym = ring[rank][ip & 63];
          if (ym >= 0) tma_prefetch_l2_3d(&k_map, 0, ym, 0);
          for (int h = 0; h < 2; ++h)
            if (ring[h][ip & 63] >= 0)
              tma_prefetch_l2_2d(&v_map, 64 * (int)rank, ring[h][ip & 63]);
        }
      }
      if (is_k) {
        const int s = i % RK;
        if (i >= RK && !all_ok(wait(&k_empty[s], ((i / RK) - 1) & 1))) return false;
        if (lane == 0) {
          const int y = ring[rank][i & 63];
          if (y >= 0) {
            mbar_arrive_expect_tx(&k_full[s], C::kKBytes);
            tma_load_3d(k_slots + s * C::kKBytes, &k_map, 0, y, 0, &k_full[s]);
          } else {
            mbar_arrive(&k_full[s]);
          }
        }
      } else {
        const int s = i % RV;
        if (i >= RV && !all_ok(wait(&v_empty[s], ((i / RV) - 1) & 1))) return false;
        if (lane == 0) {
          const int y0 = ring[0][i & 63], y1 = ring[1][i & 63];
          mbar_arrive_expect_tx(&v_full[s], y1 >= 0 ? C::kVBytes : C::kVHalfBytes);
          unsigned char* dst = v_slots + s * C::kVBytes;
          tma_load_2d(dst, &v_map, 64 * (int)rank, y0, &v_full[s]);
          if (y1 >= 0) tma_load_2d(dst + C::kVHalfBytes, &v_map, 64 * (int)rank, y1, &v_full[s]);
        }
      }
    }
    return true;
  };

  if (warp == C::kKWarp) {
    // ------------------------------------------------------------ K producer
    if (lane == 0) {
      prefetch_tensormap(&k_map);
      prefetch_tensormap(&v_map);
    }
    int ik = 0;  // K pairs streamed (all items)
    bool ok = true;
    for (int seq = 0; ok; ++seq) {
      const int d = seq & 1;
      PrefillItem& it = items[d];
      int j = 0;
      if (lead) {
        if (lane == 0) j = atomicAdd(item_counter, 1);
        j = __shfl_sync(0xffffffffu, j, 0);
        // rank 1 has read the index this slot held two items ago
        if (seq >= 2 && !all_ok(wait_remote(&j_free[d], ((seq >> 1) - 1) & 1))) break;
        if (lane == 0) {
          st_cluster_u32(cluster_map(smem_addr(const_cast<int*>(&j_slot[d])), 1), (uint32_t)j);
          mbar_arrive_cluster(cluster_map(smem_addr(&j_ready[d]), 1));
        }
      } else {
        if (!all_ok(wait_remote(&j_ready[d], (seq >> 1) & 1))) break;
        j = j_slot[d];
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(to_lead(&j_free[d]));
      }
      // the descriptor slot holds item seq - 2 until every role is done
      if (seq >= 2 && !all_ok(wait(&item_free[d], ((seq >> 1) - 1) & 1))) break;
      if (j >= n_items) {
        if (lane == 0) {
          it.valid = 0;
          mbar_arrive(&item_ready[d]);
          pairs_total = ik;  // the forwarding thread's streams end here
        }
        break;
      }
      const int blk = block_order ? block_order[j / p.hkv] : n_blocks - 1 - j / p.hkv;
      const int kvh = j % p.hkv;
      const int t_begin = blk * tokens, t_end = min(t_begin + tokens, p.rows);
      const int h0 = kvh * G;
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
        it.part = 0;  // every page of the item
        it.parts = 1;
      }
      __syncwarp();
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
      __syncwarp();
      // outputs of this CTA's tokens that no pass covers (inactive or bad run)
      for (int r = 0; r < it.runs; ++r) {
        const int rs = r == 0 ? 0 : it.run_end[r - 1], re = it.run_end[r];
        if (it.tok_row[rs] >= 0 && !it.run_bad[r]) continue;
        for (int e = lane; e < (re - rs) * G * (D / 8); e += 32) {
          const int tl = rs + e / (G * (D / 8));
          if (tl / T != (int)rank || t_begin + tl >= t_end) continue;
          const int g = (e / (D / 8)) % G, c = e % (D / 8);
          reinterpret_cast<uint4*>(p.out + ((size_t)(t_begin + tl) * p.hq + h0 + g) * D)[c] =
              make_uint4(0u, 0u, 0u, 0u);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&item_ready[d]);
      ok = stream_item(it, kvh, y_ring[0], ik, true);
    }
    // drain: this CTA's copies still in flight land before it exits
    if (lane == 0)
      for (int j = max(0, ik - RK); j < ik; ++j)
        mbar_wait_bounded(&k_full[j % RK], (j / RK) & 1, p.err);
  } else if (warp == C::kVWarp) {
    // ------------------------------------------------------------ V producer
    int iv = 0;
    for (int seq = 0;; ++seq) {
      const int d = seq & 1;
      if (!all_ok(wait(&item_ready[d], (seq >> 1) & 1))) break;
      const PrefillItem& it = items[d];
      if (!it.valid) break;
      if (!stream_item(it, it.kvh, y_ring[1], iv, false)) break;
      if (lane == 0) mbar_arrive(&item_free[d]);
    }
    if (lane == 0)
      for (int j = max(0, iv - RV); j < iv; ++j)
        mbar_wait_bounded(&v_full[j % RV], (j / RV) & 1, p.err);
  } else if (warp == C::kSWarp) {
    // ------------------------------------------------ Q copies and S issuer
    if (lane == 0) {
      const uint32_t k_addr = smem_addr(k_slots);
      const uint64_t qd = umma_desc_sw128(smem_addr(q_smem), 16, 1024);
      int i = 0;  // pair index over all items
      bool issued = false, ok = true;
      bool q_pending = false;
      int q_phase = 0;
      for (int seq = 0; ok; ++seq) {
        const int d = seq & 1;
        if (!wait(&item_ready[d], (seq >> 1) & 1)) break;
        const PrefillItem& it = items[d];
        if (!it.valid) break;
        // this CTA's Q tile, once the previous item's S products (which read
        // the same shared memory in both CTAs) are done; rank 1 forwards the
        // landing to rank 0, whose barrier then covers both tiles
        if (seq > 0 && !wait(q_free, (seq - 1) & 1)) break;
        mbar_arrive_expect_tx(q_full, 2 * T * G * 128);
        for (int bx = 0; bx < 2; ++bx)
          tma_load_3d(q_smem + bx * C::kQBoxBytes, &q_map, 64 * bx, it.kvh * G,
                      it.t_begin + (int)rank * T, q_full);
        q_pending = true;
        q_phase = seq;
        if (!lead) {
          if (!wait(q_full, seq & 1)) break;
          q_pending = false;
          mbar_arrive_cluster(to_lead(q_full));
          mbar_arrive(&item_free[d]);
          continue;
        }
        if (!wait_remote(q_full, seq & 1)) break;
        q_pending = false;
        const int n = item_pairs(it, p.window);
        for (int k = 0; k < n; ++k, ++i) {
          if (!wait_remote(&k_full[i % RK], (i / RK) & 1)) {
            ok = false;
            break;
          }
          const int b = i % SB;
          // the buffer holds P of pair i - SB until P V has read it
          if (i >= SB && !wait(&o_done[b], ((i / SB) - 1) & 1)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint64_t kd = umma_desc_sw128(k_addr + (i % RK) * C::kKBytes, 16, 1024);
          const uint32_t sb = tmem + C::kSCol + b * C::kSCols;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            umma_pair_bf16(sb, umma_desc_advance(qd, (kk >> 2) * C::kQBoxBytes + (kk & 3) * 32),
                           umma_desc_advance(kd, (kk >> 2) * kBoxBytes + (kk & 3) * 32),
                           C::kIdescS, kk > 0);
          umma_pair_commit(&s_full[b], 3);
          umma_pair_commit(&k_empty[i % RK], 3);
          issued = true;
        }
        if (ok) umma_pair_commit(q_free, 3);
        if (ok) mbar_arrive(&item_free[d]);
      }
      if (issued) {
        umma_pair_commit(fin, 1);
        mbar_wait_bounded(fin, 0, p.err);
      }
      if (q_pending) mbar_wait_bounded(q_full, q_phase & 1, p.err);
    }
  } else if (warp == C::kPvWarp) {
    if (lead) {
      // ---------------------------------------------------------- P V issuer
      if (lane == 0) {
        const uint32_t v_addr = smem_addr(v_slots);
        int i = 0;
        bool issued = false, ok = true;
        for (int seq = 0; ok; ++seq) {
          const int d = seq & 1;
          if (!wait(&item_ready[d], (seq >> 1) & 1)) break;
          const PrefillItem& it = items[d];
          if (!it.valid) break;
          ItemCursor cur{-1, 0, -1, -1, 0, 0};
          bool first = true;  // O restarts with each item
          for (bool more = item_next_run(it, p.window, cur); more && ok;
               more = item_advance_pair(it, p.window, cur), ++i) {
            const int b = i % SB;
            // both CTAs' P of the pair written and V halves landed (and zeroed)
            if (!wait_remote(&p_full[b], (i / SB) & 1)) {
              ok = false;
              break;
            }
            tc_fence_after_sync();
            const uint64_t vd = umma_desc_sw128(v_addr + (i % RV) * C::kVBytes, kBoxBytes, 1024);
            const uint32_t pb = tmem + C::kSCol + b * C::kSCols;
            const uint32_t od = tmem + C::kOCol;
            // keys 16 kk .. 16 kk + 15 of the pair: chunk kk / 2 of the P
            // columns, half kk % 2 of its 16 head (then residual) columns; V
            // rows from page kk / 4's half
            const bool two = cur.pg + 1 <= cur.last;
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              if (kk < 4 || two)
                umma_pair_bf16_tmem_a(
                    od, pb + 32 * (kk >> 1) + 8 * (kk & 1),
                    umma_desc_advance(vd, (kk >> 2) * C::kVHalfBytes + (kk & 3) * 2048),
                    C::kIdescPV, !(first && kk == 0));
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              if (kk < 4 || two)
                umma_pair_bf16_tmem_a(
                    od, pb + 32 * (kk >> 1) + 16 + 8 * (kk & 1),
                    umma_desc_advance(vd, (kk >> 2) * C::kVHalfBytes + (kk & 3) * 2048),
                    C::kIdescPV, true);
            umma_pair_commit(&o_done[b], 3);
            umma_pair_commit(&v_empty[i % RV], 3);
            first = false;
            issued = true;
          }
          if (ok) mbar_arrive(&item_free[d]);
        }
        if (issued) {
          umma_pair_commit(fin + 1, 1);
          mbar_wait_bounded(fin + 1, 0, p.err);
        }
      }
    } else if (lane == 0) {
      // ------------------------ rank 1: K landings and P signals to rank 0
      // Two streams in pair order, each forwarded as its next phase
      // completes: K landing i (the K producer streams ahead) and P signal
      // i (the softmax warps follow).  They end at the number of pairs the
      // K producer streamed in all, known once it has run out of items.
      int ik = 0, ip = 0;
      unsigned long long t0 = global_ns();
      for (uint32_t it = 1;; ++it) {
        bool moved = false;
        const int total = pairs_total;
        if ((total < 0 || ik < total) && mbar_test(&k_full[ik % RK], (ik / RK) & 1)) {
          mbar_arrive_cluster(to_lead(&k_full[ik % RK]));
          ++ik;
          moved = true;
        }
        if ((total < 0 || ip < total) && ip < ik &&
            mbar_test(&p_peer[ip % SB], (ip / SB) & 1)) {
          mbar_arrive_cluster(to_lead(&p_full[ip % SB]));
          ++ip;
          moved = true;
        }
        if (total >= 0 && ik >= total && ip >= total) break;
        if (moved) {
          t0 = global_ns();
        } else if ((it & 63u) == 0u) {
          if (abort_flag) break;
          if (global_ns() - t0 > kWaitLimitNs) {
            record_error(p.err, PGD_EDEVICE_TIMEOUT);
            abort_flag = 1;
            st_cluster_u32(peer_abort, 1u);
            break;
          }
        }
      }
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int m = tid & 127, qt = tid >> 7;  // row; quarter of the pair's keys
    const int h = qt >> 1;                   // page of the pair the quarter lies in
    constexpr int kKeys = kPage / 2;         // keys of this thread's quarter
    int xn = 0;
    const uint32_t lane_base = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
    const float c = p.q_scale_log2;
    const float cc = c > 0.f ? c : 1.f;
    int i = 0;
    // The four warpgroups exchange values at a named barrier that also ORs
    // a failure flag over them (as in the one-SM kernel), so they leave
    // their loops together.
    bool ok = true, mine = true;
    const int tl = (int)rank * T + m / G, g = m % G;  // token of the block, head of the group
    const bool in_tile = m / G < T;
    uint64_t* p_sig = lead ? p_full : p_peer;
    auto next_item = [&](int seq) -> bool {
      const int d = seq & 1;
      if (!all_ok(wait(&item_ready[d], (seq >> 1) & 1))) {
        mine = false;
        return false;
      }
      return items[d].valid != 0;
    };
    bool have = next_item(0);
    ok = !named_sync_or(1, C::kSoftmaxThreads, !mine);
    for (int seq = 0; ok && have; ++seq) {
      const int d = seq & 1;
      const PrefillItem& it = items[d];
      const int t_begin = it.t_begin, t_end = it.t_end, h0 = it.kvh * G;
      const bool row_ok = in_tile && t_begin + tl < t_end;
      int rs = 0;
      for (int r = 0; r < it.runs && ok; ++r) {
        const int re = it.run_end[r];
        const int row = it.tok_row[rs];
        if (row < 0 || it.run_bad[r]) {
          rs = re;
          continue;
        }
        const bool live = row_ok && tl >= rs && tl < re;
        const int pos = live ? it.tok_pos[tl] : -1;
        const int lo = p.window > 0 ? pos - p.window + 1 : 0;
        const int lo_run = p.window > 0 ? max(it.tok_pos[rs] - p.window + 1, 0) : 0;
        const int pos_last = it.tok_pos[re - 1];
        const int first = lo_run / kPage, last = pos_last / kPage;
        float m_run = -INFINITY;
        float l = 0.f;
        for (int pg2 = first; pg2 <= last; pg2 += 2, ++i) {
          const int b = i % SB;
          const uint32_t scol = C::kSCol + b * C::kSCols;
          const int pg = pg2 + h;  // this quarter's page (past `last`: none)
          if (!all_ok(wait(&s_full[b], (i / SB) & 1))) mine = false;
          tc_fence_after_sync();
          float sv[kKeys];
#pragma unroll
          for (int q = 0; q < kKeys / 16; ++q)
            tmem_ld16(lane_base + scol + kKeys * qt + 16 * q,
                      *reinterpret_cast<float(*)[16]>(&sv[16 * q]));
          tmem_wait_ld();
          if (!(c > 0.f)) {
#pragma unroll
            for (int k = 0; k < kKeys; ++k) sv[k] *= c;
          }
          const int pos0 = pg * kPage;
          const int pos0q = pos0 + kKeys * (qt & 1);  // this quarter's first key
          if (!(live && pg <= last && pos0q >= lo && pos0q + kKeys - 1 <= pos)) {
#pragma unroll
            for (int k = 0; k < kKeys; ++k)
              if (!(live && pg <= last && pos0q + k >= lo && pos0q + k <= pos)) sv[k] = -INFINITY;
          }
          float part[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) part[j] = sv[j];
#pragma unroll
          for (int k = 8; k + 16 <= kKeys; k += 16)
#pragma unroll
            for (int j = 0; j < 8; ++j)
              part[j] = fmax3(part[j], sv[k + 2 * j], sv[k + 2 * j + 1]);
          static_assert((kKeys - 8) % 16 == 8, "the last block holds 8 scores");
#pragma unroll
          for (int j = 0; j < 4; ++j)
            part[j] = fmax3(part[j], sv[kKeys - 8 + 2 * j], sv[kKeys - 7 + 2 * j]);
          const float mxh = fmax3(fmax3(part[0], part[1], part[2]),
                                  fmax3(part[3], part[4], part[5]), fmaxf(part[6], part[7])) *
                            cc;
          float mx;
          {
            const int sl = xn & 1;
            xval[sl][qt][m] = mxh;
            if (named_sync_or(1, C::kSoftmaxThreads, !mine)) {
              ok = false;
              break;
            }
            mx = fmax3(fmaxf(xval[sl][0][m], xval[sl][1][m]), xval[sl][2][m], xval[sl][3][m]);
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
          const float2 cc2 = make_float2(cc, cc), nml2 = make_float2(nml, nml);
          const float2 minus1 = make_float2(-1.f, -1.f);
          float2 sum2[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) sum2[j] = make_float2(0.f, 0.f);
#pragma unroll
          for (int q = 0; q < kKeys / 32; ++q) {
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
            tmem_st16(lane_base + scol + kKeys * qt + 32 * q, hw);
            tmem_st16(lane_base + scol + kKeys * qt + 32 * q + 16, lw);
          }
          const float2 s4 =
              __fadd2_rn(__fadd2_rn(sum2[0], sum2[1]), __fadd2_rn(sum2[2], sum2[3]));
          l += s4.x + s4.y;
          if (__any_sync(0xffffffffu, rose)) {
            // O holds P V up to pair i - 1, which must be done
            const int bp = (i - 1) % SB;
            if (all_ok(wait(&o_done[bp], ((i - 1) / SB) & 1))) {
              tc_fence_after_sync();
#pragma unroll
              for (int j = 0; j < D / 64; ++j) {  // this quarter's O columns
                const int q16 = qt * (D / 64) + j;
                float ov[16];
                tmem_ld16(lane_base + C::kOCol + 16 * q16, ov);
                tmem_wait_ld();
#pragma unroll
                for (int k = 0; k < 16; ++k) ov[k] *= alpha;
                tmem_st16(lane_base + C::kOCol + 16 * q16, ov);
              }
            } else {
              mine = false;
            }
          }
          if ((qt & 1) == 0 && pg <= last) {
            // this page's V half has landed (rank 0's P V issuer learns it
            // from the P signal); rows outside the run's key range on a
            // boundary page -> zero
            const int s = i % RV;
            const bool landed = all_ok(wait(&v_full[s], (i / RV) & 1));
            if (!landed) mine = false;
            const int rlo = max(lo_run - pos0, 0), rhi = min(pos_last - pos0, kPage - 1);
            if (landed && (rlo > 0 || rhi < kPage - 1)) {
              unsigned char* vt = v_slots + s * C::kVBytes + h * C::kVHalfBytes;
              for (int e = m; e < kPage * 8; e += C::kRows) {
                const int k = e >> 3, ch = e & 7;
                if (k < rlo || k > rhi)
                  *reinterpret_cast<uint4*>(vt + k * 128 + ch * 16) = make_uint4(0u, 0u, 0u, 0u);
              }
              fence_proxy_async_shared();
            }
          }
          tmem_wait_st();
          tc_fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive(&p_sig[b]);
        }
        if (!ok) break;

        // end of run: the O row once P V of the last pair is done
        const int il = i - 1;
        if (all_ok(wait(&o_done[il % SB], (il / SB) & 1)))
          tc_fence_after_sync();
        else
          mine = false;
        {
          const int sl = xn & 1;
          xval[sl][qt][m] = l;
          if (named_sync_or(1, C::kSoftmaxThreads, !mine)) {
            ok = false;
            break;
          }
          l = (xval[sl][0][m] + xval[sl][1][m]) + (xval[sl][2][m] + xval[sl][3][m]);
          ++xn;
        }
        const int hh = h0 + g;
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
        for (int j = 0; j < D / 64; ++j) {  // this quarter's output columns
          const int q16 = qt * (D / 64) + j;
          float ov[16];
          tmem_ld16(lane_base + C::kOCol + 16 * q16, ov);
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
      mbar_arrive(&item_free[d]);
      have = next_item(seq + 1);
      ok = !named_sync_or(1, C::kSoftmaxThreads, !mine);
    }
  }

  // ---------------------------------------------------------------- teardown
  // every role of both CTAs is done: no copy, product, commit or signal is
  // still headed for either CTA's shared memory or TMEM
  __syncwarp();
  tc_fence_before_sync();
  cluster_sync_all();
  tc_fence_after_sync();
  if (warp == C::kSWarp) tmem_dealloc_pair(tmem, C::kTmemCols);
}

// `prepared`: the step's write launch has already zeroed the work counter and
// written the block order (prefill_write_kernel).
template <int RK, int RV, int SB>
cudaError_t launch_prefill_pair(const DecodeParams& p, const CUtensorMap& k_map,
                                const CUtensorMap& v_map, const CUtensorMap& q_map, int sm_count,
                                bool prepared, cudaStream_t stream) {
  using C = PairPrefillCfg<RK, RV, SB>;
  auto kernel = paged_prefill_pair_kernel<RK, RV, SB>;
  static std::atomic<int> pairs_on[64];  // clusters of two resident at once, per device (+1)
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  int pairs = sm_count / 2;
  if (dev >= 0 && dev < 64 && pairs_on[dev].load(std::memory_order_acquire) > 0) {
    pairs = pairs_on[dev].load(std::memory_order_acquire) - 1;
  } else {
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * pairs);
    cfg.blockDim = dim3(C::kThreads);
    cfg.dynamicSmemBytes = C::kSmemBytes;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) == cudaSuccess && n > 0 && n < pairs)
      pairs = n;
    (void)cudaGetLastError();
    if (dev >= 0 && dev < 64) pairs_on[dev].store(pairs + 1, std::memory_order_release);
  }
  if (p.rows == 0) return cudaSuccess;
  const int tokens = 2 * (C::kRows / p.group);
  const int n_blocks = (p.rows + tokens - 1) / tokens;
  const int items = n_blocks * p.hkv;
  int* counter = reinterpret_cast<int*>(p.ws_acc);
  int* order = p.window == 0 && n_blocks <= kMaxSortedBlocks ? counter + 4 : nullptr;
  if (prepared)
    e = cudaSuccess;
  else if (order)
    e = launch_pdl(prefill_block_order_kernel<128>, dim3(1), dim3(block_order_threads(n_blocks)),
                   0, stream, p, tokens, n_blocks, counter, order);
  else
    e = cudaMemsetAsync(counter, 0, sizeof(int), stream);
  if (e != cudaSuccess) return e;
  const int grid_pairs = items < pairs ? items : pairs;
  return launch_pdl(kernel, dim3(2 * grid_pairs), dim3(C::kThreads), C::kSmemBytes, stream,
                    k_map, v_map, q_map, p, counter, static_cast<const int*>(order));
}

}  // namespace pgd
