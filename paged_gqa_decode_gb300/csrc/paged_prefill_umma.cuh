// Paged prefill attention on the 5th-generation tensor cores (tcgen05 UMMA
// with TMEM accumulators), sm_103a.
//
// What it computes is the same as the tiled prefill kernel (Mistral 7B
// Instruct v0.3 model files, src/attention.linnet, prefill_paged; window and
// sinks as GPT-OSS 20B src/attention.linnet, prefill_packed): packed token p at
// position positions[p] of table row rows[p] attends, with each query head of
// its group, over that row's keys at positions (positions[p] - window,
// positions[p]], the head's sink logit in the denominator only.
//
// Decomposition: one CTA per (block of 128 / G consecutive packed tokens, kv
// head), two CTAs per SM.  Its 128 query rows are (token, head of the group)
// pairs, row m = token * G + head, one per TMEM lane.  Tokens split into runs
// (same table row, consecutive positions); each run is one pass over the pages
// of the union of its tokens' key ranges.  Six warps:
//   warp 4      TMA producer: K and V tiles (64 x D bf16, 128-byte swizzle) of
//               each page into two rings of shared slots, and pages pulled into
//               L2 several pages ahead of their loads.
//   warp 5      MMA issuer (one thread) and TMEM owner, per page i:
//                 S_i  = Q K_i^T    M 128, N 64, K D   (Q from TMEM, K shared)
//                 O   += P_i V_i    M 128, N D,  K 64  (P from TMEM, V shared)
//               in the order S_0, PV_0, S_1, PV_1, ...
//   warps 0-3   softmax, one thread per query row (= TMEM lane): the S row
//               from TMEM, causal and window mask, online softmax in log2 units
//               with a lazy reference max (raised only when a score exceeds it
//               by more than 2^8, which then rescales that row of O in TMEM),
//               P written over S as a bf16 head and residual (two MMAs, so P V
//               keeps fp32 accuracy); at the end of a run the O row is
//               normalised with the sink and stored.
// Per CTA the page chain is serial (softmax, then P V, then the next S); the
// second CTA on the SM runs its softmax while this one's products run, and
// hides its setup and first loads.
// TMEM (256 columns): S / P [0, 64) (P per chunk of 32 keys: the bf16 head in
// the chunk's first 16 columns, the residual in the next 16, as packed pairs),
// Q [64, 64 + D / 2) as packed pairs, O [128, 128 + D).
// V rows outside the run's key range on its boundary pages are zeroed in
// shared memory before the product.  Every wait is bounded; a timeout records
// PGD_EDEVICE_TIMEOUT, stops all roles, drains in-flight copies and MMAs and
// frees TMEM before the CTA exits.
#pragma once

#include "paged_decode.cuh"
#include "pgd_umma.cuh"

namespace pgd {

template <int D, int RING>
struct UmmaPrefillCfg {
  static constexpr int kRows = 128;  // query rows per CTA (TMEM lanes)
  static constexpr int kSoftmaxThreads = 128;
  static constexpr int kProducerWarp = 4;
  static constexpr int kMmaWarp = 5;
  static constexpr int kThreads = 192;
  static constexpr int kBoxes = D / 64;
  static constexpr int kTileBytes = kPage * D * 2;  // one K or V slot (one page)
  static constexpr int kVOff = RING * kTileBytes;   // K slots at 0, V slots here
  static constexpr int kBarOff = 2 * RING * kTileBytes;
  static constexpr int kNumBars = 4 * RING + 4;
  static constexpr int kSmemBytes = 1024 + kBarOff + kNumBars * 8;
  static constexpr uint32_t kTmemCols = 256;
  static constexpr uint32_t kQCol = 64, kOCol = 128;
  static constexpr uint32_t kIdescS = umma_idesc_bf16(128, kPage, 0, 0);
  static constexpr uint32_t kIdescPV = umma_idesc_bf16(128, D, 0, 1);
  static_assert(D == 64 || D == 128, "head_dim");
  // two CTAs per SM (each with its static arrays and the 1 KB the SM reserves)
  static_assert(2 * (kSmemBytes + 4 * 1024) <= 228 * 1024, "shared memory");
};

// Reference-max slack in log2 units: P values stay below 2^8.
constexpr float kLazyRescaleLog2 = 8.0f;

// How far ahead of its load the producer pulls a page into L2.
constexpr int kL2PrefetchPages = 8;

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

template <int D, int RING>
__global__ void __launch_bounds__(192, 2)
    paged_prefill_umma_kernel(const __grid_constant__ CUtensorMap k_map,
                              const __grid_constant__ CUtensorMap v_map, const DecodeParams p) {
  using C = UmmaPrefillCfg<D, RING>;
  pdl_wait();
  pdl_allow_dependents();
  const int kvh = blockIdx.y;
  const int G = p.group;
  const int tokens = C::kRows / G;
  const int t_begin = blockIdx.x * tokens;
  const int t_end = min(t_begin + tokens, p.rows);
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int h0 = kvh * G;

  extern __shared__ unsigned char smem_raw[];
  unsigned char* base = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  unsigned char* k_slots = base;
  unsigned char* v_slots = base + C::kVOff;
  uint64_t* k_full = reinterpret_cast<uint64_t*>(base + C::kBarOff);  // TMA landed
  uint64_t* k_empty = k_full + RING;  // S of the page done (MMA commit)
  uint64_t* v_full = k_empty + RING;
  uint64_t* v_empty = v_full + RING;  // P V of the page done (MMA commit)
  uint64_t* s_full = v_empty + RING;  // S in TMEM (MMA commit; covers the previous P V)
  uint64_t* p_full = s_full + 1;      // P in TMEM, boundary V rows zeroed (softmax)
  uint64_t* o_done = p_full + 1;      // P V done (MMA commit)
  uint64_t* fin = o_done + 1;         // every MMA of the CTA done
  __shared__ int run_end[C::kRows + 1];
  __shared__ int tok_row[C::kRows], tok_pos[C::kRows], tok_run[C::kRows];
  __shared__ int run_bad[C::kRows];
  __shared__ int runs;
  __shared__ volatile int abort_flag;
  __shared__ uint32_t tmem_slot;

  // ---------------------------------------------------------------- setup
  if (tid < tokens) {
    const int t = t_begin + tid;
    int row = -1, pos = -1;
    if (t < t_end) {
      row = p.row_of ? p.row_of[t] : t;
      pos = p.positions[t];
      const bool bad = row < 0 || row >= p.table_rows || (pos >= 0 && pos / kPage >= p.maxp);
      if (bad) record_error(p.err, PGD_EDEVICE_BOUNDS);
      if (bad || pos < 0) row = -1;
    }
    tok_row[tid] = row;
    tok_pos[tid] = pos;
  }
  __syncthreads();
  if (tid == 0) {
    int r = 0;
    for (int i = 1; i <= tokens; ++i) {
      tok_run[i - 1] = r;
      const bool brk = i == tokens || tok_row[i] != tok_row[i - 1] ||
                       tok_pos[i] != tok_pos[i - 1] + 1 || tok_row[i] < 0 || tok_row[i - 1] < 0;
      if (brk) run_end[r++] = i;
    }
    runs = r;
    for (int k = 0; k < r; ++k) run_bad[k] = 0;
    for (int s = 0; s < RING; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    mbar_init(s_full, 1);
    mbar_init(p_full, C::kSoftmaxThreads);
    mbar_init(o_done, 1);
    mbar_init(fin, 1);
    mbar_init_fence();
    abort_flag = 0;
  }
  __syncthreads();
  {
    // A table entry outside the pool marks its run bad (zero outputs,
    // PGD_EDEVICE_BOUNDS); checked before any copy is issued.
    int rs = 0;
    for (int r = 0; r < runs; ++r) {
      const int re = run_end[r];
      const int row = tok_row[rs];
      if (row >= 0) {
        const int lo = p.window > 0 ? max(tok_pos[rs] - p.window + 1, 0) : 0;
        const int first = lo / kPage, last = tok_pos[re - 1] / kPage;
        for (int pg = first + tid; pg <= last; pg += C::kThreads) {
          const int page = page_of(p.table, row, pg, p.maxp);
          if (page < 0 || page >= p.num_pages) run_bad[r] = 1;
        }
      }
      rs = re;
    }
  }
  if (warp == C::kMmaWarp) {
    __syncwarp();
    tmem_alloc(&tmem_slot, C::kTmemCols);
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = tmem_slot;
  // Q rows into TMEM as packed bf16 pairs (the A operand of S); rows of no
  // token are zero.
  if (tid < C::kSoftmaxThreads) {
    const int m = tid, tl = m / G, g = m % G;
    const bool ok = tl < tokens && t_begin + tl < t_end && tok_row[tl] >= 0;
    const uint32_t lane_base = tmem + ((uint32_t)(32 * warp) << 16);
#pragma unroll
    for (int c16 = 0; c16 < D / 32; ++c16) {
      uint32_t w[16];
      if (ok) {
        const uint4* src = reinterpret_cast<const uint4*>(
            p.q + ((size_t)(t_begin + tl) * p.hq + h0 + g) * D + 32 * c16);
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          const uint4 x = src[v];
          w[4 * v] = x.x;
          w[4 * v + 1] = x.y;
          w[4 * v + 2] = x.z;
          w[4 * v + 3] = x.w;
        }
      } else {
#pragma unroll
        for (int v = 0; v < 16; ++v) w[v] = 0u;
      }
      tmem_st16(lane_base + C::kQCol + 16 * c16, w);
    }
    tmem_wait_st();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (tid == 0)
    for (int r = 0; r < runs; ++r)
      if (run_bad[r]) record_error(p.err, PGD_EDEVICE_BOUNDS);
  // Zero the outputs of tokens that no pass covers (inactive or bad run).
  for (int e = tid; e < tokens * G * (D / 8); e += C::kThreads) {
    const int tl = e / (G * (D / 8));
    if (t_begin + tl < t_end && (tok_row[tl] < 0 || run_bad[tok_run[tl]])) {
      const int g = (e / (D / 8)) % G, c = e % (D / 8);
      reinterpret_cast<uint4*>(p.out + ((size_t)(t_begin + tl) * p.hq + h0 + g) * D)[c] =
          make_uint4(0u, 0u, 0u, 0u);
    }
  }

  // Page sequence of the CTA's passes: run by run (inactive and bad runs
  // skipped), pages first..last of each.  Every role walks it in this order.
  struct Cursor {
    int r, pg, last, row;
  };
  auto next_run = [&](Cursor& c) {
    for (++c.r; c.r < runs; ++c.r) {
      const int rs = c.r == 0 ? 0 : run_end[c.r - 1];
      c.row = tok_row[rs];
      if (c.row < 0 || run_bad[c.r]) continue;
      const int lo = p.window > 0 ? max(tok_pos[rs] - p.window + 1, 0) : 0;
      c.pg = lo / kPage;
      c.last = tok_pos[run_end[c.r] - 1] / kPage;
      return;
    }
  };
  auto advance = [&](Cursor& c) {
    if (++c.pg > c.last) next_run(c);
  };

  if (warp == C::kProducerWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tensormap(&k_map);
      prefetch_tensormap(&v_map);
      auto tile_y = [&](const Cursor& c) {
        const int page = page_of(p.table, c.row, c.pg, p.maxp);
        return (int)tile_first_row(p.layout, page, kvh, p.hkv, p.num_pages, p.maxp);
      };
      Cursor kc{-1, 0, -1, -1}, vc{-1, 0, -1, -1}, pc{-1, 0, -1, -1};
      next_run(kc);
      next_run(vc);
      next_run(pc);
      int ik = 0, iv = 0, ip = 0;  // K loads, V loads, L2 prefetches issued
      // V of page j is issued before K of page j + 1: its slot frees (P V of
      // page j - RING) before K's does (S of page j + 1 - RING, issued after
      // that P V), so each wait below is for the next completion in the MMA's
      // order.
      while ((kc.r < runs || vc.r < runs) && !abort_flag) {
        if (kc.r < runs && ik <= iv) {
          // The token blocks of a request reach each page together; pulling
          // pages into L2 ahead of their loads keeps DRAM latency off the rings.
          for (; pc.r < runs && ip < ik + kL2PrefetchPages; advance(pc), ++ip) {
            const int y = tile_y(pc);
#pragma unroll
            for (int bx = 0; bx < C::kBoxes; ++bx) {
              tma_prefetch_l2_2d(&k_map, bx * 64, y);
              tma_prefetch_l2_2d(&v_map, bx * 64, y);
            }
          }
          const int s = ik % RING;
          if (ik >= RING &&
              !mbar_wait_abortable(&k_empty[s], ((ik / RING) - 1) & 1, p.err, &abort_flag))
            break;
          const int y = tile_y(kc);
          mbar_arrive_expect_tx(&k_full[s], C::kTileBytes);
#pragma unroll
          for (int bx = 0; bx < C::kBoxes; ++bx)
            tma_load_2d(k_slots + s * C::kTileBytes + bx * kBoxBytes, &k_map, bx * 64, y,
                        &k_full[s]);
          advance(kc);
          ++ik;
        } else {
          const int s = iv % RING;
          if (iv >= RING &&
              !mbar_wait_abortable(&v_empty[s], ((iv / RING) - 1) & 1, p.err, &abort_flag))
            break;
          const int y = tile_y(vc);
          mbar_arrive_expect_tx(&v_full[s], C::kTileBytes);
#pragma unroll
          for (int bx = 0; bx < C::kBoxes; ++bx)
            tma_load_2d(v_slots + s * C::kTileBytes + bx * kBoxBytes, &v_map, bx * 64, y,
                        &v_full[s]);
          advance(vc);
          ++iv;
        }
      }
      // drain: the copies still in flight land before the CTA exits
      for (int j = max(0, ik - RING); j < ik; ++j)
        mbar_wait_bounded(&k_full[j % RING], (j / RING) & 1, p.err);
      for (int j = max(0, iv - RING); j < iv; ++j)
        mbar_wait_bounded(&v_full[j % RING], (j / RING) & 1, p.err);
    }
  } else if (warp == C::kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t k_addr = smem_addr(k_slots), v_addr = smem_addr(v_slots);
      auto wait = [&](uint64_t* bar, uint32_t parity) {
        return mbar_wait_abortable(bar, parity, p.err, &abort_flag);
      };
      // S_i overwrites the P that P V_{i-1} reads: the tensor core executes
      // one thread's MMAs in issue order, reading an MMA's operands before
      // later MMAs write, so S_i is queued right behind it; its commit tells
      // the softmax that P V_{i-1} is done as well.
      auto issue_s = [&](int i) -> bool {
        if (!wait(&k_full[i % RING], (i / RING) & 1)) return false;
        tc_fence_after_sync();
        const uint32_t kt = k_addr + (i % RING) * C::kTileBytes;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          umma_bf16_tmem_a(tmem, tmem + C::kQCol + kk * 8,
                           umma_desc_sw128(kt + (kk >> 2) * kBoxBytes + (kk & 3) * 32, 16, 1024),
                           C::kIdescS, kk > 0);
        umma_commit(s_full);
        umma_commit(&k_empty[i % RING]);
        return true;
      };
      // keys 16 kk .. 16 kk + 15: chunk kk / 2 of the P columns, half kk % 2 of
      // its 16 head (then residual) columns
      auto issue_pv = [&](int i) -> bool {
        if (!wait(p_full, i & 1) || !wait(&v_full[i % RING], (i / RING) & 1)) return false;
        tc_fence_after_sync();
        const uint32_t vt = v_addr + (i % RING) * C::kTileBytes;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          umma_bf16_tmem_a(tmem + C::kOCol, tmem + 32 * (kk >> 1) + 8 * (kk & 1),
                           umma_desc_sw128(vt + kk * 2048, kBoxBytes, 1024), C::kIdescPV,
                           !(i == 0 && kk == 0));
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          umma_bf16_tmem_a(tmem + C::kOCol, tmem + 32 * (kk >> 1) + 16 + 8 * (kk & 1),
                           umma_desc_sw128(vt + kk * 2048, kBoxBytes, 1024), C::kIdescPV, true);
        umma_commit(o_done);
        umma_commit(&v_empty[i % RING]);
        return true;
      };
      Cursor c{-1, 0, -1, -1};
      next_run(c);
      int i = 0;
      bool ok = c.r < runs && issue_s(0);
      const bool issued = ok;
      while (ok) {
        if (!issue_pv(i)) break;
        advance(c);
        if (c.r >= runs) break;
        ++i;
        ok = issue_s(i);
      }
      // drain: every MMA issued so far completes before TMEM is freed
      if (issued) {
        umma_commit(fin);
        mbar_wait_bounded(fin, 0, p.err);
      }
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int m = tid, tl = m / G, g = m % G;
    const bool row_ok = tl < tokens && t_begin + tl < t_end;
    const uint32_t lane_base = tmem + ((uint32_t)(32 * warp) << 16);
    const float c = p.q_scale_log2;
    const float cc = c > 0.f ? c : 1.f;
    int i = 0, rs = 0;
    auto all_ok = [&](bool ok) { return __all_sync(0xffffffffu, ok); };
    for (int r = 0; r < runs; ++r) {
      const int re = run_end[r];
      const int row = tok_row[rs];
      if (row < 0 || run_bad[r]) {
        rs = re;
        continue;
      }
      const bool live = row_ok && tl >= rs && tl < re;
      const int pos = live ? tok_pos[tl] : -1;
      const int lo = p.window > 0 ? pos - p.window + 1 : 0;
      const int lo_run = p.window > 0 ? max(tok_pos[rs] - p.window + 1, 0) : 0;
      const int pos_last = tok_pos[re - 1];
      const int first = lo_run / kPage, last = pos_last / kPage;
      float m_ref = -INFINITY, l = 0.f;
      bool ok = true;
      for (int pg = first; pg <= last; ++pg, ++i) {
        if (!all_ok(mbar_wait_abortable(s_full, i & 1, p.err, &abort_flag))) {
          ok = false;
          break;
        }
        // the S commit also covers P V of the previous page: O is stable
        tc_fence_after_sync();
        float sv[kPage];
#pragma unroll
        for (int q = 0; q < kPage / 16; ++q)
          tmem_ld16(lane_base + 16 * q, *reinterpret_cast<float(*)[16]>(&sv[16 * q]));
        tmem_wait_ld();
        // scores stay raw: the scale is folded into the exponent's FMA (for a
        // positive scale; otherwise it is applied here)
        if (!(c > 0.f)) {
#pragma unroll
          for (int k = 0; k < kPage; ++k) sv[k] *= c;
        }
        const int pos0 = pg * kPage;
        if (!(live && pos0 >= lo && pos0 + kPage - 1 <= pos)) {
#pragma unroll
          for (int k = 0; k < kPage; ++k)
            if (!(live && pos0 + k >= lo && pos0 + k <= pos)) sv[k] = -INFINITY;
        }
        float part[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) part[j] = sv[j];
#pragma unroll
        for (int k = 8; k < kPage; k += 16)
#pragma unroll
          for (int j = 0; j < 8; ++j) part[j] = fmax3(part[j], sv[k + 2 * j], sv[k + 2 * j + 1]);
        const float mx = fmax3(fmax3(part[0], part[1], part[2]), fmax3(part[3], part[4], part[5]),
                               fmaxf(part[6], part[7])) *
                         cc;
        float alpha = 1.f;
        bool rescale_o = false;
        if (mx > m_ref + kLazyRescaleLog2) {
          if (m_ref != -INFINITY) {
            alpha = exp2_approx(m_ref - mx);
            rescale_o = true;
          }
          l *= alpha;
          m_ref = mx;
        }
        const float nml = m_ref == -INFINITY ? 0.f : -m_ref;
        // P = 2^(s - m_ref) as a bf16 head and residual over the S columns
        // (per chunk of 32 keys: head at +0, residual at +16, column j of a
        // half holding keys 2j, 2j + 1); pairs through the packed fp32 pipe
        const float2 cc2 = make_float2(cc, cc), nml2 = make_float2(nml, nml);
        const float2 minus1 = make_float2(-1.f, -1.f);
        float2 sum2[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) sum2[j] = make_float2(0.f, 0.f);
#pragma unroll
        for (int q = 0; q < kPage / 32; ++q) {
          uint32_t hw[16], lw[16];
#pragma unroll
          for (int w = 0; w < 16; ++w) {
            const float2 y =
                __ffma2_rn(make_float2(sv[32 * q + 2 * w], sv[32 * q + 2 * w + 1]), cc2, nml2);
            const float2 x = make_float2(exp2_approx(y.x), exp2_approx(y.y));
            sum2[w & 3] = __fadd2_rn(sum2[w & 3], x);
            hw[w] = pack_bf16x2(x.x, x.y);
            const float2 rr = __ffma2_rn(make_float2(bf16_lo(hw[w]), bf16_hi(hw[w])), minus1, x);
            lw[w] = pack_bf16x2(rr.x, rr.y);
          }
          tmem_st16(lane_base + 32 * q, hw);
          tmem_st16(lane_base + 32 * q + 16, lw);
        }
        const float2 s4 = __fadd2_rn(__fadd2_rn(sum2[0], sum2[1]), __fadd2_rn(sum2[2], sum2[3]));
        l += s4.x + s4.y;
        if (__any_sync(0xffffffffu, rescale_o)) {
#pragma unroll
          for (int q16 = 0; q16 < D / 16; ++q16) {
            float ov[16];
            tmem_ld16(lane_base + C::kOCol + 16 * q16, ov);
            tmem_wait_ld();
#pragma unroll
            for (int k = 0; k < 16; ++k) ov[k] *= alpha;
            tmem_st16(lane_base + C::kOCol + 16 * q16, ov);
          }
        }
        // V rows outside the run's key range on a boundary page -> zero
        const int rlo = max(lo_run - pos0, 0), rhi = min(pos_last - pos0, kPage - 1);
        if (rlo > 0 || rhi < kPage - 1) {
          const int s = i % RING;
          if (!all_ok(mbar_wait_abortable(&v_full[s], (i / RING) & 1, p.err, &abort_flag))) {
            ok = false;
            break;
          }
          unsigned char* vt = v_slots + s * C::kTileBytes;
          for (int e = m; e < kPage * (D / 8); e += C::kSoftmaxThreads) {
            const int k = e / (D / 8), ch = e % (D / 8);
            if (k < rlo || k > rhi)
              *reinterpret_cast<uint4*>(vt + (ch >> 3) * kBoxBytes + k * 128 + (ch & 7) * 16) =
                  make_uint4(0u, 0u, 0u, 0u);
          }
          fence_proxy_async_shared();  // the zeros are read by the tensor core
        }
        tmem_wait_st();
        tc_fence_before_sync();
        mbar_arrive(p_full);
      }
      if (!ok) break;

      // end of run: O rows of this run are final once P V of its last page is done
      if (!all_ok(mbar_wait_abortable(o_done, (i - 1) & 1, p.err, &abort_flag))) break;
      tc_fence_after_sync();
      const int hh = h0 + g;
      float inv = 0.f;
      if (live) {
        const float sk = p.sinks ? p.sinks[hh] * kLog2e : -INFINITY;
        const float mf = fmaxf(m_ref, sk);
        const float scl = exp2_approx(m_ref - mf);
        const float total = fmaf(l, scl, exp2_approx(sk - mf));
        inv = total > 0.f ? scl / total : 0.f;
      }
      uint16_t* orow = p.out + ((size_t)(t_begin + tl) * p.hq + hh) * D;
#pragma unroll
      for (int q16 = 0; q16 < D / 16; ++q16) {
        float ov[16];
        tmem_ld16(lane_base + C::kOCol + 16 * q16, ov);
        tmem_wait_ld();
        if (live) {
          uint32_t w[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) w[k] = pack_bf16x2(ov[2 * k] * inv, ov[2 * k + 1] * inv);
          uint4* dst = reinterpret_cast<uint4*>(orow + 16 * q16);
          dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
          dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
        }
      }
      tc_fence_before_sync();
      rs = re;
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

template <int D, int RING>
cudaError_t launch_prefill_umma(const DecodeParams& p, const CUtensorMap& k_map,
                                const CUtensorMap& v_map, cudaStream_t stream) {
  using C = UmmaPrefillCfg<D, RING>;
  static std::atomic<bool> configured[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !configured[dev].load(std::memory_order_acquire)) {
    e = cudaFuncSetAttribute(paged_prefill_umma_kernel<D, RING>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(paged_prefill_umma_kernel<D, RING>,
                             cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) configured[dev].store(true, std::memory_order_release);
  }
  if (p.rows == 0) return cudaSuccess;
  const int tokens = C::kRows / p.group;
  dim3 grid((p.rows + tokens - 1) / tokens, p.hkv);
  return launch_pdl(paged_prefill_umma_kernel<D, RING>, grid, dim3(C::kThreads), C::kSmemBytes,
                    stream, k_map, v_map, p);
}

}  // namespace pgd
