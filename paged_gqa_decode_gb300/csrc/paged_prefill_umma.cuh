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
// head).  Its 128 query rows are (token, head of the group) pairs, row
// m = token * G + head, one per TMEM lane.  Tokens split into runs (same table
// row, consecutive positions); each run is one pass over the pages of the
// union of its tokens' key ranges.  Six warps:
//   warp 4      TMA producer: K and V tiles (64 x D bf16, 128-byte swizzle)
//               of each page into a ring of shared stages.
//   warp 5      MMA issuer (one thread) and TMEM owner:
//                 S_i = Q K_i^T      M 128, N 64, K D   -> TMEM S buffer i % 2
//                 O  += P_i V_i      M 128, N D,  K 64  -> TMEM O
//               issued in the order S_0, S_1, PV_0, S_2, PV_1, ... so that
//               the next page's scores are ready when the softmax finishes.
//   warps 0-3   softmax, one thread per query row: S row from TMEM, causal
//               and window mask, online softmax in log2 units with a lazy
//               reference max (raised only when a score exceeds it by more
//               than 2^8, which then rescales that row of O in TMEM), P
//               written to shared memory as a bf16 head and residual (two
//               MMAs, so P V keeps fp32 accuracy); at the end of a run the O
//               row is normalised with the sink and stored.
// V rows outside the run's key range on its boundary pages are zeroed in
// shared memory before the product.  Every wait is bounded; a timeout records
// PGD_EDEVICE_TIMEOUT, stops all roles, drains in-flight copies and MMAs and
// frees TMEM before the CTA exits.
#pragma once

#include "paged_decode.cuh"
#include "pgd_umma.cuh"

namespace pgd {

template <int D, int STAGES>
struct UmmaPrefillCfg {
  static constexpr int kRows = 128;  // query rows per CTA (TMEM lanes)
  static constexpr int kSoftmaxThreads = 128;
  static constexpr int kProducerWarp = 4;
  static constexpr int kMmaWarp = 5;
  static constexpr int kThreads = 192;
  static constexpr int kBoxes = D / 64;
  static constexpr int kTileBytes = kPage * D * 2;
  static constexpr int kStageBytes = 2 * kTileBytes;
  static constexpr int kQBoxBytes = kRows * 128;  // 128 rows x 64 bf16
  static constexpr int kQBytes = kBoxes * kQBoxBytes;
  static constexpr int kPBytes = kRows * kPage * 2;  // one 128 x 64 bf16 tile
  static constexpr int kQOff = STAGES * kStageBytes;
  static constexpr int kPOff = kQOff + kQBytes;  // [buffer 0 hi, lo][buffer 1 hi, lo]
  static constexpr int kBarOff = kPOff + 4 * kPBytes;
  static constexpr int kNumBars = 2 * STAGES + 9;
  static constexpr int kSmemBytes = 1024 + kBarOff + kNumBars * 8;
  static constexpr uint32_t kTmemCols = 256;  // S buffers at 0 and 64, O at 128
  static constexpr uint32_t kOCol = 128;
  static constexpr uint32_t kIdescS = umma_idesc_bf16(128, 64, 0, 0);
  static constexpr uint32_t kIdescPV = umma_idesc_bf16(128, D, 0, 1);
  static_assert(D == 64 || D == 128, "head_dim");
};

// Reference-max slack in log2 units: P values stay below 2^8.
constexpr float kLazyRescaleLog2 = 8.0f;

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

template <int D, int STAGES>
__global__ void __launch_bounds__(192, 1)
    paged_prefill_umma_kernel(const __grid_constant__ CUtensorMap k_map,
                              const __grid_constant__ CUtensorMap v_map, const DecodeParams p) {
  using C = UmmaPrefillCfg<D, STAGES>;
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
  unsigned char* stages = base;
  unsigned char* q_s = base + C::kQOff;
  unsigned char* p_s = base + C::kPOff;
  uint64_t* full = reinterpret_cast<uint64_t*>(base + C::kBarOff);
  uint64_t* empty = full + STAGES;
  uint64_t* s_full = empty + STAGES;  // S_i in TMEM (MMA commit)
  uint64_t* s_free = s_full + 2;      // S_i read by all softmax threads
  uint64_t* p_full = s_free + 2;      // P_i in shared memory (softmax threads)
  uint64_t* p_free = p_full + 2;      // PV_i done (MMA commit)
  uint64_t* fin = p_free + 2;         // every MMA of the CTA done
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
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&s_full[b], 1);
      mbar_init(&s_free[b], C::kSoftmaxThreads);
      mbar_init(&p_full[b], C::kSoftmaxThreads);
      mbar_init(&p_free[b], 1);
    }
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
  // Q rows into shared memory (128-byte swizzle, K-major); rows of no token
  // are zero.
  if (tid < C::kSoftmaxThreads) {
    const int m = tid, tl = m / G, g = m % G;
    const bool ok = tl < tokens && t_begin + tl < t_end && tok_row[tl] >= 0;
    uint4 v[D / 8];
    if (ok) {
      const uint4* src =
          reinterpret_cast<const uint4*>(p.q + ((size_t)(t_begin + tl) * p.hq + h0 + g) * D);
#pragma unroll
      for (int c = 0; c < D / 8; ++c) v[c] = src[c];
    } else {
#pragma unroll
      for (int c = 0; c < D / 8; ++c) v[c] = make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int c = 0; c < D / 8; ++c)
      *reinterpret_cast<uint4*>(q_s + (c >> 3) * C::kQBoxBytes + sw128_offset(m, c & 7)) = v[c];
    fence_proxy_async_shared();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = tmem_slot;
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

  if (warp == C::kProducerWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tensormap(&k_map);
      prefetch_tensormap(&v_map);
      int i = 0, rs = 0;
      for (int r = 0; r < runs && !abort_flag; ++r) {
        const int re = run_end[r];
        const int row = tok_row[rs];
        if (row >= 0 && !run_bad[r]) {
          const int lo = p.window > 0 ? max(tok_pos[rs] - p.window + 1, 0) : 0;
          const int first = lo / kPage, last = tok_pos[re - 1] / kPage;
          for (int pg = first; pg <= last; ++pg, ++i) {
            const int s = i % STAGES;
            if (i >= STAGES &&
                !mbar_wait_abortable(&empty[s], ((i / STAGES) - 1) & 1, p.err, &abort_flag))
              break;
            const int page = page_of(p.table, row, pg, p.maxp);
            const int y = (int)tile_first_row(p.layout, page, kvh, p.hkv, p.num_pages, p.maxp);
            unsigned char* st = stages + s * C::kStageBytes;
            mbar_arrive_expect_tx(&full[s], C::kStageBytes);
#pragma unroll
            for (int bx = 0; bx < C::kBoxes; ++bx) {
              tma_load_2d(st + bx * kBoxBytes, &k_map, bx * 64, y, &full[s]);
              tma_load_2d(st + C::kTileBytes + bx * kBoxBytes, &v_map, bx * 64, y, &full[s]);
            }
          }
        }
        rs = re;
      }
      // drain: the copies still in flight land before the CTA exits
      for (int j = max(0, i - STAGES); j < i; ++j)
        mbar_wait_bounded(&full[j % STAGES], (j / STAGES) & 1, p.err);
    }
  } else if (warp == C::kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t q_addr = smem_addr(q_s), p_addr = smem_addr(p_s);
      const uint32_t st_addr = smem_addr(stages);
      auto issue_pv = [&](int j) -> bool {
        if (!mbar_wait_abortable(&p_full[j & 1], (j >> 1) & 1, p.err, &abort_flag)) return false;
        tc_fence_after_sync();
        const uint32_t vt = st_addr + (j % STAGES) * C::kStageBytes + C::kTileBytes;
        const uint32_t ph = p_addr + (j & 1) * 2 * C::kPBytes, pl = ph + C::kPBytes;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          umma_bf16(tmem + C::kOCol, umma_desc_sw128(ph + kk * 32, 16, 1024),
                    umma_desc_sw128(vt + kk * 2048, kBoxBytes, 1024), C::kIdescPV,
                    j > 0 || kk > 0);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          umma_bf16(tmem + C::kOCol, umma_desc_sw128(pl + kk * 32, 16, 1024),
                    umma_desc_sw128(vt + kk * 2048, kBoxBytes, 1024), C::kIdescPV, true);
        umma_commit(&p_free[j & 1]);
        umma_commit(&empty[j % STAGES]);
        return true;
      };
      int i = 0, rs = 0;
      bool ok = true;
      for (int r = 0; r < runs && ok; ++r) {
        const int re = run_end[r];
        const int row = tok_row[rs];
        if (row >= 0 && !run_bad[r]) {
          const int lo = p.window > 0 ? max(tok_pos[rs] - p.window + 1, 0) : 0;
          const int first = lo / kPage, last = tok_pos[re - 1] / kPage;
          for (int pg = first; pg <= last; ++pg, ++i) {
            const int s = i % STAGES;
            if (!mbar_wait_abortable(&full[s], (i / STAGES) & 1, p.err, &abort_flag) ||
                (i >= 2 &&
                 !mbar_wait_abortable(&s_free[i & 1], ((i >> 1) - 1) & 1, p.err, &abort_flag))) {
              ok = false;
              break;
            }
            tc_fence_after_sync();
            const uint32_t kt = st_addr + s * C::kStageBytes;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk)
              umma_bf16(tmem + (i & 1) * 64,
                        umma_desc_sw128(q_addr + (kk >> 2) * C::kQBoxBytes + (kk & 3) * 32, 16,
                                        1024),
                        umma_desc_sw128(kt + (kk >> 2) * kBoxBytes + (kk & 3) * 32, 16, 1024),
                        C::kIdescS, kk > 0);
            umma_commit(&s_full[i & 1]);
            if (i >= 1 && !issue_pv(i - 1)) {
              ok = false;
              break;
            }
          }
        }
        rs = re;
      }
      if (ok && i >= 1) issue_pv(i - 1);
      // drain: every MMA issued so far completes before TMEM is freed
      if (i >= 1) {
        umma_commit(fin);
        mbar_wait_bounded(fin, 0, p.err);
      }
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int m = tid, tl = m / G, g = m % G;
    const bool row_ok = tl < tokens && t_begin + tl < t_end;
    const uint32_t t_lane = tmem + ((uint32_t)(32 * warp) << 16);
    const float c = p.q_scale_log2;
    unsigned char* ph_base = p_s;
    int i = 0, rs = 0;
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
        const int b = i & 1;
        ok = mbar_wait_abortable(&s_full[b], (i >> 1) & 1, p.err, &abort_flag);
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        float sv[64];
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4)
          tmem_ld16(t_lane + b * 64 + 16 * q4, *reinterpret_cast<float(*)[16]>(&sv[16 * q4]));
        tmem_wait_ld();
        tc_fence_before_sync();
        mbar_arrive(&s_free[b]);

        const int pos0 = pg * kPage;
        float mx = -INFINITY;
        if (live && pos0 >= lo && pos0 + kPage - 1 <= pos) {
#pragma unroll
          for (int k = 0; k < 64; ++k) {
            sv[k] *= c;
            mx = fmaxf(mx, sv[k]);
          }
        } else {
#pragma unroll
          for (int k = 0; k < 64; ++k) {
            const int kp = pos0 + k;
            const bool in = live && kp >= lo && kp <= pos;
            sv[k] = in ? sv[k] * c : -INFINITY;
            mx = fmaxf(mx, sv[k]);
          }
        }
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
        const float ml = m_ref == -INFINITY ? 0.f : m_ref;
        float sum = 0.f;
#pragma unroll
        for (int k = 0; k < 64; ++k) {
          sv[k] = exp2_approx(sv[k] - ml);
          sum += sv[k];
        }
        l += sum;

        // P buffer b is free once PV_{i-2} is done
        if (i >= 2) {
          ok = mbar_wait_abortable(&p_free[b], ((i >> 1) - 1) & 1, p.err, &abort_flag);
          if (!__all_sync(0xffffffffu, ok)) {
            ok = false;
            break;
          }
        }
        if (__any_sync(0xffffffffu, rescale_o)) {
          // PV_{i-1} done before this warp's O rows are rescaled
          ok = mbar_wait_abortable(&p_free[b ^ 1], ((i - 1) >> 1) & 1, p.err, &abort_flag);
          if (!__all_sync(0xffffffffu, ok)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
#pragma unroll
          for (int q16 = 0; q16 < D / 16; ++q16) {
            float ov[16];
            tmem_ld16(t_lane + C::kOCol + 16 * q16, ov);
            tmem_wait_ld();
#pragma unroll
            for (int k = 0; k < 16; ++k) ov[k] *= alpha;
            tmem_st16(t_lane + C::kOCol + 16 * q16, ov);
          }
          tmem_wait_st();
        }
        // V rows outside the run's key range on a boundary page -> zero
        const int rlo = max(lo_run - pos0, 0), rhi = min(pos_last - pos0, kPage - 1);
        if (rlo > 0 || rhi < kPage - 1) {
          const int s = i % STAGES;
          ok = mbar_wait_abortable(&full[s], (i / STAGES) & 1, p.err, &abort_flag);
          if (!__all_sync(0xffffffffu, ok)) {
            ok = false;
            break;
          }
          unsigned char* vt = stages + s * C::kStageBytes + C::kTileBytes;
          for (int e = tid; e < kPage * (D / 8); e += C::kSoftmaxThreads) {
            const int rr = e / (D / 8), ch = e % (D / 8);
            if (rr < rlo || rr > rhi)
              *reinterpret_cast<uint4*>(vt + (ch >> 3) * kBoxBytes + rr * 128 + (ch & 7) * 16) =
                  make_uint4(0u, 0u, 0u, 0u);
          }
        }
        // P row m as bf16 head + residual, 128-byte swizzled K-major
        unsigned char* ph = ph_base + b * 2 * C::kPBytes;
        unsigned char* pl = ph + C::kPBytes;
#pragma unroll
        for (int ch = 0; ch < 8; ++ch) {
          uint32_t hw[4], lw[4];
#pragma unroll
          for (int w = 0; w < 4; ++w) {
            const float x0 = sv[8 * ch + 2 * w], x1 = sv[8 * ch + 2 * w + 1];
            hw[w] = pack_bf16x2(x0, x1);
            lw[w] = pack_bf16x2(x0 - bf16_lo(hw[w]), x1 - bf16_hi(hw[w]));
          }
          const uint32_t off = sw128_offset(m, ch);
          *reinterpret_cast<uint4*>(ph + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
          *reinterpret_cast<uint4*>(pl + off) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
        }
        fence_proxy_async_shared();
        tc_fence_before_sync();
        mbar_arrive(&p_full[b]);
      }
      if (!ok) break;

      // end of run: O rows of this run are final once PV of its last page is done
      const int jl = i - 1;
      ok = mbar_wait_abortable(&p_free[jl & 1], (jl >> 1) & 1, p.err, &abort_flag);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after_sync();
      const int h = h0 + g;
      float inv = 0.f;
      if (live) {
        const float sk = p.sinks ? p.sinks[h] * kLog2e : -INFINITY;
        const float mf = fmaxf(m_ref, sk);
        const float scl = exp2_approx(m_ref - mf);
        const float total = fmaf(l, scl, exp2_approx(sk - mf));
        inv = total > 0.f ? scl / total : 0.f;
      }
      uint16_t* orow = p.out + ((size_t)(t_begin + tl) * p.hq + h) * D;
#pragma unroll
      for (int q16 = 0; q16 < D / 16; ++q16) {
        float ov[16];
        tmem_ld16(t_lane + C::kOCol + 16 * q16, ov);
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

template <int D, int STAGES>
cudaError_t launch_prefill_umma(const DecodeParams& p, const CUtensorMap& k_map,
                                const CUtensorMap& v_map, cudaStream_t stream) {
  using C = UmmaPrefillCfg<D, STAGES>;
  static_assert(C::kSmemBytes + 4 * 1024 <= 227 * 1024, "shared memory");
  static std::atomic<bool> configured[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !configured[dev].load(std::memory_order_acquire)) {
    e = cudaFuncSetAttribute(paged_prefill_umma_kernel<D, STAGES>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) configured[dev].store(true, std::memory_order_release);
  }
  if (p.rows == 0) return cudaSuccess;
  const int tokens = C::kRows / p.group;
  dim3 grid((p.rows + tokens - 1) / tokens, p.hkv);
  return launch_pdl(paged_prefill_umma_kernel<D, STAGES>, grid, dim3(C::kThreads), C::kSmemBytes,
                    stream, k_map, v_map, p);
}

}  // namespace pgd
