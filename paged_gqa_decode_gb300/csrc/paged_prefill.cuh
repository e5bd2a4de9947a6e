// Tiled paged prefill attention for sm_103a (tensor cores).
//
// What it computes (Mistral 7B Instruct v0.3 model files, src/attention.linnet,
// prefill_paged / paged_prefill_attention; window and sinks as GPT-OSS 20B
// src/attention.linnet, prefill_packed): packed prompt token p is position
// positions[p] of the request in table row rows[p]; its query heads attend
// over that row's pages at positions (positions[p] - window, positions[p]],
// with the head's sink logit in the softmax denominator only.
//
// Decomposition: one CTA per (block of kTokens consecutive packed tokens, kv
// head).  The CTA's 64 query rows are (token, head of the group) pairs, the
// group padded to GP heads, so a block is 64 / GP tokens.  Inside a block the
// tokens split into runs -- maximal stretches with the same table row and
// consecutive positions -- and each run is one pass over the union of its
// tokens' key ranges.  (Prompt chunks are packed end to end, so a block is
// almost always one run.)  Per pass a producer warp streams the row's pages
// (K and V tiles, 64 x D bf16) with 2-D TMA loads into a ring of shared
// stages, each page loaded once for all tokens and heads of the block, and
// four consumer warps each own one m16 tile of query rows:
//   S = Q K^T      mma.sync m16n8k16 (Q as A fragments in registers, K^T as B
//                  fragments by ldmatrix from the 128-byte-swizzled tile)
//   online softmax per query row in fp32 (log2 units), per-token causal and
//                  window mask
//   O += P V       P straight from the S accumulators as A fragments, split
//                  into a bf16 head and residual (two MMAs) so P.V keeps fp32
//                  accuracy; V as B fragments by ldmatrix.trans
// V rows outside the pass's key range on its boundary pages are zeroed in
// shared memory before the product (a zero weight times a stale non-finite
// value would leak).  Outputs are written directly with the sink folded in;
// there is no split of the key range, so this kernel is chosen when there are
// enough token blocks to fill the GPU.
#pragma once

#include "paged_decode.cuh"

namespace pgd {

template <int D, int GP, int STAGES>
struct PrefillCfg {
  static constexpr int kWarps = 4;
  static constexpr int kThreads = (kWarps + 1) * 32;
  static constexpr int kRows = 16 * kWarps;  // query rows (token, head) per CTA
  static constexpr int kTokens = kRows / GP;
  static constexpr int kBoxes = D / 64;
  static constexpr int kTileBytes = kPage * D * 2;
  static constexpr int kStageBytes = 2 * kTileBytes;
  static constexpr int kStages = STAGES;
  static constexpr int kSmemBytes = 1024 + kStages * kStageBytes + 2 * kStages * 8;
  static_assert(GP == 1 || GP == 2 || GP == 4 || GP == 8, "group padding");
};

template <int D, int GP, int STAGES>
// Two CTAs per SM: at 5 warps each they fit the sub-partitions' register
// files only below ~170 registers a thread; measured 13 % faster on the
// Mistral-shaped prefill than one CTA with more registers.
__global__ void __launch_bounds__(PrefillCfg<D, GP, STAGES>::kThreads, 2)
    paged_prefill_kernel(const __grid_constant__ CUtensorMap k_map,
                         const __grid_constant__ CUtensorMap v_map, const DecodeParams p) {
  using C = PrefillCfg<D, GP, STAGES>;
  constexpr int kSteps = D / 16;   // k-steps of Q.K^T
  constexpr int kDimTiles = D / 8;  // n-tiles of P.V
  pdl_wait();
  pdl_allow_dependents();
  const int kvh = blockIdx.y;
  const int t_begin = blockIdx.x * C::kTokens;
  const int t_end = min(t_begin + C::kTokens, p.rows);
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int h0 = kvh * p.group;

  extern __shared__ unsigned char smem_raw[];
  unsigned char* stages = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(stages + C::kStages * C::kStageBytes);
  uint64_t* empty = full + C::kStages;
  __shared__ int run_end[C::kTokens + 1];  // run r covers tokens [run_end[r-1], run_end[r])
  __shared__ int runs;
  __shared__ int tok_row[C::kTokens], tok_pos[C::kTokens];
  __shared__ int run_bad[C::kTokens];
  __shared__ int abort_flag;

  // Tokens of the block, their rows and positions; bad ones are reported and
  // left out of every run (their outputs are zeroed below).
  if (tid < C::kTokens) {
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
    for (int i = 1; i <= C::kTokens; ++i) {
      const bool brk = i == C::kTokens || tok_row[i] != tok_row[i - 1] ||
                       tok_pos[i] != tok_pos[i - 1] + 1 || tok_row[i] < 0 || tok_row[i - 1] < 0;
      if (brk) run_end[r++] = i;
    }
    runs = r;
    for (int k = 0; k < C::kTokens; ++k) run_bad[k] = 0;
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], C::kWarps);
    }
    mbar_init_fence();
    abort_flag = 0;
  }
  __syncthreads();

  // Per run: pages [first, last] of the row; a table entry outside the pool
  // marks the run bad (checked by everyone before any copy is issued): its
  // tokens get zero outputs and PGD_EDEVICE_BOUNDS is recorded.
  {
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
  __syncthreads();
  if (tid == 0)
    for (int r = 0; r < runs; ++r)
      if (run_bad[r]) record_error(p.err, PGD_EDEVICE_BOUNDS);
  // Zero outputs of tokens that belong to no run (inactive or bad).
  for (int e = tid; e < C::kTokens * p.group * D; e += C::kThreads) {
    const int ti = e / (p.group * D);
    if (t_begin + ti < t_end && tok_row[ti] < 0) {
      const int g = (e / D) % p.group, d = e % D;
      p.out[((size_t)(t_begin + ti) * p.hq + h0 + g) * D + d] = 0;
    }
  }

  // ------------------------------------------------------------ producer
  if (warp == C::kWarps) {
    if (lane == 0) {
      prefetch_tensormap(&k_map);
      prefetch_tensormap(&v_map);
      int i = 0;  // page counter across runs
      int rs = 0;
      for (int r = 0; r < runs && !abort_flag; ++r) {
        const int re = run_end[r];
        const int row = tok_row[rs];
        if (row >= 0 && !run_bad[r]) {
          const int lo = p.window > 0 ? max(tok_pos[rs] - p.window + 1, 0) : 0;
          const int first = lo / kPage, last = tok_pos[re - 1] / kPage;
          for (int pg = first; pg <= last; ++pg, ++i) {
            const int s = i % C::kStages;
            // every consumer warp takes every page, in order, so each parity
            // wait targets the current phase
            if (i >= C::kStages &&
                !mbar_wait_bounded(&empty[s], ((i / C::kStages) - 1) & 1, p.err)) {
              abort_flag = 1;
              break;
            }
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
      const int issued = i;
      for (int j = max(0, issued - C::kStages); j < issued; ++j)
        mbar_wait_bounded(&full[j % C::kStages], (j / C::kStages) & 1, p.err);
    }
    return;
  }

  // ------------------------------------------------------------ consumers
  const int gid = lane >> 2, tig = lane & 3;
  // This lane's two query rows in the warp's m16 tile: rows gid and gid + 8.
  const int row_a = warp * 16 + gid, row_b = row_a + 8;
  const int ta = row_a / GP, tb = row_b / GP;  // tokens within the block
  const int ga = row_a % GP, gb = row_b % GP;  // heads within the group
  const float c = p.q_scale_log2;
  // ldmatrix row offsets: K^T B fragments (non-transposed K rows = keys):
  // matrix j: keys +8*(j>>1), dim chunk +(j&1); V B fragments (transposed):
  // matrix j: keys +8*(j&1), dim chunk +(j>>1).
  const int lj = lane >> 3, lr = lane & 7;
  uint32_t off_k[4], off_v[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    off_k[i] = ((lj >> 1) * 8 + lr) * 128 + ((((lj & 1)) ^ lr ^ (2 * i)) << 4);
    off_v[i] = ((lj & 1) * 8 + lr) * 128 + ((((lj >> 1)) ^ lr ^ (2 * i)) << 4);
  }

  int i_page = 0;
  int rs = 0;
  for (int r = 0; r < runs; ++r) {
    const int re = run_end[r];
    const int row = tok_row[rs];
    if (row < 0 || run_bad[r]) {  // bad runs: outputs zeroed below
      if (row >= 0) {
        for (int e = lane; e < (re - rs) * p.group * D; e += 32) {
          if (warp != 0) break;
          const int ti = rs + e / (p.group * D), g = (e / D) % p.group, d = e % D;
          p.out[((size_t)(t_begin + ti) * p.hq + h0 + g) * D + d] = 0;
        }
      }
      rs = re;
      continue;
    }
    const int pos_first = tok_pos[rs];
    const int lo_run = p.window > 0 ? max(pos_first - p.window + 1, 0) : 0;
    const int first = lo_run / kPage, last = tok_pos[re - 1] / kPage;
    // this lane's rows: live if their token is in the run and head < group
    const bool live_a = ta >= rs && ta < re && ga < p.group;
    const bool live_b = tb >= rs && tb < re && gb < p.group;
    const int pos_a = live_a ? tok_pos[ta] : -1, pos_b = live_b ? tok_pos[tb] : -1;
    const int lo_a = p.window > 0 ? pos_a - p.window + 1 : 0;
    const int lo_b = p.window > 0 ? pos_b - p.window + 1 : 0;

    // Q A-fragments: a0/a2 from row_a, a1/a3 from row_b; dims 16kk + 2tig (+8).
    uint32_t qa[kSteps][4];
    {
      const uint32_t* qra = reinterpret_cast<const uint32_t*>(
          p.q + ((size_t)(t_begin + (live_a ? ta : rs)) * p.hq + h0 + (live_a ? ga : 0)) * D);
      const uint32_t* qrb = reinterpret_cast<const uint32_t*>(
          p.q + ((size_t)(t_begin + (live_b ? tb : rs)) * p.hq + h0 + (live_b ? gb : 0)) * D);
#pragma unroll
      for (int kk = 0; kk < kSteps; ++kk) {
        qa[kk][0] = live_a ? qra[(16 * kk + 2 * tig) >> 1] : 0u;
        qa[kk][1] = live_b ? qrb[(16 * kk + 2 * tig) >> 1] : 0u;
        qa[kk][2] = live_a ? qra[(16 * kk + 8 + 2 * tig) >> 1] : 0u;
        qa[kk][3] = live_b ? qrb[(16 * kk + 8 + 2 * tig) >> 1] : 0u;
      }
    }
    float o[kDimTiles][4];
#pragma unroll
    for (int j = 0; j < kDimTiles; ++j)
#pragma unroll
      for (int e = 0; e < 4; ++e) o[j][e] = 0.f;
    float m_a = -INFINITY, m_b = -INFINITY, l_a = 0.f, l_b = 0.f;

    for (int pg = first; pg <= last; ++pg, ++i_page) {
      const int s = i_page % C::kStages;
      if (!mbar_wait_bounded(&full[s], (i_page / C::kStages) & 1, p.err)) {
        abort_flag = 1;
        break;
      }
      unsigned char* kt_ptr = stages + s * C::kStageBytes;
      unsigned char* vt_ptr = kt_ptr + C::kTileBytes;
      const int pos0 = pg * kPage;
      {
        const uint32_t kt = smem_addr(kt_ptr), vt = smem_addr(vt_ptr);
        // S = Q K^T over the page's 64 keys: 8 n-tiles of 8 keys.
        float sc[8][4];
#pragma unroll
        for (int j = 0; j < 8; ++j)
#pragma unroll
          for (int e = 0; e < 4; ++e) sc[j][e] = 0.f;
#pragma unroll
        for (int kk = 0; kk < kSteps; ++kk)
#pragma unroll
          for (int jp = 0; jp < 4; ++jp) {  // key tiles 2jp, 2jp+1
            uint32_t b0, b1, b2, b3;
            ldsm_x4(kt + (kk >> 2) * kBoxBytes + jp * 2048 + off_k[kk & 3], b0, b1, b2, b3);
            mma_bf16(sc[2 * jp], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b0, b1);
            mma_bf16(sc[2 * jp + 1], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b2, b3);
          }
        // mask + log2 units; row_a holds e = 0, 1, row_b e = 2, 3; key = 8j + 2tig + (e & 1)
        float mxa = -INFINITY, mxb = -INFINITY;
#pragma unroll
        for (int j = 0; j < 8; ++j)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int kp = pos0 + 8 * j + 2 * tig + (e & 1);
            const bool is_a = e < 2;
            const int pos = is_a ? pos_a : pos_b;
            const int lo = is_a ? lo_a : lo_b;
            const bool ok = kp <= pos && kp >= lo;
            const float v = ok ? sc[j][e] * c : -INFINITY;
            sc[j][e] = v;
            if (is_a) mxa = fmaxf(mxa, v); else mxb = fmaxf(mxb, v);
          }
        mxa = fmaxf(mxa, __shfl_xor_sync(0xffffffffu, mxa, 1));
        mxa = fmaxf(mxa, __shfl_xor_sync(0xffffffffu, mxa, 2));
        mxb = fmaxf(mxb, __shfl_xor_sync(0xffffffffu, mxb, 1));
        mxb = fmaxf(mxb, __shfl_xor_sync(0xffffffffu, mxb, 2));
        const float mna = fmaxf(m_a, mxa), mnb = fmaxf(m_b, mxb);
        const float ra = mna == -INFINITY ? 0.f : mna, rb = mnb == -INFINITY ? 0.f : mnb;
        const float ala = exp2_approx(m_a - ra), alb = exp2_approx(m_b - rb);
        float suma = 0.f, sumb = 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          sc[j][0] = exp2_approx(sc[j][0] - ra);
          sc[j][1] = exp2_approx(sc[j][1] - ra);
          sc[j][2] = exp2_approx(sc[j][2] - rb);
          sc[j][3] = exp2_approx(sc[j][3] - rb);
          suma += sc[j][0] + sc[j][1];
          sumb += sc[j][2] + sc[j][3];
        }
        l_a = fmaf(l_a, ala, suma);
        l_b = fmaf(l_b, alb, sumb);
        m_a = mna;
        m_b = mnb;
#pragma unroll
        for (int j = 0; j < kDimTiles; ++j) {
          o[j][0] *= ala;
          o[j][1] *= ala;
          o[j][2] *= alb;
          o[j][3] *= alb;
        }
        // V rows outside the run's key range on this page -> zero (every warp
        // zeroes the same rows with the same values; all wait below).
        // V rows outside the run's key range on this page -> zero.  Every
        // warp zeroes all of them (identical values) so that it needs no
        // barrier with the other warps; the stage is not refilled before all
        // four warps have released it.
        const int rlo = max(lo_run - pos0, 0), rhi = min(tok_pos[re - 1] - pos0, kPage - 1);
        const bool partial = rlo > 0 || rhi < kPage - 1;
        if (partial) {
          const uint4 z = make_uint4(0u, 0u, 0u, 0u);
          for (int rr = lane; rr < kPage; rr += 32)
            if (rr < rlo || rr > rhi)
#pragma unroll
              for (int bx = 0; bx < D / 64; ++bx)
#pragma unroll
                for (int ch = 0; ch < 8; ++ch)
                  *reinterpret_cast<uint4*>(vt_ptr + bx * kBoxBytes + rr * 128 + ch * 16) = z;
          __syncwarp();
        }
        // O += P V: k-step kk covers keys 16kk..16kk+15 = S tiles 2kk, 2kk+1.
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint32_t h0_ = pack_bf16x2(sc[2 * kk][0], sc[2 * kk][1]);
          const uint32_t h1_ = pack_bf16x2(sc[2 * kk][2], sc[2 * kk][3]);
          const uint32_t h2_ = pack_bf16x2(sc[2 * kk + 1][0], sc[2 * kk + 1][1]);
          const uint32_t h3_ = pack_bf16x2(sc[2 * kk + 1][2], sc[2 * kk + 1][3]);
          const uint32_t l0_ = pack_bf16x2(sc[2 * kk][0] - bf16_lo(h0_), sc[2 * kk][1] - bf16_hi(h0_));
          const uint32_t l1_ = pack_bf16x2(sc[2 * kk][2] - bf16_lo(h1_), sc[2 * kk][3] - bf16_hi(h1_));
          const uint32_t l2_ = pack_bf16x2(sc[2 * kk + 1][0] - bf16_lo(h2_),
                                           sc[2 * kk + 1][1] - bf16_hi(h2_));
          const uint32_t l3_ = pack_bf16x2(sc[2 * kk + 1][2] - bf16_lo(h3_),
                                           sc[2 * kk + 1][3] - bf16_hi(h3_));
#pragma unroll
          for (int jp = 0; jp < kDimTiles / 2; ++jp) {
            uint32_t b0, b1, b2, b3;
            ldsm_x4_trans(vt + (jp >> 2) * kBoxBytes + kk * 2048 + off_v[jp & 3], b0, b1, b2, b3);
            mma_bf16(o[2 * jp], h0_, h1_, h2_, h3_, b0, b1);
            mma_bf16(o[2 * jp], l0_, l1_, l2_, l3_, b0, b1);
            mma_bf16(o[2 * jp + 1], h0_, h1_, h2_, h3_, b2, b3);
            mma_bf16(o[2 * jp + 1], l0_, l1_, l2_, l3_, b2, b3);
          }
        }
        if (partial) fence_proxy_async_shared();
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
    if (abort_flag) break;

    // finish the run: reduce l over the quad, fold in the sink, write bf16
    l_a += __shfl_xor_sync(0xffffffffu, l_a, 1);
    l_a += __shfl_xor_sync(0xffffffffu, l_a, 2);
    l_b += __shfl_xor_sync(0xffffffffu, l_b, 1);
    l_b += __shfl_xor_sync(0xffffffffu, l_b, 2);
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const bool live = half ? live_b : live_a;
      if (!live) continue;
      const int tk = half ? tb : ta, g = half ? gb : ga;
      const float mx = half ? m_b : m_a, den = half ? l_b : l_a;
      const int h = h0 + g;
      const float sk = p.sinks ? p.sinks[h] * kLog2e : -INFINITY;
      const float mf = fmaxf(mx, sk);
      const float scl = exp2_approx(mx - mf);
      const float total = fmaf(den, scl, exp2_approx(sk - mf));
      const float inv = total > 0.f ? scl / total : 0.f;
      uint16_t* orow = p.out + ((size_t)(t_begin + tk) * p.hq + h) * D;
#pragma unroll
      for (int j = 0; j < kDimTiles; ++j) {
        const int d = 8 * j + 2 * tig;
        const float v0 = o[j][half * 2] * inv, v1 = o[j][half * 2 + 1] * inv;
        *reinterpret_cast<uint32_t*>(orow + d) = pack_bf16x2(v0, v1);
      }
    }
    rs = re;
  }
}

template <int D, int GP, int STAGES>
cudaError_t launch_prefill(const DecodeParams& p, const CUtensorMap& k_map,
                           const CUtensorMap& v_map, cudaStream_t stream) {
  using C = PrefillCfg<D, GP, STAGES>;
  static_assert(C::kSmemBytes <= 227 * 1024, "shared memory");
  static std::atomic<bool> configured[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !configured[dev].load(std::memory_order_acquire)) {
    e = cudaFuncSetAttribute(paged_prefill_kernel<D, GP, STAGES>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(paged_prefill_kernel<D, GP, STAGES>,
                             cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) configured[dev].store(true, std::memory_order_release);
  }
  if (p.rows == 0) return cudaSuccess;
  dim3 grid((p.rows + C::kTokens - 1) / C::kTokens, p.hkv);
  return launch_pdl(paged_prefill_kernel<D, GP, STAGES>, grid, dim3(C::kThreads), C::kSmemBytes,
                    stream, k_map, v_map, p);
}

template <int D>
cudaError_t launch_prefill_for_dim(const DecodeParams& p, const CUtensorMap& k_map,
                                   const CUtensorMap& v_map, int padded, cudaStream_t stream) {
  constexpr int kStages = D == 128 ? 3 : 6;
  switch (padded) {
    case 1: return launch_prefill<D, 1, kStages>(p, k_map, v_map, stream);
    case 2: return launch_prefill<D, 2, kStages>(p, k_map, v_map, stream);
    case 4: return launch_prefill<D, 4, kStages>(p, k_map, v_map, stream);
    case 8: return launch_prefill<D, 8, kStages>(p, k_map, v_map, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace pgd
