// GQA-grouped split-KV paged decode attention for sm_103a.
//
// What it computes (Mistral 7B Instruct v0.3 model files, src/attention.linnet,
// GroupedQueryAttention.decode_paged / paged_attention; GPT-OSS 20B model
// files, README "Attention sinks" and src/attention.linnet,
// SinkAttention.decode_rows): for row b with new-token position n, query
// head h and kv head g = h / G, over the attended positions
// A = { s : s <= n, s > n - window (window > 0) },
//   out = sum_{s in A} e^{x_s - m} v_s / (sum_{s in A} e^{x_s - m} + e^{sink_h - m}),
// with x_s = scale * q_h . k_s and m = max(max_s x_s, sink_h).  The sink only
// adds to the denominator.  Scores are carried in log2 units (q is
// pre-multiplied by scale * log2 e), so every exponential is one ex2.
//
// Split kernel: one CTA per (split, kv head, row).  A split is a run of
// `pages_per_split` attended pages of one row.  One producer warp streams
// each page's K and V tiles (64 x D bf16, contiguous in the pool) into a ring
// of shared-memory stages with 2-D TMA loads (128-byte swizzle, completion
// on an mbarrier); each page is read from HBM exactly once for all G query
// heads that share the kv head.  Page i goes to stage i % kStages and to
// consumer warp i % kWarps.  Because those two cycles differ, a warp could
// reach a stage's barrier a full phase early; the producer therefore
// publishes the page index it last issued into each stage (stage_seq), and a
// consumer waits for its own page index there before it waits on the stage's
// barrier, so every parity wait targets the barrier's current phase.  Four
// consumer warps take whole pages in turn, each keeping its own fp32
// online-softmax state for the G heads:
//   - scores: lane r owns tile rows r and r + 32 and forms the full dot
//     products against q (broadcast from shared memory), so no cross-lane
//     reduction is needed for Q.K^T;
//   - the page's max per head is one warp-shuffle max; the denominator stays
//     a per-lane partial until the end of the split;
//   - P.V: the probabilities go through a per-warp shared buffer and lane l
//     owns D/32 output dims, accumulating over the page's valid rows.
// At the end the four warps' states are merged through shared memory.  A row
// with one split writes its output directly (sink included); otherwise the
// split writes (m, l, acc) to the workspace and the combine kernel merges.
//
// Pages wholly outside the window are never visited (the split range starts
// at the window's first page); positions outside the window or past n inside
// a visited page are masked to -inf before the softmax and skipped in P.V, so
// their K/V values never reach the result.
#pragma once

#include <math.h>

#include "pgd_device.cuh"
#include "pgd_internal.h"

namespace pgd {

constexpr float kLog2e = 1.4426950408889634f;

template <int D, int GP>
struct DecodeCfg {
  static constexpr int kWarps = 4;  // consumer warps
  static constexpr int kThreads = (kWarps + 1) * 32;
  static constexpr int kBoxBytes = kPage * 64 * 2;  // 64 rows x 128 bytes
  static constexpr int kBoxes = D / 64;
  static constexpr int kTileBytes = kPage * D * 2;
  static constexpr int kStageBytes = 2 * kTileBytes;  // K tile then V tile
  static constexpr int kStages = D == 128 ? 3 : 6;
  static constexpr int kQFloats = GP * D;
  static constexpr int kPFloats = kWarps * kPage * GP;
  static constexpr int kDims = D / 32;  // output dims per lane
  static constexpr int kSmemBytes =
      1024 + kStages * kStageBytes + (kQFloats + kPFloats) * 4 + 2 * kStages * 8;
  static_assert(kWarps * GP * (D + 2) * 4 <= kStages * kStageBytes, "merge buffer");
  static_assert(D == 64 || D == 128, "head_dim");
};

template <int D, int GP>
__global__ void __launch_bounds__(DecodeCfg<D, GP>::kThreads, 2)
    paged_decode_split_kernel(const __grid_constant__ CUtensorMap k_map,
                              const __grid_constant__ CUtensorMap v_map, const DecodeParams p) {
  using C = DecodeCfg<D, GP>;
  const int split = blockIdx.x;
  const int kvh = blockIdx.y;
  const int b = blockIdx.z;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

  const int n = p.positions[b];
  const RowSpan span = row_span(n, p.window);
  const int nsplit = (span.pages + p.pages_per_split - 1) / p.pages_per_split;
  if (split >= nsplit) return;                 // inactive row, or past this row's splits
  if (n / kPage >= p.maxp) return;              // reported (and zeroed) by the combine kernel
  const int page0 = span.first_page + split * p.pages_per_split;
  const int npages = min(p.pages_per_split, span.pages - split * p.pages_per_split);
  const int h0 = kvh * p.group;
  const int32_t* trow = p.table + (size_t)b * p.maxp + page0;

  extern __shared__ unsigned char smem_raw[];
  unsigned char* stages = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* q_s = reinterpret_cast<float*>(stages + C::kStages * C::kStageBytes);
  float* p_s = q_s + C::kQFloats;
  uint64_t* full = reinterpret_cast<uint64_t*>(p_s + C::kPFloats);
  uint64_t* empty = full + C::kStages;
  __shared__ int abort_flag;
  __shared__ int stage_seq[C::kStages];  // page index last issued into each stage

  // Every table entry this split reads must name a pool page.
  bool bad = false;
  for (int i = tid; i < npages; i += C::kThreads) {
    const int pg = trow[i];
    bad |= (pg < 0) | (pg >= p.num_pages);
  }
  bad = __syncthreads_or(bad);
  if (bad) {
    if (tid == 0) record_error(p.err, PGD_EDEVICE_BOUNDS);
    for (int e = tid; e < GP * D; e += C::kThreads) {
      const int g = e / D, d = e % D;
      if (g >= p.group) continue;
      const size_t bh = (size_t)b * p.hq + h0 + g;
      if (nsplit == 1) {
        p.out[bh * D + d] = 0;
      } else {
        p.ws_acc[(bh * p.max_splits + split) * D + d] = 0.f;
        if (d == 0) {
          // l < 0 marks the split as skipped: the combine zeroes the row.
          p.ws_ml[(bh * p.max_splits + split) * 2 + 0] = -INFINITY;
          p.ws_ml[(bh * p.max_splits + split) * 2 + 1] = -1.f;
        }
      }
    }
    return;
  }

  if (tid == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
      stage_seq[s] = -1;
    }
    mbar_init_fence();
    abort_flag = 0;
  }
  // q for the G heads of this kv head, scaled into log2 units; padded heads are 0.
  for (int e = tid; e < GP * D; e += C::kThreads) {
    const int g = e / D, d = e % D;
    float v = 0.f;
    if (g < p.group) {
      const uint16_t bits = p.q[((size_t)b * p.hq + h0 + g) * D + d];
      v = __uint_as_float((uint32_t)bits << 16) * p.q_scale_log2;
    }
    q_s[e] = v;
  }
  __syncthreads();

  // ---------------------------------------------------------------- producer
  if (warp == C::kWarps) {
    if (lane == 0) {
      prefetch_tensormap(&k_map);
      prefetch_tensormap(&v_map);
      int issued = 0;
      for (int i = 0; i < npages; ++i) {
        const int s = i % C::kStages;
        // On a timeout the consumers time out on the pages never issued and
        // abandon the split themselves; only they write abort_flag.
        if (i >= C::kStages && !mbar_wait_bounded(&empty[s], ((i / C::kStages) - 1) & 1, p.err))
          break;
        const int page = trow[i];
        const int y = p.layout == PGD_PAGE_MAJOR ? (page * p.hkv + kvh) * kPage
                                                 : (kvh * p.num_pages + page) * kPage;
        unsigned char* st = stages + s * C::kStageBytes;
        mbar_arrive_expect_tx(&full[s], C::kStageBytes);
#pragma unroll
        for (int bx = 0; bx < C::kBoxes; ++bx) {
          tma_load_2d(st + bx * C::kBoxBytes, &k_map, bx * 64, y, &full[s]);
          tma_load_2d(st + C::kTileBytes + bx * C::kBoxBytes, &v_map, bx * 64, y, &full[s]);
        }
        *reinterpret_cast<volatile int*>(&stage_seq[s]) = i;
        issued = i + 1;
      }
      // No copy may still be landing in shared memory when the CTA exits.
      for (int i = max(0, issued - C::kStages); i < issued; ++i)
        mbar_wait_bounded(&full[i % C::kStages], (i / C::kStages) & 1, p.err);
    }
    return;
  }

  // ---------------------------------------------------------------- consumers
  float m[GP], l[GP], acc[GP][C::kDims];
#pragma unroll
  for (int g = 0; g < GP; ++g) {
    m[g] = -INFINITY;
    l[g] = 0.f;
#pragma unroll
    for (int j = 0; j < C::kDims; ++j) acc[g][j] = 0.f;
  }
  float* pw = p_s + warp * kPage * GP;
  const int r0 = lane, r1 = lane + 32;
  const int sw = lane & 7;  // swizzle phase of rows r0 and r1

  for (int i = warp; i < npages; i += C::kWarps) {
    const int s = i % C::kStages;
    if (!wait_seq_bounded(&stage_seq[s], i, p.err) ||
        !mbar_wait_bounded(&full[s], (i / C::kStages) & 1, p.err)) {
      abort_flag = 1;
      break;
    }
    const unsigned char* kt = stages + s * C::kStageBytes;
    const unsigned char* vt = kt + C::kTileBytes;
    const int pos0 = (page0 + i) * kPage;
    const int rlo = max(span.lo - pos0, 0);
    const int rhi = min(n - pos0, kPage - 1);

    // Scores for rows r0 and r1 against the G queries.
    float s0[GP], s1[GP];
#pragma unroll
    for (int g = 0; g < GP; ++g) s0[g] = s1[g] = 0.f;
#pragma unroll
    for (int c = 0; c < D / 8; ++c) {
      const unsigned char* box = kt + (c >> 3) * C::kBoxBytes;
      const int chunk = ((c & 7) ^ sw) << 4;
      const uint4 ka = *reinterpret_cast<const uint4*>(box + r0 * 128 + chunk);
      const uint4 kb = *reinterpret_cast<const uint4*>(box + r1 * 128 + chunk);
      const float fa[8] = {bf16_lo(ka.x), bf16_hi(ka.x), bf16_lo(ka.y), bf16_hi(ka.y),
                           bf16_lo(ka.z), bf16_hi(ka.z), bf16_lo(ka.w), bf16_hi(ka.w)};
      const float fb[8] = {bf16_lo(kb.x), bf16_hi(kb.x), bf16_lo(kb.y), bf16_hi(kb.y),
                           bf16_lo(kb.z), bf16_hi(kb.z), bf16_lo(kb.w), bf16_hi(kb.w)};
#pragma unroll
      for (int g = 0; g < GP; ++g) {
        const float4 qa = *reinterpret_cast<const float4*>(q_s + g * D + c * 8);
        const float4 qb = *reinterpret_cast<const float4*>(q_s + g * D + c * 8 + 4);
        const float qv[8] = {qa.x, qa.y, qa.z, qa.w, qb.x, qb.y, qb.z, qb.w};
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          s0[g] = fmaf(qv[e], fa[e], s0[g]);
          s1[g] = fmaf(qv[e], fb[e], s1[g]);
        }
      }
    }
    const bool ok0 = r0 >= rlo && r0 <= rhi;
    const bool ok1 = r1 >= rlo && r1 <= rhi;

    // Online softmax over this page (every visited page has a valid row, so
    // the new running max is finite).
#pragma unroll
    for (int g = 0; g < GP; ++g) {
      const float a0 = ok0 ? s0[g] : -INFINITY;
      const float a1 = ok1 ? s1[g] : -INFINITY;
      const float mn = fmaxf(m[g], warp_max(fmaxf(a0, a1)));
      const float alpha = exp2_approx(m[g] - mn);
      const float p0 = exp2_approx(a0 - mn);
      const float p1 = exp2_approx(a1 - mn);
      l[g] = fmaf(l[g], alpha, p0 + p1);
#pragma unroll
      for (int j = 0; j < C::kDims; ++j) acc[g][j] *= alpha;
      m[g] = mn;
      s0[g] = p0;
      s1[g] = p1;
    }
    if constexpr (GP % 4 == 0) {
#pragma unroll
      for (int g = 0; g < GP; g += 4) {
        *reinterpret_cast<float4*>(pw + r0 * GP + g) = make_float4(s0[g], s0[g + 1], s0[g + 2], s0[g + 3]);
        *reinterpret_cast<float4*>(pw + r1 * GP + g) = make_float4(s1[g], s1[g + 1], s1[g + 2], s1[g + 3]);
      }
    } else {
#pragma unroll
      for (int g = 0; g < GP; ++g) {
        pw[r0 * GP + g] = s0[g];
        pw[r1 * GP + g] = s1[g];
      }
    }
    __syncwarp();

    // P.V over the page's valid rows; lane owns dims [kDims*lane, kDims*(lane+1)).
    for (int r = rlo; r <= rhi; ++r) {
      float pr[GP];
      if constexpr (GP % 4 == 0) {
#pragma unroll
        for (int g = 0; g < GP; g += 4) {
          const float4 t = *reinterpret_cast<const float4*>(pw + r * GP + g);
          pr[g] = t.x;
          pr[g + 1] = t.y;
          pr[g + 2] = t.z;
          pr[g + 3] = t.w;
        }
      } else {
#pragma unroll
        for (int g = 0; g < GP; ++g) pr[g] = pw[r * GP + g];
      }
      float vv[C::kDims];
      if constexpr (D == 64) {
        const uint32_t w = *reinterpret_cast<const uint32_t*>(
            vt + r * 128 + ((((lane >> 2)) ^ (r & 7)) << 4) + (lane & 3) * 4);
        vv[0] = bf16_lo(w);
        vv[1] = bf16_hi(w);
      } else {
        const int l16 = lane & 15;
        const uint2 w = *reinterpret_cast<const uint2*>(
            vt + (lane >> 4) * C::kBoxBytes + r * 128 + (((l16 >> 1) ^ (r & 7)) << 4) +
            (l16 & 1) * 8);
        vv[0] = bf16_lo(w.x);
        vv[1] = bf16_hi(w.x);
        vv[2] = bf16_lo(w.y);
        vv[3] = bf16_hi(w.y);
      }
#pragma unroll
      for (int g = 0; g < GP; ++g)
#pragma unroll
        for (int j = 0; j < C::kDims; ++j) acc[g][j] = fmaf(pr[g], vv[j], acc[g][j]);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
  }

#pragma unroll
  for (int g = 0; g < GP; ++g) l[g] = warp_sum(l[g]);

  constexpr int kConsumers = C::kWarps * 32;
  named_sync(1, kConsumers);  // all pages consumed; the stages are free
  if (abort_flag) return;

  // Merge the four warps' states through shared memory (aliasing the stages).
  float* red = reinterpret_cast<float*>(stages);  // [kWarps][GP][D + 2]
#pragma unroll
  for (int g = 0; g < GP; ++g) {
    float* rw = red + (warp * GP + g) * (D + 2);
#pragma unroll
    for (int j = 0; j < C::kDims; ++j) rw[lane * C::kDims + j] = acc[g][j];
    if (lane == 0) {
      rw[D] = m[g];
      rw[D + 1] = l[g];
    }
  }
  named_sync(1, kConsumers);

  for (int e = tid; e < GP * D; e += kConsumers) {
    const int g = e / D, d = e % D;
    if (g >= p.group) continue;
    float mx = -INFINITY;
#pragma unroll
    for (int w = 0; w < C::kWarps; ++w) mx = fmaxf(mx, red[(w * GP + g) * (D + 2) + D]);
    float a = 0.f, den = 0.f;
#pragma unroll
    for (int w = 0; w < C::kWarps; ++w) {
      const float* rw = red + (w * GP + g) * (D + 2);
      const float f = exp2_approx(rw[D] - mx);  // warps without pages: m = -inf -> 0
      a = fmaf(rw[d], f, a);
      den = fmaf(rw[D + 1], f, den);
    }
    const int h = h0 + g;
    const size_t bh = (size_t)b * p.hq + h;
    if (nsplit == 1) {
      const float sk = p.sinks ? p.sinks[h] * kLog2e : -INFINITY;
      const float mf = fmaxf(mx, sk);
      const float sc = exp2_approx(mx - mf);
      const float total = fmaf(den, sc, exp2_approx(sk - mf));
      p.out[bh * D + d] = __bfloat16_as_ushort(__float2bfloat16_rn(a * sc / total));
    } else {
      p.ws_acc[(bh * p.max_splits + split) * D + d] = a;
      if (d == 0) {
        p.ws_ml[(bh * p.max_splits + split) * 2 + 0] = mx;
        p.ws_ml[(bh * p.max_splits + split) * 2 + 1] = den;
      }
    }
  }
}

// Merges the split partials of rows with two or more splits and folds in the
// sink: M = max(max_i m_i, sink), L = sum_i l_i 2^(m_i - M) + 2^(sink - M),
// out = sum_i acc_i 2^(m_i - M) / L.  Also zeroes inactive rows, rows whose
// position lies beyond their table (recording PGD_EDEVICE_BOUNDS) and rows
// with a split skipped for a bad table entry (marked l < 0).
// One warp per (row, query head); lane l owns dims [D/32 * l, D/32 * (l + 1)).
template <int D>
__global__ void __launch_bounds__(128) paged_decode_combine_kernel(const DecodeParams p) {
  constexpr int kDims = D / 32;
  const int b = blockIdx.y;
  const int h = blockIdx.x * 4 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (h >= p.hq) return;
  const size_t bh = (size_t)b * p.hq + h;
  uint16_t* o = p.out + bh * D + lane * kDims;
  const int n = p.positions[b];
  const bool beyond = n >= 0 && n / kPage >= p.maxp;
  if (n < 0 || beyond) {
    if (beyond && h == 0 && lane == 0) record_error(p.err, PGD_EDEVICE_BOUNDS);
#pragma unroll
    for (int j = 0; j < kDims; ++j) o[j] = 0;
    return;
  }
  const RowSpan span = row_span(n, p.window);
  const int nsplit = (span.pages + p.pages_per_split - 1) / p.pages_per_split;
  if (nsplit <= 1) return;  // written by the split kernel

  const float* ml = p.ws_ml + bh * p.max_splits * 2;
  const float* ac = p.ws_acc + bh * p.max_splits * D + lane * kDims;
  const float sk = p.sinks ? p.sinks[h] * kLog2e : -INFINITY;
  float mx = sk;
  bool skipped = false;
  for (int i = 0; i < nsplit; ++i) {
    mx = fmaxf(mx, ml[2 * i]);
    skipped |= ml[2 * i + 1] < 0.f;
  }
  float res[kDims];
#pragma unroll
  for (int j = 0; j < kDims; ++j) res[j] = 0.f;
  if (skipped || mx == -INFINITY) {
#pragma unroll
    for (int j = 0; j < kDims; ++j) o[j] = 0;
    return;
  }
  float den = exp2_approx(sk - mx);
  for (int i = 0; i < nsplit; ++i) {
    const float f = exp2_approx(ml[2 * i] - mx);
    den = fmaf(ml[2 * i + 1], f, den);
    if constexpr (kDims == 2) {
      const float2 a = *reinterpret_cast<const float2*>(ac + (size_t)i * D);
      res[0] = fmaf(a.x, f, res[0]);
      res[1] = fmaf(a.y, f, res[1]);
    } else {
      const float4 a = *reinterpret_cast<const float4*>(ac + (size_t)i * D);
      res[0] = fmaf(a.x, f, res[0]);
      res[1] = fmaf(a.y, f, res[1]);
      res[2] = fmaf(a.z, f, res[2]);
      res[3] = fmaf(a.w, f, res[3]);
    }
  }
  const float inv = 1.f / den;
#pragma unroll
  for (int j = 0; j < kDims; ++j) o[j] = __bfloat16_as_ushort(__float2bfloat16_rn(res[j] * inv));
}

template <int D, int GP>
cudaError_t launch_decode(const DecodeParams& p, const CUtensorMap& k_map,
                          const CUtensorMap& v_map, int grid_splits, cudaStream_t stream) {
  using C = DecodeCfg<D, GP>;
  static_assert(C::kSmemBytes <= 227 * 1024, "shared memory");
  cudaError_t e = cudaFuncSetAttribute(paged_decode_split_kernel<D, GP>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       C::kSmemBytes);
  if (e != cudaSuccess) return e;
  if (p.rows == 0) return cudaSuccess;
  dim3 grid(grid_splits, p.hkv, p.rows);
  paged_decode_split_kernel<D, GP><<<grid, C::kThreads, C::kSmemBytes, stream>>>(k_map, v_map, p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  dim3 cgrid((p.hq + 3) / 4, p.rows);
  paged_decode_combine_kernel<D><<<cgrid, 128, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace pgd
