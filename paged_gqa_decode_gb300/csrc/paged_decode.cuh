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
// adds to the denominator.  Scores are carried in log2 units (multiplied by
// scale * log2 e), so every exponential is one ex2.
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
// barrier, so every parity wait targets the barrier's current phase.
//
// Consumer warps (four; two for splits of at most three pages, so more CTAs
// share an SM) take whole pages in turn, each keeping its own fp32
// online-softmax state for the group's query heads.  Two consumers:
//   - MmaConsumer (default, group <= 8): the page's 64 x G scores are
//     S^T = K q^T on the tensor cores (mma.sync m16n8k16, bf16 in, fp32
//     accumulate; K fragments by ldmatrix from the swizzled tile, q as
//     register fragments, the group padded to 8 heads), the probabilities
//     are re-packed in registers (a bf16x2 head and residual, transposed by
//     movmatrix) as the B operand of O^T += V^T P^T (V fragments by
//     ldmatrix.trans), so P.V keeps fp32-level accuracy.
//   - ScalarConsumer: the same on CUDA cores (lane r owns tile rows r and
//     r + 32 for the scores; lane l owns D/32 output dims for P.V).
// At the end the warps' states are merged through shared memory.  A row with
// one split writes its output directly (sink included); otherwise the split
// writes (m, l, acc) to the workspace and the combine kernel merges.  When no
// row has more than one split the combine kernel is not launched at all.
//
// Decode step (the append fused in): the split holding a row's last page
// also writes the row's new K and V at the slot of its position -- the
// producer warp's other lanes store while lane 0 copies the earlier pages --
// and fences those writes before the last page's copy, which reads them.
//
// Pages wholly outside the window are never visited (the split range starts
// at the window's first page).  Positions outside the window or past n inside
// a visited page get a -inf score before the softmax; the scalar consumer
// skips them in P.V and the MMA consumer zeroes their V rows in shared memory
// first (a zero weight times a non-finite stale value would otherwise leak),
// so nothing outside the attended set reaches the result.
#pragma once

#include <math.h>

#include <atomic>
#include <type_traits>

#include "pgd_device.cuh"
#include "pgd_internal.h"

namespace pgd {

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kBoxBytes = kPage * 64 * 2;  // one TMA box: 64 rows x 128 bytes

// ------------------------------------------------------------------ tensor-core helpers

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                              uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// d += a * b for one m16n8k16 tile, bf16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
      "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Two fp32 values as a bf16x2 word (round to nearest even), `lo` in bits 0-15.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}

// Transpose of an 8x8 b16 matrix held one bf16x2 per lane.
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t a) {
  uint32_t d;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
  return d;
}

// Orders this thread's generic-proxy shared-memory writes before later
// async-proxy (TMA) accesses of the same bytes.
__device__ __forceinline__ void fence_proxy_async_shared() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ------------------------------------------------------------------ consumers

// Tensor-core consumer: one warp, whole pages, group padded to 8 heads.
// Fragment ownership (m16n8k16): lane = 4 * gid + tig.  Score tile t covers
// page rows 16t..16t+15; the lane holds rows 16t + gid (+8) of heads 2tig and
// 2tig + 1.  Output tile mt covers dims 16mt..16mt+15; the lane holds dims
// 16mt + gid (+8) of the same two heads.
template <int D>
struct MmaConsumer {
  static constexpr int kHeads = 8;
  static constexpr int kSteps = D / 16;  // k-steps of Q.K^T and dim tiles of P.V
  static constexpr int kSharedFloats = 0;

  uint32_t qb[kSteps][2];  // q^T fragments (B operand), bf16x2
  float o[kSteps][4];      // O^T accumulators
  float m[2], l[2];        // running max (log2 units) and per-lane denominator
  uint32_t off_k[4], off_v[4];
  int gid, tig;
  float c;

  __device__ static void prepare_shared(float*, const DecodeParams&, int, int, int, int) {}

  __device__ void init(const DecodeParams& p, int b, int h0, int lane, const float*) {
    gid = lane >> 2;
    tig = lane & 3;
    c = p.q_scale_log2;
    const bool live = gid < p.group;
    const uint32_t* qrow =
        reinterpret_cast<const uint32_t*>(p.q + ((size_t)b * p.hq + h0 + (live ? gid : 0)) * D);
#pragma unroll
    for (int kk = 0; kk < kSteps; ++kk) {
      qb[kk][0] = live ? qrow[(16 * kk + 2 * tig) >> 1] : 0u;
      qb[kk][1] = live ? qrow[(16 * kk + 8 + 2 * tig) >> 1] : 0u;
#pragma unroll
      for (int e = 0; e < 4; ++e) o[kk][e] = 0.f;
    }
    m[0] = m[1] = -INFINITY;
    l[0] = l[1] = 0.f;
    // ldmatrix row addresses: lane supplies row (lane & 7) of matrix (lane >> 3).
    // K (no transpose): matrix j holds rows +8*(j&1), 16-byte chunk +(j>>1).
    // V (transpose):    matrix j holds rows +8*(j>>1), chunk +(j&1).
    // Rows are 128-byte swizzled: chunk c of row r sits at chunk c ^ (r & 7).
    const int j = lane >> 3, r = lane & 7;
    const uint32_t row_k = ((j & 1) * 8 + r) * 128, x_k = (j >> 1) ^ r;
    const uint32_t row_v = ((j >> 1) * 8 + r) * 128, x_v = (j & 1) ^ r;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      off_k[i] = row_k + ((x_k ^ (2 * i)) << 4);
      off_v[i] = row_v + ((x_v ^ (2 * i)) << 4);
    }
  }

  // One page (NT = 4: 64 rows), or NT / 4 of one (the window kernel's
  // 32-row slices): kt is the shared address of its K rows, vt_ptr its V
  // rows, valid rows [rlo, rhi].  Returns true if it wrote zeros into V.
  template <int NT = 4>
  __device__ bool page(uint32_t kt, unsigned char* vt_ptr, int rlo, int rhi, int lane) {
    static_assert(NT == 2 || NT == 4, "row tiles");
    const uint32_t vt = smem_addr(vt_ptr);
    float s[NT][4];
#pragma unroll
    for (int t = 0; t < NT; ++t)
#pragma unroll
      for (int e = 0; e < 4; ++e) s[t][e] = 0.f;
#pragma unroll
    for (int kk = 0; kk < kSteps; ++kk)
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4(kt + (kk >> 2) * kBoxBytes + t * 2048 + off_k[kk & 3], a0, a1, a2, a3);
        mma_bf16(s[t], a0, a1, a2, a3, qb[kk][0], qb[kk][1]);
      }

    const bool full = rlo == 0 && rhi == 16 * NT - 1;
#pragma unroll
    for (int t = 0; t < NT; ++t)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int row = 16 * t + gid + ((e & 2) ? 8 : 0);
        const float v = s[t][e] * c;
        s[t][e] = (full || (row >= rlo && row <= rhi)) ? v : -INFINITY;
      }
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      mx0 = fmaxf(mx0, fmaxf(s[t][0], s[t][2]));
      mx1 = fmaxf(mx1, fmaxf(s[t][1], s[t][3]));
    }
#pragma unroll
    for (int x = 4; x < 32; x <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, x));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, x));
    }
    const float mn0 = fmaxf(m[0], mx0), mn1 = fmaxf(m[1], mx1);
    const float ref0 = mn0 == -INFINITY ? 0.f : mn0;
    const float ref1 = mn1 == -INFINITY ? 0.f : mn1;
    const float al0 = exp2_approx(m[0] - ref0), al1 = exp2_approx(m[1] - ref1);
    float sum0 = 0.f, sum1 = 0.f;
    // P as the B operand of P.V, split into a bf16 head and a bf16 residual
    // (p = hi + lo to ~2^-17 relative) so the products keep fp32-level
    // accuracy: one bf16 rounding of p alone would err by up to 2^-9 of
    // sum_j p_j |v_j|, far more than an output near cancellation allows.
    uint32_t pb[NT][2], pl[NT][2];
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      s[t][0] = exp2_approx(s[t][0] - ref0);
      s[t][1] = exp2_approx(s[t][1] - ref1);
      s[t][2] = exp2_approx(s[t][2] - ref0);
      s[t][3] = exp2_approx(s[t][3] - ref1);
      sum0 += s[t][0] + s[t][2];
      sum1 += s[t][1] + s[t][3];
      // rows gid / gid + 8 of heads (2tig, 2tig+1), transposed into the
      // B-operand layout (rows 2tig, 2tig+1 (+8) of head gid).
      const uint32_t h01 = pack_bf16x2(s[t][0], s[t][1]);
      const uint32_t h23 = pack_bf16x2(s[t][2], s[t][3]);
      const uint32_t l01 = pack_bf16x2(s[t][0] - bf16_lo(h01), s[t][1] - bf16_hi(h01));
      const uint32_t l23 = pack_bf16x2(s[t][2] - bf16_lo(h23), s[t][3] - bf16_hi(h23));
      pb[t][0] = movmatrix_trans(h01);
      pb[t][1] = movmatrix_trans(h23);
      pl[t][0] = movmatrix_trans(l01);
      pl[t][1] = movmatrix_trans(l23);
    }
    l[0] = fmaf(l[0], al0, sum0);
    l[1] = fmaf(l[1], al1, sum1);
    m[0] = mn0;
    m[1] = mn1;
#pragma unroll
    for (int mt = 0; mt < kSteps; ++mt) {
      o[mt][0] *= al0;
      o[mt][1] *= al1;
      o[mt][2] *= al0;
      o[mt][3] *= al1;
    }

    if (!full) {  // zero the V rows outside [rlo, rhi]
      const uint4 z = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
      for (int half = 0; half < NT / 2; ++half) {
        const int row = lane + 32 * half;
        if (row < rlo || row > rhi) {
#pragma unroll
          for (int bx = 0; bx < D / 64; ++bx)
#pragma unroll
            for (int ch = 0; ch < 8; ++ch)
              *reinterpret_cast<uint4*>(vt_ptr + bx * kBoxBytes + row * 128 + ch * 16) = z;
        }
      }
      __syncwarp();
    }

#pragma unroll
    for (int mt = 0; mt < kSteps; ++mt)
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4_trans(vt + (mt >> 2) * kBoxBytes + t * 2048 + off_v[mt & 3], a0, a1, a2, a3);
        mma_bf16(o[mt], a0, a1, a2, a3, pb[t][0], pb[t][1]);
        mma_bf16(o[mt], a0, a1, a2, a3, pl[t][0], pl[t][1]);
      }
    return !full;
  }

  __device__ void finish() {
#pragma unroll
    for (int x = 4; x < 32; x <<= 1) {
      l[0] += __shfl_xor_sync(0xffffffffu, l[0], x);
      l[1] += __shfl_xor_sync(0xffffffffu, l[1], x);
    }
  }

  // red: [warps][kHeads][D + 2] = (acc[D], m, l)
  __device__ void store(float* red, int warp, int) const {
#pragma unroll
    for (int mt = 0; mt < kSteps; ++mt)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int head = 2 * tig + (e & 1);
        const int dim = 16 * mt + gid + ((e & 2) ? 8 : 0);
        red[(warp * kHeads + head) * (D + 2) + dim] = o[mt][e];
      }
    if (gid == 0) {
      float* r0 = red + (warp * kHeads + 2 * tig) * (D + 2);
      float* r1 = r0 + (D + 2);
      r0[D] = m[0];
      r0[D + 1] = l[0];
      r1[D] = m[1];
      r1[D + 1] = l[1];
    }
  }
};

// CUDA-core consumer for a group padded to GP heads.
template <int D, int GP>
struct ScalarConsumer {
  static constexpr int kHeads = GP;
  static constexpr int kDims = D / 32;  // output dims per lane
  // q (fp32, scaled to log2 units) and a per-warp probability buffer
  static constexpr int kQFloats = GP * D;
  static constexpr int kPFloatsPerWarp = kPage * GP;
  static constexpr int kSharedFloats = kQFloats + 4 * kPFloatsPerWarp;

  float m[GP], l[GP], acc[GP][kDims];
  const float* q_s;
  float* pw;

  __device__ static void prepare_shared(float* shared, const DecodeParams& p, int b, int h0,
                                        int tid, int nthreads) {
    for (int e = tid; e < GP * D; e += nthreads) {
      const int g = e / D, d = e % D;
      float v = 0.f;
      if (g < p.group) {
        const uint16_t bits = p.q[((size_t)b * p.hq + h0 + g) * D + d];
        v = __uint_as_float((uint32_t)bits << 16) * p.q_scale_log2;
      }
      shared[e] = v;
    }
  }

  __device__ void init(const DecodeParams&, int, int, int, const float* shared) {
    q_s = shared;
    pw = const_cast<float*>(shared) + kQFloats;
#pragma unroll
    for (int g = 0; g < GP; ++g) {
      m[g] = -INFINITY;
      l[g] = 0.f;
#pragma unroll
      for (int j = 0; j < kDims; ++j) acc[g][j] = 0.f;
    }
  }

  __device__ void set_warp(int warp) { pw += warp * kPFloatsPerWarp; }

  __device__ bool page(uint32_t, unsigned char* kt_ptr, int rlo, int rhi, int lane) {
    const unsigned char* kt = kt_ptr;
    const unsigned char* vt = kt_ptr + kPage * D * 2;
    const int r0 = lane, r1 = lane + 32;
    const int sw = lane & 7;
    float s0[GP], s1[GP];
#pragma unroll
    for (int g = 0; g < GP; ++g) s0[g] = s1[g] = 0.f;
#pragma unroll
    for (int c = 0; c < D / 8; ++c) {
      const unsigned char* box = kt + (c >> 3) * kBoxBytes;
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
        const float4 qc = *reinterpret_cast<const float4*>(q_s + g * D + c * 8 + 4);
        const float qv[8] = {qa.x, qa.y, qa.z, qa.w, qc.x, qc.y, qc.z, qc.w};
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          s0[g] = fmaf(qv[e], fa[e], s0[g]);
          s1[g] = fmaf(qv[e], fb[e], s1[g]);
        }
      }
    }
    const bool ok0 = r0 >= rlo && r0 <= rhi;
    const bool ok1 = r1 >= rlo && r1 <= rhi;
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
      for (int j = 0; j < kDims; ++j) acc[g][j] *= alpha;
      m[g] = mn;
      s0[g] = p0;
      s1[g] = p1;
    }
    if constexpr (GP % 4 == 0) {
#pragma unroll
      for (int g = 0; g < GP; g += 4) {
        *reinterpret_cast<float4*>(pw + r0 * GP + g) =
            make_float4(s0[g], s0[g + 1], s0[g + 2], s0[g + 3]);
        *reinterpret_cast<float4*>(pw + r1 * GP + g) =
            make_float4(s1[g], s1[g + 1], s1[g + 2], s1[g + 3]);
      }
    } else {
#pragma unroll
      for (int g = 0; g < GP; ++g) {
        pw[r0 * GP + g] = s0[g];
        pw[r1 * GP + g] = s1[g];
      }
    }
    __syncwarp();
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
      float vv[kDims];
      if constexpr (D == 64) {
        const uint32_t w = *reinterpret_cast<const uint32_t*>(
            vt + r * 128 + ((((lane >> 2)) ^ (r & 7)) << 4) + (lane & 3) * 4);
        vv[0] = bf16_lo(w);
        vv[1] = bf16_hi(w);
      } else {
        const int l16 = lane & 15;
        const uint2 w = *reinterpret_cast<const uint2*>(
            vt + (lane >> 4) * kBoxBytes + r * 128 + (((l16 >> 1) ^ (r & 7)) << 4) +
            (l16 & 1) * 8);
        vv[0] = bf16_lo(w.x);
        vv[1] = bf16_hi(w.x);
        vv[2] = bf16_lo(w.y);
        vv[3] = bf16_hi(w.y);
      }
#pragma unroll
      for (int g = 0; g < GP; ++g)
#pragma unroll
        for (int j = 0; j < kDims; ++j) acc[g][j] = fmaf(pr[g], vv[j], acc[g][j]);
    }
    return false;
  }

  __device__ void finish() {
#pragma unroll
    for (int g = 0; g < GP; ++g) l[g] = warp_sum(l[g]);
  }

  __device__ void store(float* red, int warp, int lane) const {
#pragma unroll
    for (int g = 0; g < GP; ++g) {
      float* rw = red + (warp * GP + g) * (D + 2);
#pragma unroll
      for (int j = 0; j < kDims; ++j) rw[lane * kDims + j] = acc[g][j];
      if (lane == 0) {
        rw[D] = m[g];
        rw[D + 1] = l[g];
      }
    }
  }
};

// ------------------------------------------------------------------ split kernel

// What a split CTA leaves behind when it gives up on its pages (a table
// entry outside the pool, or a pipeline wait that timed out): with one split
// per row it writes zeros as its query heads' outputs; otherwise it marks its
// partials skipped (m = -inf, l = -1, accumulator zero), and the combine then
// writes zeros for the row's heads.  Either way nothing the CTA read reaches
// an output, and no partial a later merge reads is left from another call.
// Threads tid = 0 .. nthreads - 1 of the caller share the writes.
template <int D>
__device__ __forceinline__ void abandon_split(const DecodeParams& p, int b, int h0, int split,
                                              int nsplit, int tid, int nthreads) {
  for (int e = tid; e < p.group * D; e += nthreads) {
    const int g = e / D, d = e % D;
    const size_t bh = (size_t)b * p.hq + h0 + g;
    if (nsplit == 1) {
      p.out[bh * D + d] = 0;
    } else {
      p.ws_acc[(bh * p.max_splits + split) * D + d] = 0.f;
      if (d == 0) {
        p.ws_ml[(bh * p.max_splits + split) * 2 + 0] = -INFINITY;
        p.ws_ml[(bh * p.max_splits + split) * 2 + 1] = -1.f;
      }
    }
  }
}

template <int D, int STAGES, class Consumer, int WARPS = 4>
struct DecodeCfg {
  static constexpr int kWarps = WARPS;  // consumer warps
  static constexpr int kThreads = (kWarps + 1) * 32;
  static constexpr int kBoxes = D / 64;
  static constexpr int kTileBytes = kPage * D * 2;
  static constexpr int kStageBytes = 2 * kTileBytes;  // K tile then V tile
  static constexpr int kStages = STAGES;
  static constexpr int kHeads = Consumer::kHeads;
  static constexpr int kSmemBytes =
      1024 + kStages * kStageBytes + Consumer::kSharedFloats * 4 + 2 * kStages * 8;
  // CTAs per SM the shared memory allows (228 KB per SM) and that leave at
  // least 136 registers per thread (three 160-thread CTAs, seven 64-thread
  // ones); the CUDA-core consumer keeps its registers (no bound).
  static constexpr int kSmemBlocks = (228 * 1024) / (kSmemBytes + 1024);
  static constexpr int kRegBlocks = 65536 / (kThreads * 136);
  static constexpr int kMinBlocks =
      Consumer::kSharedFloats > 0 ? 1 : (kSmemBlocks < kRegBlocks ? kSmemBlocks : kRegBlocks);
  static_assert(kWarps * kHeads * (D + 2) * 4 <= kStages * kStageBytes, "merge buffer");
  static_assert(D == 64 || D == 128, "head_dim");
};

template <int D, int STAGES, class Consumer, int WARPS>
__global__ void __launch_bounds__(DecodeCfg<D, STAGES, Consumer, WARPS>::kThreads,
                                  DecodeCfg<D, STAGES, Consumer, WARPS>::kMinBlocks)
    paged_decode_split_kernel(const __grid_constant__ CUtensorMap k_map,
                              const __grid_constant__ CUtensorMap v_map, const DecodeParams p) {
  using C = DecodeCfg<D, STAGES, Consumer, WARPS>;
  constexpr int GP = C::kHeads;
  pdl_wait();
  pdl_allow_dependents();
  const int split = blockIdx.x;
  const int kvh = blockIdx.y;
  const int b = blockIdx.z;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

  // Without a window a split's pages start at index split * pages_per_split
  // of its table row whatever the position, so the table entries it may need
  // are loaded together with the position rather than after it.
  const bool spec = p.window == 0 && p.table != nullptr && p.row_of == nullptr;
  int pg_spec = -1;
  if (spec && tid < p.pages_per_split && split * p.pages_per_split + tid < p.maxp)
    pg_spec = p.table[(size_t)b * p.maxp + split * p.pages_per_split + tid];
  const int n = p.positions[b];
  const RowSpan span = row_span(n, p.window);
  const int nsplit = (span.pages + p.pages_per_split - 1) / p.pages_per_split;
  const int h0 = kvh * p.group;
  // With one split per row (a grid one split wide) no combine kernel runs:
  // this CTA zeroes its heads' outputs of an inactive or out-of-range row
  // itself (and the kv head 0 CTA reports the latter).
  const bool alone = gridDim.x == 1;
  auto zero_heads = [&]() {
    for (int e = tid; e < p.group * D; e += C::kThreads)
      p.out[((size_t)b * p.hq + h0 + e / D) * D + e % D] = 0;
  };
  if (split >= nsplit) {  // inactive row, or past this row's splits
    if (alone && n < 0) zero_heads();
    return;
  }
  const int table_row = p.row_of ? p.row_of[b] : b;
  if (n / kPage >= p.maxp || (p.row_of && (table_row < 0 || table_row >= p.table_rows))) {
    // otherwise reported and zeroed by the combine kernel
    if (alone) {
      zero_heads();
      if (kvh == 0 && tid == 0) record_error(p.err, PGD_EDEVICE_BOUNDS);
    }
    return;
  }
  const int page0 = span.first_page + split * p.pages_per_split;
  const int npages = min(p.pages_per_split, span.pages - split * p.pages_per_split);
  const int32_t* trow = p.table ? p.table + (size_t)table_row * p.maxp + page0 : nullptr;
  const int dense0 = table_row * p.maxp + page0;  // page of index page0 without a table

  extern __shared__ unsigned char smem_raw[];
  unsigned char* stages = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* cshared = reinterpret_cast<float*>(stages + C::kStages * C::kStageBytes);
  uint64_t* full = reinterpret_cast<uint64_t*>(cshared + Consumer::kSharedFloats);
  uint64_t* empty = full + C::kStages;
  __shared__ int abort_flag;
  __shared__ int stage_seq[C::kStages];  // page index last issued into each stage

  // Every table entry this split reads must name a pool page.
  bool bad = false;
  for (int i = tid; i < npages; i += C::kThreads) {
    const int pg = spec && i == tid ? pg_spec : (trow ? trow[i] : dense0 + i);
    bad |= (pg < 0) | (pg >= p.num_pages);
  }
  bad = __syncthreads_or(bad);
  if (bad) {
    if (tid == 0) record_error(p.err, PGD_EDEVICE_BOUNDS);
    abandon_split<D>(p, b, h0, split, nsplit, tid, C::kThreads);
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
  Consumer::prepare_shared(cshared, p, b, h0, tid, C::kThreads);
  __syncthreads();

  // ---------------------------------------------------------------- producer
  if (warp == C::kWarps) {
    // Decode step: the split holding the row's last page writes the new
    // token's K and V at their slot (position n) -- lanes 1.. store while
    // lane 0 already copies the earlier pages -- and the warp orders those
    // writes before the copy of the last page, which reads them back.
    const bool append = p.k_new != nullptr && page0 + npages - 1 == n / kPage;
    if (append) {
      const int page = trow ? trow[npages - 1] : dense0 + npages - 1;
      const size_t dst =
          ((size_t)tile_first_row(p.layout, page, kvh, p.hkv, p.num_pages, p.maxp) + n % kPage) * D;
      const size_t src = ((size_t)b * p.hkv + kvh) * D;
      for (int c = lane - 1; c >= 0 && c < D / 8; c += 31) {
        *reinterpret_cast<uint4*>(p.k_pool + dst + 8 * c) =
            *reinterpret_cast<const uint4*>(p.k_new + src + 8 * c);
        *reinterpret_cast<uint4*>(p.v_pool + dst + 8 * c) =
            *reinterpret_cast<const uint4*>(p.v_new + src + 8 * c);
      }
    }
    int issued = 0;
    bool ok = true;
    // Copies page i into its stage once the stage is free (lane 0).
    auto issue = [&](int i) {
      const int s = i % C::kStages;
      // On a timeout the consumers time out on the pages never issued and
      // abandon the split themselves; only they write abort_flag.
      if (i >= C::kStages && !mbar_wait_bounded(&empty[s], ((i / C::kStages) - 1) & 1, p.err))
        return false;
      const int page = trow ? trow[i] : dense0 + i;
      const int y = (int)tile_first_row(p.layout, page, kvh, p.hkv, p.num_pages, p.maxp);
      unsigned char* st = stages + s * C::kStageBytes;
      mbar_arrive_expect_tx(&full[s], C::kStageBytes);
#pragma unroll
      for (int bx = 0; bx < C::kBoxes; ++bx) {
        tma_load_2d(st + bx * kBoxBytes, &k_map, bx * 64, y, &full[s]);
        tma_load_2d(st + C::kTileBytes + bx * kBoxBytes, &v_map, bx * 64, y, &full[s]);
      }
      *reinterpret_cast<volatile int*>(&stage_seq[s]) = i;
      issued = i + 1;
      return true;
    };
    if (lane == 0) {
      prefetch_tensormap(&k_map);
      prefetch_tensormap(&v_map);
      for (int i = 0; i < npages - (append ? 1 : 0) && ok; ++i) ok = issue(i);
    }
    if (append) {
      asm volatile("fence.proxy.async.global;" ::: "memory");
      __syncwarp();
      if (lane == 0 && ok) issue(npages - 1);
    }
    if (lane == 0) {
      // No copy may still be landing in shared memory when the CTA exits.
      for (int i = max(0, issued - C::kStages); i < issued; ++i)
        mbar_wait_bounded(&full[i % C::kStages], (i / C::kStages) & 1, p.err);
    }
    return;
  }

  // ---------------------------------------------------------------- consumers
  Consumer cons;
  cons.init(p, b, h0, lane, cshared);
  if constexpr (Consumer::kSharedFloats > 0) cons.set_warp(warp);

  for (int i = warp; i < npages; i += C::kWarps) {
    const int s = i % C::kStages;
    if (!wait_seq_bounded(&stage_seq[s], i, p.err) ||
        !mbar_wait_bounded(&full[s], (i / C::kStages) & 1, p.err)) {
      abort_flag = 1;
      break;
    }
    unsigned char* kt = stages + s * C::kStageBytes;
    const int pos0 = (page0 + i) * kPage;
    const int rlo = max(span.lo - pos0, 0);
    const int rhi = min(n - pos0, kPage - 1);
    bool wrote;
    if constexpr (Consumer::kSharedFloats > 0)
      wrote = cons.page(0u, kt, rlo, rhi, lane);
    else
      wrote = cons.page(smem_addr(kt), kt + C::kTileBytes, rlo, rhi, lane);
    if (wrote) fence_proxy_async_shared();
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
  }
  cons.finish();

  constexpr int kConsumers = C::kWarps * 32;
  named_sync(1, kConsumers);  // all pages consumed; the stages are free
  if (abort_flag) {  // a wait timed out (recorded): the split contributes nothing
    abandon_split<D>(p, b, h0, split, nsplit, tid, kConsumers);
    return;
  }

  // Merge the warps' states through shared memory (aliasing the stages).
  float* red = reinterpret_cast<float*>(stages);  // [kWarps][GP][D + 2]
  cons.store(red, warp, lane);
  named_sync(1, kConsumers);

  for (int e = tid; e < p.group * D; e += kConsumers) {
    const int g = e / D, d = e % D;
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

// Merges nsplit >= 2 partials of one (row, query head) and folds in the
// sink: M = max(max_i m_i, sink), L = sum_i l_i 2^(m_i - M) + 2^(sink - M),
// out = sum_i acc_i 2^(m_i - M) / L, written as bf16 to o.  Partial i is
// (m, l) at ml + i * ml_stride and acc at ac + i * ac_stride (ac already
// offset to this lane's dims).  A partial marked l < 0 (skipped for a bad
// table entry or an abandoned wait) zeroes the output.
// One warp; lane l owns dims [D/32 * l, D/32 * (l + 1)).  The partials'
// (m, l) are read 32 at a time, one per lane, together with the first
// kEarly accumulators, so the merge costs about one round trip to L2; the
// weights are then broadcast by shuffle.
template <int D>
__device__ __forceinline__ void merge_partials(const float* ml, int ml_stride, const float* ac,
                                               int ac_stride, int nsplit, float sk, uint16_t* o,
                                               int lane) {
  constexpr int kDims = D / 32;
  constexpr int kEarly = 8;
  using Vec = typename std::conditional<kDims == 2, float2, float4>::type;
  Vec early[kEarly];
#pragma unroll
  for (int k = 0; k < kEarly; ++k)
    if (k < nsplit) early[k] = *reinterpret_cast<const Vec*>(ac + (size_t)k * ac_stride);
  float mx = sk;
  bool skipped = false;
  for (int base = 0; base < nsplit; base += 32) {
    const int i = base + lane;
    const float2 mli = i < nsplit ? *reinterpret_cast<const float2*>(ml + (size_t)i * ml_stride)
                                  : make_float2(-INFINITY, 0.f);
    mx = fmaxf(mx, warp_max(mli.x));
    skipped |= __any_sync(0xffffffffu, mli.y < 0.f);
  }
  if (skipped || mx == -INFINITY) {
#pragma unroll
    for (int j = 0; j < kDims; ++j) o[j] = 0;
    return;
  }
  float res[kDims];
#pragma unroll
  for (int j = 0; j < kDims; ++j) res[j] = 0.f;
  float den = 0.f;
  auto add = [&](const Vec& v, float f) {
    res[0] = fmaf(v.x, f, res[0]);
    res[1] = fmaf(v.y, f, res[1]);
    if constexpr (kDims == 4) {
      res[2] = fmaf(v.z, f, res[2]);
      res[3] = fmaf(v.w, f, res[3]);
    }
  };
  for (int base = 0; base < nsplit; base += 32) {
    const int i = base + lane;
    const float2 mli = i < nsplit ? *reinterpret_cast<const float2*>(ml + (size_t)i * ml_stride)
                                  : make_float2(-INFINITY, 0.f);
    const float fi = i < nsplit ? exp2_approx(mli.x - mx) : 0.f;
    den += warp_sum(i < nsplit ? mli.y * fi : 0.f);
    const int cnt = min(32, nsplit - base);
    int k = 0;
    if (base == 0) {
#pragma unroll
      for (; k < kEarly; ++k)
        if (k < cnt) add(early[k], __shfl_sync(0xffffffffu, fi, k));
      k = min(kEarly, cnt);
    }
#pragma unroll 4
    for (; k < cnt; ++k)
      add(*reinterpret_cast<const Vec*>(ac + (size_t)(base + k) * ac_stride),
          __shfl_sync(0xffffffffu, fi, k));
  }
  den += exp2_approx(sk - mx);
  const float inv = 1.f / den;
#pragma unroll
  for (int j = 0; j < kDims; ++j) o[j] = __bfloat16_as_ushort(__float2bfloat16_rn(res[j] * inv));
}

// Combine for the split kernel: merges the partials of rows with two or
// more splits (merge_partials).  Also zeroes inactive rows and rows whose
// position lies beyond their table or whose table row is out of range
// (recording PGD_EDEVICE_BOUNDS).  One warp per (row, query head).
template <int D>
__global__ void __launch_bounds__(128) paged_decode_combine_kernel(const DecodeParams p) {
  constexpr int kDims = D / 32;
  const int b = blockIdx.y;
  const int h = blockIdx.x * 4 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  // positions, the token rows and the sinks are inputs of the split kernel
  // as well, which reads them only after its own dependency wait; this grid
  // starts after every split CTA has passed that wait, so they are final
  // here and are read before this grid's wait, off its critical path.
  const bool live = h < p.hq;
  const size_t bh = (size_t)b * p.hq + (live ? h : 0);
  const int n = p.positions[b];
  const int table_row = p.row_of ? p.row_of[b] : b;
  const float sk = (p.sinks && live) ? p.sinks[h] * kLog2e : -INFINITY;
  pdl_wait();
  pdl_allow_dependents();
  if (!live) return;
  uint16_t* o = p.out + bh * D + lane * kDims;
  const bool beyond = n >= 0 && (n / kPage >= p.maxp ||
                                 (p.row_of && (table_row < 0 || table_row >= p.table_rows)));
  if (n < 0 || beyond) {
    if (beyond && h == 0 && lane == 0) record_error(p.err, PGD_EDEVICE_BOUNDS);
#pragma unroll
    for (int j = 0; j < kDims; ++j) o[j] = 0;
    return;
  }
  const RowSpan span = row_span(n, p.window);
  const int nsplit = (span.pages + p.pages_per_split - 1) / p.pages_per_split;
  if (nsplit <= 1) return;  // written by the split kernel
  merge_partials<D>(p.ws_ml + bh * p.max_splits * 2, 2,
                    p.ws_acc + bh * p.max_splits * D + lane * kDims, D, nsplit, sk, o, lane);
}

// ------------------------------------------------------------------ window kernel

// 16-byte copy global -> shared that bypasses the registers (and L1);
// `bytes` 0 writes 16 zero bytes and reads nothing.
__device__ __forceinline__ void cp_async16(void* dst, const void* src, uint32_t bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_addr(dst)), "l"(src),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;" ::: "memory");
}

// Sliding-window decode for windows of at most 64 * TILES positions
// (GPT-OSS 20B model files, src/attention.linnet, SinkAttention.decode_rows:
// key s is seen when n - window < s <= n).  A unit of 2 * TILES warps per
// (row, kv head) attends over exactly the window's positions, wherever they
// fall in the row's pages, so no byte outside the window is read and no split
// or combine is needed.  A CTA holds UNITS units, each on its own shared
// memory and named barrier.  Local row r holds position lo + r; warp w owns local
// rows 32 w .. 32 w + 31: it reads the row's position and the table entries
// itself, copies its rows of K and V, 16 bytes per lane at a time, straight
// into shared memory (cp.async; rows past the attended count are
// zero-filled), waits for its own copies only and runs the tensor-core
// consumer on them, so each warp computes as soon as its slice has landed.
// The rows land in the layout a TMA page tile has (64-row tiles of
// 128-byte-swizzled 64-value boxes), which the consumer reads.  The warps
// merge through shared memory (a barrier once every warp is done with the
// rows, another once their partials are stored): each thread owns a run of
// one head's output dims, forms that head's weight per warp (its running max
// against the overall one and the sink, over the total denominator) and
// stores its run with 8- or 16-byte writes.
//
// Decode step (the append fused in): the new token's row (position n, the
// window's last) is copied from k_new / v_new instead of the pool, and
// stored into the pool at its slot by the warp owning that row, so the
// kernel never reads the slot back.
template <int D, int TILES, int UNITS = 1>
struct WindowCfg {
  static constexpr int kWarps = 2 * TILES;  // one warp per 32 rows of a unit
  static constexpr int kUnitThreads = 32 * kWarps;
  static constexpr int kThreads = UNITS * kUnitThreads;
  static constexpr int kChunks = D / 8;                // 16-byte chunks per row
  static constexpr int kRowStep = 32 / kChunks;        // rows one warp pass covers
  static constexpr int kPasses = 32 / kRowStep;
  static constexpr int kTileBytes = kPage * D * 2;     // 64 rows of K (or V)
  static constexpr int kBytes = TILES * kTileBytes;    // the window's K (or V)
  static constexpr int kUnitSmem = 2 * kBytes;
  static constexpr int kSmemBytes = UNITS * kUnitSmem;
  static constexpr int kMinBlocks = UNITS == 1 ? (228 * 1024) / (kUnitSmem + 1024) : 1;
  static constexpr int kHeads = MmaConsumer<D>::kHeads;
  // output dims per thread (at least 4: with many warps, threads past
  // kHeads * D / 4 have no output run and only copy and compute)
  static constexpr int kPerThread = kHeads * D / kUnitThreads >= 4 ? kHeads * D / kUnitThreads : 4;
  static constexpr int kRun = kPerThread >= 8 ? 8 : 4;          // dims per store
  static_assert(kPerThread % kRun == 0 && D % kPerThread == 0, "output runs");
  static_assert(kWarps * kHeads * (D + 2) * 4 <= kBytes, "merge buffer");
  static_assert(UNITS >= 1 && UNITS <= 15 && kThreads <= 1024 && kSmemBytes <= 227 * 1024,
                "units per CTA");
};

// The most units one CTA can hold: shared memory, threads, and the 15 named
// barriers a CTA has besides barrier 0.
template <int D, int TILES>
constexpr int window_max_units() {
  using C = WindowCfg<D, TILES>;
  int u = (227 * 1024) / C::kUnitSmem;
  if (u > 1024 / C::kUnitThreads) u = 1024 / C::kUnitThreads;
  return u < 15 ? u : 15;
}

template <int D, int TILES, int UNITS>
__global__ void __launch_bounds__(WindowCfg<D, TILES, UNITS>::kThreads,
                                  WindowCfg<D, TILES, UNITS>::kMinBlocks)
    paged_decode_window_kernel(const DecodeParams p) {
  using C = WindowCfg<D, TILES, UNITS>;
  using Consumer = MmaConsumer<D>;
  constexpr int GP = C::kHeads;
  pdl_wait();
  pdl_allow_dependents();
  // unit u of this CTA: (row b, kv head kvh), units numbered row-major
  const int u = UNITS == 1 ? 0 : (int)threadIdx.x / C::kUnitThreads;
  const int unit = blockIdx.x * UNITS + u;
  if (unit >= p.rows * p.hkv) return;
  const int kvh = unit % p.hkv;
  const int b = unit / p.hkv;
  const int tid = UNITS == 1 ? (int)threadIdx.x : (int)threadIdx.x % C::kUnitThreads;
  // the unit's barrier: its own threads only (barrier 1 + u)
  auto unit_sync = [&]() {
    if constexpr (UNITS == 1)
      __syncthreads();
    else
      asm volatile("bar.sync %0, %1;" ::"r"(1 + u), "r"(C::kUnitThreads) : "memory");
  };
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int h0 = kvh * p.group;
  // the output run this thread merges and stores: head g, dims d0 ..
  const int g = tid / (D / C::kPerThread);
  const int d0 = (tid % (D / C::kPerThread)) * C::kPerThread;
  const bool live = g < p.group;
  const float sink = (p.sinks && live) ? p.sinks[h0 + g] * kLog2e : -INFINITY;
  uint16_t* out = p.out + ((size_t)b * p.hq + h0 + (live ? g : 0)) * D + d0;
  auto zero_run = [&]() {
    if (live)
#pragma unroll
      for (int k = 0; k < C::kPerThread; k += 4)
        *reinterpret_cast<uint2*>(out + k) = make_uint2(0u, 0u);
  };
  const int n = p.positions[b];
  const int table_row = p.row_of ? p.row_of[b] : b;
  if (n < 0) {  // inactive row
    zero_run();
    return;
  }
  if (n / kPage >= p.maxp || (p.row_of && (table_row < 0 || table_row >= p.table_rows))) {
    zero_run();
    if (kvh == 0 && tid == 0) record_error(p.err, PGD_EDEVICE_BOUNDS);
    return;
  }
  const int lo = n - p.window + 1 > 0 ? n - p.window + 1 : 0;
  const int cnt = n - lo + 1;  // attended positions, at most 64 * TILES
  const int first_page = lo / kPage;
  const int npages = n / kPage - first_page + 1;  // at most TILES + 1
  // The window's table entries: lane k of every warp loads entry k (every
  // warp reaches the same verdict).
  int pg = 0;
  if (lane < npages) pg = page_of(p.table, table_row, first_page + lane, p.maxp);
  if (__any_sync(0xffffffffu, lane < npages && (pg < 0 || pg >= p.num_pages))) {
    zero_run();
    if (tid == 0) record_error(p.err, PGD_EDEVICE_BOUNDS);
    return;
  }

  Consumer cons;
  cons.init(p, b, h0, lane, nullptr);  // q fragments load while the rows copy

  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* ks = smem_raw + u * C::kUnitSmem;
  unsigned char* vs = ks + C::kBytes;
  const bool append = p.k_new != nullptr;
  const int c = lane % C::kChunks;  // this lane's 16-byte column
  // element offset of column c of position 64 k of the window's page k
  size_t page_base[TILES + 1];
#pragma unroll
  for (int k = 0; k <= TILES; ++k)
    page_base[k] = (size_t)tile_first_row(p.layout, __shfl_sync(0xffffffffu, pg, k), kvh, p.hkv,
                                          p.num_pages, p.maxp) * D + 8 * c;
  auto pool_at = [&](int s) {
    const int k = (s >> 6) - first_page;
    size_t at = page_base[0];
#pragma unroll
    for (int q = 1; q <= TILES; ++q)
      if (k == q) at = page_base[q];
    return at + (size_t)(s & (kPage - 1)) * D;
  };
  const size_t new_at = ((size_t)b * p.hkv + kvh) * D + 8 * c;
  const int row0 = 32 * warp + lane / C::kChunks;
  const int col = (c / 8) * kBoxBytes;
#pragma unroll
  for (int j = 0; j < C::kPasses; ++j) {
    const int r = row0 + j * C::kRowStep;
    const int s = lo + r;
    const size_t at = pool_at(s);
    const bool here = r < cnt;
    const bool fresh = append && s == n;
    const int off = (r >> 6) * C::kTileBytes + col + (r & (kPage - 1)) * 128 +
                    (((c & 7) ^ (r & 7)) << 4);
    cp_async16(ks + off, !here ? (const void*)p.k_read : fresh ? (const void*)(p.k_new + new_at)
                                                              : (const void*)(p.k_read + at),
               here ? 16u : 0u);
    cp_async16(vs + off, !here ? (const void*)p.v_read : fresh ? (const void*)(p.v_new + new_at)
                                                              : (const void*)(p.v_read + at),
               here ? 16u : 0u);
  }
  if (append && (cnt - 1) / 32 == warp && lane < C::kChunks) {  // the new token into the pool
    const size_t at = pool_at(n);
    *reinterpret_cast<uint4*>(p.k_pool + at) = *reinterpret_cast<const uint4*>(p.k_new + new_at);
    *reinterpret_cast<uint4*>(p.v_pool + at) = *reinterpret_cast<const uint4*>(p.v_new + new_at);
  }
  cp_async_wait_all();
  __syncwarp();

  const int rhi = min(cnt - 1 - 32 * warp, 31);
  if (rhi >= 0) {
    const int slice = (warp >> 1) * C::kTileBytes + (warp & 1) * 32 * 128;
    cons.template page<2>(smem_addr(ks + slice), vs + slice, 0, rhi, lane);
  }
  cons.finish();
  unit_sync();  // every warp of the unit is done with the rows

  float* red = reinterpret_cast<float*>(ks);  // [kWarps][GP][D + 2]
  cons.store(red, warp, lane);
  unit_sync();
  if (!live) return;
  float mx = sink, f[C::kWarps];
#pragma unroll
  for (int w = 0; w < C::kWarps; ++w) {
    f[w] = red[(w * GP + g) * (D + 2) + D];
    mx = fmaxf(mx, f[w]);
  }
  float total = exp2_approx(sink - mx);
#pragma unroll
  for (int w = 0; w < C::kWarps; ++w) {
    f[w] = exp2_approx(f[w] - mx);  // a warp without rows: m = -inf -> 0
    total = fmaf(red[(w * GP + g) * (D + 2) + D + 1], f[w], total);
  }
  const float inv = 1.f / total;
#pragma unroll
  for (int w = 0; w < C::kWarps; ++w) f[w] *= inv;
  constexpr int R = C::kRun;
#pragma unroll
  for (int k = 0; k < C::kPerThread; k += R) {
    float a[R];
#pragma unroll
    for (int e = 0; e < R; ++e) a[e] = 0.f;
#pragma unroll
    for (int w = 0; w < C::kWarps; ++w) {
      const float* rw = red + (w * GP + g) * (D + 2) + d0 + k;
#pragma unroll
      for (int e = 0; e < R; e += 2) {
        const float2 v = *reinterpret_cast<const float2*>(rw + e);
        a[e] = fmaf(v.x, f[w], a[e]);
        a[e + 1] = fmaf(v.y, f[w], a[e + 1]);
      }
    }
    if constexpr (R == 8)
      *reinterpret_cast<uint4*>(out + k) =
          make_uint4(pack_bf16x2(a[0], a[1]), pack_bf16x2(a[2], a[3]), pack_bf16x2(a[4], a[5]),
                     pack_bf16x2(a[6], a[7]));
    else
      *reinterpret_cast<uint2*>(out + k) = make_uint2(pack_bf16x2(a[0], a[1]),
                                                      pack_bf16x2(a[2], a[3]));
  }
}

template <int D, int TILES, int UNITS>
cudaError_t launch_window_units(const DecodeParams& p, cudaStream_t stream) {
  using C = WindowCfg<D, TILES, UNITS>;
  auto kern = paged_decode_window_kernel<D, TILES, UNITS>;
  static std::atomic<bool> configured[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !configured[dev].load(std::memory_order_acquire)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) configured[dev].store(true, std::memory_order_release);
  }
  if (p.rows == 0) return cudaSuccess;
  const int units = p.rows * p.hkv;
  return launch_pdl(kern, dim3((units + UNITS - 1) / UNITS), dim3(C::kThreads), C::kSmemBytes,
                    stream, p);
}

// One unit (row, kv head) per CTA lets the block scheduler fill each SM with
// kMinBlocks CTAs.  When that takes two rounds but the units fit one round of
// CTAs holding as many units as shared memory allows (the hardware reserves
// shared memory per CTA, so one large CTA per SM holds a unit more), the large
// CTAs are launched instead: one round, no second wave of late units.
template <int D, int TILES>
cudaError_t launch_window(const DecodeParams& p, cudaStream_t stream) {
  constexpr int kUnits = window_max_units<D, TILES>();
  if constexpr (kUnits > WindowCfg<D, TILES>::kMinBlocks) {
    static std::atomic<int> sms[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    int n = dev >= 0 && dev < 64 ? sms[dev].load(std::memory_order_relaxed) : 0;
    if (n == 0) {
      e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
      if (e != cudaSuccess) return e;
      if (dev >= 0 && dev < 64) sms[dev].store(n, std::memory_order_relaxed);
    }
    const long long units = (long long)p.rows * p.hkv;
    if (units > (long long)n * WindowCfg<D, TILES>::kMinBlocks && units <= (long long)n * kUnits)
      return launch_window_units<D, TILES, kUnits>(p, stream);
  }
  return launch_window_units<D, TILES, 1>(p, stream);
}

template <int D, int STAGES, class Consumer, int WARPS = 4>
cudaError_t launch_decode(const DecodeParams& p, const CUtensorMap& k_map,
                          const CUtensorMap& v_map, int grid_splits, cudaStream_t stream) {
  using C = DecodeCfg<D, STAGES, Consumer, WARPS>;
  auto kern = paged_decode_split_kernel<D, STAGES, Consumer, WARPS>;
  static_assert(C::kSmemBytes <= 227 * 1024, "shared memory");
  // The shared-memory opt-in is per device; set it once on each.
  static std::atomic<bool> configured[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !configured[dev].load(std::memory_order_acquire)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) configured[dev].store(true, std::memory_order_release);
  }
  if (p.rows == 0) return cudaSuccess;
  dim3 grid(grid_splits, p.hkv, p.rows);
  e = launch_pdl(kern, grid, dim3(C::kThreads), C::kSmemBytes, stream, k_map, v_map, p);
  if (e != cudaSuccess || grid_splits == 1) return e;  // one split: written directly
  dim3 cgrid((p.hq + 3) / 4, p.rows);
  return launch_pdl(paged_decode_combine_kernel<D>, cgrid, dim3(128), 0, stream, p);
}

// Splits of at most 3 pages (windows, short tables) are latency-bound: they
// run with kShortWarps consumer warps and a ring of kShortStages3 stages for
// 3 pages, so more CTAs share an SM.
constexpr int kShortWarps = 2;
constexpr int kShortStages3 = 3;

// Kernel choice for one head_dim: the tensor-core consumer unless the caller
// asks for the CUDA-core one.
template <int D>
cudaError_t launch_decode_for_dim(const DecodeParams& p, const CUtensorMap& k_map,
                                  const CUtensorMap& v_map, int padded, int kernel,
                                  int grid_splits, int pages_per_cta, bool short_rows,
                                  cudaStream_t stream) {
  constexpr int kStages = D == 128 ? 3 : 6;
  if (kernel == PGD_KERNEL_AUTO && p.window > 0 && p.window <= kMaxWindowKernel)
    return p.window <= kPage ? launch_window<D, 1>(p, stream) : launch_window<D, 2>(p, stream);
  if (short_rows && p.window == 0) {
    // Full attention over a table of a few pages: the window kernel with the
    // whole table as its window (every row's positions 0 .. n are then in
    // it: n < 64 x the table width, which the kernel checks).
    DecodeParams q = p;
    switch (short_row_tiles(D, p.maxp)) {
      case 1: q.window = kPage; return launch_window<D, 1>(q, stream);
      case 2: q.window = 2 * kPage; return launch_window<D, 2>(q, stream);
      case 4: q.window = 4 * kPage; return launch_window<D, 4>(q, stream);
      case 10:
        if constexpr (D == 64) {
          q.window = 10 * kPage;
          return launch_window<D, 10>(q, stream);
        }
        break;
      default: break;
    }
  }
  if (kernel != PGD_KERNEL_CUDA_CORE) {
    // A ring no deeper than the pages a split can stream: shallower rings let
    // more CTAs share an SM when splits are short (windows, small contexts).
    if (pages_per_cta <= 1)
      return launch_decode<D, 1, MmaConsumer<D>, kShortWarps>(p, k_map, v_map, grid_splits, stream);
    if (pages_per_cta <= 2)
      return launch_decode<D, 2, MmaConsumer<D>, kShortWarps>(p, k_map, v_map, grid_splits, stream);
    if (D == 64 && pages_per_cta <= 3)
      return launch_decode<D, kShortStages3, MmaConsumer<D>, kShortWarps>(p, k_map, v_map, grid_splits, stream);
    return launch_decode<D, kStages, MmaConsumer<D>>(p, k_map, v_map, grid_splits, stream);
  }
  switch (padded) {
    case 1: return launch_decode<D, kStages, ScalarConsumer<D, 1>>(p, k_map, v_map, grid_splits, stream);
    case 2: return launch_decode<D, kStages, ScalarConsumer<D, 2>>(p, k_map, v_map, grid_splits, stream);
    case 4: return launch_decode<D, kStages, ScalarConsumer<D, 4>>(p, k_map, v_map, grid_splits, stream);
    case 8: return launch_decode<D, kStages, ScalarConsumer<D, 8>>(p, k_map, v_map, grid_splits, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace pgd
