// Decode kernels for head_dim 64 (gpt-oss, Qwen2.5 shapes).
#include "paged_decode.cuh"

namespace pgd {

cudaError_t launch_decode_d64(const DecodeParams& p, const CUtensorMap& k_map,
                              const CUtensorMap& v_map, int padded, int kernel, int grid_splits,
                              int pages_per_cta, bool short_rows, cudaStream_t stream) {
  return launch_decode_for_dim<64>(p, k_map, v_map, padded, kernel, grid_splits, pages_per_cta,
                                    short_rows, stream);
}

// Self-test of failure handling.  Thread 0 waits on an mbarrier phase that
// nothing completes and then on a shared word that nothing writes; each wait
// gives up after its limit, records PGD_EDEVICE_TIMEOUT and returns, exactly
// as the decode and prefill kernels' waits do.  The warp then does what a
// decode split CTA does after such a timeout (abandon_split) to a fake row of
// two query heads held in shared memory, whose outputs start as NaN and whose
// partials all start valid: once as the row's only split (its outputs must
// become zero), and once as split 0 of two, after which the combine's merge
// (merge_partials) of the row must give zero although split 1 is valid.
__global__ void bounded_wait_selftest_kernel(unsigned int* err, int* outcome) {
  constexpr int D = 64, G = 2, S = 2;
  constexpr uint16_t kNaN = 0x7fc0;
  __shared__ uint64_t bar;
  __shared__ int word, wait_bits;
  __shared__ __align__(16) float acc[G * S * D];
  __shared__ __align__(16) float ml[G * S * 2];
  __shared__ __align__(16) uint16_t out[G * D];
  const int lane = threadIdx.x;
  if (lane == 0) {
    mbar_init(&bar, 1);
    mbar_init_fence();
    word = 0;
    const bool a = mbar_wait_bounded(&bar, 0, err);  // phase 0 never completes
    const bool b = wait_seq_bounded(&word, 1, err);   // nobody writes 1
    wait_bits = (a ? 1 : 0) | (b ? 2 : 0);
  }
  for (int e = lane; e < G * D; e += 32) out[e] = kNaN;
  for (int e = lane; e < G * S * D; e += 32) acc[e] = 1.f;
  for (int e = lane; e < G * S; e += 32) {
    ml[2 * e] = 0.f;
    ml[2 * e + 1] = 1.f;
  }
  __syncwarp();
  DecodeParams p = {};
  p.out = out;
  p.ws_acc = acc;
  p.ws_ml = ml;
  p.hq = G;
  p.group = G;
  p.max_splits = S;
  int bad = 0;
  abandon_split<D>(p, 0, 0, 0, 1, lane, 32);  // the row's only split
  __syncwarp();
  for (int e = lane; e < G * D; e += 32) bad |= out[e] != 0 ? 1 : 0;
  __syncwarp();
  for (int e = lane; e < G * D; e += 32) out[e] = kNaN;
  __syncwarp();
  abandon_split<D>(p, 0, 0, 0, S, lane, 32);  // split 0 of two
  __syncwarp();
  for (int g = 0; g < G; ++g)
    merge_partials<D>(ml + g * S * 2, 2, acc + g * S * D + lane * (D / 32), D, S, -INFINITY,
                      out + g * D + lane * (D / 32), lane);
  __syncwarp();
  for (int e = lane; e < G * D; e += 32) bad |= out[e] != 0 ? 2 : 0;
  bad = __reduce_or_sync(0xffffffffu, bad);
  if (lane == 0) {
    outcome[0] = wait_bits;
    outcome[1] = bad;
  }
}

cudaError_t launch_bounded_wait_selftest(unsigned int* err, int* outcome, cudaStream_t stream) {
  bounded_wait_selftest_kernel<<<1, 32, 0, stream>>>(err, outcome);
  return cudaGetLastError();
}

}  // namespace pgd
