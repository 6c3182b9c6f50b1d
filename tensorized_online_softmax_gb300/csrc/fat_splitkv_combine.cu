// Merge of split-KV partial results: every split s of the key range produced
// O_s (normalised over its keys) and LSE_s for each query row; the full
// result is the LSE-weighted average
//     LSE = ln sum_s exp(LSE_s),   O = sum_s exp(LSE_s - LSE) O_s,
// which is exactly softmax attention over the union of the key ranges.
// One warp per query row; memory bound (reads S partial rows, writes one).
#include <cuda_runtime.h>

#include <cstdint>

#include "fat_launch.cuh"

namespace fat {

namespace {

template <int D>
__global__ void __launch_bounds__(256) splitkv_combine_kernel(const float* __restrict__ o_part,
                                                              const float* __restrict__ lse_part,
                                                              float* __restrict__ o,
                                                              float* __restrict__ lse,
                                                              long long rows, int splits) {
  constexpr int kCols = D / 32;  // columns per lane
  const long long row = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  // maximum over the splits' LSE (empty splits hold -inf)
  float m = -INFINITY;
  for (int s = lane; s < splits; s += 32) m = fmaxf(m, lse_part[s * rows + row]);
#pragma unroll
  for (int o_ = 16; o_ > 0; o_ >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o_));
  float acc[kCols];
#pragma unroll
  for (int c = 0; c < kCols; ++c) acc[c] = 0.f;
  float wsum = 0.f;
  for (int s = 0; s < splits; ++s) {
    const float ls = lse_part[s * rows + row];
    if (ls == -INFINITY) continue;  // warp-uniform
    const float w = __expf(ls - m);
    wsum += w;
    const float* src = o_part + (s * rows + row) * D + lane * kCols;
#pragma unroll
    for (int c = 0; c < kCols; ++c) acc[c] = fmaf(w, src[c], acc[c]);
  }
  // a row that no split reaches is empty: O = 0 and LSE = -inf, as the
  // unsplit kernel writes it
  const bool empty = !(wsum > 0.f);
  const float inv = empty ? 0.f : 1.f / wsum;
  float* dst = o + row * D + lane * kCols;
#pragma unroll
  for (int c = 0; c < kCols; ++c) dst[c] = acc[c] * inv;
  if (lane == 0) lse[row] = empty ? -INFINITY : m + __logf(wsum);
}

}  // namespace

// rows = B * H * Nq.  Returns 0 or -4 (launch error).
int launch_splitkv_combine(const float* o_part, const float* lse_part, float* o, float* lse,
                           long long rows, int splits, int d, cudaStream_t stream) {
  const unsigned blocks = static_cast<unsigned>((rows + 7) / 8);
  if (d == 128)
    splitkv_combine_kernel<128><<<blocks, 256, 0, stream>>>(o_part, lse_part, o, lse, rows, splits);
  else
    splitkv_combine_kernel<64><<<blocks, 256, 0, stream>>>(o_part, lse_part, o, lse, rows, splits);
  return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

}  // namespace fat
