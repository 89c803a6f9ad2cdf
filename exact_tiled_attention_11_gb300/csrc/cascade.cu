// Merge of key-chunk partials for cascade decode (sm_103a).
//
// "3.4 Attention Kernels" (llm-learning-path), "Decode attention and Flash-Decoding"
// and "Online softmax": partial results over disjoint key sets combine exactly
// through their log-sum-exps.  The
// shared prefix of a cascade decode is computed as C chunks of keys, each a
// normalised partial (O_c, LSE_c) per (request, head) row; this kernel folds them
// into one (O, LSE) per row:
//     m = max_c LSE_c,  w_c = exp(LSE_c - m),  O = sum_c w_c O_c / sum_c w_c,
//     LSE = m + ln sum_c w_c,
// with a partial of LSE_c = -inf (no keys) weighing nothing.  The result is the
// prefix partial the decode's merge then combines with each request's own keys.
// One warp per row, d / 32 elements per lane.
//
// The prefix pass takes its query rows per KV head: the g = H / Hkv query heads of
// every request that share KV head kvh form rows (request, head in group) of one
// plane, so that a 128-row tile is full and both chains of a CTA work on the same
// K/V tiles.  group_queries_kernel copies q [B, H, d] into that order,
// [Hkv][B * g][d]; the merge writes each row back to its [B, H] position.
#include <cuda_bf16.h>

#include "common.cuh"
#include "kernels.h"

namespace attn {
namespace {

template <int D>
__global__ void __launch_bounds__(256) merge_chunks_kernel(const __nv_bfloat16 *__restrict__ o_parts,
                                                           const float *__restrict__ lse_parts, int C, int rows,
                                                           long long o_stride, long long l_stride, int B, int g,
                                                           __nv_bfloat16 *__restrict__ o, float *__restrict__ lse) {
  constexpr int E = D / 32;
  const int row = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;  // (kvh, request, head in group)
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const int kvh = row / (B * g), rb = row % (B * g);
  const int out_row = (rb / g) * (rows / B) + kvh * g + rb % g;  // (request, head) of [B, H]
  float m = -INFINITY;
  for (int c = 0; c < C; ++c) m = fmaxf(m, lse_parts[c * l_stride + row]);
  float l = 0.f;
  float acc[E];
#pragma unroll
  for (int j = 0; j < E; ++j) acc[j] = 0.f;
  if (m != -INFINITY) {
    for (int c = 0; c < C; ++c) {
      const float lc = lse_parts[c * l_stride + row];
      if (lc == -INFINITY) continue;
      const float w = expf(lc - m);
      l += w;
      const __nv_bfloat16 *src = o_parts + c * o_stride + static_cast<long long>(row) * D + lane * E;
#pragma unroll
      for (int j = 0; j < E; ++j) acc[j] += w * __bfloat162float(src[j]);
    }
  }
  const float inv = l > 0.f ? 1.f / l : 0.f;
  __nv_bfloat16 *dst = o + static_cast<size_t>(out_row) * D + lane * E;
#pragma unroll
  for (int j = 0; j < E; ++j) dst[j] = __float2bfloat16_rn(acc[j] * inv);
  if (lane == 0) lse[out_row] = l > 0.f ? m + logf(l) : -INFINITY;
}

// q [B, H, d] -> qg [Hkv][B * g][d]: 16 bytes per thread
__global__ void __launch_bounds__(256) group_queries_kernel(const uint4 *__restrict__ q, uint4 *__restrict__ qg, int B,
                                                            int H, int g, int chunks_per_row) {
  const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long total = static_cast<long long>(B) * H * chunks_per_row;
  if (i >= total) return;
  const int ch = static_cast<int>(i % chunks_per_row);
  const long long src_row = i / chunks_per_row;  // b * H + h
  const int b = static_cast<int>(src_row / H), h = static_cast<int>(src_row % H);
  const long long dst_row = static_cast<long long>(h / g) * B * g + static_cast<long long>(b) * g + h % g;
  qg[dst_row * chunks_per_row + ch] = q[i];
}

}  // namespace

cudaError_t launch_group_queries(const void *q, void *qg, int B, int H, int Hkv, int d, cudaStream_t stream) {
  const int chunks_per_row = d * 2 / 16;
  const long long total = static_cast<long long>(B) * H * chunks_per_row;
  if (total == 0) return cudaSuccess;
  const int threads = 256;
  group_queries_kernel<<<static_cast<unsigned>((total + threads - 1) / threads), threads, 0, stream>>>(
      static_cast<const uint4 *>(q), static_cast<uint4 *>(qg), B, H, H / Hkv, chunks_per_row);
  return cudaGetLastError();
}

cudaError_t launch_merge_chunks(const void *o_parts, const float *lse_parts, int C, int rows, long long o_stride,
                                long long l_stride, int B, int g, int d, void *o, float *lse, cudaStream_t stream) {
  if (rows <= 0) return cudaSuccess;
  const int threads = 256;
  const int blocks = static_cast<int>((static_cast<long long>(rows) * 32 + threads - 1) / threads);
  const auto *src = static_cast<const __nv_bfloat16 *>(o_parts);
  auto *dst = static_cast<__nv_bfloat16 *>(o);
  if (d == 64)
    merge_chunks_kernel<64><<<blocks, threads, 0, stream>>>(src, lse_parts, C, rows, o_stride, l_stride, B, g, dst,
                                                            lse);
  else
    merge_chunks_kernel<128><<<blocks, threads, 0, stream>>>(src, lse_parts, C, rows, o_stride, l_stride, B, g, dst,
                                                             lse);
  return cudaGetLastError();
}

}  // namespace attn
