// Precise fp32 exact-attention forward pass (SIMT), for fp32 inputs.
//
// Same block-wise algorithm as the bf16 kernel ("3.4 Attention Kernels",
// "FlashAttention: tiling"; "FlashAttention and Optimized Kernels", "The
// online softmax"): K/V tiles staged in shared memory, a running max m,
// denominator l and unnormalised output o~ per query row, rescaled by
// exp(m - m') whenever the maximum grows, O = o~ / l and LSE = m + ln l at the
// end, causal tiles after the query skipped.
//
// Precision: with queries scaled by 30 the scores reach the hundreds, and an
// fp32 dot product then carries absolute errors around 1e-5 into exp().  This
// kernel therefore forms every q.k in fp64 (the fp32 products are exact in
// fp64), keeps m, l and o~ in fp64, and evaluates exp in fp32 on the fp64
// difference s - m' rounded once to fp32.  One warp owns one query row: lane j
// computes the score of key j of the tile; the lanes then share the
// probabilities to accumulate the d / 32 output elements each lane owns.
#include "common.cuh"
#include "kernels.h"

namespace attn {
namespace {

constexpr int kRowsPerCta = 8;  // warps per CTA, one query row each
constexpr int kTile = 32;       // keys per tile (one per lane)

template <int D>
__global__ void __launch_bounds__(kRowsPerCta * 32)
    prefill_f32_kernel(const float *__restrict__ q, const float *__restrict__ k, const float *__restrict__ v,
                       PrefillOut out, int H, int Hkv, int Nq, int Nk, int causal, float scale) {
  constexpr int E = D / 32;
  __shared__ float ks[kTile][D + 1];  // +1: lane j reads row j without bank conflicts
  __shared__ float vs[kTile][D];
  __shared__ float qs[kRowsPerCta][D];

  const int b = blockIdx.z;
  const int h = blockIdx.y;
  const int kvh = h / (H / Hkv);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int row0 = blockIdx.x * kRowsPerCta;
  const int row = row0 + warp;
  const bool live_row = row < Nq;

  const float *qh = q + (static_cast<size_t>(b) * H + h) * Nq * D;
  const float *kh = k + (static_cast<size_t>(b) * Hkv + kvh) * Nk * D;
  const float *vh = v + (static_cast<size_t>(b) * Hkv + kvh) * Nk * D;
  const int shift = Nk - Nq;  // causal: query row i attends keys j <= i + shift (aligned to the last key)

  for (int e = lane; e < D; e += 32) qs[warp][e] = live_row ? qh[static_cast<size_t>(row) * D + e] : 0.f;

  double m = -INFINITY, l = 0.0;
  double acc[E];
#pragma unroll
  for (int j = 0; j < E; ++j) acc[j] = 0.0;

  const int last_row = min(Nq, row0 + kRowsPerCta) - 1;
  // tiles wholly after the CTA's last row are skipped
  const int key_end = causal ? max(0, min(Nk, last_row + shift + 1)) : Nk;
  for (int t0 = 0; t0 < key_end; t0 += kTile) {
    __syncthreads();
    for (int idx = threadIdx.x; idx < kTile * D; idx += kRowsPerCta * 32) {
      const int r = idx / D, e = idx % D;
      const bool in = t0 + r < Nk;
      ks[r][e] = in ? kh[static_cast<size_t>(t0 + r) * D + e] : 0.f;
      vs[r][e] = in ? vh[static_cast<size_t>(t0 + r) * D + e] : 0.f;
    }
    __syncthreads();

    const int key = t0 + lane;
    const bool attend = live_row && key < Nk && (!causal || key <= row + shift);
    double s = -INFINITY;
    if (attend) {
      double dot = 0.0;
#pragma unroll 8
      for (int e = 0; e < D; ++e) dot = fma(static_cast<double>(qs[warp][e]), static_cast<double>(ks[lane][e]), dot);
      s = dot * static_cast<double>(scale);
    }
    double tmax = s;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) tmax = fmax(tmax, __shfl_xor_sync(0xffffffffu, tmax, off));
    if (tmax == -INFINITY) continue;  // nothing attended in this tile (warp-uniform)
    const double m_new = fmax(m, tmax);
    const double corr = (m == -INFINITY) ? 0.0 : static_cast<double>(expf(static_cast<float>(m - m_new)));
    const float p = attend ? expf(static_cast<float>(s - m_new)) : 0.f;
    double psum = p;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) psum += __shfl_xor_sync(0xffffffffu, psum, off);
    l = l * corr + psum;
#pragma unroll
    for (int j = 0; j < E; ++j) acc[j] *= corr;
    for (int jj = 0; jj < kTile; ++jj) {
      const float pj = __shfl_sync(0xffffffffu, p, jj);
      if (pj == 0.f) continue;
#pragma unroll
      for (int j = 0; j < E; ++j) acc[j] = fma(static_cast<double>(pj), static_cast<double>(vs[jj][lane + 32 * j]), acc[j]);
    }
    m = m_new;
  }

  if (!live_row) return;
  float *oh = static_cast<float *>(out.o) + b * out.o_b + h * out.o_h + row * out.o_r;
  const double inv = (l > 0.0) ? 1.0 / l : 0.0;
#pragma unroll
  for (int j = 0; j < E; ++j) oh[lane + 32 * j] = static_cast<float>(acc[j] * inv);
  if (out.lse != nullptr && lane == 0) {
    out.lse[b * out.l_b + h * out.l_h + row * out.l_r] = (l > 0.0) ? static_cast<float>(m + log(l)) : -INFINITY;
  }
}

}  // namespace

ATTN_DEFINE_ERROR_ACCESSOR(device_error_prefill_f32)

cudaError_t launch_prefill_f32(const float *q, const float *k, const float *v, const PrefillOut &out, int B, int H,
                               int Hkv, int Nq, int Nk, int d, bool causal, float scale, cudaStream_t stream) {
  dim3 grid((Nq + kRowsPerCta - 1) / kRowsPerCta, H, B);
  if (d == 64) {
    prefill_f32_kernel<64><<<grid, kRowsPerCta * 32, 0, stream>>>(q, k, v, out, H, Hkv, Nq, Nk, causal ? 1 : 0, scale);
  } else {
    prefill_f32_kernel<128><<<grid, kRowsPerCta * 32, 0, stream>>>(q, k, v, out, H, Hkv, Nq, Nk, causal ? 1 : 0, scale);
  }
  return cudaGetLastError();
}

}  // namespace attn
