// FP8 inputs of the attention: the random orthogonal transform of Q and K and
// the block quantisation of Q', K' and V to e4m3 (sm_103a).
//
// "3.4 Attention Kernels" (llm-learning-path), "FlashAttention-2 and -3":
// FlashAttention-3's FP8 attention quantises by blocks and applies
// "incoherent processing" first, a random orthogonal transform that spreads
// outlier channels before the 8-bit rounding.  Here the transform is
// M = diag(signs) H_d / sqrt(d) (H_d the Sylvester Hadamard matrix), applied to
// the rows of Q and K (Q' K'^T = Q K^T); a block is one 128-row tile of one
// head with one fp32 scale = amax / 448, and each value is stored as the e4m3
// code of x / scale (round to nearest even, saturating).
//
// One CTA per (tensor, head plane, 128-row block), 512 threads (64 registers
// each, so two CTAs per SM): warp w holds rows 8w .. 8w + 7 of the block, lane l
// holds columns 4l .. 4l + 3 of each row (d = 128).  The Hadamard transform is the fast Walsh-Hadamard butterfly
// over the 7 bits of the column index: bits 0-1 inside a lane, bits 2-6 across
// lanes with shuffles.  The 1/sqrt(d) normalisation does not change the codes
// (the block's scale absorbs it), so it is only folded into the stored scale.
// V is written transposed, v8t [plane, d, Nk_pad], so that both MMAs of the
// attention read K-major operands; keys in [Nk, Nk_pad) are zero.
#include "common.cuh"
#include "kernels.h"

namespace attn {
namespace {

constexpr int kRows = 128;
constexpr int kD = 128;
constexpr int kThreads = 512;
constexpr int kRowsPerWarp = kRows / (kThreads / 32);
constexpr float kE4m3Max = 448.f;

// four fp32 values to four e4m3 codes (round to nearest even, saturating), a in the lowest byte
__device__ __forceinline__ uint32_t pack_e4m3x4(float a, float b, float c, float d) {
  uint32_t r;
  asm("{\n\t.reg .b16 lo, hi;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 lo, %2, %1;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 hi, %4, %3;\n\t"
      "mov.b32 %0, {lo, hi};\n\t}"
      : "=r"(r)
      : "f"(a), "f"(b), "f"(c), "f"(d));
  return r;
}

__global__ void __launch_bounds__(kThreads) fp8_quantize_kernel(Fp8QuantJob jq, Fp8QuantJob jk, Fp8QuantJob jv,
                                                                 const float *signs, float transform_norm) {
  __shared__ float warp_max[kThreads / 32];
  __shared__ uint8_t tile[kRows][kD + 4];  // V codes, padded rows for the transposed read
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ---- which tensor and block
  long long id = blockIdx.x;
  const long long nq = static_cast<long long>(jq.planes) * ((jq.N + kRows - 1) / kRows);
  const long long nk = static_cast<long long>(jk.planes) * ((jk.N + kRows - 1) / kRows);
  int which = 0;  // 0: Q, 1: K, 2: V
  if (id >= nq) {
    id -= nq;
    which = 1;
    if (id >= nk) {
      id -= nk;
      which = 2;
    }
  }
  const Fp8QuantJob job = which == 0 ? jq : (which == 1 ? jk : jv);
  const bool transposed = which == 2;
  const bool transform = !transposed && signs != nullptr;
  const int nb = (job.N + kRows - 1) / kRows;
  const long long plane = id / nb;
  const int blk = static_cast<int>(id % nb);
  if (plane >= job.planes) return;

  // ---- load 16 rows x 4 columns per lane (rows past N read as zero)
  float x[kRowsPerWarp][4];
  float sg[4] = {1.f, 1.f, 1.f, 1.f};
  if (transform) {
    const float4 s4 = reinterpret_cast<const float4 *>(signs)[lane];
    sg[0] = s4.x, sg[1] = s4.y, sg[2] = s4.z, sg[3] = s4.w;
  }
#pragma unroll
  for (int r = 0; r < kRowsPerWarp; ++r) {
    const int row = blk * kRows + warp * kRowsPerWarp + r;
    uint2 raw = make_uint2(0u, 0u);
    if (row < job.N) raw = reinterpret_cast<const uint2 *>(job.x + (plane * job.N + row) * kD)[lane];
    x[r][0] = __uint_as_float(raw.x << 16) * sg[0];
    x[r][1] = __uint_as_float(raw.x & 0xFFFF0000u) * sg[1];
    x[r][2] = __uint_as_float(raw.y << 16) * sg[2];
    x[r][3] = __uint_as_float(raw.y & 0xFFFF0000u) * sg[3];
  }
  // ---- x diag(signs) H_d: butterflies over column bits 0, 1 (in lane) and 2..6 (across lanes)
  if (transform) {
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) {
      float a0 = x[r][0] + x[r][1], a1 = x[r][0] - x[r][1];
      float a2 = x[r][2] + x[r][3], a3 = x[r][2] - x[r][3];
      x[r][0] = a0 + a2, x[r][2] = a0 - a2;
      x[r][1] = a1 + a3, x[r][3] = a1 - a3;
#pragma unroll
      for (int m = 1; m < 32; m <<= 1) {
        // lower lane: x + other, upper lane: other - x; fma with +-1 rounds exactly as the add
        const float sgn = (lane & m) ? -1.f : 1.f;
#pragma unroll
        for (int t = 0; t < 4; ++t) x[r][t] = fmaf(sgn, x[r][t], __shfl_xor_sync(0xffffffffu, x[r][t], m));
      }
    }
  }
  // ---- block amax
  float amax = 0.f;
#pragma unroll
  for (int r = 0; r < kRowsPerWarp; ++r)
#pragma unroll
    for (int t = 0; t < 4; ++t) amax = fmaxf(amax, fabsf(x[r][t]));
#pragma unroll
  for (int m = 16; m > 0; m >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, m));
  if (lane == 0) warp_max[warp] = amax;
  __syncthreads();
  amax = warp_max[0];
#pragma unroll
  for (int w = 1; w < kThreads / 32; ++w) amax = fmaxf(amax, warp_max[w]);
  const float inv = amax > 0.f ? kE4m3Max / amax : 0.f;
  if (threadIdx.x == 0) job.scale[plane * nb + blk] = amax / kE4m3Max * (transform ? transform_norm : 1.f);

  // ---- codes
#pragma unroll
  for (int r = 0; r < kRowsPerWarp; ++r) {
    const int rr = warp * kRowsPerWarp + r;
    const int row = blk * kRows + rr;
    const uint32_t c = pack_e4m3x4(x[r][0] * inv, x[r][1] * inv, x[r][2] * inv, x[r][3] * inv);
    if (!transposed) {
      if (row < job.N) reinterpret_cast<uint32_t *>(job.out + (plane * job.N + row) * kD)[lane] = c;
    } else {
      *reinterpret_cast<uint32_t *>(&tile[rr][4 * lane]) = c;
    }
  }
  if (!transposed) return;
  __syncthreads();
  // ---- V^T: row dd of the plane holds the block's keys; 16 keys (one 16-byte store) per step
  const int n_pad = job.n_pad;
#pragma unroll
  for (int i = 0; i < (kD * kRows / 16) / kThreads; ++i) {
    const int chunk = threadIdx.x + i * kThreads;
    const int dd = chunk / (kRows / 16);
    const int kc = chunk % (kRows / 16);
    const int key0 = blk * kRows + kc * 16;
    if (key0 >= n_pad) continue;
    uint32_t w[4];
#pragma unroll
    for (int q = 0; q < 4; ++q)
      w[q] = static_cast<uint32_t>(tile[kc * 16 + 4 * q][dd]) | (static_cast<uint32_t>(tile[kc * 16 + 4 * q + 1][dd]) << 8) |
             (static_cast<uint32_t>(tile[kc * 16 + 4 * q + 2][dd]) << 16) |
             (static_cast<uint32_t>(tile[kc * 16 + 4 * q + 3][dd]) << 24);
    *reinterpret_cast<uint4 *>(job.out + (plane * kD + dd) * n_pad + key0) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

}  // namespace

cudaError_t launch_fp8_quantize(const Fp8QuantJob &q, const Fp8QuantJob &k, const Fp8QuantJob &v, const float *signs,
                                float transform_norm, cudaStream_t stream) {
  auto blocks = [](const Fp8QuantJob &j) {
    return static_cast<long long>(j.planes) * ((j.N + kRows - 1) / kRows);
  };
  const long long total = blocks(q) + blocks(k) + blocks(v);
  if (total == 0) return cudaSuccess;
  if (total > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  fp8_quantize_kernel<<<static_cast<unsigned>(total), kThreads, 0, stream>>>(q, k, v, signs, transform_norm);
  return cudaGetLastError();
}

}  // namespace attn
