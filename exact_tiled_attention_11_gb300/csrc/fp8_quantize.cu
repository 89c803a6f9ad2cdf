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
// One CTA per (tensor, head plane, 128-row block), 512 threads: warp w holds
// rows 8w .. 8w + 7 of the block, two rows per pass, sixteen lanes per row, lane l
// columns 8 (l mod 16) .. + 7 (d = 128; one 16-byte load per lane and row).  The
// Hadamard transform is the fast Walsh-Hadamard butterfly over the 7 bits of the
// column index: bits 0-2 inside the lane (bits 1-2 on packed f32x2 pairs), bits 3-6
// across the row's sixteen lanes with shuffles.  The 1/sqrt(d) normalisation does not change the codes
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

// packed fp32 pairs (Blackwell f32x2 forms)
__device__ __forceinline__ uint64_t f2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_split(uint64_t r, float &lo, float &hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(r));
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t sub2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

__global__ void __launch_bounds__(kThreads) fp8_quantize_kernel(Fp8QuantJob jq, Fp8QuantJob jk, Fp8QuantJob jv,
                                                                 const float *signs, float transform_norm) {
  __shared__ float warp_max[kThreads / 32];
  __shared__ uint8_t tile[kRows][kD + 4];  // V codes; a 132-byte pitch keeps the column reads conflict-free
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int seg = lane & 15;      // this lane's columns: 8 seg .. 8 seg + 7
  const int half = lane >> 4;     // which of the pass's two rows

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

  // ---- rows 8 warp + 2 p + half (p = 0..3), 8 columns each, times the signs; rows past N read as zero
  float sg[8] = {1.f, 1.f, 1.f, 1.f, 1.f, 1.f, 1.f, 1.f};
  if (transform) {
    const float4 s0 = reinterpret_cast<const float4 *>(signs + seg * 8)[0];
    const float4 s1 = reinterpret_cast<const float4 *>(signs + seg * 8)[1];
    sg[0] = s0.x, sg[1] = s0.y, sg[2] = s0.z, sg[3] = s0.w, sg[4] = s1.x, sg[5] = s1.y, sg[6] = s1.z, sg[7] = s1.w;
  }
  float x[kRowsPerWarp / 2][8];
#pragma unroll
  for (int p = 0; p < kRowsPerWarp / 2; ++p) {
    const int row = blk * kRows + warp * kRowsPerWarp + 2 * p + half;
    uint4 raw = make_uint4(0u, 0u, 0u, 0u);
    if (row < job.N) raw = reinterpret_cast<const uint4 *>(job.x + (plane * job.N + row) * kD)[seg];
    const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      x[p][2 * k] = __uint_as_float(w[k] << 16) * sg[2 * k];
      x[p][2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u) * sg[2 * k + 1];
    }
  }
  // ---- x diag(signs) H_d: column bits 0..2 in the lane, bits 3..6 across the row's 16 lanes
  if (transform) {
#pragma unroll
    for (int p = 0; p < kRowsPerWarp / 2; ++p) {
#pragma unroll
      for (int i = 0; i < 8; i += 2) {  // bit 0
        const float a = x[p][i], c = x[p][i + 1];
        x[p][i] = a + c, x[p][i + 1] = a - c;
      }
#pragma unroll
      for (int st = 2; st < 8; st <<= 1) {  // bits 1, 2 on packed pairs (i, i + 1)
#pragma unroll
        for (int i = 0; i < 8; i += 2) {
          if (i & st) continue;
          const uint64_t lo = f2(x[p][i], x[p][i + 1]), hi = f2(x[p][i + st], x[p][i + st + 1]);
          f2_split(add2(lo, hi), x[p][i], x[p][i + 1]);
          f2_split(sub2(lo, hi), x[p][i + st], x[p][i + st + 1]);
        }
      }
#pragma unroll
      for (int m = 1; m < 16; m <<= 1) {  // bits 3..6: lanes seg ^ m of the same row
        // lower lane: x + other, upper lane: other - x; fma with +-1 rounds exactly as the add
        const float sgn = (seg & m) ? -1.f : 1.f;
#pragma unroll
        for (int t = 0; t < 8; ++t) x[p][t] = fmaf(sgn, x[p][t], __shfl_xor_sync(0xffffffffu, x[p][t], m));
      }
    }
  }
  // ---- block amax
  float amax = 0.f;
#pragma unroll
  for (int p = 0; p < kRowsPerWarp / 2; ++p)
#pragma unroll
    for (int t = 0; t < 8; ++t) amax = fmaxf(amax, fabsf(x[p][t]));
#pragma unroll
  for (int m = 16; m > 0; m >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, m));
  if (lane == 0) warp_max[warp] = amax;
  __syncthreads();
  amax = warp_max[0];
#pragma unroll
  for (int w = 1; w < kThreads / 32; ++w) amax = fmaxf(amax, warp_max[w]);
  const float inv = amax > 0.f ? kE4m3Max / amax : 0.f;
  if (threadIdx.x == 0) job.scale[plane * nb + blk] = amax / kE4m3Max * (transform ? transform_norm : 1.f);

  // ---- codes: 8 bytes per lane and row
#pragma unroll
  for (int p = 0; p < kRowsPerWarp / 2; ++p) {
    const int row_in = warp * kRowsPerWarp + 2 * p + half;
    const int row = blk * kRows + row_in;
    const uint32_t c0 = pack_e4m3x4(x[p][0] * inv, x[p][1] * inv, x[p][2] * inv, x[p][3] * inv);
    const uint32_t c1 = pack_e4m3x4(x[p][4] * inv, x[p][5] * inv, x[p][6] * inv, x[p][7] * inv);
    if (!transposed) {
      if (row < job.N) reinterpret_cast<uint2 *>(job.out + (plane * job.N + row) * kD)[seg] = make_uint2(c0, c1);
    } else {
      uint32_t *t = reinterpret_cast<uint32_t *>(&tile[row_in][8 * seg]);
      t[0] = c0;
      t[1] = c1;
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
