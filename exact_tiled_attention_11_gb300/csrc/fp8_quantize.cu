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
// One CTA per (tensor, head plane, 128-row block), 128 threads, thread t = row t of the
// block.  The block's 32 KB of bf16 is contiguous in memory: it is staged in shared memory
// with coalesced 16-byte cp.async copies (a 272-byte row pitch keeps both the staging
// writes and each thread's row reads free of bank conflicts), each thread takes its row
// into registers, applies the signs to the bf16 sign bits, and runs the whole 128-point
// Walsh-Hadamard butterfly in registers: values are held as packed f32x2 pairs
// (x[k], x[k + 64]), the stage on column bit 6 is the scalar first stage and the six
// stages on bits 0..5 are packed add/sub between pairs k and k ^ 2^b.  The 1/sqrt(d)
// normalisation does not change the codes (the block's scale absorbs it), so it is only
// folded into the stored scale.  Codes are staged in shared memory and written out
// coalesced.  V is written transposed, v8t [plane, d, Nk_pad], so that both MMAs of the
// attention read K-major operands; keys in [Nk, Nk_pad) are zero.
#include "common.cuh"
#include "kernels.h"

namespace attn {
namespace {

constexpr int kRows = 128;
constexpr int kD = 128;
constexpr int kThreads = 128;   // one per row
constexpr int kInPitch = 272;   // bytes per staged bf16 row (256 + 16)
constexpr int kOutPitch = 144;  // bytes per staged code row (128 + 16)
constexpr int kVPitch = 132;    // bytes per staged V code row for the transposed copy-out
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
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

struct alignas(16) QuantSmem {
  uint8_t rows[kRows * kInPitch];  // staged bf16 rows; later the codes (kOutPitch or kVPitch rows)
  uint32_t sign_bits[kD / 2];      // per bf16 pair: the sign bits the transform's signs flip
  float warp_max[kThreads / 32];
};

__global__ void __launch_bounds__(kThreads, 3) fp8_quantize_kernel(Fp8QuantJob jq, Fp8QuantJob jk, Fp8QuantJob jv,
                                                                    const float *signs, float transform_norm) {
  __shared__ QuantSmem sm;
  const int t = threadIdx.x;
  const int warp = t >> 5;
  const int lane = t & 31;

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
  const int rows = min(kRows, job.N - blk * kRows);  // rows of this block inside the tensor

  // ---- stage the block: 16-byte chunk c = row c / 16, bytes 16 (c mod 16) .. + 15
  const uint8_t *src = reinterpret_cast<const uint8_t *>(job.x + (plane * job.N + static_cast<long long>(blk) * kRows) * kD);
  const uint32_t rows_s = smem_u32(sm.rows);
#pragma unroll
  for (int i = 0; i < kRows * kD * 2 / 16 / kThreads; ++i) {
    const int c = t + i * kThreads;
    if ((c >> 4) < rows) cp_async16(rows_s + (c >> 4) * kInPitch + (c & 15) * 16, src + c * 16);
  }
  if (transform && t < kD / 2)
    sm.sign_bits[t] = (signs[2 * t] < 0.f ? 0x8000u : 0u) | (signs[2 * t + 1] < 0.f ? 0x80000000u : 0u);
  asm volatile("cp.async.wait_all;" ::: "memory");
  __syncthreads();

  // ---- this row: x[k] and x[k + 64] as one packed pair, signs applied to the bf16 sign bits
  uint64_t x[kD / 2];
  {
    uint32_t w[kD / 2];  // bf16 pairs (columns 2j, 2j + 1)
#pragma unroll
    for (int i = 0; i < kD / 8; ++i) {
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (t < rows) v = *reinterpret_cast<const uint4 *>(sm.rows + t * kInPitch + i * 16);
      w[4 * i] = v.x, w[4 * i + 1] = v.y, w[4 * i + 2] = v.z, w[4 * i + 3] = v.w;
    }
    if (transform) {
#pragma unroll
      for (int i = 0; i < kD / 8; ++i) {
        const uint4 m = reinterpret_cast<const uint4 *>(sm.sign_bits)[i];
        w[4 * i] ^= m.x, w[4 * i + 1] ^= m.y, w[4 * i + 2] ^= m.z, w[4 * i + 3] ^= m.w;
      }
    }
#pragma unroll
    for (int k = 0; k < kD / 2; ++k) {
      // column k is the low or high half of word k / 2, column k + 64 of word 32 + k / 2
      const uint32_t a = w[k >> 1], b = w[32 + (k >> 1)];
      const float xa = __uint_as_float((k & 1) ? (a & 0xFFFF0000u) : (a << 16));
      const float xb = __uint_as_float((k & 1) ? (b & 0xFFFF0000u) : (b << 16));
      // column bit 6 first (scalar): (x[k], x[k + 64]) -> (x[k] + x[k + 64], x[k] - x[k + 64])
      x[k] = transform ? f2(xa + xb, xa - xb) : f2(xa, xb);
    }
  }
  if (transform) {
    // column bits 0..5: packed butterflies between pairs k and k ^ m
#pragma unroll
    for (int m = 1; m < kD / 2; m <<= 1) {
#pragma unroll
      for (int k = 0; k < kD / 2; ++k) {
        if (k & m) continue;
        const uint64_t lo = x[k], hi = x[k | m];
        x[k] = add2(lo, hi);
        x[k | m] = sub2(lo, hi);
      }
    }
  }
  // ---- block amax
  float amax = 0.f;
#pragma unroll
  for (int k = 0; k < kD / 2; ++k) {
    float a, b;
    f2_split(x[k], a, b);
    amax = fmaxf(amax, fmaxf(fabsf(a), fabsf(b)));
  }
#pragma unroll
  for (int m = 16; m > 0; m >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, m));
  if (lane == 0) sm.warp_max[warp] = amax;
  __syncthreads();  // also: every row has been read out of the staging buffer
  amax = fmaxf(fmaxf(sm.warp_max[0], sm.warp_max[1]), fmaxf(sm.warp_max[2], sm.warp_max[3]));
  const float inv = amax > 0.f ? kE4m3Max / amax : 0.f;
  if (t == 0) job.scale[plane * nb + blk] = amax / kE4m3Max * (transform ? transform_norm : 1.f);

  // ---- codes of this row: columns 16 i .. 16 i + 15 -> one 16-byte word
  const uint64_t inv2 = f2(inv, inv);
  const int pitch = transposed ? kVPitch : kOutPitch;
#pragma unroll
  for (int i = 0; i < kD / 16; ++i) {
    uint32_t c[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      // columns 16 i + 4 q .. + 3: the low (i < 4) or high (i >= 4) halves of pairs (16 i + 4 q) mod 64 ..
      const int k0 = (16 * i + 4 * q) & 63;
      float v[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float lo, hi;
        f2_split(mul2(x[k0 + e], inv2), lo, hi);
        v[e] = i < 4 ? lo : hi;
      }
      c[q] = pack_e4m3x4(v[0], v[1], v[2], v[3]);
    }
    uint8_t *dst = sm.rows + t * pitch + i * 16;
    if (transposed) {  // 4-byte aligned rows (the 132-byte pitch)
#pragma unroll
      for (int q = 0; q < 4; ++q) reinterpret_cast<uint32_t *>(dst)[q] = c[q];
    } else {
      *reinterpret_cast<uint4 *>(dst) = make_uint4(c[0], c[1], c[2], c[3]);
    }
  }
  __syncthreads();

  if (!transposed) {
    // ---- row-major codes, coalesced: chunk c = row c / 8, bytes 16 (c mod 8) .. + 15
    uint8_t *dst = job.out + (plane * job.N + static_cast<long long>(blk) * kRows) * kD;
#pragma unroll
    for (int i = 0; i < kRows * kD / 16 / kThreads; ++i) {
      const int c = t + i * kThreads;
      if ((c >> 3) < rows)
        *reinterpret_cast<uint4 *>(dst + c * 16) =
            *reinterpret_cast<const uint4 *>(sm.rows + (c >> 3) * kOutPitch + (c & 7) * 16);
    }
    return;
  }
  // ---- V^T: row dd of the plane holds the block's keys.  Warp w takes key groups kc = w, w + 4
  // (16 keys each) and lane l dims 4 l .. 4 l + 3: 32-bit reads of four keys' four codes
  // (conflict-free: the 132-byte pitch puts the 32 lanes' words in 32 banks), a 4 x 4 byte
  // transpose in registers, one 16-byte store of 16 keys per dim.
  const int n_pad = job.n_pad;
#pragma unroll
  for (int g = 0; g < kRows / 16 / (kThreads / 32); ++g) {
    const int kc = warp + g * (kThreads / 32);
    const int key0 = blk * kRows + kc * 16;
    if (key0 >= n_pad) continue;  // warp-uniform
    uint32_t col[4][4];  // [dim j][4-key group]: keys 4 group .. + 3 of dim 4 lane + j
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      // keys past N (a partial last block) were quantised from zeros: zero codes
      const uint8_t *p = sm.rows + (kc * 16 + 4 * q) * kVPitch + 4 * lane;
      const uint32_t r0 = *reinterpret_cast<const uint32_t *>(p);
      const uint32_t r1 = *reinterpret_cast<const uint32_t *>(p + kVPitch);
      const uint32_t r2 = *reinterpret_cast<const uint32_t *>(p + 2 * kVPitch);
      const uint32_t r3 = *reinterpret_cast<const uint32_t *>(p + 3 * kVPitch);
      const uint32_t t0 = __byte_perm(r0, r1, 0x5140), t1 = __byte_perm(r0, r1, 0x7362);
      const uint32_t t2 = __byte_perm(r2, r3, 0x5140), t3 = __byte_perm(r2, r3, 0x7362);
      col[0][q] = __byte_perm(t0, t2, 0x5410);
      col[1][q] = __byte_perm(t0, t2, 0x7632);
      col[2][q] = __byte_perm(t1, t3, 0x5410);
      col[3][q] = __byte_perm(t1, t3, 0x7632);
    }
#pragma unroll
    for (int j = 0; j < 4; ++j)
      *reinterpret_cast<uint4 *>(job.out + (plane * kD + 4 * lane + j) * n_pad + key0) =
          make_uint4(col[j][0], col[j][1], col[j][2], col[j][3]);
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
