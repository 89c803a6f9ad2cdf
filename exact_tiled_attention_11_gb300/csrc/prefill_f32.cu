// Precise fp32 exact-attention forward pass (SIMT), for fp32 inputs.
//
// Same block-wise algorithm as the bf16 kernel ("3.4 Attention Kernels",
// "FlashAttention: tiling"; "FlashAttention and Optimized Kernels", "The
// online softmax"): keys in tiles of 32, a running max m, denominator l and
// unnormalised output o~ per query row, rescaled by exp(m - m') whenever the
// maximum grows, O = o~ / l and LSE = m + ln l at the end, keys after the
// query skipped when causal.  The keys of a row are split among the CTA's
// warps (warp w takes tiles w, w + 4, ...), and the warps' partial results
// (m_w, l_w, o~_w) are merged at the end by the exact rule
//     m = max m_w,  l = sum_w e^(m_w - m) l_w,  o~ = sum_w e^(m_w - m) o~_w
// ("3.4 Attention Kernels", "Online softmax": the merge of two partial
// results).
//
// Precision without fp64 (this GPU runs fp64 at a small fraction of its fp32
// rate).  With queries scaled by 30 the scores reach the hundreds, and a plain
// fp32 dot product then carries absolute errors around 1e-5 into exp().
// Every q.k is therefore a compensated dot product (Ogita, Rump and Oishi,
// "Accurate sum and dot product", 2005, algorithm Dot2): each product is split
// exactly into p + e with one FMA (e = fma(a, b, -p)), the p are summed with
// the error-free TwoSum (Knuth), and the e and the TwoSum errors are summed
// apart, which gives the score as an unevaluated pair s_hi + s_lo accurate to
// a few units in the last place of fp32.  exp is taken of (s_hi - m) + s_lo.
// The row sum l and o~ are pairs (hi, lo) as well: each tile's contribution is
// added with TwoSum, so the rounding of a long row's sums stays at fp32 level
// per tile rather than growing with the number of keys.
#include "common.cuh"
#include "kernels.h"

namespace attn {
namespace {

constexpr int kTile = 32;       // keys per tile (one per lane)

// error-free transformations (exact: a + b = s + err, a * b = p + err)
__device__ __forceinline__ void two_sum(float a, float b, float &s, float &err) {
  s = a + b;
  const float z = s - a;
  err = (a - (s - z)) + (b - z);
}
__device__ __forceinline__ void fast_two_sum(float a, float b, float &s, float &err) {  // needs |a| >= |b|
  s = a + b;
  err = b - (s - a);
}

// (hi, lo) += x as a compensated pair
__device__ __forceinline__ void pair_add(float &hi, float &lo, float x) {
  float s, e;
  two_sum(hi, x, s, e);
  hi = s;
  lo += e;
}

// 16-byte global -> shared copy that does not pass through registers; src_bytes = 0
// writes zeros (the source is not read).
__device__ __forceinline__ void cp_async16(void *dst, const void *src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Per head dimension: the warps per CTA (each takes every kSplits-th key tile of the row) and
// where a tile's V lives.  At d = 64 each lane holds its two columns of the tile's 32 V rows
// in registers (64 values, read with coalesced loads while K is staged), so that only K
// takes shared memory and eight warps still leave room for several CTAs per SM (a 256-key
// row is then one tile per warp); at d = 128 V is staged in shared memory beside K.
template <int D>
struct F32Cfg {
  static constexpr int kSplits = D == 64 ? 8 : 4;
  static constexpr bool kVRegs = D == 64;
};

template <int D>
struct F32Smem {
  static constexpr int kSplits = F32Cfg<D>::kSplits;
  static constexpr int kStride = D + 4;   // padded K row: float4 reads of 8 lanes hit 8 distinct bank groups
  float k[kSplits][kTile * kStride];      // each warp's own key tile (lane j reads key j)
  float v[F32Cfg<D>::kVRegs ? 1 : kSplits][F32Cfg<D>::kVRegs ? 4 : kTile * D];  // each warp's value tile
  float q[D];
};

template <int D>
__global__ void __launch_bounds__(F32Cfg<D>::kSplits * 32)
    prefill_f32_kernel(const float *__restrict__ q, const float *__restrict__ k, const float *__restrict__ v,
                       PrefillOut out, int H, int Hkv, int Nq, int Nk, int causal, float scale) {
  constexpr int E = D / 32;                // output elements per lane
  constexpr int kStride = F32Smem<D>::kStride;
  constexpr int kSplits = F32Cfg<D>::kSplits;
  constexpr bool kVRegs = F32Cfg<D>::kVRegs;
  extern __shared__ float4 smem_f4[];
  F32Smem<D> &sm = *reinterpret_cast<F32Smem<D> *>(smem_f4);

  const int row = blockIdx.x;
  const int h = blockIdx.y;
  const int b = blockIdx.z;
  const int kvh = h / (H / Hkv);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  const float *qh = q + ((static_cast<size_t>(b) * H + h) * Nq + row) * D;
  const float *kh = k + (static_cast<size_t>(b) * Hkv + kvh) * static_cast<size_t>(Nk) * D;
  const float *vh = v + (static_cast<size_t>(b) * Hkv + kvh) * static_cast<size_t>(Nk) * D;
  // keys [0, key_end) are attended; causal: j <= row + (Nk - Nq), the mask aligned to the last key
  const int key_end = causal ? max(0, min(Nk, row + (Nk - Nq) + 1)) : Nk;

  for (int e = 4 * threadIdx.x; e < D; e += 4 * kSplits * 32) cp_async16(sm.q + e, qh + e, 16);

  float *ks = sm.k[warp];
  float *vs = sm.v[kVRegs ? 0 : warp];
  float vr[kVRegs ? kTile : 1][E];         // d = 64: lane's columns lane + 32 j of the tile's V rows
  float m = -INFINITY;                     // running max of s_hi (warp-uniform)
  float l_hi = 0.f, l_lo = 0.f;            // row sum over this warp's keys (warp-uniform)
  float acc_hi[E], acc_lo[E];              // o~ elements lane + 32 j
#pragma unroll
  for (int j = 0; j < E; ++j) acc_hi[j] = acc_lo[j] = 0.f;

  // Stage the K and V rows of the tile at t0: every 16-byte copy of the tile in flight
  // at once (rows past key_end are written as zeros), and the warp's next tile brought
  // into L2 meanwhile.
  auto stage = [&](int t0) {
#pragma unroll 4
    for (int i = lane; i < kTile * D / 4; i += 32) {
      const int r = (4 * i) / D, c = (4 * i) % D;
      const bool in = t0 + r < key_end;
      const size_t off = in ? static_cast<size_t>(t0 + r) * D + c : 0;
      cp_async16(ks + r * kStride + c, kh + off, in ? 16 : 0);
      if (!kVRegs) cp_async16(vs + r * D + c, vh + off, in ? 16 : 0);
    }
    if (kVRegs) {  // rows past key_end read as zeros (their p is 0)
#pragma unroll
      for (int jj = 0; jj < (kVRegs ? kTile : 0); ++jj) {
        const bool in = t0 + jj < key_end;
#pragma unroll
        for (int j = 0; j < E; ++j)
          vr[jj][j] = in ? __ldg(vh + static_cast<size_t>(t0 + jj) * D + lane + 32 * j) : 0.f;
      }
    }
    const int t_next = t0 + kSplits * kTile;
    if (t_next + lane < key_end) {
      const size_t row_off = static_cast<size_t>(t_next + lane) * D;
#pragma unroll
      for (int c = 0; c < D; c += 32) {  // 128-byte lines
        asm volatile("prefetch.global.L2 [%0];" ::"l"(kh + row_off + c));
        asm volatile("prefetch.global.L2 [%0];" ::"l"(vh + row_off + c));
      }
    }
  };
  if (warp * kTile < key_end) stage(warp * kTile);
  cp_async_wait_all();
  __syncthreads();  // q (copied by the whole CTA) and each warp's first tile have landed

  for (int t0 = warp * kTile; t0 < key_end; t0 += kSplits * kTile) {
    if (t0 != warp * kTile) {
      __syncwarp();  // the previous tile's reads are done before its buffers are refilled
      stage(t0);
      cp_async_wait_all();
      __syncwarp();
    }

    // ---- s = scale * q . k_lane as s_hi + s_lo (Dot2, four interleaved accumulators)
    const int key = t0 + lane;
    const bool attend = key < key_end;
    float sh[4] = {0.f, 0.f, 0.f, 0.f}, sl[4] = {0.f, 0.f, 0.f, 0.f};
    const float *krow = ks + lane * kStride;
#pragma unroll 4
    for (int e = 0; e < D; e += 4) {
      const float4 a = *reinterpret_cast<const float4 *>(sm.q + e);
      const float4 c = *reinterpret_cast<const float4 *>(krow + e);
      const float av[4] = {a.x, a.y, a.z, a.w}, cv[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float p = av[u] * cv[u];
        const float pe = fmaf(av[u], cv[u], -p);
        float s, err;
        two_sum(sh[u], p, s, err);
        sh[u] = s;
        sl[u] += err + pe;
      }
    }
    // combine the four accumulators, then scale (hi * scale split exactly with one FMA)
    float s01, e01, s23, e23, s, es;
    two_sum(sh[0], sh[1], s01, e01);
    two_sum(sh[2], sh[3], s23, e23);
    two_sum(s01, s23, s, es);
    const float lo_sum = ((sl[0] + sl[1]) + (sl[2] + sl[3])) + ((e01 + e23) + es);
    const float hs = s * scale;
    const float hs_err = fmaf(s, scale, -hs) + lo_sum * scale;
    float s_hi, s_lo;
    fast_two_sum(hs, hs_err, s_hi, s_lo);
    if (!attend) {
      s_hi = -INFINITY;
      s_lo = 0.f;
    }

    // ---- online softmax over the tile
    float tmax = s_hi;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, off));
    const float m_new = fmaxf(m, tmax);     // finite: the tile's first key is always attended
    const float corr = (m == -INFINITY) ? 0.f : expf(m - m_new);
    const float p = attend ? expf((s_hi - m_new) + s_lo) : 0.f;
    // tile sum of p, compensated across the shuffle tree
    float ps_hi = p, ps_lo = 0.f;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float oh = __shfl_xor_sync(0xffffffffu, ps_hi, off);
      const float ol = __shfl_xor_sync(0xffffffffu, ps_lo, off);
      float t, te;
      two_sum(ps_hi, oh, t, te);
      ps_hi = t;
      ps_lo += ol + te;
    }
    l_hi *= corr;
    l_lo *= corr;
    pair_add(l_hi, l_lo, ps_hi);
    l_lo += ps_lo;
    // o~ = corr * o~ + sum_j p_j v_j: the tile's sum in plain fp32, added to the pair
    float tile[E];
#pragma unroll
    for (int j = 0; j < E; ++j) tile[j] = 0.f;
    if (kVRegs) {
      // keys past key_end contribute p = 0 times v = 0: the sum is unchanged
#pragma unroll
      for (int jj = 0; jj < (kVRegs ? kTile : 0); ++jj) {
        const float pj = __shfl_sync(0xffffffffu, p, jj);
#pragma unroll
        for (int j = 0; j < E; ++j) tile[j] = fmaf(pj, vr[jj][j], tile[j]);
      }
    } else {
      const int n_keys = min(kTile, key_end - t0);
      for (int jj = 0; jj < n_keys; ++jj) {
        const float pj = __shfl_sync(0xffffffffu, p, jj);
#pragma unroll
        for (int j = 0; j < E; ++j) tile[j] = fmaf(pj, vs[jj * D + lane + 32 * j], tile[j]);
      }
    }
#pragma unroll
    for (int j = 0; j < E; ++j) {
      acc_hi[j] *= corr;
      acc_lo[j] *= corr;
      pair_add(acc_hi[j], acc_lo[j], tile[j]);
    }
    m = m_new;
  }

  // ---- merge the warps' partials (m_w, l_w, o~_w) in shared memory, reusing the K tiles
  __syncthreads();
  float *part = &sm.k[0][0];               // per warp: m, l_hi, l_lo, then o~ hi [D], lo [D]
  float *mine = part + warp * (3 + 2 * D);
  if (lane == 0) {
    mine[0] = m;
    mine[1] = l_hi;
    mine[2] = l_lo;
  }
#pragma unroll
  for (int j = 0; j < E; ++j) {
    mine[3 + lane + 32 * j] = acc_hi[j];
    mine[3 + D + lane + 32 * j] = acc_lo[j];
  }
  __syncthreads();
  if (warp != 0) return;
  float M = -INFINITY;
#pragma unroll
  for (int w = 0; w < kSplits; ++w) M = fmaxf(M, part[w * (3 + 2 * D)]);
  float L = 0.f, o[E];
#pragma unroll
  for (int j = 0; j < E; ++j) o[j] = 0.f;
  if (M != -INFINITY) {
#pragma unroll
    for (int w = 0; w < kSplits; ++w) {
      const float *pw = part + w * (3 + 2 * D);
      const float mw = pw[0];
      if (mw == -INFINITY) continue;      // a warp that met no key
      const float f = expf(mw - M);
      L += f * (pw[1] + pw[2]);
#pragma unroll
      for (int j = 0; j < E; ++j) o[j] += f * (pw[3 + lane + 32 * j] + pw[3 + D + lane + 32 * j]);
    }
  }
  float *oh = static_cast<float *>(out.o) + b * out.o_b + h * out.o_h + static_cast<long long>(row) * out.o_r;
#pragma unroll
  for (int j = 0; j < E; ++j) oh[lane + 32 * j] = (L > 0.f) ? o[j] / L : 0.f;
  if (out.lse != nullptr && lane == 0)
    out.lse[b * out.l_b + h * out.l_h + static_cast<long long>(row) * out.l_r] =
        (L > 0.f) ? M + logf(L) : -INFINITY;
}

template <int D>
cudaError_t launch_d(const float *q, const float *k, const float *v, const PrefillOut &out, int B, int H, int Hkv,
                     int Nq, int Nk, bool causal, float scale, cudaStream_t stream) {
  constexpr int kSplits = F32Cfg<D>::kSplits;
  const size_t smem = sizeof(F32Smem<D>);
  auto kern = prefill_f32_kernel<D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  // one CTA per query row; rows on x (up to 2^31 - 1), heads on y, batch on z
  if (H > 65535 || B > 65535) return cudaErrorInvalidConfiguration;
  kern<<<dim3(Nq, H, B), kSplits * 32, smem, stream>>>(q, k, v, out, H, Hkv, Nq, Nk, causal ? 1 : 0, scale);
  return cudaGetLastError();
}

}  // namespace

ATTN_DEFINE_ERROR_ACCESSOR(device_error_prefill_f32)

cudaError_t launch_prefill_f32(const float *q, const float *k, const float *v, const PrefillOut &out, int B, int H,
                               int Hkv, int Nq, int Nk, int d, bool causal, float scale, cudaStream_t stream) {
  if (d == 64) return launch_d<64>(q, k, v, out, B, H, Hkv, Nq, Nk, causal, scale, stream);
  return launch_d<128>(q, k, v, out, B, H, Hkv, Nq, Nk, causal, scale, stream);
}

}  // namespace attn
