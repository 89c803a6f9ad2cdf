// FP8 (e4m3) exact-attention forward pass on the 5th-generation tensor cores (sm_103a).
//
// "3.4 Attention Kernels" (llm-learning-path), "FlashAttention-2 and -3":
// FlashAttention-3 adds FP8 attention with block quantisation and an
// incoherent-processing transform.  The inputs come from fp8_quantize.cu:
// Q' = Q M and K' = K M (M orthogonal, so Q' K'^T = Q K^T) and V, each in
// 128-row blocks of e4m3 codes with one fp32 scale per block.  Both products
// run as tcgen05.mma kind::f8f6f4 (e4m3 x e4m3 -> fp32 in tensor memory):
//     S_c(j) = (Q8_c K8_j^T) * sq_c * sk_j          (scores of the dequantised blocks)
//     O_c   += P8_c(j) V8_j                          (P rounded to e4m3)
// with the same block-wise online softmax, causal tile skipping, warp roles
// and tensor-memory plan as the bf16 kernel (prefill_bf16.cu): one CTA per
// pair of 128-row query tiles, a TMA warp for Q and K (3-stage ring), a TMA
// warp for V (2-stage ring), one MMA warp per chain, and two softmax
// warpgroups.  The e4m3 tiles are half the bf16 size, which leaves room for two
// P buffers per chain: softmax writes P(j) while P(j-1) V is still running and
// waits for that product only when it must rescale o~ (the lazy rescale makes
// that rare).  As in the bf16 kernel, the two softmax warpgroups take turns for
// their exponentials (an mbarrier token passed after each tile's exponentials).
//
// V's per-block scale sv_j enters through P: softmax writes
// p'_j = p * r_j with r_j = sv_j / max_i sv_i <= 1 (a shift of the exponent,
// so it costs no instruction), the row sum keeps p itself (it adds
// rowsum(p') / r_j), and the epilogue multiplies by max_i sv_i / l.  With
// the lazy rescale p <= 2^8, so p' <= 256 stays inside e4m3's range (448).
// V is stored transposed (V^T [d, keys]) so that the P V product reads both
// operands K-major, like Q K^T.
#include <algorithm>

#include "common.cuh"
#include "tc05.cuh"
#include "kernels.h"

namespace attn {
namespace {

constexpr int BM = 128;      // query rows per tile (= TMEM lanes)
constexpr int BN = 128;      // keys per K/V tile
constexpr int D = 128;       // head dimension (one 128-byte e4m3 row)
constexpr int kKStages = 3;
constexpr int kVStages = 2;
constexpr int kPBufs = 2;                  // P buffers per chain
constexpr int kThreads = 384;
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr int kTileBytes = 128 * 128;      // 128 rows x 128 one-byte elements, one swizzled TMA box

struct Fp8Smem {
  alignas(1024) uint8_t q[2][kTileBytes];
  alignas(1024) uint8_t k[kKStages][kTileBytes];
  alignas(1024) uint8_t v[kVStages][kTileBytes];    // V^T tiles: 128 rows (d) x 128 keys
  alignas(1024) uint8_t p[2][kPBufs][kTileBytes];   // P of chains A and B: 128 rows x 128 keys
  uint64_t q_full;
  uint64_t k_full[kKStages], k_empty[2][kKStages];  // empty: per chain, committed by its MMA warp
  uint64_t v_full[kVStages], v_empty[2][kVStages];
  uint64_t s_full[2], s_free[2];
  uint64_t p_full[2][kPBufs], pv_done[2][kPBufs];   // per P buffer, so phases never alias
  uint64_t turn[2];  // turn[c]: the other chain's softmax has finished its exponentials
  uint64_t mma_done[2];
  uint32_t tmem_base;
  int abort;
};

// Instruction descriptor for kind::f8f6f4 with e4m3 A and B (format 0), fp32 D,
// both operands K-major: [4,6) D format 1 = f32, [7,10) A format, [10,13) B format,
// [17,23) N >> 3, [24,29) M >> 4.
__host__ __device__ constexpr uint32_t idesc_e4m3_f32(int M, int N) {
  return (1u << 4) | (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

__device__ __forceinline__ void mma_f8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                       bool accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate ? 1u : 0u)
      : "memory");
}

// ---- packed fp32 pairs (Blackwell f32x2 ALU forms)
__device__ __forceinline__ uint64_t f2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_split(uint64_t r, float &lo, float &hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(r));
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

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

__device__ __forceinline__ bool elect_one() {
  uint32_t pred;
  asm volatile(
      "{\n\t.reg .pred P;\n\t"
      "elect.sync _|P, 0xffffffff;\n\t"
      "selp.u32 %0, 1, 0, P;\n\t}"
      : "=r"(pred));
  return pred != 0;
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

__device__ __forceinline__ void rescale_o_chunk(uint32_t taddr, float corr) {
  uint32_t r[32];
  tc05::tmem_ld_x32(taddr, r);
  tc05::tmem_ld_wait(r);
  const uint64_t c2 = f2(corr, corr);
#pragma unroll
  for (int e = 0; e < 32; e += 2) {
    float a, b;
    f2_split(mul2(f2(__uint_as_float(r[e]), __uint_as_float(r[e + 1])), c2), a, b);
    r[e] = __float_as_uint(a);
    r[e + 1] = __float_as_uint(b);
  }
  tc05::tmem_st_x32(taddr, r);
}

__global__ void __launch_bounds__(kThreads, 1)
    prefill_fp8_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_vt, const float *__restrict__ q_scale,
                       const float *__restrict__ k_scale, const float *__restrict__ v_scale, const PrefillOut out,
                       int B, int H, int Hkv, int Nq, int Nk, int causal, float scale_log2) {
  extern __shared__ uint8_t smem_raw[];
  Fp8Smem &sm = *reinterpret_cast<Fp8Smem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ---- which (query-tile pair, batch, head): heaviest causal pairs first
  const int n_pairs = (Nq + 2 * BM - 1) / (2 * BM);
  const int bh_count = B * H;
  const int rank = blockIdx.x / bh_count;
  const int bh = blockIdx.x % bh_count;
  const int t = causal ? (n_pairs - 1 - rank) : rank;
  const int b = bh / H;
  const int h = bh % H;
  const int kvh = h / (H / Hkv);
  const int q_plane = b * H + h;
  const int kv_plane = b * Hkv + kvh;
  const int row0[2] = {2 * t * BM, (2 * t + 1) * BM};
  const bool has_b = row0[1] < Nq;
  const int n_kt_all = (Nk + BN - 1) / BN;
  const int n_qt_all = (Nq + BM - 1) / BM;
  const int shift = Nk - Nq;
  auto tiles_of = [&](int r0) {
    if (!causal) return n_kt_all;
    const int last_key = min(r0 + BM, Nq) - 1 + shift;
    return last_key < 0 ? 0 : min(n_kt_all, last_key / BN + 1);
  };
  const int n_tiles[2] = {tiles_of(row0[0]), has_b ? tiles_of(row0[1]) : 0};
  const int n_kv = max(n_tiles[0], n_tiles[1]);

  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&sm.q_full), 1);
    for (int s = 0; s < kKStages; ++s) {
      mbar_init(smem_u32(&sm.k_full[s]), 1);
      mbar_init(smem_u32(&sm.k_empty[0][s]), 1);
      mbar_init(smem_u32(&sm.k_empty[1][s]), 1);
    }
    for (int s = 0; s < kVStages; ++s) {
      mbar_init(smem_u32(&sm.v_full[s]), 1);
      mbar_init(smem_u32(&sm.v_empty[0][s]), 1);
      mbar_init(smem_u32(&sm.v_empty[1][s]), 1);
    }
    for (int c = 0; c < 2; ++c) {
      mbar_init(smem_u32(&sm.s_full[c]), 1);
      mbar_init(smem_u32(&sm.s_free[c]), 128);
      mbar_init(smem_u32(&sm.turn[c]), 128);
      for (int pb = 0; pb < kPBufs; ++pb) {
        mbar_init(smem_u32(&sm.p_full[c][pb]), 128);
        mbar_init(smem_u32(&sm.pv_done[c][pb]), 1);
      }
    }
    mbar_init(smem_u32(&sm.mma_done[0]), 1);
    mbar_init(smem_u32(&sm.mma_done[1]), 1);
    sm.abort = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tc05::tmem_alloc(smem_u32(&sm.tmem_base), kTmemCols);
    tc05::tmem_relinquish();
  }
  tc05::fence_before_sync();
  __syncthreads();
  tc05::fence_after_sync();
  const uint32_t tmem = sm.tmem_base;

  // Register split as in the bf16 kernel: 128 x 56 + 256 x 224 = 64,512 = 384 x 168.
  if (warp < 4) asm volatile("setmaxnreg.dec.sync.aligned.u32 56;" ::: "memory");
  if (warp == 0) {
    // ================================================================ TMA: Q and K
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      const uint64_t keep = l2_policy_evict_last();
      const uint64_t once = l2_policy_evict_first();
      const uint32_t qbar = smem_u32(&sm.q_full);
      mbar_arrive_expect_tx(qbar, (has_b ? 2 : 1) * kTileBytes);
      for (int c = 0; c < (has_b ? 2 : 1); ++c)
        tma_load_3d_hint(smem_u32(sm.q[c]), &tm_q, qbar, 0, row0[c], q_plane, once);
      int issued = 0;
      for (int j = 0; j < n_kv; ++j) {
        const int ks = j % kKStages;
        // the stage's previous tile must have been read by each chain that used it
        bool free_ok = true;
        for (int c = 0; c < 2 && free_ok; ++c)
          if (j >= kKStages && j - kKStages < n_tiles[c])
            free_ok = mbar_wait(smem_u32(&sm.k_empty[c][ks]), ((j / kKStages) - 1) & 1, &sm.abort);
        if (!free_ok) break;
        const uint32_t kbar = smem_u32(&sm.k_full[ks]);
        mbar_arrive_expect_tx(kbar, kTileBytes);
        tma_load_3d_hint(smem_u32(sm.k[ks]), &tm_k, kbar, 0, j * BN, kv_plane, keep);
        ++issued;
      }
      mbar_wait(qbar, 0, nullptr);
      for (int s = 0; s < kKStages && s < issued; ++s) {
        const int last = s + ((issued - 1 - s) / kKStages) * kKStages;
        mbar_wait(smem_u32(&sm.k_full[s]), (last / kKStages) & 1, nullptr);
      }
    }
    __syncwarp();
  } else if (warp == 2) {
    // ================================================================ TMA: V^T (2-stage ring)
    if (lane == 0) {
      tma_prefetch_desc(&tm_vt);
      const uint64_t keep = l2_policy_evict_last();
      int issued = 0;
      for (int j = 0; j < n_kv; ++j) {
        const int vs = j % kVStages;
        bool free_ok = true;
        for (int c = 0; c < 2 && free_ok; ++c)
          if (j >= kVStages && j - kVStages < n_tiles[c])
            free_ok = mbar_wait(smem_u32(&sm.v_empty[c][vs]), ((j / kVStages) - 1) & 1, &sm.abort);
        if (!free_ok) break;
        const uint32_t vbar = smem_u32(&sm.v_full[vs]);
        mbar_arrive_expect_tx(vbar, kTileBytes);
        tma_load_3d_hint(smem_u32(sm.v[vs]), &tm_vt, vbar, j * BN, 0, kv_plane, keep);
        ++issued;
      }
      for (int s = 0; s < kVStages && s < issued; ++s) {
        const int last = s + ((issued - 1 - s) / kVStages) * kVStages;
        mbar_wait(smem_u32(&sm.v_full[s]), (last / kVStages) & 1, nullptr);
      }
    }
    __syncwarp();
  } else if (warp == 1 || warp == 3) {
    // ================================================================ MMA warps, one per chain
    // Warp 1 issues chain A's MMAs and warp 3 chain B's, each in the order
    //   S_c(0), S_c(1), P_c(0) V_0, S_c(2), P_c(1) V_1, ...
    // after bounded blocking waits: S_c(j) once softmax has taken S_c(j-1) out of
    // tensor memory and K_j has landed, P_c(j-1) V_{j-1} once P_c(j-1) is written
    // and V_{j-1} has landed.
    const int c = warp == 1 ? 0 : 1;
    const int n_c = n_tiles[c];
    constexpr uint32_t idesc = idesc_e4m3_f32(BM, BN);  // N = BN = D = 128 for both products
    bool ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&sm.q_full), 0, &sm.abort));
    tc05::fence_after_sync();
    const uint64_t dq = tc05::sdesc_sw128(smem_u32(sm.q[c]), 16, 1024);
    for (int j = 0; ok && j <= n_c; ++j) {
      if (j < n_c) {
        // S_c(j) = Q_c K_j^T
        const int ks = j % kKStages;
        ok = __all_sync(0xffffffffu, (j == 0 || mbar_wait(smem_u32(&sm.s_free[c]), (j - 1) & 1, &sm.abort)) &&
                                         mbar_wait(smem_u32(&sm.k_full[ks]), (j / kKStages) & 1, &sm.abort));
        if (!ok) break;
        tc05::fence_after_sync();
        const uint64_t db = tc05::sdesc_sw128(smem_u32(sm.k[ks]), 16, 1024);
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < D / 32; ++kk)  // K = 32 e4m3 elements (32 bytes, descriptor +2) per MMA
            mma_f8(tmem + c * BN, dq + 2 * kk, db + 2 * kk, idesc, kk > 0);
          tc05::commit(smem_u32(&sm.s_full[c]));
          tc05::commit(smem_u32(&sm.k_empty[c][ks]));
        }
        __syncwarp();
      }
      if (j > 0) {
        // O_c += P_c(j-1) V_{j-1}
        const int jp = j - 1;
        const int pb = jp % kPBufs, vs = jp % kVStages;
        ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&sm.p_full[c][pb]), (jp / kPBufs) & 1, &sm.abort) &&
                                         mbar_wait(smem_u32(&sm.v_full[vs]), (jp / kVStages) & 1, &sm.abort));
        if (!ok) break;
        tc05::fence_after_sync();
        const uint64_t da = tc05::sdesc_sw128(smem_u32(sm.p[c][pb]), 16, 1024);
        const uint64_t db = tc05::sdesc_sw128(smem_u32(sm.v[vs]), 16, 1024);
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < BN / 32; ++kk)
            mma_f8(tmem + 2 * BN + c * BN, da + 2 * kk, db + 2 * kk, idesc, (jp > 0) || (kk > 0));
          tc05::commit(smem_u32(&sm.pv_done[c][pb]));
          tc05::commit(smem_u32(&sm.v_empty[c][vs]));
        }
        __syncwarp();
      }
    }
    // every MMA this warp issued must complete before tensor memory is released
    if (elect_one()) tc05::commit(smem_u32(&sm.mma_done[c]));
    __syncwarp();
    mbar_wait(smem_u32(&sm.mma_done[c]), 0, nullptr);
  } else if (warp >= 4) {
    // ================================================================ softmax warpgroups
    asm volatile("setmaxnreg.inc.sync.aligned.u32 224;" ::: "memory");
    const int c = (warp - 4) >> 2;
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const int q_row = row0[c] + row;
    const int n_c = n_tiles[c];
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t s_addr = tmem + lane_addr + c * BN;
    const uint32_t o_addr = tmem + lane_addr + 2 * BN + c * BN;
    const uint32_t p_row0 = smem_u32(sm.p[c][0]) + row * 128;  // this row of P buffer 0 (buffer 1 follows)
    const int lim = causal ? min(q_row + shift + 1, Nk) : Nk;
    const float *ks = k_scale + static_cast<long long>(kv_plane) * n_kt_all;
    const float *vs = v_scale + static_cast<long long>(kv_plane) * n_kt_all;
    // score factor of this query tile, and the largest V block scale of the head
    // (chain B of the last pair may lie past Nq: its block has no scale, and it runs no tile)
    const float sq_log2 =
        row0[c] < Nq ? scale_log2 * q_scale[static_cast<long long>(q_plane) * n_qt_all + row0[c] / BM] : 0.f;
    float v_max = 0.f;
    for (int i = lane; i < n_kt_all; i += 32) v_max = fmaxf(v_max, vs[i]);
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) v_max = fmaxf(v_max, __shfl_xor_sync(0xffffffffu, v_max, m));
    float m_ref = -INFINITY;
    float l = 0.f;
    bool ok = true;
    float sk_next = n_c > 0 ? ks[0] : 0.f;
    float sv_next = n_c > 0 ? vs[0] : 0.f;
    for (int j = 0; j < n_c; ++j) {
      const float sk = sk_next, sv = sv_next;
      if (j + 1 < n_c) {  // next tile's scales, loaded while this one is processed
        sk_next = ks[j + 1];
        sv_next = vs[j + 1];
      }
      if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&sm.s_full[c]), j & 1, &sm.abort))) {
        ok = false;
        break;
      }
      tc05::fence_after_sync();
      uint32_t sr[4][32];
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) tc05::tmem_ld_x32(s_addr + q4 * 32, sr[q4]);
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) tc05::tmem_ld_wait(sr[q4]);
      tc05::fence_before_sync();
      mbar_arrive(smem_u32(&sm.s_free[c]));

      // s' = acc * c_j in log2 units; c_j > 0 (a zero block has acc = 0 exactly,
      // and the floor keeps -inf * c_j = -inf for masked keys)
      const float c_j = fmaxf(sq_log2 * sk, 1.17549435e-38f);
      // V block scale relative to the head's largest: p' = p * r_j, r_j in [2^-20, 1].
      // The floor keeps p' and the row sum rowsum(p') / r_j in fp32 range; a block
      // below it holds values under 2^-20 * max|V|, which it then overstates by
      // at most that much.  A zero block takes r_j = 1 (its codes are 0).
      const float r_j = (sv > 0.f && v_max > 0.f) ? fmaxf(sv / v_max, 0x1p-20f) : 1.f;
      const float log2_r = __log2f(r_j);

      const int kv0 = j * BN;
      if (kv0 + BN > lim) {
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4)
#pragma unroll
          for (int e = 0; e < 32; ++e)
            if (kv0 + q4 * 32 + e >= lim) sr[q4][e] = __float_as_uint(-INFINITY);
      }
      // p' = 2^(acc * c_j - m_ref + log2 r_j), summed, packed to e4m3.  First relative to the
      // current reference without a row maximum: if the row sum of p stays <= 2^8, every p
      // does, so the row maximum has not outgrown the reference by more than 2^8 and the
      // reference stays.  Otherwise (and on a row's first scores) the maximum decides.
      const uint64_t c2 = f2(c_j, c_j);
      uint32_t pr[32];
      float sum = 0.f;
      auto exp_pass = [&](float neg_m_ref) {
        const uint64_t negm2 = f2(neg_m_ref + log2_r, neg_m_ref + log2_r);
        uint64_t acc2[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
#pragma unroll
          for (int e = 0; e < 32; e += 4) {
            float x0, x1, x2, x3;
            f2_split(fma2(f2(__uint_as_float(sr[q4][e]), __uint_as_float(sr[q4][e + 1])), c2, negm2), x0, x1);
            f2_split(fma2(f2(__uint_as_float(sr[q4][e + 2]), __uint_as_float(sr[q4][e + 3])), c2, negm2), x2, x3);
            const float p0 = ex2_approx(x0), p1 = ex2_approx(x1), p2 = ex2_approx(x2), p3 = ex2_approx(x3);
            acc2[(e >> 2) & 3] = add2(acc2[(e >> 2) & 3], add2(f2(p0, p1), f2(p2, p3)));
            pr[q4 * 8 + (e >> 2)] = pack_e4m3x4(p0, p1, p2, p3);
          }
        }
        float lo, hi;
        f2_split(add2(add2(acc2[0], acc2[1]), add2(acc2[2], acc2[3])), lo, hi);
        sum = lo + hi;
      };
      // ping-pong: chain A's exponentials of tile j follow chain B's of tile j-1, and
      // chain B's of tile j follow chain A's of tile j
      {
        const int need = c == 0 ? j - 1 : j;  // the other chain's step to wait for
        if (need >= 0 && need < n_tiles[1 - c] &&
            !__all_sync(0xffffffffu, mbar_wait(smem_u32(&sm.turn[c]), need & 1, &sm.abort))) {
          ok = false;
          break;
        }
      }
      bool need_max = m_ref == -INFINITY;
      if (!need_max) {
        exp_pass(-m_ref);
        need_max = sum > 256.f * r_j;
      }
      bool move = false;
      float corr = 1.f;
      if (need_max) {
        float mq[4];
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          float m = __uint_as_float(sr[q4][0]);
#pragma unroll
          for (int e = 1; e < 31; e += 2) m = max3(m, __uint_as_float(sr[q4][e]), __uint_as_float(sr[q4][e + 1]));
          mq[q4] = fmaxf(m, __uint_as_float(sr[q4][31]));
        }
        const float m_new = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3])) * c_j;
        move = m_new > m_ref + kRescaleThreshold;
        if (move) {
          corr = (m_ref == -INFINITY) ? 0.f : ex2_approx(m_ref - m_new);
          m_ref = m_new;
          exp_pass(-m_ref);
        } else if (m_ref == -INFINITY) {
          exp_pass(0.f);  // no key of the row met yet: every s is -inf and p = 0
        }
      }
      l = l * corr + sum / r_j;
      mbar_arrive(smem_u32(&sm.turn[1 - c]));

      // P buffer pb was last read by P(j-2) V_{j-2}; o~ is rescaled in place (when this
      // warp's rows moved their reference) only once P(j-1) V_{j-1} has completed
      const int pb = j % kPBufs;
      if (j >= kPBufs &&
          !__all_sync(0xffffffffu, mbar_wait(smem_u32(&sm.pv_done[c][pb]), ((j / kPBufs) - 1) & 1, &sm.abort))) {
        ok = false;
        break;
      }
      if (j > 0 && __any_sync(0xffffffffu, move)) {
        const int jb = (j - 1) % kPBufs;
        if (!__all_sync(0xffffffffu,
                        mbar_wait(smem_u32(&sm.pv_done[c][jb]), ((j - 1) / kPBufs) & 1, &sm.abort))) {
          ok = false;
          break;
        }
        tc05::fence_after_sync();
#pragma unroll
        for (int q4 = 0; q4 < D / 32; ++q4) rescale_o_chunk(o_addr + q4 * 32, corr);
      }
      // P row -> shared memory: keys 16ch .. 16ch+15 at chunk ch, chunk index XOR (row mod 8)
      const uint32_t p_row = p_row0 + pb * kTileBytes;
#pragma unroll
      for (int ch = 0; ch < 8; ++ch)
        st_shared_v4(p_row + (((ch ^ row) & 7) << 4), pr[4 * ch], pr[4 * ch + 1], pr[4 * ch + 2], pr[4 * ch + 3]);
      fence_proxy_async_smem();
      tc05::tmem_wait_st();
      tc05::fence_before_sync();
      mbar_arrive(smem_u32(&sm.p_full[c][pb]));
    }

    // ---- epilogue: O = o~ * max sv / l, LSE = m + ln l
    if (ok && n_c > 0) {
      ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&sm.pv_done[c][(n_c - 1) % kPBufs]),
                                             ((n_c - 1) / kPBufs) & 1, &sm.abort));
      if (ok) {
        tc05::fence_after_sync();
        const float inv = (l > 0.f) ? v_max / l : 0.f;
        const uint64_t inv2 = f2(inv, inv);
        const bool store = q_row < Nq;
        __nv_bfloat16 *orow = static_cast<__nv_bfloat16 *>(out.o) + b * out.o_b + h * out.o_h +
                              static_cast<long long>(store ? q_row : 0) * out.o_r;
#pragma unroll
        for (int q4 = 0; q4 < D / 32; ++q4) {
          uint32_t orr[32];
          tc05::tmem_ld_x32(o_addr + q4 * 32, orr);
          tc05::tmem_ld_wait(orr);
          uint32_t packed[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            float a, bb;
            f2_split(mul2(f2(__uint_as_float(orr[2 * e]), __uint_as_float(orr[2 * e + 1])), inv2), a, bb);
            packed[e] = pack_bf16x2(a, bb);
          }
          if (store) {
            uint4 *dst = reinterpret_cast<uint4 *>(orow + q4 * 32);
#pragma unroll
            for (int e = 0; e < 4; ++e)
              dst[e] = make_uint4(packed[4 * e], packed[4 * e + 1], packed[4 * e + 2], packed[4 * e + 3]);
          }
        }
        if (store && out.lse != nullptr)
          out.lse[b * out.l_b + h * out.l_h + static_cast<long long>(q_row) * out.l_r] =
              (l > 0.f) ? m_ref * kLn2 + logf(l) : -INFINITY;
      }
    } else if (n_c == 0 && q_row < Nq) {
      uint4 *dst = reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(out.o) + b * out.o_b + h * out.o_h +
                                             static_cast<long long>(q_row) * out.o_r);
#pragma unroll
      for (int e = 0; e < D / 8; ++e) dst[e] = make_uint4(0u, 0u, 0u, 0u);
      if (out.lse != nullptr) out.lse[b * out.l_b + h * out.l_h + static_cast<long long>(q_row) * out.l_r] = -INFINITY;
    }
  }

  tc05::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc05::fence_after_sync();
    tc05::tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

ATTN_DEFINE_ERROR_ACCESSOR(device_error_prefill_fp8)

cudaError_t launch_prefill_fp8(const Fp8Maps &maps, const float *q_scale, const float *k_scale, const float *v_scale,
                               const PrefillOut &out, int B, int H, int Hkv, int Nq, int Nk, bool causal, float scale,
                               cudaStream_t stream) {
  const size_t smem = sizeof(Fp8Smem) + 1024;
  cudaError_t e = cudaFuncSetAttribute(prefill_fp8_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const long long n_pairs = (Nq + 2 * BM - 1) / (2 * BM);
  const long long blocks = n_pairs * B * H;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  prefill_fp8_kernel<<<static_cast<unsigned>(blocks), kThreads, smem, stream>>>(
      maps.q, maps.k, maps.vt, q_scale, k_scale, v_scale, out, B, H, Hkv, Nq, Nk, causal ? 1 : 0, scale * kLog2e);
  return cudaGetLastError();
}

}  // namespace attn
