// bf16 exact-attention forward pass on the 5th-generation tensor cores (sm_103a).
//
// The algorithm is the block-wise one of "3.4 Attention Kernels"
// (llm-learning-path), "FlashAttention: tiling" and "FlashAttention-2 and -3",
// and "FlashAttention and Optimized Kernels" (programmer.ie), "The online
// softmax": per 128-row query tile, stream 128-key K/V tiles, S = scale Q K^T,
// running row max m and denominator l, p = exp(S - m), o~ += p V with the
// exp(m - m') rescale, and O = o~ / l, LSE = m + ln l at the end.  With causal
// masking only key tiles j <= i are visited and the diagonal tile is masked.
//
// GB300 mapping: one CTA per PAIR of 128-row query tiles (A and B) of one
// (batch, head), 384 threads, one CTA per SM.  The two tiles form two
// independent chains  S_c(j) -> softmax_c(j) -> P_c(j) -> O_c += P_c(j) V_j ->
// S_c(j+1) ... and the tensor core alternates between them, so that the
// softmax of one tile runs while the MMAs of the other tile execute (the
// FlashAttention-3 overlap, here with tcgen05 and tensor memory).
//   warp 0      TMA producer: Q_A, Q_B once, then K_j / V_j into 2-stage rings
//               (128-byte-swizzled tiles, completion on mbarriers).
//   warps 1, 2  one MMA warp per chain (warp 1 also allocates tensor memory):
//                 S_c = Q_c K_j^T  (SS form; Q, K K-major in SMEM)
//                 O_c += P_c V_j   (TS form; P from TMEM, V MN-major in SMEM)
//               issued by an elected lane of the converged warp, completion
//               tracked by tcgen05.commit on mbarriers.  Two issuing warps
//               keep the tensor core fed while each waits on its own chain.
//   warps 4-7   softmax warpgroup of tile A, warps 8-11 of tile B; one thread
//               per query row (= TMEM lane): load S, mask, row max, p = 2^(s'-m),
//               row sum, write P = bf16(p) over the first 64 columns of S,
//               rescale O in TMEM lazily (the reference maximum moves only
//               when the row max outgrows it by more than 2^8; the result does
//               not depend on the reference, and p stays <= 256), and at the
//               end write O = o~ / l (bf16, round to nearest even) and the LSE.
// Tensor memory, 512 columns: S_A [0,128), S_B [128,256), O_A [256,256+d),
// O_B [384,384+d).  Query-tile pairs are ordered heaviest causal pair first.
#include <algorithm>

#include "common.cuh"
#include "tc05.cuh"
#include "kernels.h"

namespace attn {
namespace {

constexpr int BM = 128;      // query rows per tile (= TMEM lanes)
constexpr int BN = 128;      // keys per K/V tile
constexpr int kKStages = 2;
constexpr int kVStages = 2;
constexpr int kThreads = 384;
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr int kBoxBytes = BN * 64 * 2;     // one 128-row x 64-column bf16 TMA box: 16 KiB

template <int D>
struct PrefillSmem {
  static constexpr int kTileBytes = BN * D * 2;
  alignas(1024) uint8_t q[2][BM * D * 2];
  alignas(1024) uint8_t k[kKStages][kTileBytes];
  alignas(1024) uint8_t v[kVStages][kTileBytes];
  uint64_t q_full;
  uint64_t k_full[kKStages], k_empty[kKStages];
  uint64_t v_full[kVStages], v_empty[kVStages];
  uint64_t s_full[2], p_full[2], pv_done[2];
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort;
};

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

// One lane of a converged warp (the MMA instructions are issued by it while
// the whole warp runs the control flow, so their operands stay warp-uniform).
__device__ __forceinline__ bool elect_one() {
  uint32_t pred;
  asm volatile(
      "{\n\t.reg .pred P;\n\t"
      "elect.sync _|P, 0xffffffff;\n\t"
      "selp.u32 %0, 1, 0, P;\n\t}"
      : "=r"(pred));
  return pred != 0;
}

// Scale a 32-column chunk of O (one row per thread) in tensor memory.
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

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_bf16_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v, __nv_bfloat16 *__restrict__ o,
                        float *__restrict__ lse, int B, int H, int Hkv, int N, int causal, float scale_log2) {
  using Smem = PrefillSmem<D>;
  extern __shared__ uint8_t smem_raw[];
  Smem &sm = *reinterpret_cast<Smem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ---- which (query-tile pair, batch, head): heaviest causal pairs first
  const int n_pairs = (N + 2 * BM - 1) / (2 * BM);
  const int bh_count = B * H;
  const int rank = blockIdx.x / bh_count;
  const int bh = blockIdx.x % bh_count;
  const int t = causal ? (n_pairs - 1 - rank) : rank;
  const int b = bh / H;
  const int h = bh % H;
  const int kvh = h / (H / Hkv);
  const int row0[2] = {2 * t * BM, (2 * t + 1) * BM};
  const bool has_b = row0[1] < N;
  const int n_kt_all = (N + BN - 1) / BN;
  // key tiles each chain visits: causal tile i attends tiles 0..i
  const int n_tiles[2] = {causal ? 2 * t + 1 : n_kt_all, has_b ? (causal ? 2 * t + 2 : n_kt_all) : 0};
  const int n_kv = max(n_tiles[0], n_tiles[1]);

  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&sm.q_full), 1);
    // a stage is handed back once both chains' MMAs have read it
    for (int s = 0; s < kKStages; ++s) {
      mbar_init(smem_u32(&sm.k_full[s]), 1);
      mbar_init(smem_u32(&sm.k_empty[s]), 2);
    }
    for (int s = 0; s < kVStages; ++s) {
      mbar_init(smem_u32(&sm.v_full[s]), 1);
      mbar_init(smem_u32(&sm.v_empty[s]), 2);
    }
    for (int c = 0; c < 2; ++c) {
      mbar_init(smem_u32(&sm.s_full[c]), 1);
      mbar_init(smem_u32(&sm.p_full[c]), 128);
      mbar_init(smem_u32(&sm.pv_done[c]), 1);
    }
    mbar_init(smem_u32(&sm.mma_done), 2);
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

  // Register split: the CTA is launched with 384 threads x 168 registers =
  // 64,512.  Warpgroup 0 (producer, MMA issuer, two idle warps) gives up to
  // 56 per thread and the two softmax warpgroups take 224:
  // 128 x 56 + 256 x 224 = 64,512, exactly the launch's allocation.
  if (warp < 4) asm volatile("setmaxnreg.dec.sync.aligned.u32 56;" ::: "memory");
  if (warp == 0) {
    // ================================================================ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      const uint64_t keep = l2_policy_evict_last();    // K/V tiles are re-read by other query tiles
      const uint64_t once = l2_policy_evict_first();   // each Q tile is read once
      const uint32_t qbar = smem_u32(&sm.q_full);
      mbar_arrive_expect_tx(qbar, (has_b ? 2 : 1) * BM * D * 2);
      for (int c = 0; c < (has_b ? 2 : 1); ++c)
#pragma unroll
        for (int x = 0; x < D / 64; ++x)
          tma_load_3d_hint(smem_u32(sm.q[c]) + x * kBoxBytes, &tm_q, qbar, x * 64, row0[c], b * H + h, once);
      int k_issued = 0, v_issued = 0;
      for (int j = 0; j < n_kv; ++j) {
        const int ks = j % kKStages;
        if (j >= kKStages && !mbar_wait(smem_u32(&sm.k_empty[ks]), ((j / kKStages) - 1) & 1, &sm.abort)) break;
        const uint32_t kbar = smem_u32(&sm.k_full[ks]);
        mbar_arrive_expect_tx(kbar, Smem::kTileBytes);
#pragma unroll
        for (int x = 0; x < D / 64; ++x)
          tma_load_3d_hint(smem_u32(sm.k[ks]) + x * kBoxBytes, &tm_k, kbar, x * 64, j * BN, b * Hkv + kvh, keep);
        ++k_issued;
        const int vs = j % kVStages;
        if (j >= kVStages && !mbar_wait(smem_u32(&sm.v_empty[vs]), ((j / kVStages) - 1) & 1, &sm.abort)) break;
        const uint32_t vbar = smem_u32(&sm.v_full[vs]);
        mbar_arrive_expect_tx(vbar, Smem::kTileBytes);
#pragma unroll
        for (int x = 0; x < D / 64; ++x)
          tma_load_3d_hint(smem_u32(sm.v[vs]) + x * kBoxBytes, &tm_v, vbar, x * 64, j * BN, b * Hkv + kvh, keep);
        ++v_issued;
      }
      // drain: every issued copy must land before the CTA's shared memory is released
      mbar_wait(qbar, 0, nullptr);
      for (int s = 0; s < kKStages && s < k_issued; ++s) {
        const int last = s + ((k_issued - 1 - s) / kKStages) * kKStages;
        mbar_wait(smem_u32(&sm.k_full[s]), (last / kKStages) & 1, nullptr);
      }
      for (int s = 0; s < kVStages && s < v_issued; ++s) {
        const int last = s + ((v_issued - 1 - s) / kVStages) * kVStages;
        mbar_wait(smem_u32(&sm.v_full[s]), (last / kVStages) & 1, nullptr);
      }
    }
    __syncwarp();
  } else if (warp == 1 || warp == 2) {
    // ================================================================ MMA warps, one per chain
    const int c = warp - 1;
    const int n_c = n_tiles[c];
    constexpr uint32_t idesc_qk = tc05::idesc_bf16_f32(BM, BN, false);
    constexpr uint32_t idesc_pv = tc05::idesc_bf16_f32(BM, D, true);
    const uint32_t q_addr = smem_u32(sm.q[c]);
    const uint32_t s_tmem = tmem + c * BN;
    const uint32_t o_tmem = tmem + 2 * BN + c * BN;
    // key tiles the other chain does not visit are handed back with two arrivals from this chain
    const int n_other = n_tiles[1 - c];
    bool ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&sm.q_full), 0, &sm.abort));
    for (int j = 0; ok && j < n_c; ++j) {
      // S_c(j) = Q_c K_j^T, once O_c += P_c(j-1) V_{j-1} has completed (S_c holds P_c(j-1))
      if (j > 0 && !__all_sync(0xffffffffu, mbar_wait(smem_u32(&sm.pv_done[c]), (j - 1) & 1, &sm.abort))) break;
      const int ks = j % kKStages;
      if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&sm.k_full[ks]), (j / kKStages) & 1, &sm.abort))) break;
      tc05::fence_after_sync();
      const uint32_t k_addr = smem_u32(sm.k[ks]);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t off = (kk >> 2) * kBoxBytes + (kk & 3) * 32;
        const uint64_t da = tc05::sdesc_sw128(q_addr + off, 16, 1024);
        const uint64_t db = tc05::sdesc_sw128(k_addr + off, 16, 1024);
        if (elect_one()) tc05::mma_ss(s_tmem, da, db, idesc_qk, kk > 0);
        __syncwarp();
      }
      if (elect_one()) {
        tc05::commit(smem_u32(&sm.s_full[c]));
        tc05::commit(smem_u32(&sm.k_empty[ks]));
        if (j >= n_other) tc05::commit(smem_u32(&sm.k_empty[ks]));
      }
      __syncwarp();
      // O_c += P_c(j) V_j, once softmax has written P_c(j)
      const int vs = j % kVStages;
      if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&sm.p_full[c]), j & 1, &sm.abort))) break;
      if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&sm.v_full[vs]), (j / kVStages) & 1, &sm.abort))) break;
      tc05::fence_after_sync();
      const uint32_t v_addr = smem_u32(sm.v[vs]);
#pragma unroll
      for (int kk = 0; kk < BN / 16; ++kk) {
        const uint64_t db = tc05::sdesc_sw128(v_addr + kk * 2048, kBoxBytes, 1024);
        if (elect_one()) tc05::mma_ts(o_tmem, s_tmem + kk * 8, db, idesc_pv, (j > 0) || (kk > 0));
        __syncwarp();
      }
      if (elect_one()) {
        tc05::commit(smem_u32(&sm.pv_done[c]));
        tc05::commit(smem_u32(&sm.v_empty[vs]));
        if (j >= n_other) tc05::commit(smem_u32(&sm.v_empty[vs]));
      }
      __syncwarp();
    }
    // every MMA this warp issued must complete before tensor memory is released
    if (elect_one()) tc05::commit(smem_u32(&sm.mma_done));
    __syncwarp();
    mbar_wait(smem_u32(&sm.mma_done), 0, nullptr);
  } else if (warp >= 4) {
    // ================================================================ softmax warpgroups
    asm volatile("setmaxnreg.inc.sync.aligned.u32 224;" ::: "memory");
    const int c = (warp - 4) >> 2;              // 0: tile A, 1: tile B
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;        // row within the tile = TMEM lane
    const int q_row = row0[c] + row;
    const int n_c = n_tiles[c];
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t s_addr = tmem + lane_addr + c * BN;
    const uint32_t o_addr = tmem + lane_addr + 2 * BN + c * BN;
    const int lim = causal ? min(q_row + 1, N) : N;  // keys [0, lim) are attended by this row
    const uint64_t scale2 = f2(scale_log2, scale_log2);
    float m_ref = -INFINITY;  // reference maximum (log2 units) that p and o~ are relative to
    float l = 0.f;
    bool ok = true;
    for (int j = 0; j < n_c; ++j) {
      // wait outcomes are made warp-uniform: tcgen05.ld/st are warp-collective
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

      const int kv0 = j * BN;
      if (kv0 + BN > lim) {  // diagonal tile or ragged tail: mask keys >= lim
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4)
#pragma unroll
          for (int e = 0; e < 32; ++e)
            if (kv0 + q4 * 32 + e >= lim) sr[q4][e] = __float_as_uint(-INFINITY);
      }
      // row max: four independent 3-input max chains
      float mq[4];
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        float m = __uint_as_float(sr[q4][0]);
#pragma unroll
        for (int e = 1; e < 31; e += 2) m = max3(m, __uint_as_float(sr[q4][e]), __uint_as_float(sr[q4][e + 1]));
        mq[q4] = fmaxf(m, __uint_as_float(sr[q4][31]));
      }
      const float m_new = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3])) * scale_log2;
      // move the reference only when the row maximum outgrows it by more than 2^8
      const bool move = m_new > m_ref + kRescaleThreshold;
      const float m_next = move ? m_new : m_ref;
      const float corr = ex2_approx(m_ref - m_next);  // 1 when kept; 0 on the first tile
      m_ref = m_next;

      // p = 2^(s * scale * log2(e) - m_ref), summed in eight partial sums, packed to bf16
      const uint64_t negm2 = f2(-m_ref, -m_ref);
      uint64_t acc2[4] = {0ull, 0ull, 0ull, 0ull};
      uint32_t pr[2][32];
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          float x0, x1;
          f2_split(fma2(f2(__uint_as_float(sr[q4][e]), __uint_as_float(sr[q4][e + 1])), scale2, negm2), x0, x1);
          const float p0 = ex2_approx(x0);
          const float p1 = ex2_approx(x1);
          acc2[(e >> 1) & 3] = add2(acc2[(e >> 1) & 3], f2(p0, p1));
          pr[q4 >> 1][(q4 & 1) * 16 + (e >> 1)] = pack_bf16x2(p0, p1);
        }
      }
      tc05::tmem_st_x32(s_addr, pr[0]);
      tc05::tmem_st_x32(s_addr + 32, pr[1]);
      float sum_lo, sum_hi;
      f2_split(add2(add2(acc2[0], acc2[1]), add2(acc2[2], acc2[3])), sum_lo, sum_hi);
      l = l * corr + (sum_lo + sum_hi);

      if (__any_sync(0xffffffffu, move) && j > 0) {
        // o~ must hold the complete P_{j-1} V_{j-1} before it is rescaled; the MMA
        // issuer only started S_c(j) after that product completed, so this wait
        // returns at once
        if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&sm.pv_done[c]), (j - 1) & 1, &sm.abort))) {
          ok = false;
          break;
        }
        tc05::fence_after_sync();
#pragma unroll
        for (int q4 = 0; q4 < D / 32; ++q4) rescale_o_chunk(o_addr + q4 * 32, corr);
      }
      tc05::tmem_wait_st();
      tc05::fence_before_sync();
      mbar_arrive(smem_u32(&sm.p_full[c]));
    }

    // ---- epilogue: O = o~ / l, LSE = m + ln l
    if (ok && n_c > 0) {
      ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&sm.pv_done[c]), (n_c - 1) & 1, &sm.abort));
      if (ok) {
        tc05::fence_after_sync();
        const float inv = (l > 0.f) ? 1.f / l : 0.f;
        const uint64_t inv2 = f2(inv, inv);
        const bool store = q_row < N;
        __nv_bfloat16 *orow = o + ((static_cast<size_t>(b) * H + h) * N + (store ? q_row : 0)) * D;
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
        if (store && lse != nullptr)
          lse[(static_cast<size_t>(b) * H + h) * N + q_row] = (l > 0.f) ? m_ref * kLn2 + logf(l) : -INFINITY;
      }
    }
  }

  tc05::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc05::fence_after_sync();
    tc05::tmem_dealloc(tmem, kTmemCols);
  }
}

template <int D>
cudaError_t launch_d(const PrefillMaps &maps, void *o, float *lse, int B, int H, int Hkv, int N, bool causal,
                     float scale, cudaStream_t stream) {
  // One CTA per SM: the kernel holds all 512 tensor-memory columns.
  const size_t smem = std::max<size_t>(sizeof(PrefillSmem<D>) + 1024, 120 * 1024);
  auto kern = prefill_bf16_kernel<D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const long long n_pairs = (N + 2 * BM - 1) / (2 * BM);
  const long long blocks = n_pairs * B * H;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  kern<<<static_cast<unsigned>(blocks), kThreads, smem, stream>>>(maps.q, maps.k, maps.v,
                                                                   static_cast<__nv_bfloat16 *>(o), lse, B, H, Hkv, N,
                                                                   causal ? 1 : 0, scale * kLog2e);
  return cudaGetLastError();
}

}  // namespace

ATTN_DEFINE_ERROR_ACCESSOR(device_error_prefill_bf16)

cudaError_t launch_prefill_bf16(const PrefillMaps &maps, void *o, float *lse, int B, int H, int Hkv, int N, int d,
                                bool causal, float scale, int /*num_sms*/, cudaStream_t stream) {
  if (d == 64) return launch_d<64>(maps, o, lse, B, H, Hkv, N, causal, scale, stream);
  return launch_d<128>(maps, o, lse, B, H, Hkv, N, causal, scale, stream);
}

}  // namespace attn
