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
// GB300 mapping (one CTA per query tile, 256 threads):
//   warp 0      TMA producer: Q once, then K_j / V_j into a 2-stage ring each
//               (128-byte-swizzled tiles, completion on mbarriers).
//   warp 1      allocates tensor memory; lane 0 issues every tcgen05.mma:
//               S_j = Q K_j^T  (SS form, A = Q and B = K both K-major in SMEM)
//               O  += P_j V_j  (TS form, A = P_j from TMEM, B = V MN-major in SMEM)
//               and tracks completion with tcgen05.commit.
//   warps 4-7   softmax warpgroup, one thread per query row (TMEM lane): loads
//               S_j from TMEM, masks, updates m and l, writes P_j = bf16(p)
//               back into the same TMEM columns, and rescales O in TMEM
//               lazily: the reference maximum only moves when the new row max
//               exceeds it by more than 2^8 (the result does not depend on
//               which reference is used; p stays <= 256).  Finally writes
//               O = o~ / l (bf16, round to nearest even) and the LSE.
// Tensor memory (512 columns x 128 lanes x 32 bit): three S buffers of 128
// columns (P_j aliases the first 64 columns of S_j) and O (d columns), so
// S_{j+1} and S_{j+2} can be computed while softmax works on S_j.
// Query-tile order: heaviest causal tiles first across all (batch, head).
#include <algorithm>

#include "common.cuh"
#include "tc05.cuh"
#include "kernels.h"

namespace attn {
namespace {

constexpr int BM = 128;      // query rows per tile (= TMEM lanes)
constexpr int BN = 128;      // keys per K/V tile
constexpr int kSBuf = 3;     // S buffers in tensor memory
constexpr int kKStages = 2;
constexpr int kVStages = 2;
constexpr int kThreads = 256;
constexpr int kSoftmaxWarp0 = 4;
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr int kBoxBytes = BN * 64 * 2;     // one 128-row x 64-column bf16 TMA box: 16 KiB

template <int D>
struct PrefillSmem {
  static constexpr int kTileBytes = BN * D * 2;
  alignas(1024) uint8_t q[BM * D * 2];
  alignas(1024) uint8_t k[kKStages][kTileBytes];
  alignas(1024) uint8_t v[kVStages][kTileBytes];
  uint64_t q_full;
  uint64_t k_full[kKStages], k_empty[kKStages];
  uint64_t v_full[kVStages], v_empty[kVStages];
  uint64_t s_full[kSBuf], p_full[kSBuf], pv_done[kSBuf];
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort;
};

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

  // ---- which (query tile, batch, head): heaviest causal tiles first
  const int n_qt = (N + BM - 1) / BM;
  const int bh_count = B * H;
  const int qt_rank = blockIdx.x / bh_count;
  const int bh = blockIdx.x % bh_count;
  const int qt = causal ? (n_qt - 1 - qt_rank) : qt_rank;
  const int b = bh / H;
  const int h = bh % H;
  const int kvh = h / (H / Hkv);
  const int n_kt = causal ? (qt + 1) : (N + BN - 1) / BN;  // key tiles visited

  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&sm.q_full), 1);
    for (int s = 0; s < kKStages; ++s) {
      mbar_init(smem_u32(&sm.k_full[s]), 1);
      mbar_init(smem_u32(&sm.k_empty[s]), 1);
    }
    for (int s = 0; s < kVStages; ++s) {
      mbar_init(smem_u32(&sm.v_full[s]), 1);
      mbar_init(smem_u32(&sm.v_empty[s]), 1);
    }
    for (int s = 0; s < kSBuf; ++s) {
      mbar_init(smem_u32(&sm.s_full[s]), 1);
      mbar_init(smem_u32(&sm.p_full[s]), 128);
      mbar_init(smem_u32(&sm.pv_done[s]), 1);
    }
    mbar_init(smem_u32(&sm.mma_done), 1);
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
  const uint32_t tmem_o = tmem + kSBuf * BN;

  if (warp == 0) {
    // ================================================================ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      const uint64_t keep = l2_policy_evict_last();  // K/V tiles are re-read by other query tiles
      const uint32_t qbar = smem_u32(&sm.q_full);
      mbar_arrive_expect_tx(qbar, BM * D * 2);
#pragma unroll
      for (int x = 0; x < D / 64; ++x) tma_load_3d(smem_u32(sm.q) + x * kBoxBytes, &tm_q, qbar, x * 64, qt * BM, b * H + h);
      int k_issued = 0, v_issued = 0;
      for (int j = 0; j < n_kt; ++j) {
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
  } else if (warp == 1) {
    // ================================================================ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_qk = tc05::idesc_bf16_f32(BM, BN, false);
      constexpr uint32_t idesc_pv = tc05::idesc_bf16_f32(BM, D, true);
      const uint32_t q_addr = smem_u32(sm.q);
      bool ok = mbar_wait(smem_u32(&sm.q_full), 0, &sm.abort);
      auto issue_qk = [&](int j) -> bool {
        const int sb = j % kSBuf;
        const int ks = j % kKStages;
        if (!mbar_wait(smem_u32(&sm.k_full[ks]), (j / kKStages) & 1, &sm.abort)) return false;
        tc05::fence_after_sync();
        const uint32_t k_addr = smem_u32(sm.k[ks]);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kBoxBytes + (kk & 3) * 32;
          tc05::mma_ss(tmem + sb * BN, tc05::sdesc_sw128(q_addr + off, 16, 1024),
                       tc05::sdesc_sw128(k_addr + off, 16, 1024), idesc_qk, kk > 0);
        }
        tc05::commit(smem_u32(&sm.s_full[sb]));
        tc05::commit(smem_u32(&sm.k_empty[ks]));
        return true;
      };
      if (ok) ok = issue_qk(0);
      if (ok && n_kt > 1) ok = issue_qk(1);
      for (int j = 0; ok && j < n_kt; ++j) {
        const int sb = j % kSBuf;
        const int vs = j % kVStages;
        if (!mbar_wait(smem_u32(&sm.p_full[sb]), (j / kSBuf) & 1, &sm.abort)) break;
        if (!mbar_wait(smem_u32(&sm.v_full[vs]), (j / kVStages) & 1, &sm.abort)) break;
        tc05::fence_after_sync();
        const uint32_t v_addr = smem_u32(sm.v[vs]);
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk) {
          tc05::mma_ts(tmem_o, tmem + sb * BN + kk * 8, tc05::sdesc_sw128(v_addr + kk * 2048, kBoxBytes, 1024),
                       idesc_pv, (j > 0) || (kk > 0));
        }
        tc05::commit(smem_u32(&sm.pv_done[sb]));
        tc05::commit(smem_u32(&sm.v_empty[vs]));
        if (j + 2 < n_kt) {
          // S buffer (j + 2) % 3 held P_{j-1}: P.V of tile j - 1 must have finished
          if (j >= 1 && !mbar_wait(smem_u32(&sm.pv_done[(j - 1) % kSBuf]), ((j - 1) / kSBuf) & 1, &sm.abort)) break;
          ok = issue_qk(j + 2);
        }
      }
      // every MMA this thread issued must complete before tensor memory is released
      tc05::commit(smem_u32(&sm.mma_done));
      mbar_wait(smem_u32(&sm.mma_done), 0, nullptr);
    }
    __syncwarp();
  } else if (warp >= kSoftmaxWarp0) {
    // ================================================================ softmax warpgroup
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;          // row within the tile = TMEM lane
    const int q_row = qt * BM + row;
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    float m_ref = -INFINITY;  // reference maximum (log2 units) that p and o~ are relative to
    float l = 0.f;
    bool ok = true;
    for (int j = 0; j < n_kt; ++j) {
      const int sb = j % kSBuf;
      // wait outcomes are made warp-uniform: tcgen05.ld/st are warp-collective
      if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&sm.s_full[sb]), (j / kSBuf) & 1, &sm.abort))) {
        ok = false;
        break;
      }
      tc05::fence_after_sync();
      const uint32_t s_addr = tmem + lane_addr + sb * BN;
      uint32_t sr[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tc05::tmem_ld_x32(s_addr + c * 32, sr[c]);
#pragma unroll
      for (int c = 0; c < 4; ++c) tc05::tmem_ld_wait(sr[c]);

      const int kv0 = j * BN;
      const bool edge = (causal && j == qt) || (kv0 + BN > N);
      if (edge) {
        const int lim = causal ? min(q_row + 1, N) : N;  // keys [kv0, lim) are attended
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int e = 0; e < 32; ++e)
            if (kv0 + c * 32 + e >= lim) sr[c][e] = __float_as_uint(-INFINITY);
      }
      float mx = -INFINITY;
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int e = 0; e < 32; ++e) mx = fmaxf(mx, __uint_as_float(sr[c][e]));
      const float m_new = mx * scale_log2;
      // move the reference only when the row maximum outgrows it by more than 2^8
      const bool move = m_new > m_ref + kRescaleThreshold;
      const float m_next = move ? m_new : m_ref;
      if (__any_sync(0xffffffffu, move) && j > 0) {
        const float corr = ex2_approx(m_ref - m_next);  // 1 for rows that keep their reference
        // o~ in TMEM must hold the complete P_{j-1} V_{j-1} before it is rescaled
        if (!__all_sync(0xffffffffu,
                        mbar_wait(smem_u32(&sm.pv_done[(j - 1) % kSBuf]), ((j - 1) / kSBuf) & 1, &sm.abort))) {
          ok = false;
          break;
        }
        tc05::fence_after_sync();
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t orr[32];
          tc05::tmem_ld_x32(tmem_o + lane_addr + c * 32, orr);
          tc05::tmem_ld_wait(orr);
#pragma unroll
          for (int e = 0; e < 32; ++e) orr[e] = __float_as_uint(__uint_as_float(orr[e]) * corr);
          tc05::tmem_st_x32(tmem_o + lane_addr + c * 32, orr);
        }
        l *= corr;
      }
      m_ref = m_next;
      // p = exp2(s * scale * log2(e) - m_ref), rounded to bf16 into TMEM over S_j
      const float neg_m = -m_ref;
      float rowsum = 0.f;
      uint32_t pr[2][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const float p0 = ex2_approx(fmaf(__uint_as_float(sr[c][e]), scale_log2, neg_m));
          const float p1 = ex2_approx(fmaf(__uint_as_float(sr[c][e + 1]), scale_log2, neg_m));
          rowsum += p0 + p1;
          pr[c >> 1][(c & 1) * 16 + (e >> 1)] = pack_bf16x2(p0, p1);
        }
      }
      l += rowsum;
      tc05::tmem_st_x32(s_addr, pr[0]);
      tc05::tmem_st_x32(s_addr + 32, pr[1]);
      tc05::tmem_wait_st();
      tc05::fence_before_sync();
      mbar_arrive(smem_u32(&sm.p_full[sb]));
    }

    // ---- epilogue: O = o~ / l, LSE = m + ln l
    if (ok) {
      const int last = n_kt - 1;
      ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&sm.pv_done[last % kSBuf]), (last / kSBuf) & 1, &sm.abort));
    }
    if (ok) {
      tc05::fence_after_sync();
      const float inv = (l > 0.f) ? 1.f / l : 0.f;
      const bool store = q_row < N;
      __nv_bfloat16 *orow = o + ((static_cast<size_t>(b) * H + h) * N + (store ? q_row : 0)) * D;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t orr[32];
        tc05::tmem_ld_x32(tmem_o + lane_addr + c * 32, orr);
        tc05::tmem_ld_wait(orr);
        uint32_t packed[16];
#pragma unroll
        for (int e = 0; e < 16; ++e)
          packed[e] = pack_bf16x2(__uint_as_float(orr[2 * e]) * inv, __uint_as_float(orr[2 * e + 1]) * inv);
        if (store) {
          uint4 *dst = reinterpret_cast<uint4 *>(orow + c * 32);
#pragma unroll
          for (int e = 0; e < 4; ++e)
            dst[e] = make_uint4(packed[4 * e], packed[4 * e + 1], packed[4 * e + 2], packed[4 * e + 3]);
        }
      }
      if (store && lse != nullptr)
        lse[(static_cast<size_t>(b) * H + h) * N + q_row] = (l > 0.f) ? m_ref * kLn2 + logf(l) : -INFINITY;
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
  const long long n_qt = (N + BM - 1) / BM;
  const long long blocks = n_qt * B * H;
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
