// Split-KV paged decode and the exact merge of partial results (sm_103a).
//
// "3.4 Attention Kernels" (llm-learning-path), "Decode attention and
// Flash-Decoding": the keys of each sequence are split into chunks, one CTA
// per (sequence, KV head, chunk) computes the partial (m_c, l_c, o~_c) of all
// query heads of the GQA group against that chunk, and a small reduction
// kernel merges the partials with the log-sum-exp rule of "Online softmax".
// "Paged and ragged layouts: FlashInfer": K/V are gathered page by page
// through the page table.
//
// Data movement: a single producer thread streams each page of the chunk
// (K and V, 16 tokens x d dims bf16 each: 4 KiB + 4 KiB at d = 128) into a ring of
// shared-memory stages with TMA tensor loads (128-byte swizzle), completion
// signalled on mbarriers.  Four consumer warps take pages round-robin, each
// keeping its own online-softmax state; the four states are merged exactly in
// shared memory at the end.  Per page a consumer warp does the two small
// contractions S = Q K^T (16 heads-rows x 16 tokens x d) and O += P V
// (16 x d x 16 tokens) with warp-level bf16 tensor-core MMAs; the GQA
// group's g <= 16 query heads are the rows, so every K/V byte loaded is used
// g times.  Only the running row max m, the partial row sums and the output
// fragments live in registers.
#include "common.cuh"
#include "kernels.h"

namespace attn {

namespace {

constexpr int kPage = 16;               // tokens per page
constexpr int kConsumerWarps = 4;
constexpr int kHalfBytes = kPage * 64 * 2;        // one 64-column block of a K or V page: 2 KiB
constexpr int kThreads = (kConsumerWarps + 1) * 32;

// Sizes for head dimension D (64 or 128): a stage holds one page of K and one of V;
// the ring keeps 32 KiB in flight per CTA whatever D is (64 KiB measured 7 % slower on
// the 64-sequence workload: three CTAs per SM either way, set by the registers, but
// the smaller ring leaves more of each SM's unified L1 / shared storage to the cache).
template <int D>
struct DecodeGeom {
  static constexpr int kPageBytes = (D / 64) * kHalfBytes;  // 4 KiB at d = 128
  static constexpr int kStageBytes = 2 * kPageBytes;        // K page + V page
  static constexpr int kStages = (32 * 1024) / kStageBytes;  // 4 at d = 128, 8 at d = 64
  // Consumer warp w takes pages w, w + 4, ... and page i uses stage i mod kStages, so
  // with kStages a multiple of the consumer count every use of a stage falls to the same
  // warp, which then waits on that stage's barrier phases strictly in order.  Otherwise a
  // warp could wait on a phase two ahead of the barrier, which a parity wait reports as
  // already complete.
  static_assert(kStages % kConsumerWarps == 0, "each ring stage must belong to one consumer warp");
  // the per-warp output fragments are merged through the (then idle) ring at the end
  static_assert(kConsumerWarps * 16 * D * 4 <= kStages * kStageBytes, "merge scratch must fit in the ring");
};

template <int D>
struct DecodeSmem {
  using G = DecodeGeom<D>;
  alignas(1024) uint8_t stage[G::kStages][G::kStageBytes];
  uint64_t full[G::kStages];
  uint64_t empty[G::kStages];
  float warp_m[kConsumerWarps][16];
  float warp_l[kConsumerWarps][16];
  int abort;
};
// The per-warp output fragments are merged through the (then idle) stage
// buffers: 4 warps x 16 rows x d fp32 (32 KiB at d = 128), the ring's 32 KiB
// (checked in DecodeGeom).

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void mma_bf16_16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Byte offset of the 16-byte chunk holding (row, col) of a 64-column half tile
// written by TMA with the 128-byte swizzle: chunk index XOR (row mod 8).
__device__ __forceinline__ uint32_t swz(int row, int col) {
  return static_cast<uint32_t>(row * 128 + ((((col >> 3) ^ row) & 7) << 4));
}

// Rows 0..7 of the MMA tile hold query heads 0..7 of the group, rows 8..15
// heads 8..15; kHiRows says whether any head lands in rows 8..15 (g > 8).
// Four CTAs per SM (at most 96 registers a thread, a few spilled) measured 2.7 % faster than
// three; the instance for groups of more than 8 query heads keeps three (it would spill more).
template <int D, bool kHiRows>
__global__ void __launch_bounds__(kThreads, kHiRows ? 3 : 4)
    decode_split_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                        const __nv_bfloat16 *__restrict__ q, const int32_t *__restrict__ page_table,
                        const int32_t *__restrict__ kv_lens, float *__restrict__ ws_m, float *__restrict__ ws_l,
                        float *__restrict__ ws_o, int H, int Hkv, int max_pages, int num_pages, int chunk_pages,
                        int S, float scale_log2) {
  using G = DecodeGeom<D>;
  constexpr int kStages = G::kStages;
  constexpr int kPageBytes = G::kPageBytes;
  constexpr int kStageBytes = G::kStageBytes;
  extern __shared__ uint8_t smem_raw[];
  DecodeSmem<D> &sm =
      *reinterpret_cast<DecodeSmem<D> *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  // the grid is (KV head, sequence, split) with the split slowest: CTAs are dispatched
  // chunk 0 of every sequence first, and the last ones dispatched are the final
  // chunks of the longest sequences
  const int split = blockIdx.z;
  const int kvh = blockIdx.x;
  const int b = blockIdx.y;
  const int g = H / Hkv;
  int L = kv_lens[b];
  if (L < 0 || L > max_pages * kPage) {
    // a length the page table cannot hold: attend to what the table covers
    if (threadIdx.x == 0) record_device_error(ATTN_DEVERR_BAD_PAGE);
    L = max(0, min(L, max_pages * kPage));
  }
  const int pages_b = (L + kPage - 1) / kPage;
  const int first = split * chunk_pages;
  if (first >= pages_b) return;  // this sequence needs fewer partials; the merge never reads this slot
  const int npg = min(pages_b, first + chunk_pages) - first;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&sm.full[s]), 1);
      mbar_init(smem_u32(&sm.empty[s]), 1);
    }
    sm.abort = 0;
    fence_barrier_init();
  }
  __syncthreads();

  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------ producer
    // The warp reads the chunk's page ids 32 at a time (one coalesced load,
    // the next batch fetched while the current one is issued); lane 0 issues
    // the TMA copies.
    if (lane == 0) {
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
    }
    const uint64_t policy = l2_policy_evict_first();
    const int32_t *row = page_table + static_cast<size_t>(b) * max_pages + first;
    int issued = 0;
    bool ok = true;
    int next_ids = lane < npg ? row[lane] : 0;
    for (int base = 0; ok && base < npg; base += 32) {
      const int ids = next_ids;
      if (base + 32 < npg) next_ids = (base + 32 + lane < npg) ? row[base + 32 + lane] : 0;
      const int n = min(32, npg - base);
      for (int t = 0; t < n; ++t) {
        const int i = base + t;
        const int page = __shfl_sync(0xffffffffu, ids, t);
        int good = 1;
        if (lane == 0) {
          const int s = i % kStages;
          if (i >= kStages && !mbar_wait(smem_u32(&sm.empty[s]), ((i / kStages) - 1) & 1, &sm.abort)) {
            good = 0;
          } else {
            if (page < 0 || page >= num_pages) {
              // out of the pool: TMA fills an out-of-range box with zeros; record it
              record_device_error(ATTN_DEVERR_BAD_PAGE);
            }
            const int c2 = page * Hkv + kvh;
            const uint32_t bar = smem_u32(&sm.full[s]);
            const uint32_t dst = smem_u32(&sm.stage[s][0]);
            mbar_arrive_expect_tx(bar, kStageBytes);
#pragma unroll
            for (int x = 0; x < D / 64; ++x) {
              tma_load_3d_hint(dst + x * kHalfBytes, &tm_k, bar, x * 64, 0, c2, policy);
              tma_load_3d_hint(dst + kPageBytes + x * kHalfBytes, &tm_v, bar, x * 64, 0, c2, policy);
            }
            ++issued;
          }
        }
        if (!__shfl_sync(0xffffffffu, good, 0)) {
          ok = false;
          break;
        }
      }
    }
    // Teardown: the ring is reused as merge scratch, and the CTA may exit
    // early, only after every issued copy has landed.  Wait (bounded) for
    // the last phase of each stage this thread armed.
    if (lane == 0) {
      for (int s = 0; s < kStages && s < issued; ++s) {
        const int last_i = s + ((issued - 1 - s) / kStages) * kStages;
        mbar_wait(smem_u32(&sm.full[s]), (last_i / kStages) & 1, nullptr);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ consumers
    const int r0 = lane >> 2;           // MMA rows r0 and r0 + 8
    const int cpair = (lane & 3) * 2;   // column pair within an 8-wide n tile
    // Q fragments (A operand, rows = the group's query heads), loaded once.
    uint32_t qa[D / 16][4];
    {
      const int h_lo = kvh * g + r0;
      const int h_hi = kvh * g + r0 + 8;
      const bool v_lo = r0 < g;
      const bool v_hi = kHiRows && (r0 + 8 < g);
      const uint32_t *q_lo = reinterpret_cast<const uint32_t *>(q + (static_cast<size_t>(b) * H + h_lo) * D);
      const uint32_t *q_hi = reinterpret_cast<const uint32_t *>(q + (static_cast<size_t>(b) * H + h_hi) * D);
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        const int c = ks * 16 + cpair;
        qa[ks][0] = v_lo ? q_lo[c / 2] : 0u;
        qa[ks][1] = v_hi ? q_hi[c / 2] : 0u;
        qa[ks][2] = v_lo ? q_lo[(c + 8) / 2] : 0u;
        qa[ks][3] = v_hi ? q_hi[(c + 8) / 2] : 0u;
      }
    }
    float acc[D / 8][4];
#pragma unroll
    for (int i = 0; i < D / 8; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
    float m_lo = -INFINITY, m_hi = -INFINITY;  // running max (log2 units) of rows r0, r0 + 8
    float l_lo = 0.f, l_hi = 0.f;              // this lane's share of the running sums

    // ldmatrix lane roles
    const int mi = lane >> 3;   // which of the four 8x8 matrices this lane addresses
    const int mr = lane & 7;    // row within it

    for (int i = warp; i < npg; i += kConsumerWarps) {
      const int s = i % kStages;
      const bool landed = mbar_wait(smem_u32(&sm.full[s]), (i / kStages) & 1, &sm.abort);
      if (!__all_sync(0xffffffffu, landed)) break;  // keep the warp converged for ldmatrix / mma
      const uint32_t kbase = smem_u32(&sm.stage[s][0]);
      const uint32_t vbase = kbase + kPageBytes;

      // ---- S = Q K^T for the 16 tokens of this page (two n tiles of 8)
      float sc[2][4];
#pragma unroll
      for (int n = 0; n < 2; ++n) sc[n][0] = sc[n][1] = sc[n][2] = sc[n][3] = 0.f;
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        // matrices: (tok 0-7, d lo), (tok 0-7, d hi), (tok 8-15, d lo), (tok 8-15, d hi)
        const int tok = ((mi >> 1) << 3) + mr;
        const int col = ks * 16 + ((mi & 1) << 3);
        const uint32_t addr = kbase + (col >> 6) * kHalfBytes + swz(tok, col & 63);
        uint32_t b0, b1, b2, b3;
        ldsm_x4(addr, b0, b1, b2, b3);
        mma_bf16_16816(sc[0], qa[ks], b0, b1);
        mma_bf16_16816(sc[1], qa[ks], b2, b3);
      }

      // ---- online softmax update (log2 units), masking tokens past the sequence end
      const int tok0 = (first + i) * kPage;
      float mx_lo = -INFINITY, mx_hi = -INFINITY;
#pragma unroll
      for (int n = 0; n < 2; ++n) {
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const bool live = tok0 + n * 8 + cpair + j < L;
          sc[n][j] = live ? sc[n][j] * scale_log2 : -INFINITY;
          sc[n][2 + j] = live ? sc[n][2 + j] * scale_log2 : -INFINITY;
          mx_lo = fmaxf(mx_lo, sc[n][j]);
          mx_hi = fmaxf(mx_hi, sc[n][2 + j]);
        }
      }
      mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, 1));
      mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, 2));
      if (kHiRows) {
        mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, 1));
        mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, 2));
      }
      const float mn_lo = fmaxf(m_lo, mx_lo);
      const float mn_hi = kHiRows ? fmaxf(m_hi, mx_hi) : 0.f;
      // rescale the running state only when some row's maximum grew
      const bool grow = (mn_lo > m_lo) || (kHiRows && mn_hi > m_hi);
      if (__any_sync(0xffffffffu, grow)) {
        const float c_lo = ex2_approx(m_lo - mn_lo);  // exp2(-inf) = 0 on the first page
        const float c_hi = kHiRows ? ex2_approx(m_hi - mn_hi) : 0.f;
        l_lo *= c_lo;
        l_hi *= c_hi;
#pragma unroll
        for (int t = 0; t < D / 8; ++t) {
          acc[t][0] *= c_lo;
          acc[t][1] *= c_lo;
          acc[t][2] *= c_hi;
          acc[t][3] *= c_hi;
        }
        m_lo = mn_lo;
        m_hi = mn_hi;
      }
      float p[2][4];
#pragma unroll
      for (int n = 0; n < 2; ++n) {
        p[n][0] = ex2_approx(sc[n][0] - m_lo);
        p[n][1] = ex2_approx(sc[n][1] - m_lo);
        p[n][2] = kHiRows ? ex2_approx(sc[n][2] - m_hi) : 0.f;
        p[n][3] = kHiRows ? ex2_approx(sc[n][3] - m_hi) : 0.f;
        l_lo += p[n][0] + p[n][1];
        l_hi += p[n][2] + p[n][3];
      }
      // P as the A operand of the P.V MMA (k = tokens 0..15)
      uint32_t pa[4];
      pa[0] = pack_bf16x2(p[0][0], p[0][1]);
      pa[1] = pack_bf16x2(p[0][2], p[0][3]);
      pa[2] = pack_bf16x2(p[1][0], p[1][1]);
      pa[3] = pack_bf16x2(p[1][2], p[1][3]);

      // ---- slots of the sequence's last page past its length may hold anything (stale
      //      tokens, or non-finite values in a pool that was never written): their weights
      //      are exact zeros, but 0 x NaN is NaN in the MMA, so their V rows are zeroed first
      //      (whole 128-byte rows of each 64-column half; the swizzle only permutes chunks
      //      within a row).  The proxy fence orders these writes before the TMA that later
      //      refills the stage.
      const int valid = L - tok0;
      if (valid < kPage) {
        const int n16 = (kPage - valid) * 8;  // 16-byte chunks per half
        for (int idx = lane; idx < n16 * (D / 64); idx += 32) {
          const int half = idx / n16, rem = idx % n16;
          *reinterpret_cast<uint4 *>(&sm.stage[s][kPageBytes + half * kHalfBytes + (valid + rem / 8) * 128 +
                                                  (rem % 8) * 16]) = make_uint4(0u, 0u, 0u, 0u);
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
      }

      // ---- O += P V over the 16 n tiles of the head dimension
#pragma unroll
      for (int dt = 0; dt < D / 8; dt += 2) {
        // matrices: (tok 0-7, d dt), (tok 8-15, d dt), (tok 0-7, d dt+1), (tok 8-15, d dt+1)
        const int tok = ((mi & 1) << 3) + mr;
        const int col = (dt + (mi >> 1)) * 8;
        const uint32_t addr = vbase + (col >> 6) * kHalfBytes + swz(tok, col & 63);
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(addr, b0, b1, b2, b3);
        mma_bf16_16816(acc[dt], pa, b0, b1);
        mma_bf16_16816(acc[dt + 1], pa, b2, b3);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sm.empty[s]));
    }

    // full row sums of this warp's state
    l_lo += __shfl_xor_sync(0xffffffffu, l_lo, 1);
    l_lo += __shfl_xor_sync(0xffffffffu, l_lo, 2);
    l_hi += __shfl_xor_sync(0xffffffffu, l_hi, 1);
    l_hi += __shfl_xor_sync(0xffffffffu, l_hi, 2);
    if ((lane & 3) == 0) {
      sm.warp_m[warp][r0] = m_lo;
      sm.warp_l[warp][r0] = l_lo;
      sm.warp_m[warp][r0 + 8] = kHiRows ? m_hi : -INFINITY;
      sm.warp_l[warp][r0 + 8] = kHiRows ? l_hi : 0.f;
    }
    // Stash this warp's unnormalised output rows for the cross-warp merge.
    // The ring is reused as scratch: wait until every warp has finished reading it.
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
    float *scratch = reinterpret_cast<float *>(&sm.stage[0][0]) + warp * 16 * D;
#pragma unroll
    for (int dt = 0; dt < D / 8; ++dt) {
      const int col = dt * 8 + cpair;
      scratch[r0 * D + col] = acc[dt][0];
      scratch[r0 * D + col + 1] = acc[dt][1];
      if (kHiRows) {
        scratch[(r0 + 8) * D + col] = acc[dt][2];
        scratch[(r0 + 8) * D + col + 1] = acc[dt][3];
      }
    }
  }
  __syncthreads();
  if (sm.abort) return;

  // ---- merge the four warp states exactly and write this chunk's partial
  //      (m in natural-log units of the scaled scores, l, o~)
  const float *scratch = reinterpret_cast<const float *>(&sm.stage[0][0]);
  for (int idx = threadIdx.x; idx < g * D; idx += kThreads) {
    const int r = idx / D;
    const int e = idx % D;
    float m = -INFINITY;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) m = fmaxf(m, sm.warp_m[w][r]);
    float l = 0.f, o = 0.f;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) {
      const float mw = sm.warp_m[w][r];
      if (mw == -INFINITY) continue;  // a warp that saw no page contributes nothing
      const float c = ex2_approx(mw - m);
      l += c * sm.warp_l[w][r];
      o += c * scratch[(w * 16 + r) * D + e];
    }
    const size_t slot = (static_cast<size_t>(b) * H + kvh * g + r) * S + split;
    ws_o[slot * D + e] = o;
    if (e == 0) {
      ws_m[slot] = m * kLn2;
      ws_l[slot] = l;
    }
  }
}

// One warp per (sequence, head): m = max m_s, l = sum exp(m_s - m) l_s,
// o~ = sum exp(m_s - m) o~_s, O = o~ / l, LSE = m + ln l.
// The partial count is num_parts[b], S when num_parts is null, or -- for the
// decode path -- derived from kv_lens as ceil(ceil(L / page) / chunk).
// An optional extra partial per (sequence, head) comes as a normalised output
// with its log-sum-exp: (m, l, o~) = (LSE, 1, O) -- e.g. the shared-prefix
// part of cascade attention.
template <int D, typename OutT>
__global__ void __launch_bounds__(256)
    merge_kernel(const float *__restrict__ m_in, const float *__restrict__ l_in, const float *__restrict__ o_in,
                 const int32_t *__restrict__ num_parts, const int32_t *__restrict__ kv_lens, int page_size,
                 int chunk_pages, int B, int H, int S, OutT *__restrict__ o_out, float *__restrict__ lse_out,
                 const __nv_bfloat16 *__restrict__ extra_o, const float *__restrict__ extra_lse) {
  constexpr int E = D / 32;  // elements per lane
  // Launched as a programmatic dependent of the split kernel in the decode path:
  // wait here until that grid has finished and its partials are visible (a no-op
  // for an ordinary launch).
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int warp_global = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (warp_global >= B * H) return;
  const int b = warp_global / H;
  int n = S;
  if (kv_lens != nullptr) {
    const int pages = (kv_lens[b] + page_size - 1) / page_size;
    n = (pages + chunk_pages - 1) / chunk_pages;
  } else if (num_parts != nullptr) {
    n = num_parts[b];
  }
  n = max(0, min(n, S));
  const size_t base = static_cast<size_t>(warp_global) * S;

  float m = -INFINITY;
  for (int s = lane; s < n; s += 32) m = fmaxf(m, m_in[base + s]);
  const float m_extra = extra_lse != nullptr ? extra_lse[warp_global] : -INFINITY;
  m = fmaxf(m, m_extra);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));

  float l = 0.f;
  float o[E];
#pragma unroll
  for (int j = 0; j < E; ++j) o[j] = 0.f;
  if (m != -INFINITY) {
    // four partials per step: their loads are independent and overlap
    for (int s0 = 0; s0 < n; s0 += 4) {
      float w[4], lv[4], ov[4][E];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int s = s0 + u;
        const bool in = s < n;
        const float ms = in ? m_in[base + s] : -INFINITY;
        lv[u] = in ? l_in[base + s] : 0.f;
        const float *src = o_in + (base + (in ? s : 0)) * D + lane * E;
        if constexpr (E == 4) {
          const float4 v = *reinterpret_cast<const float4 *>(src);
          ov[u][0] = v.x;
          ov[u][1] = v.y;
          ov[u][2] = v.z;
          ov[u][3] = v.w;
        } else {
          const float2 v = *reinterpret_cast<const float2 *>(src);
          ov[u][0] = v.x;
          ov[u][1] = v.y;
        }
        w[u] = (ms == -INFINITY) ? 0.f : expf(ms - m);  // an empty partial weighs nothing
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        l += w[u] * lv[u];
#pragma unroll
        for (int j = 0; j < E; ++j) o[j] += w[u] * ov[u][j];
      }
    }
  }
  if (m != -INFINITY && m_extra != -INFINITY) {
    const float w = expf(m_extra - m);
    l += w;
    const __nv_bfloat16 *src = extra_o + static_cast<size_t>(warp_global) * D + lane * E;
#pragma unroll
    for (int j = 0; j < E; ++j) o[j] += w * __bfloat162float(src[j]);
  }
  const float inv = (l > 0.f) ? 1.f / l : 0.f;
  OutT *dst = o_out + static_cast<size_t>(warp_global) * D + lane * E;
#pragma unroll
  for (int j = 0; j < E; ++j) {
    if constexpr (sizeof(OutT) == 2) {
      dst[j] = __float2bfloat16_rn(o[j] * inv);
    } else {
      dst[j] = o[j] * inv;
    }
  }
  if (lse_out != nullptr && lane == 0) lse_out[warp_global] = (l > 0.f) ? m + logf(l) : -INFINITY;
}

}  // namespace

size_t decode_smem_bytes(int d) { return (d == 64 ? sizeof(DecodeSmem<64>) : sizeof(DecodeSmem<128>)) + 1024; }

ATTN_DEFINE_ERROR_ACCESSOR(device_error_decode)

namespace {
template <int D, bool kHiRows>
cudaError_t launch_split_d(const CUtensorMap &tm_k, const CUtensorMap &tm_v, const void *q,
                           const int32_t *page_table, const int32_t *kv_lens, float *ws_m, float *ws_l, float *ws_o,
                           int B, int H, int Hkv, int max_pages, int num_pages, int chunk_pages, int S, float scale,
                           cudaStream_t stream) {
  const size_t smem = sizeof(DecodeSmem<D>) + 1024;
  auto kern = decode_split_kernel<D, kHiRows>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  kern<<<dim3(Hkv, B, S), kThreads, smem, stream>>>(tm_k, tm_v, static_cast<const __nv_bfloat16 *>(q), page_table,
                                                    kv_lens, ws_m, ws_l, ws_o, H, Hkv, max_pages, num_pages,
                                                    chunk_pages, S, scale * kLog2e);
  return cudaGetLastError();
}
}  // namespace

cudaError_t launch_decode_split(const CUtensorMap &tm_k, const CUtensorMap &tm_v, const void *q,
                                const int32_t *page_table, const int32_t *kv_lens, float *ws_m, float *ws_l,
                                float *ws_o, int B, int H, int Hkv, int d, int max_pages, int num_pages,
                                int chunk_pages, int S, float scale, cudaStream_t stream) {
  const bool hi = H / Hkv > 8;
#define ATTN_SPLIT(DD, HI)                                                                                     \
  launch_split_d<DD, HI>(tm_k, tm_v, q, page_table, kv_lens, ws_m, ws_l, ws_o, B, H, Hkv, max_pages, num_pages, \
                         chunk_pages, S, scale, stream)
  if (d == 64) return hi ? ATTN_SPLIT(64, true) : ATTN_SPLIT(64, false);
  return hi ? ATTN_SPLIT(128, true) : ATTN_SPLIT(128, false);
#undef ATTN_SPLIT
}

cudaError_t launch_merge(const float *m, const float *l, const float *o_tilde, const int32_t *num_parts,
                         const int32_t *kv_lens, int page_size, int chunk_pages, int B, int H, int S, int d, void *o,
                         bool out_bf16, float *lse, const void *extra_o, const float *extra_lse,
                         cudaStream_t stream, bool after_split) {
  const int warps = B * H;
  const int threads = 256;
  const int blocks = (warps * 32 + threads - 1) / threads;
  if (blocks == 0) return cudaSuccess;
  // Right after the split kernel the merge is launched as its programmatic
  // dependent, so that its launch overlaps the split kernel's last CTAs.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(blocks);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = after_split ? 1 : 0;
#define ATTN_MERGE_LAUNCH(DD, T)                                                                              \
  cudaLaunchKernelEx(&cfg, merge_kernel<DD, T>, m, l, o_tilde, num_parts, kv_lens, page_size, chunk_pages, B, H, \
                     S, static_cast<T *>(o), lse, static_cast<const __nv_bfloat16 *>(extra_o), extra_lse)
  cudaError_t e;
  if (d == 128)
    e = out_bf16 ? ATTN_MERGE_LAUNCH(128, __nv_bfloat16) : ATTN_MERGE_LAUNCH(128, float);
  else
    e = out_bf16 ? ATTN_MERGE_LAUNCH(64, __nv_bfloat16) : ATTN_MERGE_LAUNCH(64, float);
#undef ATTN_MERGE_LAUNCH
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace attn
