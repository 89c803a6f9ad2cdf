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
// (batch, head), 384 threads, one CTA per SM.  Each tile is a chain
//     S_c(j) = Q_c K_j^T -> softmax_c(j) -> P_c(j) -> O_c += P_c(j) V_j
// over Nq query rows and Nk keys; with causal masking query row i attends
// keys j <= i + (Nk - Nq), i.e. the mask is aligned to the last key (for
// self-attention, Nq = Nk, this is j <= i).  Because P lives in shared
// memory rather than over S, S_c(j+1) can be computed as soon as softmax has
// loaded S_c(j) into registers: the tensor core works on the next score tile
// (and on the other chain) while the exponentials of this one are evaluated
// (the FlashAttention-3 overlap, here with tcgen05, tensor memory and TMA).
//   warp 0      TMA: Q_A, Q_B once, then K_j into a 2-stage ring
//   warp 2      TMA: V_j into a single stage (it is needed only after softmax;
//               V_{j+1} is prefetched into L2 meanwhile)
//   warps 1, 3  one MMA warp per chain (warp 1 also allocates tensor memory):
//               an elected lane of the converged warp issues its chain's MMAs
//               in the order S_c(0), S_c(1), P_c(0) V_0, S_c(2), P_c(1) V_1, ...
//                 S_c = Q_c K_j^T  (SS; Q, K K-major in SMEM; D in TMEM)
//                 O_c += P_c V_j   (SS; P K-major, V MN-major in SMEM; D in TMEM;
//                                   TS at d = 64: P in TMEM)
//               after bounded blocking waits on mbarriers; completion is tracked
//               by tcgen05.commit.  Issuing a group of MMAs blocks while the
//               tensor pipe holds earlier groups, so a separate issuer per
//               chain keeps one chain's issue from holding up the other's.
//   warps 4-7   softmax warpgroup of tile A, warps 8-11 of tile B; one thread
//               per query row (= TMEM lane): load S, release it, mask, row
//               max, p = 2^(s' - m), row sum, write P = bf16(p) (round to
//               nearest even) to shared memory in the 128-byte-swizzled
//               K-major layout (to tensor memory at d = 64), rescale O in
//               TMEM lazily (the reference
//               maximum moves only when the row max outgrows it by more than
//               2^8; the result does not depend on the reference, and p stays
//               <= 256), and at the end write O = o~ / l and the LSE.
//               At d = 128 the two warpgroups take turns for the exponentials (an
//               mbarrier token: A's of tile j after B's of tile j-1, B's of tile j
//               after A's of tile j, passed on once the ex2 instructions are
//               issued), so that one chain's exponentials run while the other packs
//               and stores P and loads its next S, instead of both competing for the
//               same sub-partitions' quarter-rate pipe at once.  At d = 64, with half
//               the tensor work per exponential, they run without turns.
// Tensor memory, 512 columns: S_A [0,128), S_B [128,256), O_A [256,256+d),
// O_B [384,384+d).  At d = 64 the columns after each O hold that chain's P
// (128 keys as 64 columns of packed bf16 pairs, written with tcgen05.st), and
// P V is the TS form (A from tensor memory): no P round trip through shared
// memory and no async-proxy fence on the softmax's path.  At d = 128 there is
// no room beside O, and P goes through shared memory.
// Query-tile pairs are ordered heaviest causal pair first.
// One kernel instance per sequence layout: dense [B, heads, N, d] blocks,
// ragged token-major tensors with indptr offsets, ragged queries against
// a paged K/V cache (each 128-key tile gathered as eight 16-token pages), or
// one shared key set split into chunks, each chunk a partial for a later merge
// (the shared prefix of cascade decode).
#include <algorithm>

#include "common.cuh"
#include "tc05.cuh"
#include "kernels.h"

namespace attn {
namespace {

constexpr int BM = 128;      // query rows per tile (= TMEM lanes)
constexpr int BN = 128;      // keys per K/V tile
constexpr int kKStages = 2;
constexpr int kThreads = 384;
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr int kBoxBytes = BN * 64 * 2;     // one 128-row x 64-column bf16 TMA box: 16 KiB

template <int D>
struct PrefillSmem {
  static constexpr int kTileBytes = BN * D * 2;
  alignas(1024) uint8_t q[2][BM * D * 2];
  alignas(1024) uint8_t k[kKStages][kTileBytes];
  alignas(1024) uint8_t v[kTileBytes];
  // P_A, P_B: 128 rows x 128 keys bf16, two 64-key swizzled boxes (at d = 64 P lives in
  // tensor memory and these are placeholders)
  alignas(1024) uint8_t p[2][D == 64 ? 1024 : BM * BN * 2];
  uint64_t q_full, q_empty;  // q_empty: both chains' S products of an item are done (persistent form)
  uint64_t k_full[kKStages], k_empty[2][kKStages];  // empty: per chain, committed by its MMA warp
  uint64_t v_full, v_empty[2];
  uint64_t v_tail;   // paged layout: the last V tile with its tail slots zeroed
  uint64_t s_full[2], s_free[2], p_full[2], pv_done[2];
  uint64_t turn[2];  // turn[c]: the other chain's softmax has finished its exponentials
  uint64_t mma_done[2];
  uint32_t tmem_base;
  int abort;
  // one item per CTA at d = 128: the first 64-key box of P_c is in shared memory
  alignas(8) uint64_t p_half[2];
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

// maximum of the 128 values of a score row (sr[q4][e] = column 32 q4 + e, fp32 bits) by a
// balanced tree of 3-input maxima: 43, 15, 5, 2 and 1 at the five levels
__device__ __forceinline__ float row_max128(const uint32_t (&sr)[4][32]) {
  float l1[43];
#pragma unroll
  for (int i = 0; i < 42; ++i) {
    const int a = 3 * i;
    l1[i] = max3(__uint_as_float(sr[a >> 5][a & 31]), __uint_as_float(sr[(a + 1) >> 5][(a + 1) & 31]),
                 __uint_as_float(sr[(a + 2) >> 5][(a + 2) & 31]));
  }
  l1[42] = fmaxf(__uint_as_float(sr[3][30]), __uint_as_float(sr[3][31]));
  float l2[15];
#pragma unroll
  for (int i = 0; i < 14; ++i) l2[i] = max3(l1[3 * i], l1[3 * i + 1], l1[3 * i + 2]);
  l2[14] = l1[42];
  float l3[5];
#pragma unroll
  for (int i = 0; i < 5; ++i) l3[i] = max3(l2[3 * i], l2[3 * i + 1], l2[3 * i + 2]);
  return fmaxf(max3(l3[0], l3[1], l3[2]), fmaxf(l3[3], l3[4]));
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

// Generic-proxy shared-memory writes made visible to the tensor core (async proxy).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
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

// Where each sequence's rows live: one dense block per (batch, head), ragged
// (indptr offsets into token-major q/k/v), or ragged queries against a paged cache.
enum { kDense = 0, kRagged = 1, kPaged = 2, kKeyChunks = 3 };

// One work item: a pair of 128-row query tiles of one (batch, head) and the keys they attend.
struct PrefillItem {
  int t, b, h, kvh;        // pair index, batch (sequence), query head, KV head
  int Nq, Nk, q_base, k_base, q_plane, kv_plane, shift;
  int row0[2], n_tiles[2], n_kv;
  bool has_b, v_tail_fix, valid;
};

template <int D, int kLay, bool kPersistent>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_bf16_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v, const PrefillOut out, const PrefillLayout lay,
                        int B, int H, int Hkv, int Nq_max, int Nk_dense, int causal, float scale_log2,
                        int q_rows_outer, int resident_ctas, int n_items, int plane_group) {
  constexpr bool kRaggedQ = kLay != kDense;  // query rows are the outer dimension (q_plane = head)
  constexpr bool kIndptrQ = kLay == kRagged || kLay == kPaged;  // query offsets from qo_indptr
  constexpr bool kChunkK = kLay == kKeyChunks;  // batch b: keys [b * key_chunk, ...) of one shared set
  constexpr bool kRaggedK = kLay == kRagged;  // key offsets from kv_indptr (rows-outer K/V maps)
  constexpr bool kPagedK = kLay == kPaged;    // keys gathered page by page
  constexpr bool kPInTmem = D == 64;          // P_c kept in tensor memory for a TS-form P V
  // P_c through shared memory in two 64-key boxes, each with its own ready barrier, so that
  // P V starts on the first box while the second is stored (one item per CTA only)
  constexpr bool kSplitP = !kPInTmem && !kPersistent;
  // Persistent form (dense layout, chosen by the host for many short items): each CTA takes
  // items blockIdx.x, 2G-1-blockIdx.x, 2G+blockIdx.x, ... (G CTAs, a snake over the
  // heaviest-first item order), so that one item's Q and first tiles load and its first
  // scores are computed while the previous item finishes.  Otherwise one item per CTA.
  static_assert(!kPersistent || kLay == kDense, "the persistent form is for the dense layout");
  // The two softmax warpgroups take turns for their exponentials at d = 128; at d = 64 they
  // run them concurrently (measured: +2 % with turns at d = 128, +7 % without them at d = 64).
  constexpr bool kPingPong = D == 128;
  using Smem = PrefillSmem<D>;
  extern __shared__ uint8_t smem_raw[];
  Smem &sm = *reinterpret_cast<Smem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n_pairs = (Nq_max + 2 * BM - 1) / (2 * BM);
  const int bh_count = B * H;

  // the k-th item of this CTA, or -1 past the last
  auto item_index = [&](int k) {
    if (!kPersistent) return k == 0 ? static_cast<int>(blockIdx.x) : -1;
    const int G = gridDim.x;
    const int idx = k * G + ((k & 1) ? G - 1 - static_cast<int>(blockIdx.x) : static_cast<int>(blockIdx.x));
    return idx < n_items ? idx : -1;
  };
  // Item idx: pair t of (batch, head) bh, heaviest causal pairs first, over all planes or,
  // one item per CTA with plane_group > 0, over groups of that many consecutive planes in
  // turn (so that the CTAs running at once read the K and V of one group, which fits in L2;
  // the persistent instance does without the mapping: its code then runs 3-10 % faster).
  // A sequence whose
  // offsets leave [0, total) or exceed the host's max_q_len is not computed (its rows stay
  // unwritten) and sets BAD_LENGTH.  Every thread computes the same values.
  auto make_item = [&](int idx, bool record) {
    PrefillItem it;
    if (idx < 0) {  // past the CTA's last item
      it.t = it.b = it.h = it.kvh = it.Nq = it.Nk = it.q_base = it.k_base = it.q_plane = it.kv_plane = it.shift = 0;
      it.row0[0] = it.row0[1] = it.n_tiles[0] = it.n_tiles[1] = it.n_kv = 0;
      it.has_b = it.v_tail_fix = it.valid = false;
      return it;
    }
    int rank, bh;
    if (!kPersistent && plane_group > 0 && plane_group < bh_count) {  // one item per CTA only
      const int per_group = plane_group * n_pairs;
      const int g = idx / per_group, r = idx - g * per_group;
      const int in_group = min(plane_group, bh_count - g * plane_group);  // the last group may be smaller
      rank = r / in_group;
      bh = g * plane_group + r % in_group;
    } else {
      rank = idx / bh_count;
      bh = idx % bh_count;
    }
    it.t = causal ? (n_pairs - 1 - rank) : rank;
    it.b = bh / H;
    it.h = bh % H;
    it.kvh = it.h / (H / Hkv);
    it.Nq = Nq_max;
    it.Nk = Nk_dense;
    it.q_base = 0;
    it.k_base = 0;
    bool bad = false;
    if (kIndptrQ) {
      it.q_base = lay.qo_indptr[it.b];
      it.Nq = lay.qo_indptr[it.b + 1] - it.q_base;
      bad |= it.q_base < 0 || it.Nq < 0 || it.Nq > Nq_max || static_cast<long long>(it.q_base) + it.Nq > lay.total_q;
    }
    if (kRaggedK) {
      it.k_base = lay.kv_indptr[it.b];
      it.Nk = lay.kv_indptr[it.b + 1] - it.k_base;
      bad |= it.k_base < 0 || it.Nk < 0 || static_cast<long long>(it.k_base) + it.Nk > lay.total_k;
    }
    if (bad && record && it.t == 0) record_device_error(ATTN_DEVERR_BAD_LENGTH);
    if (kChunkK) {
      it.k_base = it.b * lay.key_chunk;
      it.Nk = max(0, min(lay.key_chunk, Nk_dense - it.k_base));
    }
    if (kPagedK) {
      const int L = lay.kv_lens[it.b];
      if (L < 0 || L > lay.max_pages * 16) {  // beyond the table: clamped, as in paged decode
        if (record && it.t == 0) record_device_error(ATTN_DEVERR_BAD_PAGE);
      }
      it.Nk = max(0, min(L, lay.max_pages * 16));
    }
    it.valid = !bad && 2 * it.t * BM < it.Nq;  // else the pair lies past the sequence's queries
    it.q_plane = kRaggedQ ? it.h : it.b * H + it.h;
    it.kv_plane = (kRaggedK || kChunkK) ? it.kvh : it.b * Hkv + it.kvh;
    it.row0[0] = 2 * it.t * BM;
    it.row0[1] = (2 * it.t + 1) * BM;
    it.has_b = it.row0[1] < it.Nq;
    it.shift = it.Nk - it.Nq;
    const int n_kt_all = (it.Nk + BN - 1) / BN;
    // key tiles each chain visits: causal, up to the tile of its last row's last key
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      int n = n_kt_all;
      if (causal) {
        const int last_key = min(it.row0[c] + BM, it.Nq) - 1 + it.shift;
        n = last_key < 0 ? 0 : min(n_kt_all, last_key / BN + 1);
      }
      it.n_tiles[c] = (c == 0 || it.has_b) ? n : 0;
    }
    if (!it.valid) it.n_tiles[0] = it.n_tiles[1] = 0;
    it.n_kv = max(it.n_tiles[0], it.n_tiles[1]);
    // paged layout: keys [Nk, Nk rounded up to a page) of the last tile are the unused slots
    // of the sequence's last page, which may hold anything; their V rows are zeroed before
    // P V reads them (their weights are exact zeros, but 0 x NaN is NaN in the MMA).  Later
    // pages of the tile read as zeros already (page id -1 lies outside the pool).
    it.v_tail_fix = kPagedK && (it.Nk % 16) != 0 && it.n_kv > 0 && (it.n_kv - 1) * BN < it.Nk;
    return it;
  };

  // the first item; a one-item CTA whose item is empty or invalid leaves at once
  const PrefillItem first = make_item(item_index(0), threadIdx.x == 0);
  if (!kPersistent && !first.valid) return;

  // Key tile j of item `it` into shared memory: one box per 64 columns, or, paged, eight
  // 16-token pages per 64 columns (a page id past the sequence or outside the pool reads as
  // zeros: TMA fills out-of-range boxes).
  auto load_kv_tile = [&](const PrefillItem &it, uint32_t dst, const CUtensorMap *map, uint32_t bar, int j,
                          uint64_t policy, const int (&pages)[8]) {
#pragma unroll
    for (int x = 0; x < D / 64; ++x) {
      if (!kPagedK) {
        if (kRaggedK)
          tma_load_3d_hint(dst + x * kBoxBytes, map, bar, x * 64, it.kv_plane, it.k_base + j * BN, policy);
        else
          tma_load_3d_hint(dst + x * kBoxBytes, map, bar, x * 64, it.k_base + j * BN, it.kv_plane, policy);
      } else {
#pragma unroll
        for (int pg = 0; pg < 8; ++pg)
          tma_load_3d_hint(dst + x * kBoxBytes + pg * 16 * 128, map, bar, x * 64, 0, pages[pg] * Hkv + it.kvh,
                           policy);
      }
    }
  };
  // page ids of key tile j (paged layout; -1 past the sequence's pages)
  auto tile_pages = [&](const PrefillItem &it, int j, int (&pages)[8]) {
    const int pages_b = (it.Nk + 15) / 16;
#pragma unroll
    for (int pg = 0; pg < 8; ++pg) {
      const int i = j * 8 + pg;
      int id = -1;
      if (kPagedK && i < pages_b) {
        id = lay.page_table[static_cast<size_t>(it.b) * lay.max_pages + i];
        if (id < 0 || id >= lay.num_pages) {
          record_device_error(ATTN_DEVERR_BAD_PAGE);
          id = -1;
        }
      }
      pages[pg] = id;
    }
  };
  auto load_q = [&](const PrefillItem &it, uint64_t policy) {
    const uint32_t qbar = smem_u32(&sm.q_full);
    mbar_arrive_expect_tx(qbar, (it.has_b ? 2 : 1) * BM * D * 2);
#pragma unroll
    for (int c = 0; c < 2; ++c)
      if (c == 0 || it.has_b)
#pragma unroll
      for (int x = 0; x < D / 64; ++x)
        // Q map dimensions: (d, rows, planes), or (d, planes, rows) when the query rows are the outer dimension
        tma_load_3d_hint(smem_u32(sm.q[c]) + x * kBoxBytes, &tm_q, qbar, x * 64,
                         q_rows_outer ? it.q_plane : it.q_base + it.row0[c],
                         q_rows_outer ? it.q_base + it.row0[c] : it.q_plane, policy);
  };

  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&sm.q_full), 1);
    mbar_init(smem_u32(&sm.q_empty), 2);
    for (int s = 0; s < kKStages; ++s) {
      mbar_init(smem_u32(&sm.k_full[s]), 1);
      mbar_init(smem_u32(&sm.k_empty[0][s]), 1);
      mbar_init(smem_u32(&sm.k_empty[1][s]), 1);
    }
    mbar_init(smem_u32(&sm.v_full), 1);
    mbar_init(smem_u32(&sm.v_tail), 1);
    mbar_init(smem_u32(&sm.v_empty[0]), 1);
    mbar_init(smem_u32(&sm.v_empty[1]), 1);
    for (int c = 0; c < 2; ++c) {
      mbar_init(smem_u32(&sm.s_full[c]), 1);
      mbar_init(smem_u32(&sm.s_free[c]), 128);
      mbar_init(smem_u32(&sm.p_full[c]), 128);
      if (kSplitP) mbar_init(smem_u32(&sm.p_half[c]), 128);
      mbar_init(smem_u32(&sm.pv_done[c]), 1);
      mbar_init(smem_u32(&sm.turn[c]), 128);
    }
    mbar_init(smem_u32(&sm.mma_done[0]), 1);
    mbar_init(smem_u32(&sm.mma_done[1]), 1);
    sm.abort = 0;
    fence_barrier_init();
    // the first item's Q, first K tile and first V tile at once, while tensor memory is
    // allocated and the warps take their roles (the TMA warps' loops continue from there)
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    if (first.valid) {
      const uint64_t keep = l2_policy_evict_last();
      load_q(first, l2_policy_evict_first());
      if (first.n_kv > 0) {
        int pages[8];
        tile_pages(first, 0, pages);
        mbar_arrive_expect_tx(smem_u32(&sm.k_full[0]), Smem::kTileBytes);
        load_kv_tile(first, smem_u32(sm.k[0]), &tm_k, smem_u32(&sm.k_full[0]), 0, keep, pages);
        mbar_arrive_expect_tx(smem_u32(&sm.v_full), Smem::kTileBytes);
        load_kv_tile(first, smem_u32(sm.v), &tm_v, smem_u32(&sm.v_full), 0, keep, pages);
      }
    }
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
  // 64,512.  Warpgroup 0 (two TMA warps, two MMA warps) gives up to
  // 56 per thread and the two softmax warpgroups take 224:
  // 128 x 56 + 256 x 224 = 64,512, exactly the launch's allocation.  The persistent form's
  // item bookkeeping needs more in warpgroup 0: 128 x 72 + 256 x 216 = 64,512.
  //
  // Barrier phases run on across items: every role counts the uses of each barrier it
  // waits on (K tiles, V tiles, S and P V products of its chain, items), and no barrier
  // can be more than one phase ahead of a waiter.
  if (warp < 4) {
    if (kPersistent)
      asm volatile("setmaxnreg.dec.sync.aligned.u32 72;" ::: "memory");
    else
      asm volatile("setmaxnreg.dec.sync.aligned.u32 56;" ::: "memory");
  }
  if (warp == 0) {
    // ================================================================ TMA: Q and K
    if (lane == 0) {
      const uint64_t keep = l2_policy_evict_last();    // K tiles are re-read by other query tiles
      const uint64_t once = l2_policy_evict_first();   // each Q tile is read once
      // K stage s: which chains read the tile last placed there and have not yet released it,
      // and how many releases each chain has committed on it in all
      bool in_use[kKStages][2] = {};
      int releases[kKStages][2] = {};
      int g = 0;        // K tiles issued by this CTA
      int q_loads = first.valid ? 1 : 0;  // Q loads issued (the first with the barrier set-up)
      bool ok = true;
      int k = 0;
      for (PrefillItem it = first; ok && it.valid; it = make_item(item_index(++k), false)) {
        // the item after this one needs its Q tiles next: bring them into L2 now (dense
        // layout; a one-item CTA prefetches for the CTA that will probably run next on this SM)
        {
          const int nb = kPersistent ? item_index(k + 1) : static_cast<int>(blockIdx.x) + resident_ctas;
          if (!kRaggedQ && nb >= 0 && nb < (kPersistent ? n_items : static_cast<int>(gridDim.x))) {
            const PrefillItem nx = make_item(nb, false);
#pragma unroll
            for (int c = 0; c < 2; ++c)
              if (nx.row0[c] < nx.Nq)
#pragma unroll
                for (int x = 0; x < D / 64; ++x) tma_prefetch_l2(&tm_q, x * 64, nx.row0[c], nx.q_plane);
          }
        }
        if (k > 0) {
          // Q of the previous item must no longer be read by either chain's S products
          if (!(ok = mbar_wait(smem_u32(&sm.q_empty), (k - 1) & 1, &sm.abort))) break;
          load_q(it, once);
          ++q_loads;
        }
        for (int j = 0; j < it.n_kv; ++j, ++g) {
          const int ks = g % kKStages;
          const bool issued_early = k == 0 && j == 0;  // issued with the barrier set-up
          if (!issued_early) {
            int pages[8];
            tile_pages(it, j, pages);  // before the wait: the ids do not depend on the stage
            // the stage's previous tile must have been read by each chain that used it
#pragma unroll
            for (int c = 0; c < 2; ++c)
              if (ok && in_use[ks][c]) ok = mbar_wait(smem_u32(&sm.k_empty[c][ks]), (releases[ks][c] - 1) & 1, &sm.abort);
            if (!ok) break;
            const uint32_t kbar = smem_u32(&sm.k_full[ks]);
            mbar_arrive_expect_tx(kbar, Smem::kTileBytes);
            load_kv_tile(it, smem_u32(sm.k[ks]), &tm_k, kbar, j, keep, pages);
          }
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            in_use[ks][c] = j < it.n_tiles[c];
            releases[ks][c] += in_use[ks][c] ? 1 : 0;
          }
        }
      }
      // drain: every issued copy must land before the CTA's shared memory is released
      if (q_loads > 0) mbar_wait(smem_u32(&sm.q_full), (q_loads - 1) & 1, nullptr);
      for (int s = 0; s < kKStages && s < g; ++s) {
        const int last = s + ((g - 1 - s) / kKStages) * kKStages;
        mbar_wait(smem_u32(&sm.k_full[s]), (last / kKStages) & 1, nullptr);
      }
    }
    __syncwarp();
  } else if (warp == 2) {
    // ================================================================ TMA: V (single stage)
    if (lane == 0) {
      const uint64_t keep = l2_policy_evict_last();
      const uint32_t vbar = smem_u32(&sm.v_full);
      bool in_use[2] = {false, false};  // chains that read the tile in the stage and have not released it
      int releases[2] = {0, 0};
      int g = 0;  // V tiles issued by this CTA
      bool ok = true;
      int k = 0;
      for (PrefillItem it = first; ok && it.valid; it = make_item(item_index(++k), false)) {
        // V has one stage, so each tile's copy waits for the previous tile's P V: bring the
        // next tile into L2 meanwhile (dense and ragged layouts; for the paged layout the
        // extra page-id loads and per-page prefetches cost more than they save)
        auto prefetch_l2 = [&](int j) {
          if (!kPagedK && j < it.n_kv) {
#pragma unroll
            for (int x = 0; x < D / 64; ++x) {
              if (kRaggedK)
                tma_prefetch_l2(&tm_v, x * 64, it.kv_plane, it.k_base + j * BN);
              else
                tma_prefetch_l2(&tm_v, x * 64, it.k_base + j * BN, it.kv_plane);
            }
          }
        };
        for (int j = 0; j < it.n_kv; ++j, ++g) {
          const bool issued_early = k == 0 && j == 0;  // issued with the barrier set-up
          if (!issued_early) {
            int pages[8];
            tile_pages(it, j, pages);  // before the wait: the ids do not depend on the stage
#pragma unroll
            for (int c = 0; c < 2; ++c)
              if (ok && in_use[c]) ok = mbar_wait(smem_u32(&sm.v_empty[c]), (releases[c] - 1) & 1, &sm.abort);
            if (!ok) break;
            mbar_arrive_expect_tx(vbar, Smem::kTileBytes);
            load_kv_tile(it, smem_u32(sm.v), &tm_v, vbar, j, keep, pages);
          }
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            in_use[c] = j < it.n_tiles[c];
            releases[c] += in_use[c] ? 1 : 0;
          }
          if (it.v_tail_fix && j == it.n_kv - 1) {
            // paged layout, last tile (one item per CTA): wait for it, zero the tail slots'
            // rows in each 64-column box, make the writes visible to the tensor core, and
            // release the tile to the MMA warps
            if (!(ok = mbar_wait(vbar, g & 1, &sm.abort))) break;
            const int r0 = it.Nk - j * BN, r1 = min(BN, ((it.Nk + 15) / 16) * 16 - j * BN);
            for (int x = 0; x < D / 64; ++x)
              for (int r = r0; r < r1; ++r)
                for (int c = 0; c < 8; ++c)
                  st_shared_v4(smem_u32(sm.v) + x * kBoxBytes + r * 128 + c * 16, 0, 0, 0, 0);
            fence_proxy_async_smem();
            mbar_arrive(smem_u32(&sm.v_tail));
          }
          prefetch_l2(j + 1);
        }
      }
      if (g > 0) mbar_wait(vbar, (g - 1) & 1, nullptr);
    }
    __syncwarp();
  } else if (warp == 1 || warp == 3) {
    // ================================================================ MMA warps, one per chain
    // Warp 1 issues chain A's MMAs and warp 3 chain B's, each in the order
    //   S_c(0), S_c(1), P_c(0) V_0, S_c(2), P_c(1) V_1, ...
    // with blocking (bounded) waits: S_c(j) once softmax has taken S_c(j-1) out of
    // tensor memory and K_j has landed, P_c(j-1) V_{j-1} once P_c(j-1) is written and
    // V_{j-1} has landed.  A warp blocked in one chain's MMA issue does not hold up
    // the other chain.
    const int c = warp == 1 ? 0 : 1;
    constexpr uint32_t idesc_qk = tc05::idesc_bf16_f32(BM, BN, false);
    constexpr uint32_t idesc_pv = tc05::idesc_bf16_f32(BM, D, true);
    const uint32_t q_addr = smem_u32(sm.q[c]);
    const uint32_t p_addr = smem_u32(sm.p[c]);
    const uint32_t v_addr = smem_u32(sm.v);
    int gk = 0;    // K (and V) tiles of the items before this one
    int ts = 0;    // S products of this chain so far
    bool ok = true;
    int k = 0;
    for (PrefillItem it = first; ok && it.valid; it = make_item(item_index(++k), false)) {
      const int n_c = c == 0 ? it.n_tiles[0] : it.n_tiles[1];
      ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&sm.q_full), k & 1, &sm.abort));
      tc05::fence_after_sync();
      for (int j = 0; ok && j <= n_c; ++j) {
        if (j < n_c) {
          const int g = gk + j, ks = g % kKStages;
          ok = __all_sync(0xffffffffu,
                          (ts + j == 0 || mbar_wait(smem_u32(&sm.s_free[c]), (ts + j - 1) & 1, &sm.abort)) &&
                              mbar_wait(smem_u32(&sm.k_full[ks]), (g / kKStages) & 1, &sm.abort));
          if (!ok) break;
          tc05::fence_after_sync();
          const uint32_t k_addr = smem_u32(sm.k[ks]);
          if (elect_one()) {
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t off = (kk >> 2) * kBoxBytes + (kk & 3) * 32;
              tc05::mma_ss(tmem + c * BN, tc05::sdesc_sw128(q_addr + off, 16, 1024),
                           tc05::sdesc_sw128(k_addr + off, 16, 1024), idesc_qk, kk > 0);
            }
            tc05::commit(smem_u32(&sm.s_full[c]));
            tc05::commit(smem_u32(&sm.k_empty[c][ks]));
            // the item's last S product: its Q tile may be replaced once this completes
            if (j == n_c - 1) tc05::commit(smem_u32(&sm.q_empty));
          }
          __syncwarp();
        }
        if (j > 0) {
          const int jp = j - 1;
          const bool tail = it.v_tail_fix && jp == it.n_kv - 1;  // the last tile, tail slots zeroed
          ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(kSplitP ? &sm.p_half[c] : &sm.p_full[c]), (ts + jp) & 1, &sm.abort) &&
                                           (tail ? mbar_wait(smem_u32(&sm.v_tail), 0, &sm.abort)
                                                 : mbar_wait(smem_u32(&sm.v_full), (gk + jp) & 1, &sm.abort)));
          if (!ok) break;
          tc05::fence_after_sync();
          if (elect_one()) {
#pragma unroll
            for (int kk = 0; kk < (kSplitP ? BN / 32 : BN / 16); ++kk) {
              if (kPInTmem)  // P_c in tensor memory beside O_c: 16 keys = 8 columns of packed bf16 pairs
                tc05::mma_ts(tmem + 2 * BN + c * BN, tmem + 2 * BN + c * BN + D + kk * 8,
                             tc05::sdesc_sw128(v_addr + kk * 2048, kBoxBytes, 1024), idesc_pv, (jp > 0) || (kk > 0));
              else
                tc05::mma_ss(tmem + 2 * BN + c * BN,
                             tc05::sdesc_sw128(p_addr + (kk >> 2) * kBoxBytes + (kk & 3) * 32, 16, 1024),
                             tc05::sdesc_sw128(v_addr + kk * 2048, kBoxBytes, 1024), idesc_pv, (jp > 0) || (kk > 0));
            }
          }
          __syncwarp();
          if (kSplitP) {  // the second 64-key box of P
            if (!(ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&sm.p_full[c]), (ts + jp) & 1, &sm.abort)))) break;
            tc05::fence_after_sync();
            if (elect_one()) {
#pragma unroll
              for (int kk = BN / 32; kk < BN / 16; ++kk)
                tc05::mma_ss(tmem + 2 * BN + c * BN,
                             tc05::sdesc_sw128(p_addr + (kk >> 2) * kBoxBytes + (kk & 3) * 32, 16, 1024),
                             tc05::sdesc_sw128(v_addr + kk * 2048, kBoxBytes, 1024), idesc_pv, true);
            }
            __syncwarp();
          }
          if (elect_one()) {
            tc05::commit(smem_u32(&sm.pv_done[c]));
            tc05::commit(smem_u32(&sm.v_empty[c]));
          }
          __syncwarp();
        }
      }
      if (ok && n_c == 0 && elect_one()) mbar_arrive(smem_u32(&sm.q_empty));  // this chain reads no Q here
      __syncwarp();
      gk += it.n_kv;
      ts += n_c;
    }
    // every MMA this warp issued must complete before tensor memory is released
    if (elect_one()) tc05::commit(smem_u32(&sm.mma_done[c]));
    __syncwarp();
    mbar_wait(smem_u32(&sm.mma_done[c]), 0, nullptr);
  } else if (warp >= 4) {
    // ================================================================ softmax warpgroups
    if (kPersistent)
      asm volatile("setmaxnreg.inc.sync.aligned.u32 216;" ::: "memory");
    else
      asm volatile("setmaxnreg.inc.sync.aligned.u32 224;" ::: "memory");
    const int c = (warp - 4) >> 2;              // 0: tile A, 1: tile B
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;        // row within the tile = TMEM lane
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t s_addr = tmem + lane_addr + c * BN;
    const uint32_t o_addr = tmem + lane_addr + 2 * BN + c * BN;
    const uint32_t p_tm = o_addr + D;  // P_c in tensor memory (d = 64: the columns after O_c are free)
    const uint32_t p_row = smem_u32(sm.p[c]) + row * 128;  // this row in each 64-key swizzled box
    const uint64_t scale2 = f2(scale_log2, scale_log2);
    int ts = 0;      // S products of this chain so far
    int t_other = 0; // exponential phases of the other chain so far (ping-pong token count)
    bool ok = true;
    int k = 0;
    for (PrefillItem it = first; ok && it.valid; it = make_item(item_index(++k), false)) {
      const int q_row = (c == 0 ? it.row0[0] : it.row0[1]) + row;
      const int n_c = c == 0 ? it.n_tiles[0] : it.n_tiles[1];
      const int n_other = c == 0 ? it.n_tiles[1] : it.n_tiles[0];
      const int lim = causal ? min(q_row + it.shift + 1, it.Nk) : it.Nk;  // keys [0, lim) are attended by this row
      float m_ref = -INFINITY;  // reference maximum (log2 units) that p and o~ are relative to
      float l = 0.f;
      for (int j = 0; j < n_c; ++j) {
        // wait outcomes are made warp-uniform: tcgen05.ld/st are warp-collective
        if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&sm.s_full[c]), (ts + j) & 1, &sm.abort))) {
          ok = false;
          break;
        }
        tc05::fence_after_sync();
        uint32_t sr[4][32];
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) tc05::tmem_ld_x32(s_addr + q4 * 32, sr[q4]);
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) tc05::tmem_ld_wait(sr[q4]);
        // S_c is in registers: its MMA warp may compute S_c(j+1) into it now
        tc05::fence_before_sync();
        mbar_arrive(smem_u32(&sm.s_free[c]));

        const int kv0 = j * BN;
        if (kv0 + BN > lim) {  // diagonal tile or ragged tail: mask keys >= lim
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4)
#pragma unroll
            for (int e = 0; e < 32; ++e)
              if (kv0 + q4 * 32 + e >= lim) sr[q4][e] = __float_as_uint(-INFINITY);
        }
        // row max.  Persistent form (causal d = 128): a balanced tree, +1.2 % at N = 8192 causal,
        // -1 % with Q x30/x40; one-item form: the chains (the tree there: +3 % at N = 16384, but
        // -6 to -10 % with Q x40 and -3 to -7 % at d = 64)
        float m_row;
        if (kPersistent) {
          m_row = row_max128(sr);
        } else {
          // row max: four independent 3-input max chains
          float mq[4];
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            float m = __uint_as_float(sr[q4][0]);
#pragma unroll
            for (int e = 1; e < 31; e += 2) m = max3(m, __uint_as_float(sr[q4][e]), __uint_as_float(sr[q4][e + 1]));
            mq[q4] = fmaxf(m, __uint_as_float(sr[q4][31]));
          }
          m_row = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3]));
        }
        const float m_new = m_row * scale_log2;
        // move the reference only when the row maximum outgrows it by more than 2^8
        const bool move = m_new > m_ref + kRescaleThreshold;
        const float m_next = move ? m_new : m_ref;
        // 1 when kept (also while the row has met no key at all); 0 on the row's first key
        const float corr = (m_next == m_ref) ? 1.f : ex2_approx(m_ref - m_next);
        m_ref = m_next;
        // ping-pong (d = 128): chain A's exponentials of tile j follow chain B's of tile j-1,
        // and chain B's of tile j follow chain A's of tile j.  Counted over all items: A's first
        // tile of an item follows B's last tile of the items before, so that neither chain can
        // run two token phases ahead of the other at an item boundary, where the chains' tile
        // counts differ (by at most one).
        if (kPingPong) {
          const int need = c == 0 ? j - 1 : j;  // the other chain's step to wait for (this item)
          if (t_other + need >= 0 && need < n_other &&
              !__all_sync(0xffffffffu, mbar_wait(smem_u32(&sm.turn[c]), (t_other + need) & 1, &sm.abort))) {
            ok = false;
            break;
          }
        }

        // p = 2^(s * scale * log2(e) - m_ref), in place (a row that has met no key yet has
        // every s = -inf and takes reference 0: p = 0).  The turn passes to the other chain
        // as soon as the exponentials are issued: the bf16 packs below use the same
        // quarter-rate pipe as ex2, and run while the other chain starts its exponentials.
        const float neg_m = (m_ref == -INFINITY) ? 0.f : -m_ref;
        const uint64_t negm2 = f2(neg_m, neg_m);
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            float x0, x1;
            f2_split(fma2(f2(__uint_as_float(sr[q4][e]), __uint_as_float(sr[q4][e + 1])), scale2, negm2), x0, x1);
            sr[q4][e] = __float_as_uint(ex2_approx(x0));
            sr[q4][e + 1] = __float_as_uint(ex2_approx(x1));
          }
        }
        if (kPingPong) mbar_arrive(smem_u32(&sm.turn[1 - c]));
        // the row sum in eight partial sums, and P packed to bf16 (round to nearest even)
        uint64_t acc2[4] = {0ull, 0ull, 0ull, 0ull};
        uint32_t pr[2][32];
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const float p0 = __uint_as_float(sr[q4][e]), p1 = __uint_as_float(sr[q4][e + 1]);
            acc2[(e >> 1) & 3] = add2(acc2[(e >> 1) & 3], f2(p0, p1));
            pr[q4 >> 1][(q4 & 1) * 16 + (e >> 1)] = pack_bf16x2(p0, p1);
          }
        }
        float sum_lo, sum_hi;
        f2_split(add2(add2(acc2[0], acc2[1]), add2(acc2[2], acc2[3])), sum_lo, sum_hi);
        l = l * corr + (sum_lo + sum_hi);

        // P_c(j-1) V_{j-1} must have completed: it reads the P buffer written below
        // and o~ is rescaled in place (at j = 0 the previous item's epilogue waited for it)
        if (j > 0) {
          if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&sm.pv_done[c]), (ts + j - 1) & 1, &sm.abort))) {
            ok = false;
            break;
          }
          tc05::fence_after_sync();
          if (__any_sync(0xffffffffu, move)) {
#pragma unroll
            for (int q4 = 0; q4 < D / 32; ++q4) rescale_o_chunk(o_addr + q4 * 32, corr);
          }
        }
        if (kPInTmem) {
          // P row -> tensor memory beside O_c: column 32x + k holds keys 64x + 2k, 64x + 2k + 1
          tc05::tmem_st_x32(p_tm, pr[0]);
          tc05::tmem_st_x32(p_tm + 32, pr[1]);
        } else {
          // P row -> shared memory: keys 64x + 8ch .. +7 at chunk ch of box x, chunk index XOR (row mod 8)
#pragma unroll
          for (int x = 0; x < 2; ++x) {
#pragma unroll
            for (int ch = 0; ch < 8; ++ch)
              st_shared_v4(p_row + x * kBoxBytes + (((ch ^ row) & 7) << 4), pr[x][4 * ch], pr[x][4 * ch + 1],
                           pr[x][4 * ch + 2], pr[x][4 * ch + 3]);
            if (kSplitP) {  // P V may start on the first 64 keys
              fence_proxy_async_smem();
              if (x == 0) mbar_arrive(smem_u32(&sm.p_half[c]));
            }
          }
          if (!kSplitP) fence_proxy_async_smem();
        }
        tc05::tmem_wait_st();
        tc05::fence_before_sync();
        mbar_arrive(smem_u32(&sm.p_full[c]));
      }

      // ---- epilogue: O = o~ / l, LSE = m + ln l
      if (ok && n_c > 0) {
        ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&sm.pv_done[c]), (ts + n_c - 1) & 1, &sm.abort));
        if (ok) {
          tc05::fence_after_sync();
          const float inv = (l > 0.f) ? 1.f / l : 0.f;
          const uint64_t inv2 = f2(inv, inv);
          const bool store = q_row < it.Nq;
          __nv_bfloat16 *orow = static_cast<__nv_bfloat16 *>(out.o) + it.b * out.o_b + it.h * out.o_h +
                                static_cast<long long>(it.q_base + (store ? q_row : 0)) * out.o_r;
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
            out.lse[it.b * out.l_b + it.h * out.l_h + static_cast<long long>(it.q_base + q_row) * out.l_r] =
                (l > 0.f) ? m_ref * kLn2 + logf(l) : -INFINITY;
        }
      } else if (ok && n_c == 0 && q_row < it.Nq) {
        // a tile whose rows attend no key (causal, Nq > Nk): O = 0, LSE = -inf
        uint4 *dst = reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(out.o) + it.b * out.o_b +
                                               it.h * out.o_h + static_cast<long long>(it.q_base + q_row) * out.o_r);
#pragma unroll
        for (int e = 0; e < D / 8; ++e) dst[e] = make_uint4(0u, 0u, 0u, 0u);
        if (out.lse != nullptr)
          out.lse[it.b * out.l_b + it.h * out.l_h + static_cast<long long>(it.q_base + q_row) * out.l_r] = -INFINITY;
      }
      ts += n_c;
      t_other += n_other;
    }
  }

  tc05::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc05::fence_after_sync();
    tc05::tmem_dealloc(tmem, kTmemCols);
  }
}

template <int D, int kLay, bool kPersistent>
cudaError_t launch_d(const PrefillMaps &maps, const PrefillOut &out, const PrefillLayout &lay, int B, int H, int Hkv,
                     int Nq, int Nk, bool causal, float scale, long long items, int sms, cudaStream_t stream,
                     int plane_group = 0) {
  // One CTA per SM: the kernel holds all 512 tensor-memory columns.
  const size_t smem = std::max<size_t>(sizeof(PrefillSmem<D>) + 1024, 120 * 1024);
  auto kern = prefill_bf16_kernel<D, kLay, kPersistent>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const long long blocks = kPersistent ? std::min<long long>(items, sms) : items;
  kern<<<static_cast<unsigned>(blocks), kThreads, smem, stream>>>(maps.q, maps.k, maps.v, out, lay, B, H, Hkv, Nq,
                                                                   Nk, causal ? 1 : 0, scale * kLog2e,
                                                                   maps.q_rows_outer ? 1 : 0, sms,
                                                                   static_cast<int>(items), plane_group);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_layout(const PrefillMaps &maps, const PrefillOut &out, const PrefillLayout &lay, int B, int H,
                          int Hkv, int Nq, int Nk, bool causal, float scale, cudaStream_t stream) {
  const long long n_pairs = (Nq + 2 * BM - 1) / (2 * BM);
  const long long items = n_pairs * B * H;
  if (items > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  if (lay.key_chunk > 0)
    return launch_d<D, kKeyChunks, false>(maps, out, lay, B, H, Hkv, Nq, Nk, causal, scale, items, sms, stream);
  if (lay.kv_lens != nullptr)
    return launch_d<D, kPaged, false>(maps, out, lay, B, H, Hkv, Nq, Nk, causal, scale, items, sms, stream);
  if (lay.kv_indptr != nullptr)
    return launch_d<D, kRagged, false>(maps, out, lay, B, H, Hkv, Nq, Nk, causal, scale, items, sms, stream);
  // Dense: the persistent form pays for causal d = 128 when items are many (at least four per
  // SM) and short (at most 48 key tiles on average): then the ~2.5 tiles' worth of set-up,
  // first loads and epilogue per item that it overlaps outweigh its ~1 % per tile of
  // bookkeeping.  Measured on GB300 against the one-item form (with its split P store):
  // +0.8 % at N = 8192 causal GQA (1024 items of 33 tiles on average), -0.7 % at N = 16384
  // causal (65 tiles), -3 % at N = 2048 (2.5 items per SM); non-causal N = 4096: -1 % at
  // d = 128, -3.5 % at d = 64; d = 64 N = 8192 causal: -1.5 %.
  const long long kt = (Nk + BN - 1) / BN;
  const long long avg_tiles = causal ? (kt + 1) / 2 : kt;
  if constexpr (D == 128) {
    if (causal && items >= 4LL * sms && avg_tiles <= 48)
      return launch_d<D, kDense, true>(maps, out, lay, B, H, Hkv, Nq, Nk, causal, scale, items, sms, stream);
  }
  // One item per CTA, heaviest first: the CTAs running at once take the same pairs of every
  // (batch, head) plane.  When all planes' K and V exceed half of L2, take the planes in
  // groups whose K and V fit there (whole GQA groups), so that K and V are read from DRAM
  // about once instead of once per few query-tile pairs.
  int l2 = 0;
  if (cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev) != cudaSuccess) l2 = 0;
  const long long kv_plane_bytes = static_cast<long long>(Nk) * D * 2 * 2;  // K and V of one KV head
  int plane_group = 0;
  if (l2 > 0 && kv_plane_bytes * B * Hkv > l2 / 2) {
    const long long kv_planes = std::max<long long>(1, (l2 / 2) / std::max<long long>(kv_plane_bytes, 1));
    plane_group = static_cast<int>(std::min<long long>(kv_planes * (H / Hkv), static_cast<long long>(B) * H));
  }
  return launch_d<D, kDense, false>(maps, out, lay, B, H, Hkv, Nq, Nk, causal, scale, items, sms, stream,
                                    plane_group);
}

}  // namespace

ATTN_DEFINE_ERROR_ACCESSOR(device_error_prefill_bf16)

cudaError_t launch_prefill_bf16(const PrefillMaps &maps, const PrefillOut &out, int B, int H, int Hkv, int Nq,
                                int Nk, int d, bool causal, float scale, cudaStream_t stream,
                                const PrefillLayout &layout) {
  if (d == 64) return launch_layout<64>(maps, out, layout, B, H, Hkv, Nq, Nk, causal, scale, stream);
  return launch_layout<128>(maps, out, layout, B, H, Hkv, Nq, Nk, causal, scale, stream);
}

}  // namespace attn
