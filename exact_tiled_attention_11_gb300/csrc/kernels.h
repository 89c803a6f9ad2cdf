// Internal host-side launchers, one per kernel family (not part of the C ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace attn {

// decode.cu (d = 64 or 128)
size_t decode_smem_bytes(int d);
cudaError_t launch_decode_split(const CUtensorMap &tm_k, const CUtensorMap &tm_v, const void *q,
                                const int32_t *page_table, const int32_t *kv_lens, float *ws_m, float *ws_l,
                                float *ws_o, int B, int H, int Hkv, int d, int max_pages, int num_pages,
                                int chunk_pages, int S, float scale, cudaStream_t stream);
// extra_o / extra_lse (nullable): one more partial per (sequence, head), given as a
// normalised output O [B, H, d] bf16 with its LSE [B, H], i.e. (m, l, o~) = (LSE, 1, O).
cudaError_t launch_merge(const float *m, const float *l, const float *o_tilde, const int32_t *num_parts,
                         const int32_t *kv_lens, int page_size, int chunk_pages, int B, int H, int S, int d, void *o,
                         bool out_bf16, float *lse, const void *extra_o, const float *extra_lse,
                         cudaStream_t stream, bool after_split = false);

// Where the prefill kernels write O and the LSE: element strides of the batch,
// head and query-row dimensions (d is contiguous).  The plain [B, H, Nq, d] /
// [B, H, Nq] layout is {H*Nq*d, Nq*d, d} / {H*Nq, Nq, 1}.
struct PrefillOut {
  void *o;
  float *lse;  // may be null
  long long o_b, o_h, o_r;
  long long l_b, l_h, l_r;
};

// prefill_f32.cu (q [B, H, Nq, d], k/v [B, Hkv, Nk, d])
cudaError_t launch_prefill_f32(const float *q, const float *k, const float *v, const PrefillOut &out, int B, int H,
                               int Hkv, int Nq, int Nk, int d, bool causal, float scale, cudaStream_t stream);

// prefill_bf16.cu: Q, K, V through TMA maps whose dimensions are (d, rows, B * heads);
// with q_rows_outer the Q map is (d, heads, rows) instead (box (64, 1, 128)): ragged
// queries [tokens, H, d], or q [B, H, d] read as one batch of B rows.
struct PrefillMaps {
  CUtensorMap q, k, v;
  bool q_rows_outer = false;
};
// Per-sequence layout, chosen by which pointers are set (one kernel instance each):
//  * dense (all null): sequence b's rows are rows [0, Nq) / [0, Nk) of plane b;
//  * ragged (qo_indptr and kv_indptr): queries are rows [qo_indptr[b], qo_indptr[b+1])
//    and keys rows [kv_indptr[b], kv_indptr[b+1]) of token-major tensors; the K/V maps
//    are (d, Hkv, total_k) like a rows-outer Q map, and Nq is the longest sequence's
//    query count (it sizes the grid);
//  * paged (qo_indptr and kv_lens): ragged queries; keys are the kv_lens[b] tokens
//    gathered through page_table[b, :] from a pool of num_pages pages of 16 tokens,
//    the K/V maps spanning the pool as (d, 16, num_pages * Hkv).  With max_pages 0 no
//    page is ever read (page_table may then be null);
//  * key chunks (key_chunk > 0): one shared set of Nk keys (the dense K/V maps, one plane
//    per KV head) split into chunks; batch b takes keys [b * key_chunk, (b + 1) *
//    key_chunk) against the same Nq query rows (rows-outer Q map), and writes its own
//    normalised O and LSE (a partial for a later merge) at batch stride o_b / l_b.
struct PrefillLayout {
  const int32_t *qo_indptr = nullptr;
  const int32_t *kv_indptr = nullptr;
  const int32_t *page_table = nullptr;
  const int32_t *kv_lens = nullptr;
  int max_pages = 0;
  int num_pages = 0;
  int total_q = 0;  // rows of q / o (bounds every indptr range)
  int total_k = 0;  // rows of k / v
  int key_chunk = 0;  // keys per chunk (key-chunk layout), a multiple of 128
};
// cascade.cu: q [B, H, d] bf16 -> qg [Hkv][B * g][d] (the query rows of each KV head)
cudaError_t launch_group_queries(const void *q, void *qg, int B, int H, int Hkv, int d, cudaStream_t stream);
// cascade.cu: merge C normalised partials (O bf16, partial c at o_parts + c * o_stride
// elements, rows x d in the [Hkv][B * g] row order; LSE at lse_parts + c * l_stride) of
// each row into one (O bf16 [B, H, d], LSE [B, H]); a partial with LSE = -inf weighs nothing
cudaError_t launch_merge_chunks(const void *o_parts, const float *lse_parts, int C, int rows, long long o_stride,
                                long long l_stride, int B, int g, int d, void *o, float *lse, cudaStream_t stream);
cudaError_t launch_prefill_bf16(const PrefillMaps &maps, const PrefillOut &out, int B, int H, int Hkv, int Nq,
                                int Nk, int d, bool causal, float scale, cudaStream_t stream,
                                const PrefillLayout &layout = PrefillLayout());

// fp8_quantize.cu: one tensor of the FP8 inputs (d = 128).  x [planes, N, 128]
// bf16 (raw bits); codes [planes, N, 128] e4m3, or, for V, transposed
// [planes, 128, n_pad] (n_pad a multiple of 16, keys N .. n_pad-1 zero);
// scale [planes, ceil(N / 128)] fp32.
struct Fp8QuantJob {
  const uint16_t *x = nullptr;
  uint8_t *out = nullptr;
  float *scale = nullptr;
  long long planes = 0;
  int N = 0;
  int n_pad = 0;
};
// q and k are multiplied by diag(signs) H_128 first unless signs is null; their
// stored scales then carry transform_norm (1 / sqrt(128)).  v is never transformed.
cudaError_t launch_fp8_quantize(const Fp8QuantJob &q, const Fp8QuantJob &k, const Fp8QuantJob &v, const float *signs,
                                float transform_norm, cudaStream_t stream);

// prefill_fp8.cu: exact-attention forward over e4m3 blocks (d = 128): q8 [B, H, Nq, 128],
// k8 [B, Hkv, Nk, 128] and v8t [B, Hkv, 128, Nk_pad] through 128 x 128-byte TMA boxes,
// per-block scales as written by launch_fp8_quantize; O and LSE as PrefillOut.
struct Fp8Maps {
  CUtensorMap q, k, vt;
};
cudaError_t launch_prefill_fp8(const Fp8Maps &maps, const float *q_scale, const float *k_scale, const float *v_scale,
                               const PrefillOut &out, int B, int H, int Hkv, int Nq, int Nk, bool causal, float scale,
                               cudaStream_t stream);

// Per-translation-unit device error words (see common.cuh).
cudaError_t device_error_decode(unsigned int *value, bool clear);
cudaError_t device_error_prefill_f32(unsigned int *value, bool clear);
cudaError_t device_error_prefill_bf16(unsigned int *value, bool clear);
cudaError_t device_error_prefill_fp8(unsigned int *value, bool clear);
cudaError_t device_error_selftest(unsigned int *value, bool clear);
// one CTA whose two warps wait on mbarriers that nothing arrives on (selftest.cu);
// gave_up[w] = 1 once warp w's bounded wait has given up
cudaError_t launch_wait_timeout_selftest(int *gave_up, cudaStream_t stream);
// {globaltimer, clock64, smid} of one SM (the SM of `match`'s probe when given); selftest.cu
cudaError_t launch_clock_probe(unsigned long long *out, const unsigned long long *match, int blocks,
                               cudaStream_t stream);

}  // namespace attn
