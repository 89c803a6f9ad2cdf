/*
 * attn.h -- C ABI of the exact tiled attention library for GB300 (sm_103a).
 *
 * Exact block-wise (Flash) attention: the prefill forward pass and split-KV
 * paged decode with the exact merge of partial results.  Every entry point
 * takes plain device pointers and sizes, launches on the caller's CUDA
 * stream and returns without synchronising.  The library allocates no
 * device memory: the caller owns every buffer (including the decode
 * workspace) and keeps it alive until the launched work has finished.
 *
 * Common rules
 *  - Device pointers must be 16-byte aligned (log-sum-exp outputs: 4-byte)
 *    and tensors dense, last dimension contiguous, in the layouts stated per
 *    call.
 *  - Argument errors are detected on the host and returned before anything
 *    is launched (ATTN_ERR_INVALID_ARG, ATTN_ERR_UNSUPPORTED,
 *    ATTN_ERR_WORKSPACE).  A failed launch returns ATTN_ERR_CUDA.  Kernel
 *    faults surface, as with any CUDA call, at the next synchronising call.
 *  - Kernels never trap.  Their pipeline waits are bounded; a wait that runs
 *    out sets a device-wide error word and the kernel returns early.
 *    attn_device_error() reads (and optionally clears) that word.
 *  - Grouped-query attention: query head h reads KV head h / (H / Hkv); H
 *    must be a multiple of Hkv.
 *  - The log-sum-exp (LSE) is the natural logarithm of the sum of exp of the
 *    scaled scores of a row; a row that attends to no key has O = 0 and
 *    LSE = -inf.
 */
#ifndef ATTN_H_
#define ATTN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* cudaStream_t without including the CUDA headers; NULL is the legacy default stream. */
typedef struct CUstream_st *attn_stream_t;

typedef enum {
  ATTN_OK = 0,
  ATTN_ERR_INVALID_ARG = 1,  /* null/misaligned pointer, negative size, H % Hkv != 0, ... */
  ATTN_ERR_UNSUPPORTED = 2,  /* a valid request this build has no kernel for (d, dtype, page size) */
  ATTN_ERR_WORKSPACE = 3,    /* decode workspace smaller than attn_decode_workspace_size() */
  ATTN_ERR_CUDA = 4,         /* a CUDA runtime/driver call or a launch failed */
  ATTN_ERR_DEVICE_CHECK = 5  /* a kernel recorded a failed in-kernel check (see attn_device_error) */
} attn_status_t;

typedef enum { ATTN_F32 = 0, ATTN_BF16 = 1 } attn_dtype_t;

/*
 * attn_fwd -- exact attention forward pass (prefill).
 *
 * Follows "3.4 Attention Kernels" (llm-learning-path), sections "Online
 * softmax" and "FlashAttention: tiling": Q is cut into row tiles, K and V are
 * streamed tile by tile through on-chip memory, each score tile
 * S_ij = scale * Q_i K_j^T is folded into a running row maximum m, running
 * denominator l and unnormalised output o~ with the online-softmax rescale
 * exp(m - m'), and O_i = o~ / l and LSE_i = m + ln l are written once.  With
 * causal = 1, key tiles wholly after a query tile are skipped and the
 * diagonal tile is masked (key j is attended by query i iff j <= i).  Also
 * "FlashAttention and Optimized Kernels" (programmer.ie), "The online
 * softmax".
 *
 *  q     [B, H, N, d]    dtype       queries
 *  k, v  [B, Hkv, N, d]  dtype       keys and values
 *  o     [B, H, N, d]    dtype       output (written)
 *  lse   [B, H, N]       float32     log-sum-exp per row (written; may be NULL)
 *  scale                              score scale (1/sqrt(d) for standard attention)
 *  dtype ATTN_BF16: d in {64, 128}; tcgen05 tensor-core kernel, fp32
 *                   accumulation, P rounded to bf16 before P.V, O rounded
 *                   to nearest-even bf16.
 *        ATTN_F32:  d in {64, 128}; precise SIMT kernel: dot products and
 *                   the softmax sums accumulated in fp64, exp in fp32.
 *  B, H, Hkv, N >= 0; N == 0 or B == 0 or H == 0 is a no-op returning ATTN_OK.
 */
attn_status_t attn_fwd(const void *q, const void *k, const void *v, void *o, float *lse,
                       int B, int H, int Hkv, int N, int d, int causal, float scale,
                       attn_dtype_t dtype, attn_stream_t stream);

/*
 * attn_fwd_host -- attn_fwd on inputs and outputs in HOST memory: the call
 * copies Q, K, V in, computes, and copies O (and the LSE) out, pipelined so
 * that the copies overlap the attention (no counterpart on the pages; it is
 * the end-to-end form of attn_fwd for callers whose tensors live on the host,
 * e.g. offloaded activations on a Grace-Blackwell node).
 *
 * The (batch, KV head) planes are cut into up to four contiguous groups (a KV
 * head and its g = H / Hkv query heads are contiguous in the layouts below).
 * Group i: host-to-device copies of its Q, K, V rows on copy_in; attention of
 * the group on `stream` once they have landed; device-to-host copies of its O
 * and LSE rows on copy_out once that attention is done.  One cudaMemcpyAsync
 * per contiguous range; no memory is allocated.  The ten CUDA events that
 * order the three streams are created on a thread's first call for a device
 * and reused by its later calls (a thread's calls must not be captured into
 * graphs that run concurrently with each other).
 *
 *  q_host, k_host, v_host, o_host, lse_host   host pointers, layouts and dtype as attn_fwd
 *             (lse_host may be NULL); page-locked memory is needed for the copies to
 *             overlap the computation, pageable memory still gives correct results
 *  q_dev, k_dev, v_dev, o_dev, lse_dev          device buffers of the same sizes (the
 *             caller's; lse_dev may be NULL only if lse_host is)
 *  stream     the compute stream (NULL: the default stream); the call is ordered after the
 *             work already queued on it, and everything the call does (copies included) is
 *             complete once `stream` has reached the point of the call's return
 *  copy_in, copy_out   two more streams, distinct from each other and from `stream`
 * Errors: as attn_fwd; ATTN_ERR_INVALID_ARG also for NULL or coinciding copy streams.
 */
attn_status_t attn_fwd_host(const void *q_host, const void *k_host, const void *v_host, void *o_host,
                            float *lse_host, void *q_dev, void *k_dev, void *v_dev, void *o_dev, float *lse_dev,
                            int B, int H, int Hkv, int N, int d, int causal, float scale, attn_dtype_t dtype,
                            attn_stream_t stream, attn_stream_t copy_in, attn_stream_t copy_out);

/*
 * attn_fwd_cross -- attn_fwd with Nq query rows against Nk keys (Nq may differ
 * from Nk: cross attention, or a chunk of new queries against a cache that
 * ends with them).  With causal = 1 the mask is aligned to the last key:
 * query row i attends key j iff j <= i + (Nk - Nq), the alignment of the
 * naive causal attention in "3.4 Attention Kernels", "Code"; rows that attend
 * no key get O = 0 and LSE = -inf.  Same algorithm and citations as attn_fwd.
 *
 *  q     [B, H, Nq, d]    k, v [B, Hkv, Nk, d]    o [B, H, Nq, d]    lse [B, H, Nq]
 *  Nq, Nk >= 0; Nq == 0 (or B == 0, H == 0) is a no-op.
 */
attn_status_t attn_fwd_cross(const void *q, const void *k, const void *v, void *o, float *lse,
                             int B, int H, int Hkv, int Nq, int Nk, int d, int causal, float scale,
                             attn_dtype_t dtype, attn_stream_t stream);

/*
 * attn_fwd_varlen -- exact attention over a batch of sequences of different
 * lengths packed without padding (ragged tensors).
 *
 * Follows "3.4 Attention Kernels", "Paged and ragged layouts: FlashInfer":
 * all sequences' tokens are concatenated and an offsets array (indptr) marks
 * where each sequence starts.  Sequence b's queries are rows
 * [qo_indptr[b], qo_indptr[b+1]) of q and its keys/values rows
 * [kv_indptr[b], kv_indptr[b+1]) of k and v; each sequence is attended on its
 * own with the tcgen05 prefill kernel (same algorithm as attn_fwd).  With
 * causal = 1 the mask is aligned to each sequence's last key (query row i of
 * a sequence with Lq queries and Lk keys attends keys j <= i + Lk - Lq).
 *
 *  q         [total_q, H, d]    bf16    k, v [total_k, Hkv, d] bf16
 *  o         [total_q, H, d]    bf16    lse  [total_q, H] fp32 (may be NULL)
 *  qo_indptr, kv_indptr  [B + 1] int32, device, non-decreasing, within [0, total_q] / [0, total_k]
 *  max_q_len  the longest sequence's query count (sizes the grid on the host)
 *  d in {64, 128}.
 * The offsets stay on the device (no copy, so the call can be graph-captured);
 * the kernel checks them: a sequence with more than max_q_len queries, or whose
 * offsets leave those ranges, is not computed (its rows of o and lse are left
 * unwritten) and sets ATTN_DEVERR_BAD_LENGTH in attn_device_error.
 */
attn_status_t attn_fwd_varlen(const void *q, const void *k, const void *v, void *o, float *lse,
                              const int32_t *qo_indptr, const int32_t *kv_indptr, int B, int H, int Hkv,
                              int max_q_len, int total_q, int total_k, int d, int causal, float scale,
                              attn_stream_t stream);

/*
 * attn_fwd_paged -- prefill of ragged query chunks against a paged KV cache
 * (continuous batching: new tokens of several sequences in one launch).
 *
 * Follows "3.4 Attention Kernels", "Paged and ragged layouts: FlashInfer"
 * (ragged queries through indptr; K/V gathered through the block table and
 * the sequence lengths).  Sequence b's queries are rows
 * [qo_indptr[b], qo_indptr[b+1]) of q; its keys are the kv_lens[b] tokens of
 * its pages, with the query chunk being the last tokens of the sequence:
 * with causal = 1, query row i of a chunk of Lq rows attends keys
 * j <= i + kv_lens[b] - Lq.  The K/V tiles are gathered page by page by TMA.
 *
 *  q          [total_q, H, d] bf16     o [total_q, H, d] bf16   lse [total_q, H] fp32 (nullable)
 *  k_pages, v_pages, page_table, kv_lens, num_pages: as attn_decode_paged (page_size 16;
 *             bad page ids and kv_lens values beyond the table are handled the same way)
 *  qo_indptr  [B + 1] int32, device, checked as in attn_fwd_varlen (with total_q);
 *  max_q_len  as attn_fwd_varlen;  d in {64, 128}.
 * Each 128-key tile is loaded as whole 16-token pages; the slots past
 * kv_lens[b] in a sequence's last page may hold anything (stale tokens, NaN,
 * Inf): their scores are masked and their V rows are zeroed in shared memory
 * before P V, so they never reach O or the LSE.
 */
attn_status_t attn_fwd_paged(const void *q, const void *k_pages, const void *v_pages, const int32_t *page_table,
                             const int32_t *kv_lens, const int32_t *qo_indptr, void *o, float *lse,
                             int B, int H, int Hkv, int max_q_len, int total_q, int d, int page_size,
                             int max_pages_per_seq, int num_pages, int causal, float scale, attn_stream_t stream);

/*
 * FP8 attention: attn_fp8_quantize then attn_fwd_fp8.
 *
 * Follows "3.4 Attention Kernels", "FlashAttention-2 and -3": FlashAttention-3's
 * FP8 attention, with block quantisation and "incoherent processing" (a random
 * orthogonal transform against outliers).  Readings of that prose: the
 * transform is M = diag(signs) H_d / sqrt(d) (H_d Sylvester's Hadamard matrix,
 * signs a random +-1 vector) applied to Q and K, which leaves Q K^T unchanged;
 * a block is one 128-row tile of one head, with one fp32 scale = amax / 448
 * and e4m3 codes of x / scale (round to nearest even, saturating).  d = 128 only.
 *
 * attn_fp8_quantize -- quantise bf16 q [B, H, Nq, 128], k and v [B, Hkv, Nk, 128]:
 *  signs     [128] fp32 +-1, device, 16-byte aligned; NULL = no transform
 *  q8        [B, H, Nq, 128]        e4m3 codes of q M (written)
 *  k8        [B, Hkv, Nk, 128]      e4m3 codes of k M (written)
 *  v8t       [B, Hkv, 128, Nk_pad]  e4m3 codes of v, TRANSPOSED (keys contiguous),
 *                                   Nk_pad = attn_fp8_padded_keys(Nk); keys Nk.. are 0
 *  q_scale   [B, H, ceil(Nq / 128)]   fp32 block scales (dequantised x' = code * scale)
 *  k_scale, v_scale [B, Hkv, ceil(Nk / 128)]
 * All buffers are the caller's (nothing is allocated); one kernel launch.
 */
int attn_fp8_padded_keys(int Nk);
attn_status_t attn_fp8_quantize(const void *q, const void *k, const void *v, const float *signs, void *q8,
                                void *k8, void *v8t, float *q_scale, float *k_scale, float *v_scale, int B, int H,
                                int Hkv, int Nq, int Nk, int d, attn_stream_t stream);

/*
 * attn_fwd_fp8 -- exact attention forward over the FP8 blocks written by
 * attn_fp8_quantize: S = scale * (q8 k8^T) * sq * sk per block pair, the online
 * softmax of attn_fwd (causal tile skipping, mask aligned to the last key when
 * Nq != Nk, GQA), P rounded to e4m3 for P V (tcgen05 kind::f8f6f4 for both
 * products).  o [B, H, Nq, 128] bf16, lse [B, H, Nq] fp32 (nullable).  The
 * result equals attention of the dequantised blocks up to P's 8-bit rounding
 * (|error| <= 2^-4 of the attended values' magnitude per key weight).
 */
attn_status_t attn_fwd_fp8(const void *q8, const void *k8, const void *v8t, const float *q_scale,
                           const float *k_scale, const float *v_scale, void *o, float *lse, int B, int H, int Hkv,
                           int Nq, int Nk, int d, int causal, float scale, attn_stream_t stream);

/*
 * attn_decode_workspace_size -- bytes of device workspace attn_decode_paged
 * needs for up to max_splits partial results per (sequence, query head):
 * fp32 m and l [B, H, max_splits] and fp32 o~ [B, H, max_splits, d], each
 * region 256-byte aligned.  Returns 0 for invalid arguments.
 */
size_t attn_decode_workspace_size(int B, int H, int d, int max_splits);

/*
 * attn_decode_paged -- one query token per sequence against a paged,
 * ragged KV cache, split along the keys (split-KV / Flash-Decoding), then
 * merged exactly.
 *
 * Follows "3.4 Attention Kernels", sections "Decode attention and
 * Flash-Decoding" (split the cache into chunks, one partial (m_c, l_c, o~_c)
 * per chunk, merged by the log-sum-exp merge in a small reduction kernel;
 * all query heads of a GQA group share each loaded K/V tile) and "Paged and
 * ragged layouts: FlashInfer" (the kernel gathers K/V through a page table).
 *
 *  q           [B, H, d]                   bf16   one query token per sequence
 *  k_pages     [P, Hkv, page_size, d]      bf16   shared pool of K pages
 *  v_pages     [P, Hkv, page_size, d]      bf16   shared pool of V pages
 *  page_table  [B, max_pages_per_seq]      int32  page ids (< num_pages) of each sequence, in token order
 *  kv_lens     [B]                         int32  tokens of each sequence, 0 <= kv_lens[b] <= max_pages_per_seq * page_size
 *  o           [B, H, d]                   bf16   output (written)
 *  lse         [B, H]                      fp32   log-sum-exp (written; may be NULL)
 *  num_pages   P, the pool size (the tensor-map extent).  A page id outside [0, P)
 *              reads as zeros (TMA fills out-of-range boxes) and is recorded as
 *              ATTN_DEVERR_BAD_PAGE; so is a kv_lens value beyond the table.
 *              Slots past kv_lens[b] in a sequence's last page may hold
 *              anything (NaN and Inf included): their scores are masked and
 *              their V rows zeroed in shared memory before P V.
 *  num_splits  upper bound on the key chunks per sequence; <= 0 picks one from
 *              B, Hkv, max_pages_per_seq and the SM count.  The chunk is
 *              ceil(max_pages_per_seq / num_splits) pages; sequence b uses
 *              ceil(pages_b / chunk) partials.  No device-to-host copy is made.
 *  workspace   >= attn_decode_workspace_size(B, H, d, num_splits used) bytes;
 *              with num_splits <= 0 pass the size for attn_decode_max_splits().
 *  Supported: d in {64, 128}, page_size == 16, H / Hkv <= 16.  Results are
 *  deterministic for a given num_splits.
 */
attn_status_t attn_decode_paged(const void *q, const void *k_pages, const void *v_pages,
                                const int32_t *page_table, const int32_t *kv_lens, void *o, float *lse,
                                int B, int H, int Hkv, int d, int page_size, int max_pages_per_seq,
                                int num_pages, float scale, int num_splits,
                                void *workspace, size_t workspace_bytes, attn_stream_t stream);

/*
 * attn_decode_max_splits -- the split count attn_decode_paged picks when
 * called with num_splits <= 0 on the current device (for sizing the
 * workspace).  Returns 0 for invalid arguments.
 */
int attn_decode_max_splits(int B, int H, int Hkv, int max_pages_per_seq);

/*
 * attn_cascade_workspace_size -- bytes of device workspace attn_cascade_decode
 * needs: the decode partials for max_splits chunks, the shared-prefix result
 * (bf16 O [B, H, d] and fp32 LSE [B, H]), up to 16 key-chunk partials of the
 * same shape and a copy of q grouped by KV head, each region 256-byte aligned.
 * Returns 0 for invalid arguments.
 */
size_t attn_cascade_workspace_size(int B, int H, int d, int max_splits);

/*
 * attn_cascade_decode -- decode for B requests that share one prefix of
 * prefix_len tokens and each have their own paged suffix (cascade attention).
 *
 * Follows "3.4 Attention Kernels", "Paged and ragged layouts: FlashInfer"
 * (attention over the shared prefix is computed once for all requests' queries
 * and merged with each request's own-suffix attention by the merge operator)
 * and "Check your understanding" (attention over prefix U suffix is the
 * log-sum-exp merge of the two).  The prefix pass is attention, per KV head,
 * whose query rows are the B requests' query heads of that head's group,
 * against the prefix keys, on the tensor-core prefill kernel, split into up to
 * 16 chunks of keys (about two CTAs per SM) whose normalised partials are
 * merged into one prefix result;
 * the suffix pass is attn_decode_paged's split kernel; the merge kernel
 * combines the suffix chunks' partials with the prefix result taken as the
 * partial (m, l, o~) = (LSE_prefix, 1, O_prefix).
 *
 *  q                     [B, H, d]                  bf16   one query token per request
 *  prefix_k, prefix_v    [Hkv, prefix_len, d]       bf16   the shared prefix's keys/values
 *  k_pages ... kv_lens   the requests' own suffixes, exactly as attn_decode_paged
 *                        (kv_lens counts suffix tokens only; 0 is allowed)
 *  o [B, H, d] bf16, lse [B, H] fp32 (may be NULL): attention over prefix + suffix
 *  workspace             >= attn_cascade_workspace_size(B, H, d, splits used)
 *  prefix_len >= 0 (0: plain paged decode).  Supported as attn_decode_paged.
 */
attn_status_t attn_cascade_decode(const void *q, const void *prefix_k, const void *prefix_v, int prefix_len,
                                  const void *k_pages, const void *v_pages, const int32_t *page_table,
                                  const int32_t *kv_lens, void *o, float *lse,
                                  int B, int H, int Hkv, int d, int page_size, int max_pages_per_seq,
                                  int num_pages, float scale, int num_splits,
                                  void *workspace, size_t workspace_bytes, attn_stream_t stream);

/*
 * merge_partials -- exact merge of per-chunk partial results.
 *
 * Follows "3.4 Attention Kernels", section "Online softmax" (the merge of two
 * partial results computed on disjoint key sets), applied over S partials:
 * m = max_s m_s, l = sum_s exp(m_s - m) l_s, o~ = sum_s exp(m_s - m) o~_s,
 * then O = o~ / l and LSE = m + ln l.  "FlashAttention and Optimized
 * Kernels", "The decode shape: splitting the keys" names the operation.
 * An empty partial is (m, l, o~) = (-inf, 0, 0) and contributes nothing.
 *
 *  m, l        [B, H, S]     fp32   per-partial running max (natural-log units of the
 *                                   scaled scores) and denominator
 *  o_tilde     [B, H, S, d]  fp32   per-partial unnormalised output
 *  num_parts   [B]           int32  partials used for sequence b (first num_parts[b]
 *                                   of S); NULL means all S
 *  o           [B, H, d]     o_dtype  merged output (written)
 *  lse         [B, H]        fp32   merged log-sum-exp (written; may be NULL)
 *  d in {64, 128}; S >= 1.
 */
attn_status_t merge_partials(const float *m, const float *l, const float *o_tilde,
                             const int32_t *num_parts, int B, int H, int S, int d,
                             void *o, attn_dtype_t o_dtype, float *lse, attn_stream_t stream);

/*
 * attn_decode_paged_noalloc -- attn_decode_paged for callers that cannot
 * allocate device memory.  The pages this library follows have no
 * counterpart to it; it exists for callers such as a plugin or custom op
 * inside another runtime that is handed only its input and output buffers
 * (no allocator, no workspace), or a latency-critical serving loop that must
 * not call cudaMalloc because it can synchronise the device.
 *
 * Arguments, layouts, results and errors are those of attn_decode_paged,
 * without workspace and workspace_bytes: the per-chunk partials go to a fixed
 * array in device global memory that belongs to this library,
 * ATTN_DECODE_NOALLOC_SCRATCH_BYTES long, which every GPU that loads the
 * library holds until the process exits.  A request whose partials,
 * attn_decode_workspace_size(B, H, d, splits used), exceed that size returns
 * ATTN_ERR_WORKSPACE before anything is launched (with num_splits <= 0 the
 * automatic split count decides the size; pass a smaller num_splits to fit).
 * It calls no cudaMalloc, cudaFree or other allocating routine.
 *
 * The first call on a device looks up the array's device address on that
 * device (cudaGetSymbolAddress, with the caller's current device); make that
 * first call before any stream capture.  The address is kept for the life of
 * the process: after cudaDeviceReset, or any other end of the device's
 * primary context, it no longer names the array, so no call may follow such a
 * reset on that device.  All calls on a device share the one
 * array and it keeps the previous call's contents; nothing in it needs to
 * start at zero, because every partial the merge reads is written earlier in
 * the same call.  Calls that overlap on the GPU (on different streams, or
 * from several host threads without ordering) race on the array: order them.
 */
#define ATTN_DECODE_NOALLOC_SCRATCH_BYTES (40u * 1024u * 1024u)
attn_status_t attn_decode_paged_noalloc(const void *q, const void *k_pages, const void *v_pages,
                                        const int32_t *page_table, const int32_t *kv_lens, void *o, float *lse,
                                        int B, int H, int Hkv, int d, int page_size, int max_pages_per_seq,
                                        int num_pages, float scale, int num_splits, attn_stream_t stream);

/* attn_status_string -- a static, human-readable name for a status code. */
const char *attn_status_string(attn_status_t status);

/*
 * attn_device_error -- read the device-wide error word of the current device
 * (synchronises the device).  0 means no kernel has recorded a failure; a
 * non-zero value is a bit set of ATTN_DEVERR_* codes.  clear != 0 resets it.
 * Returns ATTN_ERR_CUDA if the read itself failed.
 */
attn_status_t attn_device_error(uint32_t *code, int clear);

/*
 * attn_selftest_wait_timeout -- exercise the bounded pipeline waits.  Launches
 * one CTA on `stream` whose two warps wait on mbarriers that nothing ever
 * arrives on, through the same bounded wait the attention kernels use.  The
 * first wait to run out (after about 2 s) records ATTN_DEVERR_WAIT_TIMEOUT and
 * raises the CTA's abort flag; the other warp then gives up through that flag.
 * The kernel returns without trapping, so the context stays usable.
 *   gave_up  [2] int32, device, written with 1 for each warp whose wait gave up
 *            (0 would mean a barrier completed, which nothing here allows)
 * Returns ATTN_ERR_INVALID_ARG for a null pointer and ATTN_ERR_CUDA if the
 * launch failed.  Like every entry point it does not synchronise; read the
 * error word with attn_device_error afterwards.
 */
attn_status_t attn_selftest_wait_timeout(int32_t *gave_up, attn_stream_t stream);

/*
 * attn_clock_probe -- the SM clock over a stretch of work, measured on the device
 * (a diagnostic; no counterpart on the pages).  Records, on `stream`, the global
 * timer (ns) and one SM's cycle counter %clock64:
 *   out    [4] uint64, device, 8-byte aligned: {global timer ns, clock64, SM id, claim};
 *          zeroed by the call, then written by the first probe block on the chosen SM
 *          (claim = 1 once written; 0 means no block ran there)
 *   match  NULL: any SM (one block); or an earlier probe's `out` (read on the device
 *          when this probe runs): record on the same SM, since clock64 is a per-SM
 *          counter (blocks on every SM; those on other SMs return at once)
 * Two probes around work on one stream give its average SM clock in MHz:
 * 1000 * (clock64 difference) / (timer difference).  Returns ATTN_ERR_INVALID_ARG
 * for a null or misaligned pointer, ATTN_ERR_CUDA if the launch failed.
 */
attn_status_t attn_clock_probe(uint64_t *out, const uint64_t *match, attn_stream_t stream);

#define ATTN_DEVERR_WAIT_TIMEOUT 0x1u   /* a pipeline wait gave up after its iteration limit */
#define ATTN_DEVERR_BAD_PAGE     0x2u   /* a page id outside [0, num_pages) was skipped */
#define ATTN_DEVERR_TMEM_ALLOC   0x4u   /* tensor memory allocation returned an unusable address */
#define ATTN_DEVERR_BAD_LENGTH   0x8u   /* a ragged sequence's offsets were out of range or exceeded max_q_len */

#ifdef __cplusplus
}
#endif

#endif /* ATTN_H_ */
