// Host side of the C ABI declared in include/attn.h: argument validation,
// TMA tensor-map encoding, the split-KV plan, and kernel launches.  Nothing
// here allocates device memory or synchronises (except attn_device_error).
#include <algorithm>
#include <mutex>

#include <cudaTypedefs.h>

#include "attn.h"
#include "common.cuh"
#include "kernels.h"

namespace {

using attn::PrefillMaps;
using attn::PrefillOut;

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }  // the LSE (scalar stores)

// cuTensorMapEncodeTiled through the runtime's driver entry point (no -lcuda).
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 3-D bf16 tensor [d2][d1][d0] (d0 contiguous, nested strides) with a box of
// (64, box1, box2) and 128-byte swizzle.
bool make_map_3d(CUtensorMap *map, const void *base, uint64_t d0, uint64_t d1, uint64_t d2, uint32_t box1,
                 uint32_t box2 = 1) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[3] = {d0, std::max<uint64_t>(d1, 1), std::max<uint64_t>(d2, 1)};
  cuuint64_t strides[2] = {d0 * 2, d0 * dims[1] * 2};
  cuuint32_t box[3] = {64, box1, box2};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 3-D byte tensor [d2][d1][d0] (d0 contiguous, a multiple of 16 bytes) with a
// box of (128, 128, 1) bytes and 128-byte swizzle: one e4m3 tile.
bool make_map_u8(CUtensorMap *map, const void *base, uint64_t d0, uint64_t d1, uint64_t d2) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[3] = {d0, std::max<uint64_t>(d1, 1), std::max<uint64_t>(d2, 1)};
  cuuint64_t strides[2] = {d0, d0 * dims[1]};
  cuuint32_t box[3] = {128, 128, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

int device_sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

int ceil_div(long long a, long long b) { return static_cast<int>((a + b - 1) / b); }

// The shared prefix of a cascade decode runs as at most this many key chunks.
constexpr int kMaxPrefixChunks = 16;

// Split-KV plan from arguments only (no device-to-host copy): chunks of at
// most 256 pages (2 MiB of one KV head's K and V at d = 128, long enough to
// amortise a CTA's set-up), more splits when that gives fewer than ~6 CTAs per
// SM with every sequence as long as the longest, and chunks of at least 8 pages.
int auto_splits(int B, int Hkv, int max_pages, int num_sms) {
  const int want_ctas = 6 * std::max(num_sms, 1);
  int s = ceil_div(max_pages, 256);
  s = std::max(s, ceil_div(want_ctas, static_cast<long long>(B) * Hkv));
  s = std::min(s, ceil_div(max_pages, 8));
  return std::max(s, 1);
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

size_t decode_ws_bytes(int B, int H, int d, int splits) {
  const size_t n = static_cast<size_t>(B) * H * splits;
  return 2 * align256(n * sizeof(float)) + align256(n * d * sizeof(float));
}

// ---------------------------------------------------------------------------
// prefill over Nq query rows and Nk keys (Nq == Nk for attn_fwd)
// ---------------------------------------------------------------------------
attn_status_t fwd_impl(const void *q, const void *k, const void *v, void *o, float *lse, int B, int H, int Hkv,
                       int Nq, int Nk, int d, int causal, float scale, attn_dtype_t dtype, attn_stream_t stream) {
  if (B < 0 || H < 0 || Hkv < 0 || Nq < 0 || Nk < 0) return ATTN_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !(scale < INFINITY)) return ATTN_ERR_INVALID_ARG;
  if (dtype != ATTN_F32 && dtype != ATTN_BF16) return ATTN_ERR_INVALID_ARG;
  if (B == 0 || H == 0 || Nq == 0) return ATTN_OK;
  if (Hkv == 0 || H % Hkv != 0) return ATTN_ERR_INVALID_ARG;
  if (q == nullptr || o == nullptr || (Nk > 0 && (k == nullptr || v == nullptr))) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || (lse && !aligned4(lse)))
    return ATTN_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  PrefillOut out;
  out.o = o;
  out.lse = lse;
  out.o_b = static_cast<long long>(H) * Nq * d;
  out.o_h = static_cast<long long>(Nq) * d;
  out.o_r = d;
  out.l_b = static_cast<long long>(H) * Nq;
  out.l_h = Nq;
  out.l_r = 1;
  cudaError_t e;
  if (dtype == ATTN_F32) {
    e = attn::launch_prefill_f32(static_cast<const float *>(q), static_cast<const float *>(k),
                                 static_cast<const float *>(v), out, B, H, Hkv, Nq, Nk, d, causal != 0, scale, st);
  } else {
    // with Nk == 0 the K/V maps are never read; they only need a valid shape
    const void *kb = Nk > 0 ? k : q;
    const void *vb = Nk > 0 ? v : q;
    PrefillMaps maps;
    if (!make_map_3d(&maps.q, q, d, Nq, static_cast<uint64_t>(B) * H, 128) ||
        !make_map_3d(&maps.k, kb, d, Nk, static_cast<uint64_t>(B) * Hkv, 128) ||
        !make_map_3d(&maps.v, vb, d, Nk, static_cast<uint64_t>(B) * Hkv, 128))
      return ATTN_ERR_CUDA;
    e = attn::launch_prefill_bf16(maps, out, B, H, Hkv, Nq, Nk, d, causal != 0, scale, st);
  }
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

// ---------------------------------------------------------------------------
// paged split-KV decode; optional extra partial (O, LSE) per (sequence, head)
// ---------------------------------------------------------------------------
struct DecodePlan {
  int splits;      // partial slots per (sequence, head)
  int chunk;       // pages per chunk
  bool has_pages;  // anything to stream at all
};

attn_status_t decode_check(const void *q, const void *k_pages, const void *v_pages, const int32_t *page_table,
                           const int32_t *kv_lens, const void *o, const float *lse, int B, int H, int Hkv, int d,
                           int page_size, int max_pages_per_seq, int num_pages, float scale, const void *workspace) {
  if (B < 0 || H < 0 || Hkv < 0 || max_pages_per_seq < 0 || num_pages < 0) return ATTN_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !(scale < INFINITY)) return ATTN_ERR_INVALID_ARG;
  if (B == 0 || H == 0) return ATTN_OK;
  if (Hkv == 0 || H % Hkv != 0) return ATTN_ERR_INVALID_ARG;
  if (q == nullptr || o == nullptr || kv_lens == nullptr || workspace == nullptr) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(o) || (lse && !aligned4(lse)) || !aligned16(workspace)) return ATTN_ERR_INVALID_ARG;
  if ((d != 64 && d != 128) || page_size != 16 || H / Hkv > 16) return ATTN_ERR_UNSUPPORTED;
  if (max_pages_per_seq > 0 && num_pages > 0) {
    if (k_pages == nullptr || v_pages == nullptr || page_table == nullptr) return ATTN_ERR_INVALID_ARG;
    if (!aligned16(k_pages) || !aligned16(v_pages)) return ATTN_ERR_INVALID_ARG;
  }
  return ATTN_OK;
}

DecodePlan decode_plan(int B, int Hkv, int max_pages_per_seq, int num_pages, int num_splits) {
  const int mp = std::max(max_pages_per_seq, 1);
  const int S = num_splits > 0 ? std::min(num_splits, mp) : auto_splits(B, Hkv, mp, device_sm_count());
  const int chunk = ceil_div(mp, S);
  DecodePlan p;
  p.splits = ceil_div(mp, chunk);  // partial slots any sequence can need
  p.chunk = chunk;
  p.has_pages = max_pages_per_seq > 0 && num_pages > 0;
  return p;
}

attn_status_t decode_launch(const DecodePlan &plan, const void *q, const void *k_pages, const void *v_pages,
                            const int32_t *page_table, const int32_t *kv_lens, void *o, float *lse, int B, int H,
                            int Hkv, int d, int page_size, int max_pages_per_seq, int num_pages, float scale,
                            void *workspace, const void *extra_o, const float *extra_lse, cudaStream_t st) {
  const size_t n = static_cast<size_t>(B) * H * plan.splits;
  float *ws_m = static_cast<float *>(workspace);
  float *ws_l = reinterpret_cast<float *>(static_cast<char *>(workspace) + align256(n * sizeof(float)));
  float *ws_o = reinterpret_cast<float *>(static_cast<char *>(workspace) + 2 * align256(n * sizeof(float)));
  if (plan.has_pages) {
    CUtensorMap tm_k, tm_v;
    const uint64_t rows = static_cast<uint64_t>(num_pages) * Hkv;
    if (!make_map_3d(&tm_k, k_pages, d, page_size, rows, page_size) ||
        !make_map_3d(&tm_v, v_pages, d, page_size, rows, page_size))
      return ATTN_ERR_CUDA;
    cudaError_t e = attn::launch_decode_split(tm_k, tm_v, q, page_table, kv_lens, ws_m, ws_l, ws_o, B, H, Hkv, d,
                                              max_pages_per_seq, num_pages, plan.chunk, plan.splits, scale, st);
    if (e != cudaSuccess) return ATTN_ERR_CUDA;
  }
  // with no pages at all every sequence's own keys are empty: only the extra partial (if any) counts
  cudaError_t e = attn::launch_merge(ws_m, ws_l, ws_o, nullptr, kv_lens, page_size,
                                     plan.has_pages ? plan.chunk : 1 << 30, B, H, plan.splits, d, o, true, lse,
                                     extra_o, extra_lse, st, plan.has_pages);
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace

extern "C" {

const char *attn_status_string(attn_status_t s) {
  switch (s) {
    case ATTN_OK: return "ATTN_OK";
    case ATTN_ERR_INVALID_ARG: return "ATTN_ERR_INVALID_ARG";
    case ATTN_ERR_UNSUPPORTED: return "ATTN_ERR_UNSUPPORTED";
    case ATTN_ERR_WORKSPACE: return "ATTN_ERR_WORKSPACE";
    case ATTN_ERR_CUDA: return "ATTN_ERR_CUDA";
    case ATTN_ERR_DEVICE_CHECK: return "ATTN_ERR_DEVICE_CHECK";
  }
  return "ATTN_STATUS_UNKNOWN";
}

attn_status_t attn_fwd(const void *q, const void *k, const void *v, void *o, float *lse, int B, int H, int Hkv, int N,
                       int d, int causal, float scale, attn_dtype_t dtype, attn_stream_t stream) {
  return fwd_impl(q, k, v, o, lse, B, H, Hkv, N, N, d, causal, scale, dtype, stream);
}

// attn_fwd_host: groups of (batch, KV head) planes in flight at once
constexpr int kHostGroups = 4;

// The events that order attn_fwd_host's three streams, created once per host thread and
// device and reused by every call from that thread: a thread's calls are queued one after
// another, and a stream wait binds to the event's latest record at the time it is queued.
// They are released when the thread moves to another device, and otherwise kept until the
// device's context goes away (no CUDA call from a thread-exit destructor, which may run
// after the runtime has shut down).
struct HostCallEvents {
  int device = -1;
  cudaEvent_t ev[2 + 2 * kHostGroups] = {};
  void release() {
    for (cudaEvent_t &e : ev)
      if (e != nullptr) {
        cudaEventDestroy(e);
        e = nullptr;
      }
    device = -1;
  }
  // the events for the current device, or nullptr if they cannot be created
  cudaEvent_t *get() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
    if (dev == device) return ev;
    release();
    for (cudaEvent_t &e : ev)
      if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) {
        release();
        return nullptr;
      }
    device = dev;
    return ev;
  }
};

attn_status_t attn_fwd_host(const void *q_host, const void *k_host, const void *v_host, void *o_host,
                            float *lse_host, void *q_dev, void *k_dev, void *v_dev, void *o_dev, float *lse_dev,
                            int B, int H, int Hkv, int N, int d, int causal, float scale, attn_dtype_t dtype,
                            attn_stream_t stream, attn_stream_t copy_in, attn_stream_t copy_out) {
  if (B < 0 || H < 0 || Hkv < 0 || N < 0) return ATTN_ERR_INVALID_ARG;
  if (dtype != ATTN_F32 && dtype != ATTN_BF16) return ATTN_ERR_INVALID_ARG;
  if (copy_in == nullptr || copy_out == nullptr || stream == copy_in || stream == copy_out || copy_in == copy_out)
    return ATTN_ERR_INVALID_ARG;
  if (B == 0 || H == 0 || N == 0) return ATTN_OK;
  if (Hkv == 0 || H % Hkv != 0) return ATTN_ERR_INVALID_ARG;
  if (q_host == nullptr || k_host == nullptr || v_host == nullptr || o_host == nullptr || q_dev == nullptr ||
      k_dev == nullptr || v_dev == nullptr || o_dev == nullptr || (lse_host != nullptr && lse_dev == nullptr))
    return ATTN_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !(scale < INFINITY)) return ATTN_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaStream_t cin = reinterpret_cast<cudaStream_t>(copy_in);
  cudaStream_t cout = reinterpret_cast<cudaStream_t>(copy_out);
  const int g = H / Hkv;
  const long long planes = static_cast<long long>(B) * Hkv;  // (batch, KV head) planes
  const int groups = static_cast<int>(std::min<long long>(kHostGroups, planes));
  const size_t es = dtype == ATTN_BF16 ? 2 : 4;
  const size_t kv_plane = static_cast<size_t>(N) * d * es;   // bytes of one K (or V) plane
  const size_t q_plane = kv_plane * g;                       // bytes of the plane's g query heads
  const size_t l_plane = static_cast<size_t>(N) * g * sizeof(float);

  static thread_local HostCallEvents pool;
  cudaEvent_t *ev = pool.get();
  if (ev == nullptr) return ATTN_ERR_CUDA;
  cudaEvent_t start = ev[0], out_done = ev[1];
  cudaEvent_t *in_done = ev + 2, *fwd_done = ev + 2 + kHostGroups;
  attn_status_t status = ATTN_OK;
  auto check = [&](cudaError_t e) {
    if (e != cudaSuccess && status == ATTN_OK) status = ATTN_ERR_CUDA;
  };
  // the copies may only touch the device buffers once earlier work on `stream` is done
  check(cudaEventRecord(start, st));
  check(cudaStreamWaitEvent(cin, start, 0));
  check(cudaStreamWaitEvent(cout, start, 0));
  auto bytes = [](const void *p, size_t off) { return static_cast<const char *>(p) + off; };
  auto wbytes = [](void *p, size_t off) { return static_cast<char *>(p) + off; };
  for (int i = 0; i < groups && status == ATTN_OK; ++i) {
    const long long p0 = planes * i / groups, p1 = planes * (i + 1) / groups;
    const size_t np = static_cast<size_t>(p1 - p0);
    check(cudaMemcpyAsync(wbytes(q_dev, p0 * q_plane), bytes(q_host, p0 * q_plane), np * q_plane,
                          cudaMemcpyHostToDevice, cin));
    check(cudaMemcpyAsync(wbytes(k_dev, p0 * kv_plane), bytes(k_host, p0 * kv_plane), np * kv_plane,
                          cudaMemcpyHostToDevice, cin));
    check(cudaMemcpyAsync(wbytes(v_dev, p0 * kv_plane), bytes(v_host, p0 * kv_plane), np * kv_plane,
                          cudaMemcpyHostToDevice, cin));
    check(cudaEventRecord(in_done[i], cin));
    check(cudaStreamWaitEvent(st, in_done[i], 0));
    // the group as np batches of g query heads sharing one KV head
    const attn_status_t s = fwd_impl(bytes(q_dev, p0 * q_plane), bytes(k_dev, p0 * kv_plane),
                                     bytes(v_dev, p0 * kv_plane), wbytes(o_dev, p0 * q_plane),
                                     lse_dev ? lse_dev + p0 * (l_plane / sizeof(float)) : nullptr,
                                     static_cast<int>(np), g, 1, N, N, d, causal, scale, dtype, stream);
    if (s != ATTN_OK) status = s;
    check(cudaEventRecord(fwd_done[i], st));
    check(cudaStreamWaitEvent(cout, fwd_done[i], 0));
    check(cudaMemcpyAsync(wbytes(o_host, p0 * q_plane), bytes(o_dev, p0 * q_plane), np * q_plane,
                          cudaMemcpyDeviceToHost, cout));
    if (lse_host != nullptr)
      check(cudaMemcpyAsync(lse_host + p0 * (l_plane / sizeof(float)), lse_dev + p0 * (l_plane / sizeof(float)),
                            np * l_plane, cudaMemcpyDeviceToHost, cout));
  }
  // `stream` covers everything the call queued
  check(cudaEventRecord(out_done, cout));
  check(cudaStreamWaitEvent(st, out_done, 0));
  return status;
}

attn_status_t attn_fwd_cross(const void *q, const void *k, const void *v, void *o, float *lse, int B, int H, int Hkv,
                             int Nq, int Nk, int d, int causal, float scale, attn_dtype_t dtype, attn_stream_t stream) {
  return fwd_impl(q, k, v, o, lse, B, H, Hkv, Nq, Nk, d, causal, scale, dtype, stream);
}

attn_status_t attn_fwd_varlen(const void *q, const void *k, const void *v, void *o, float *lse,
                              const int32_t *qo_indptr, const int32_t *kv_indptr, int B, int H, int Hkv,
                              int max_q_len, int total_q, int total_k, int d, int causal, float scale,
                              attn_stream_t stream) {
  if (B < 0 || H < 0 || Hkv < 0 || max_q_len < 0 || total_q < 0 || total_k < 0) return ATTN_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !(scale < INFINITY)) return ATTN_ERR_INVALID_ARG;
  if (B == 0 || H == 0 || max_q_len == 0 || total_q == 0) return ATTN_OK;
  if (Hkv == 0 || H % Hkv != 0) return ATTN_ERR_INVALID_ARG;
  if (q == nullptr || o == nullptr || qo_indptr == nullptr || kv_indptr == nullptr) return ATTN_ERR_INVALID_ARG;
  if (total_k > 0 && (k == nullptr || v == nullptr)) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || (lse && !aligned4(lse)))
    return ATTN_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
  PrefillMaps maps;
  maps.q_rows_outer = true;
  const void *kb = total_k > 0 ? k : q;
  const void *vb = total_k > 0 ? v : q;
  if (!make_map_3d(&maps.q, q, d, H, total_q, 1, 128) || !make_map_3d(&maps.k, kb, d, Hkv, total_k, 1, 128) ||
      !make_map_3d(&maps.v, vb, d, Hkv, total_k, 1, 128))
    return ATTN_ERR_CUDA;
  PrefillOut out;
  out.o = o;
  out.lse = lse;
  out.o_b = 0;
  out.o_h = d;
  out.o_r = static_cast<long long>(H) * d;
  out.l_b = 0;
  out.l_h = 1;
  out.l_r = H;
  attn::PrefillLayout lay;
  lay.qo_indptr = qo_indptr;
  lay.kv_indptr = kv_indptr;
  lay.total_q = total_q;
  lay.total_k = total_k;
  cudaError_t e = attn::launch_prefill_bf16(maps, out, B, H, Hkv, max_q_len, 0, d, causal != 0, scale,
                                            reinterpret_cast<cudaStream_t>(stream), lay);
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

attn_status_t attn_fwd_paged(const void *q, const void *k_pages, const void *v_pages, const int32_t *page_table,
                             const int32_t *kv_lens, const int32_t *qo_indptr, void *o, float *lse, int B, int H,
                             int Hkv, int max_q_len, int total_q, int d, int page_size, int max_pages_per_seq,
                             int num_pages, int causal, float scale, attn_stream_t stream) {
  if (B < 0 || H < 0 || Hkv < 0 || max_q_len < 0 || total_q < 0 || max_pages_per_seq < 0 || num_pages < 0)
    return ATTN_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !(scale < INFINITY)) return ATTN_ERR_INVALID_ARG;
  if (B == 0 || H == 0 || max_q_len == 0 || total_q == 0) return ATTN_OK;
  if (Hkv == 0 || H % Hkv != 0) return ATTN_ERR_INVALID_ARG;
  if (q == nullptr || o == nullptr || qo_indptr == nullptr || kv_lens == nullptr) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(o) || (lse && !aligned4(lse))) return ATTN_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
  if (page_size != 16) return ATTN_ERR_UNSUPPORTED;
  const bool has_pages = max_pages_per_seq > 0 && num_pages > 0;
  if (has_pages && (k_pages == nullptr || v_pages == nullptr || page_table == nullptr)) return ATTN_ERR_INVALID_ARG;
  if (has_pages && (!aligned16(k_pages) || !aligned16(v_pages))) return ATTN_ERR_INVALID_ARG;
  PrefillMaps maps;
  maps.q_rows_outer = true;
  const void *kb = has_pages ? k_pages : q;
  const void *vb = has_pages ? v_pages : q;
  const uint64_t planes = static_cast<uint64_t>(std::max(num_pages, 1)) * Hkv;
  if (!make_map_3d(&maps.q, q, d, H, total_q, 1, 128) || !make_map_3d(&maps.k, kb, d, page_size, planes, page_size) ||
      !make_map_3d(&maps.v, vb, d, page_size, planes, page_size))
    return ATTN_ERR_CUDA;
  PrefillOut out;
  out.o = o;
  out.lse = lse;
  out.o_b = 0;
  out.o_h = d;
  out.o_r = static_cast<long long>(H) * d;
  out.l_b = 0;
  out.l_h = 1;
  out.l_r = H;
  attn::PrefillLayout lay;
  lay.qo_indptr = qo_indptr;
  lay.page_table = has_pages ? page_table : nullptr;
  lay.kv_lens = kv_lens;
  lay.max_pages = has_pages ? max_pages_per_seq : 0;
  lay.num_pages = has_pages ? num_pages : 0;
  lay.total_q = total_q;
  // with no pages at all no page is read: every sequence has zero keys (and a
  // positive kv_lens is recorded as beyond the table)
  cudaError_t e = attn::launch_prefill_bf16(maps, out, B, H, Hkv, max_q_len, 0, d, causal != 0, scale,
                                            reinterpret_cast<cudaStream_t>(stream), lay);
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

int attn_fp8_padded_keys(int Nk) { return Nk < 0 ? -1 : (Nk + 15) / 16 * 16; }

attn_status_t attn_fp8_quantize(const void *q, const void *k, const void *v, const float *signs, void *q8, void *k8,
                                void *v8t, float *q_scale, float *k_scale, float *v_scale, int B, int H, int Hkv,
                                int Nq, int Nk, int d, attn_stream_t stream) {
  if (B < 0 || H < 0 || Hkv < 0 || Nq < 0 || Nk < 0) return ATTN_ERR_INVALID_ARG;
  if (d != 128) return ATTN_ERR_UNSUPPORTED;
  const bool has_q = B > 0 && H > 0 && Nq > 0;
  const bool has_kv = B > 0 && Hkv > 0 && Nk > 0;
  if (has_q && (q == nullptr || q8 == nullptr || q_scale == nullptr)) return ATTN_ERR_INVALID_ARG;
  if (has_kv && (k == nullptr || v == nullptr || k8 == nullptr || v8t == nullptr || k_scale == nullptr ||
                 v_scale == nullptr))
    return ATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(q8) || !aligned16(k8) || !aligned16(v8t) ||
      !aligned16(signs))
    return ATTN_ERR_INVALID_ARG;
  attn::Fp8QuantJob jq, jk, jv;
  if (has_q) {
    jq.x = static_cast<const uint16_t *>(q);
    jq.out = static_cast<uint8_t *>(q8);
    jq.scale = q_scale;
    jq.planes = static_cast<long long>(B) * H;
    jq.N = Nq;
  }
  if (has_kv) {
    jk.x = static_cast<const uint16_t *>(k);
    jk.out = static_cast<uint8_t *>(k8);
    jk.scale = k_scale;
    jk.planes = static_cast<long long>(B) * Hkv;
    jk.N = Nk;
    jv = jk;
    jv.x = static_cast<const uint16_t *>(v);
    jv.out = static_cast<uint8_t *>(v8t);
    jv.scale = v_scale;
    jv.n_pad = attn_fp8_padded_keys(Nk);
  }
  cudaError_t e = attn::launch_fp8_quantize(jq, jk, jv, signs, 1.0f / sqrtf(static_cast<float>(d)),
                                            reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

attn_status_t attn_fwd_fp8(const void *q8, const void *k8, const void *v8t, const float *q_scale,
                           const float *k_scale, const float *v_scale, void *o, float *lse, int B, int H, int Hkv,
                           int Nq, int Nk, int d, int causal, float scale, attn_stream_t stream) {
  if (B < 0 || H < 0 || Hkv < 0 || Nq < 0 || Nk < 0) return ATTN_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !(scale < INFINITY)) return ATTN_ERR_INVALID_ARG;
  if (B == 0 || H == 0 || Nq == 0) return ATTN_OK;
  if (Hkv == 0 || H % Hkv != 0) return ATTN_ERR_INVALID_ARG;
  if (d != 128) return ATTN_ERR_UNSUPPORTED;
  if (q8 == nullptr || q_scale == nullptr || o == nullptr) return ATTN_ERR_INVALID_ARG;
  if (Nk > 0 && (k8 == nullptr || v8t == nullptr || k_scale == nullptr || v_scale == nullptr))
    return ATTN_ERR_INVALID_ARG;
  if (!aligned16(q8) || !aligned16(k8) || !aligned16(v8t) || !aligned16(o) || (lse && !aligned4(lse)))
    return ATTN_ERR_INVALID_ARG;
  attn::Fp8Maps maps;
  // with Nk == 0 the K/V maps are never read; they only need a valid shape
  const void *kb = Nk > 0 ? k8 : q8;
  const void *vb = Nk > 0 ? v8t : q8;
  if (!make_map_u8(&maps.q, q8, d, Nq, static_cast<uint64_t>(B) * H) ||
      !make_map_u8(&maps.k, kb, d, Nk, static_cast<uint64_t>(B) * Hkv) ||
      !make_map_u8(&maps.vt, vb, Nk > 0 ? attn_fp8_padded_keys(Nk) : 16, d, static_cast<uint64_t>(B) * Hkv))
    return ATTN_ERR_CUDA;
  PrefillOut out;
  out.o = o;
  out.lse = lse;
  out.o_b = static_cast<long long>(H) * Nq * d;
  out.o_h = static_cast<long long>(Nq) * d;
  out.o_r = d;
  out.l_b = static_cast<long long>(H) * Nq;
  out.l_h = Nq;
  out.l_r = 1;
  cudaError_t e = attn::launch_prefill_fp8(maps, q_scale, k_scale, v_scale, out, B, H, Hkv, Nq, Nk, causal != 0,
                                           scale, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

size_t attn_decode_workspace_size(int B, int H, int d, int max_splits) {
  if (B <= 0 || H <= 0 || d <= 0 || max_splits <= 0) return 0;
  return decode_ws_bytes(B, H, d, max_splits);
}

int attn_decode_max_splits(int B, int H, int Hkv, int max_pages_per_seq) {
  if (B <= 0 || H <= 0 || Hkv <= 0 || H % Hkv != 0 || max_pages_per_seq <= 0) return 0;
  return auto_splits(B, Hkv, max_pages_per_seq, device_sm_count());
}

attn_status_t attn_decode_paged(const void *q, const void *k_pages, const void *v_pages, const int32_t *page_table,
                                const int32_t *kv_lens, void *o, float *lse, int B, int H, int Hkv, int d,
                                int page_size, int max_pages_per_seq, int num_pages, float scale, int num_splits,
                                void *workspace, size_t workspace_bytes, attn_stream_t stream) {
  attn_status_t s = decode_check(q, k_pages, v_pages, page_table, kv_lens, o, lse, B, H, Hkv, d, page_size,
                                 max_pages_per_seq, num_pages, scale, workspace);
  if (s != ATTN_OK || B == 0 || H == 0) return s;
  const DecodePlan plan = decode_plan(B, Hkv, max_pages_per_seq, num_pages, num_splits);
  if (workspace_bytes < decode_ws_bytes(B, H, d, plan.splits)) return ATTN_ERR_WORKSPACE;
  if (plan.splits > 65535 || B > 65535) return ATTN_ERR_UNSUPPORTED;
  return decode_launch(plan, q, k_pages, v_pages, page_table, kv_lens, o, lse, B, H, Hkv, d, page_size,
                       max_pages_per_seq, num_pages, scale, workspace, nullptr, nullptr,
                       reinterpret_cast<cudaStream_t>(stream));
}

size_t attn_cascade_workspace_size(int B, int H, int d, int max_splits) {
  if (B <= 0 || H <= 0 || d <= 0 || max_splits <= 0) return 0;
  const size_t rows = static_cast<size_t>(B) * H;
  // the decode partials, the merged prefix partial, up to kMaxPrefixChunks chunk partials,
  // and the queries regrouped by KV head
  return decode_ws_bytes(B, H, d, max_splits) +
         (1 + kMaxPrefixChunks) * (align256(rows * d * 2) + align256(rows * sizeof(float))) + align256(rows * d * 2);
}

attn_status_t attn_cascade_decode(const void *q, const void *prefix_k, const void *prefix_v, int prefix_len,
                                  const void *k_pages, const void *v_pages, const int32_t *page_table,
                                  const int32_t *kv_lens, void *o, float *lse, int B, int H, int Hkv, int d,
                                  int page_size, int max_pages_per_seq, int num_pages, float scale, int num_splits,
                                  void *workspace, size_t workspace_bytes, attn_stream_t stream) {
  if (prefix_len < 0) return ATTN_ERR_INVALID_ARG;
  attn_status_t s = decode_check(q, k_pages, v_pages, page_table, kv_lens, o, lse, B, H, Hkv, d, page_size,
                                 max_pages_per_seq, num_pages, scale, workspace);
  if (s != ATTN_OK || B == 0 || H == 0) return s;
  if (prefix_len > 0) {
    if (prefix_k == nullptr || prefix_v == nullptr) return ATTN_ERR_INVALID_ARG;
    if (!aligned16(prefix_k) || !aligned16(prefix_v)) return ATTN_ERR_INVALID_ARG;
  }
  const DecodePlan plan = decode_plan(B, Hkv, max_pages_per_seq, num_pages, num_splits);
  if (workspace_bytes < attn_cascade_workspace_size(B, H, d, plan.splits)) return ATTN_ERR_WORKSPACE;
  if (plan.splits > 65535 || B > 65535) return ATTN_ERR_UNSUPPORTED;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);

  const size_t rows = static_cast<size_t>(B) * H;
  const size_t o_bytes = align256(rows * d * 2), l_bytes = align256(rows * sizeof(float));
  char *prefix_area = static_cast<char *>(workspace) + decode_ws_bytes(B, H, d, plan.splits);
  void *o_prefix = prefix_area;                                         // [B, H, d] bf16
  float *lse_prefix = reinterpret_cast<float *>(prefix_area + o_bytes);  // [B, H] fp32
  char *chunk_area = prefix_area + o_bytes + l_bytes;
  void *o_chunks = chunk_area;                                                                  // [C][B, H, d]
  float *lse_chunks = reinterpret_cast<float *>(chunk_area + kMaxPrefixChunks * o_bytes);       // [C][Hkv, B * g]
  void *q_grouped = chunk_area + kMaxPrefixChunks * (o_bytes + l_bytes);                        // [Hkv][B * g][d]
  if (prefix_len > 0) {
    // The shared prefix once for every request: per KV head, one attention whose query
    // rows are the B requests' g query heads of that group (B * g rows) against the
    // prefix keys, in C chunks of keys (about two CTAs per SM in all), each a
    // normalised partial, then merged into one.
    const int g = H / Hkv;
    const int q_tiles = ceil_div(ceil_div(static_cast<long long>(B) * g, 128), 2);  // query-tile pairs per KV head
    const int want = ceil_div(2LL * std::max(device_sm_count(), 1), static_cast<long long>(Hkv) * q_tiles);
    const int key_tiles = ceil_div(prefix_len, 128);
    const int c_try = std::max(1, std::min({want, key_tiles, kMaxPrefixChunks}));
    const int chunk = ceil_div(key_tiles, c_try) * 128;
    const int C = ceil_div(prefix_len, chunk);
    const int group_rows = B * g;
    PrefillMaps maps;  // Q planes are the KV heads, each with its B * g query rows
    if (!make_map_3d(&maps.q, q_grouped, d, group_rows, Hkv, 128) ||
        !make_map_3d(&maps.k, prefix_k, d, prefix_len, Hkv, 128) ||
        !make_map_3d(&maps.v, prefix_v, d, prefix_len, Hkv, 128))
      return ATTN_ERR_CUDA;
    PrefillOut out;  // chunk partials [C][Hkv][B * g][d] and [C][Hkv][B * g]
    out.o = o_chunks;
    out.lse = lse_chunks;
    out.o_b = static_cast<long long>(o_bytes / 2);
    out.o_h = static_cast<long long>(group_rows) * d;
    out.o_r = d;
    out.l_b = static_cast<long long>(l_bytes / sizeof(float));
    out.l_h = group_rows;
    out.l_r = 1;
    attn::PrefillLayout lay;
    lay.key_chunk = chunk;
    if (attn::launch_group_queries(q, q_grouped, B, H, Hkv, d, st) != cudaSuccess ||
        attn::launch_prefill_bf16(maps, out, C, Hkv, Hkv, group_rows, prefix_len, d, false, scale, st, lay) !=
            cudaSuccess ||
        attn::launch_merge_chunks(o_chunks, lse_chunks, C, static_cast<int>(rows), out.o_b, out.l_b, B, g, d,
                                  o_prefix, lse_prefix, st) != cudaSuccess)
      return ATTN_ERR_CUDA;
  }
  // each request's own suffix, merged with the prefix result as one more partial
  return decode_launch(plan, q, k_pages, v_pages, page_table, kv_lens, o, lse, B, H, Hkv, d, page_size,
                       max_pages_per_seq, num_pages, scale, workspace, prefix_len > 0 ? o_prefix : nullptr,
                       prefix_len > 0 ? lse_prefix : nullptr, st);
}

attn_status_t merge_partials(const float *m, const float *l, const float *o_tilde, const int32_t *num_parts, int B,
                             int H, int S, int d, void *o, attn_dtype_t o_dtype, float *lse, attn_stream_t stream) {
  if (B < 0 || H < 0 || S < 1) return ATTN_ERR_INVALID_ARG;
  if (o_dtype != ATTN_F32 && o_dtype != ATTN_BF16) return ATTN_ERR_INVALID_ARG;
  if (B == 0 || H == 0) return ATTN_OK;
  if (m == nullptr || l == nullptr || o_tilde == nullptr || o == nullptr) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(o_tilde) || !aligned16(o) || (lse && !aligned4(lse))) return ATTN_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
  cudaError_t e = attn::launch_merge(m, l, o_tilde, num_parts, nullptr, 0, 1, B, H, S, d, o, o_dtype == ATTN_BF16,
                                     lse, nullptr, nullptr, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

attn_status_t attn_device_error(uint32_t *code, int clear) {
  if (code == nullptr) return ATTN_ERR_INVALID_ARG;
  if (cudaDeviceSynchronize() != cudaSuccess) return ATTN_ERR_CUDA;
  unsigned int a = 0, b = 0, c = 0, f = 0, t = 0;
  if (attn::device_error_decode(&a, clear != 0) != cudaSuccess ||
      attn::device_error_prefill_f32(&b, clear != 0) != cudaSuccess ||
      attn::device_error_prefill_bf16(&c, clear != 0) != cudaSuccess ||
      attn::device_error_prefill_fp8(&f, clear != 0) != cudaSuccess ||
      attn::device_error_selftest(&t, clear != 0) != cudaSuccess)
    return ATTN_ERR_CUDA;
  *code = a | b | c | f | t;
  return ATTN_OK;
}

attn_status_t attn_selftest_wait_timeout(int32_t *gave_up, attn_stream_t stream) {
  if (gave_up == nullptr) return ATTN_ERR_INVALID_ARG;
  return attn::launch_wait_timeout_selftest(gave_up, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? ATTN_OK
             : ATTN_ERR_CUDA;
}

attn_status_t attn_clock_probe(uint64_t *out, const uint64_t *match, attn_stream_t stream) {
  if (out == nullptr || (reinterpret_cast<uintptr_t>(out) & 7u) != 0 ||
      (match != nullptr && (reinterpret_cast<uintptr_t>(match) & 7u) != 0))
    return ATTN_ERR_INVALID_ARG;
  // without `match` one block records on whichever SM runs it; with `match`, every SM gets
  // blocks so that one of them runs on the recorded SM (the others return at once)
  const int blocks = match == nullptr ? 1 : 16 * std::max(device_sm_count(), 1);
  return attn::launch_clock_probe(reinterpret_cast<unsigned long long *>(out),
                                  reinterpret_cast<const unsigned long long *>(match), blocks,
                                  reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? ATTN_OK
             : ATTN_ERR_CUDA;
}

}  // extern "C"
