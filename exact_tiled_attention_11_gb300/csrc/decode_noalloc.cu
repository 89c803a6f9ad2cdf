// attn_decode_paged_noalloc: paged split-KV decode for callers that cannot
// allocate device memory.
//
// Some callers have no way to provide the decode workspace: code running as a
// plugin or custom op inside another runtime that hands it only its input and
// output buffers (no allocator, no workspace hook), and latency-critical
// serving loops that must not call cudaMalloc, which can synchronise the
// device and stall every other stream.  For them the per-chunk partials live
// in one fixed array in device global memory that is part of this library
// (ATTN_DECODE_NOALLOC_SCRATCH_BYTES, held by every GPU that loads the library
// until the process exits), and this entry point forwards to
// attn_decode_paged with that array as the workspace.  Nothing here calls
// cudaMalloc, cudaFree or any allocating routine.
#include <mutex>

#include <cuda_runtime.h>

#include "attn.h"

namespace {

constexpr size_t kScratchBytes = ATTN_DECODE_NOALLOC_SCRATCH_BYTES;

// The decode partials (m, l, o~) of every call to attn_decode_paged_noalloc.
static __device__ __align__(256) unsigned char g_decode_scratch[kScratchBytes];

// Device address of g_decode_scratch, per device.  In host code the name
// g_decode_scratch is only a host-side stand-in for the symbol, never a
// device address; the real address comes from cudaGetSymbolAddress with the
// device current.  It is looked up once per device and kept, so it is valid
// only while that device's primary context lives (no cudaDeviceReset between
// calls).
constexpr int kMaxDevices = 128;
std::mutex g_mutex;
void *g_scratch_addr[kMaxDevices] = {};

attn_status_t scratch_on_current_device(void **out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return ATTN_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (g_scratch_addr[dev] == nullptr) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr) return ATTN_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return ATTN_OK;
}

}  // namespace

extern "C" attn_status_t attn_decode_paged_noalloc(const void *q, const void *k_pages, const void *v_pages,
                                                   const int32_t *page_table, const int32_t *kv_lens, void *o,
                                                   float *lse, int B, int H, int Hkv, int d, int page_size,
                                                   int max_pages_per_seq, int num_pages, float scale, int num_splits,
                                                   attn_stream_t stream) {
  void *scratch = nullptr;
  const attn_status_t s = scratch_on_current_device(&scratch);
  if (s != ATTN_OK) return s;
  // attn_decode_paged returns ATTN_ERR_WORKSPACE, before launching anything,
  // when the partials of this request do not fit in the fixed array.
  return attn_decode_paged(q, k_pages, v_pages, page_table, kv_lens, o, lse, B, H, Hkv, d, page_size,
                           max_pages_per_seq, num_pages, scale, num_splits, scratch, kScratchBytes, stream);
}
