// Internal host-side launchers, one per kernel family (not part of the C ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace attn {

// decode.cu
size_t decode_smem_bytes();
cudaError_t launch_decode_split(const CUtensorMap &tm_k, const CUtensorMap &tm_v, const void *q,
                                const int32_t *page_table, const int32_t *kv_lens, float *ws_m, float *ws_l,
                                float *ws_o, int B, int H, int Hkv, int max_pages, int num_pages, int chunk_pages,
                                int S, float scale, cudaStream_t stream);
cudaError_t launch_merge(const float *m, const float *l, const float *o_tilde, const int32_t *num_parts,
                         const int32_t *kv_lens, int page_size, int chunk_pages, int B, int H, int S, int d, void *o,
                         bool out_bf16, float *lse, cudaStream_t stream);

// prefill_f32.cu
cudaError_t launch_prefill_f32(const float *q, const float *k, const float *v, float *o, float *lse, int B, int H,
                               int Hkv, int N, int d, bool causal, float scale, cudaStream_t stream);

// prefill_bf16.cu
struct PrefillMaps {
  CUtensorMap q, k, v;
};
cudaError_t launch_prefill_bf16(const PrefillMaps &maps, void *o, float *lse, int B, int H, int Hkv, int N, int d,
                                bool causal, float scale, int num_sms, cudaStream_t stream);

// Per-translation-unit device error words (see common.cuh).
cudaError_t device_error_decode(unsigned int *value, bool clear);
cudaError_t device_error_prefill_f32(unsigned int *value, bool clear);
cudaError_t device_error_prefill_bf16(unsigned int *value, bool clear);

}  // namespace attn
