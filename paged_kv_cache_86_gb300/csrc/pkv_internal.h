// pkv_internal.h -- launchers shared between the C ABI (api.cu) and the kernel
// translation units. Host-side only; argument checking happens in api.cu.
#pragma once

#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>

#include "pkv.h"

namespace pkv {

// Device error word of the current device (lazily resolved, cached per device).
uint32_t *device_error_word(cudaError_t *status);

int sm_count(int device);

// ---- store
cudaError_t launch_store_kvcache(const void *key, const void *value, void *k_cache, void *v_cache,
                                 const int32_t *slot_mapping, int32_t num_tokens,
                                 int32_t row_elems, int64_t key_stride, int64_t value_stride,
                                 int64_t num_slots, uint32_t *err, cudaStream_t stream);

// ---- decode
struct DecodeArgs {
  void *out;
  const void *q;
  const void *k_cache;
  const void *v_cache;
  const int32_t *block_tables;
  int32_t max_blocks_per_seq;
  const int32_t *context_lens;
  int32_t num_seqs;
  int32_t max_context_len;
  int32_t num_q_heads;
  int32_t num_kv_heads;
  int32_t block_size;
  int32_t num_blocks;
  float scale;
  void *workspace;
  size_t workspace_bytes;
  uint32_t *err;
};

// Grid size (CTAs) of the split-decode kernel for this head configuration on
// the current device, or 0 if the configuration is unsupported.
int decode_grid(int num_q_heads, int num_kv_heads, cudaError_t *status);
size_t decode_workspace_bytes(int num_seqs, int num_q_heads, int num_kv_heads, int grid);
cudaError_t launch_paged_decode(const DecodeArgs &a, int grid, cudaStream_t stream);

// ---- prefill
struct PrefillArgs {
  void *out;
  const void *q;
  const void *k_cache;
  const void *v_cache;
  const int32_t *cu_seqlens_q;
  const int32_t *cu_seqlens_k;
  int32_t max_seqlen_q;
  int32_t max_seqlen_k;
  const int32_t *block_tables;
  int32_t max_blocks_per_seq;
  int32_t num_seqs;
  int32_t total_q;
  int32_t num_q_heads;
  int32_t num_kv_heads;
  int32_t block_size;
  int32_t num_blocks;
  float scale;
  int32_t causal;
  uint32_t *err;
};

bool prefill_supported(int num_q_heads, int num_kv_heads, int block_size);
cudaError_t launch_paged_prefill(const PrefillArgs &a, cudaStream_t stream);

}  // namespace pkv
