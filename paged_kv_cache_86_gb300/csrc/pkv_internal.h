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

// fp8 E4M3 caches [NB, bs, Hkv, 128] uint8 with fp32 scales [NB * bs, Hkv];
// head_dim 128; strides in elements of the bf16 key/value rows.
cudaError_t launch_store_kvcache_fp8(const void *key, const void *value, void *k_cache,
                                     void *v_cache, float *k_scales, float *v_scales,
                                     const int32_t *slot_mapping, int32_t num_tokens,
                                     int32_t num_kv_heads, int64_t key_stride, int64_t value_stride,
                                     int64_t num_slots, uint32_t *err, cudaStream_t stream);

// ---- block copy (copy-on-write)
cudaError_t launch_copy_blocks(void *k_cache, void *v_cache, const int32_t *src,
                               const int32_t *dst, const int32_t *rows, int32_t num_pairs,
                               int32_t block_size, int32_t num_blocks, int32_t row_elems,
                               uint32_t *err, cudaStream_t stream);

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
  // Decode step only (nullptr otherwise): the newest token of each sequence,
  // [num_seqs, Hkv, 128] bf16 rows with these token strides in elements, is
  // written to the cache at logical position min(context_len, max_context_len) - 1
  // before it is attended to.
  const void *key_new = nullptr;
  const void *value_new = nullptr;
  int64_t key_stride = 0;
  int64_t value_stride = 0;
  // mixed batch: a prefill launched between the tcgen05 attention kernel and
  // the combine, so that it fills the SMs the attention kernel's tail leaves
  // (nullptr otherwise)
  const struct PrefillArgs *interleave = nullptr;
  // all-heads tcgen05 kernel: CTAs to launch instead of one per SM (0: one per
  // SM), leaving the other SMs to a kernel that runs beside it
  int grid_override = 0;
  // fp8 E4M3 caches (uint8 codes) with fp32 row scales [NB * bs, Hkv]
  bool fp8 = false;
  const float *k_scales = nullptr;
  const float *v_scales = nullptr;
};

// Context lengths of the decode sequences 0..D-1 of a mixed batch from
// cu_seqlens_k (checks that each has exactly one query row).
cudaError_t launch_mixed_decode_lens(const int32_t *cu_q, const int32_t *cu_k, int num_decode,
                                     int32_t *lens, uint32_t *err, cudaStream_t stream);

// Which decode kernel runs and on how many CTAs. Block sizes that are a
// multiple of 8 (and at most 16 query heads per KV head) run the tcgen05
// kernel; other shapes the CUDA-core split kernel.
struct DecodePlan {
  int kind;  // 3: tcgen05, all KV heads per stage; 2: tcgen05, one KV head per CTA range; 1: CUDA cores
  bool tc;   // records keyed by (slot, query head of the group) -- kind 2 only
  int grid;
};

bool choose_decode_plan(int num_q_heads, int num_kv_heads, int block_size, DecodePlan *plan,
                        cudaError_t *status, bool fp8 = false);
size_t decode_workspace_bytes(int num_seqs, int num_q_heads, int num_kv_heads,
                              const DecodePlan &plan);
// The largest workspace any block size needs for this head configuration.
size_t decode_workspace_upper_bound(int num_seqs, int num_q_heads, int num_kv_heads,
                                    cudaError_t *status);
cudaError_t launch_paged_decode(const DecodeArgs &a, const DecodePlan &plan, cudaStream_t stream);

// tcgen05 decode kernel, all KV heads of a block per stage (decode_tcg.cu)
bool decode_tcg_supported(int num_q_heads, int num_kv_heads, int block_size, bool fp8 = false);
// The all-heads tcgen05 decode kernel splits the concatenated contexts into
// equal CTA ranges; every sequence segment a CTA handles also costs a fixed
// amount of time (its first stage's Q load and reference maximum, its last
// stage's row sums, output rows and partly filled stage). The plan counts that
// cost as this many extra tokens in front of each non-empty sequence, so that
// a CTA given many short sequences gets fewer tokens. Measured on GB300 over
// 0, 16, 32, 64 and 128: 64 was best for the 512-sequence lognormal batch
// (386 -> 378 us) and near best for 8 x 32768 + 248 x 200 (230 -> 206 us).
constexpr int kDecodeSegmentCost = 64;

// seg_cost: extra units in front of each non-empty sequence's tokens in the
// flat space the CTA ranges cut. The kernel plans the call itself (every CTA
// computes the prefix sums; CTA 0 leaves them in the workspace for the
// combine, the others in cu_copies, cu_stride ints apart) and writes a decode
// step's new rows (decode.cu, launch_paged_decode).
cudaError_t launch_decode_tcg(const DecodeArgs &a, int grid, float2 *ml, float *po, int seg_cost,
                              int *cu_copies, int cu_stride, cudaStream_t stream);
// ints between the per-CTA prefix-sum copies of the tcgen05 decode kernel
inline int tcg_cu_stride(int num_seqs) { return (num_seqs + 1 + 63) / 64 * 64; }

// tcgen05 decode kernel, one KV head per CTA range (decode_tc.cu)
bool decode_tc_supported(int num_q_heads, int num_kv_heads, int block_size);
int decode_tc_grid();
cudaError_t launch_decode_tc(const DecodeArgs &a, int grid, float2 *ml, float *po,
                             cudaStream_t stream);

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
  // kPrefillWorkspace bytes of device scratch (the work ticket of the
  // persistent kernel), 256-byte aligned
  void *workspace = nullptr;
  // the caller has zeroed the work ticket already (earlier on the stream)
  bool ticket_zeroed = false;
  // launch as a programmatic dependent of the previous kernel on the stream
  // without waiting for it: the caller guarantees that the prefill reads
  // nothing that kernel writes. The kernel still waits for it before it
  // exits, so a later dependent sees both finished.
  bool overlap_previous = false;
  // CTAs of the persistent kernel (0: one per SM); items are claimed from the
  // work ticket, so two launches sharing one ticket split the items between them
  int max_ctas = 0;
};

constexpr size_t kPrefillWorkspace = 256;

bool prefill_supported(int num_q_heads, int num_kv_heads, int block_size);
cudaError_t launch_paged_prefill(const PrefillArgs &a, cudaStream_t stream);

// two query heads per CTA in ping-pong (prefill_pp.cu): even GQA groups
bool prefill_pp_supported(int num_q_heads, int num_kv_heads, int block_size);
cudaError_t launch_prefill_pp(const PrefillArgs &a, cudaStream_t stream);

}  // namespace pkv
