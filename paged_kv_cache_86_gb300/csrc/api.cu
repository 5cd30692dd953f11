// api.cu -- the extern "C" entry points of libpkv: host-side argument checks,
// workspace sizing and kernel launches on the caller's stream. The contract of
// each call is documented in include/pkv.h.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "pkv.h"
#include "pkv_internal.h"

namespace {

__device__ uint32_t g_device_errors;  // PKV_DEVERR_* bits, one word per device

constexpr int kMaxDevices = 64;
std::mutex g_mu;
uint32_t *g_err_ptr[kMaxDevices] = {};
int g_sms[kMaxDevices] = {};

// The share of the SMs a mixed round gives to the prefill launch that runs
// beside its decode kernel: kMixedSideGain times the prefill's share of an
// estimate of the round's work -- with equal key counts per query row, decode
// moves Hkv * 512 bytes per sequence and key at ~45 GB/s per SM, and prefill
// does Hq * 512 flops per chunk row and key at ~8.5 TFLOP/s per SM -- capped at
// kMixedSideMax. The estimate undercounts the prefill's share (the decode kernel
// keeps most of its bandwidth on fewer SMs, and the prefill launch after the
// decode kernel takes what is left), hence the gain, set by measurement.
constexpr float kMixedSideGain = 1.6f;
constexpr float kMixedSideMax = 0.45f;

float mixed_side_share(int num_decode, int64_t chunk_rows, int num_q_heads, int num_kv_heads) {
  const double dec = double(num_decode) * num_kv_heads * 512.0 / 45e9;
  const double pre = double(chunk_rows) * num_q_heads * 512.0 / 8.5e12;
  if (dec + pre <= 0.0) return 0.f;
  const double share = kMixedSideGain * pre / (dec + pre);
  return static_cast<float>(share < kMixedSideMax ? share : kMixedSideMax);
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// A second stream per device on which a mixed round runs part of its prefill
// beside the decode kernel, forked from and joined back into the caller's
// stream by two events. Created on first use; the fork-launch-join sequence
// is issued under g_side_mu so that concurrent callers do not interleave their
// event records.
struct SideStream {
  cudaStream_t stream = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
};
std::mutex g_side_mu;
SideStream g_side[kMaxDevices];

cudaError_t side_stream_locked(int dev, SideStream **out) {
  SideStream &s = g_side[dev];
  if (s.stream == nullptr) {
    cudaError_t e = cudaStreamCreateWithFlags(&s.stream, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&s.fork, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&s.join, cudaEventDisableTiming);
    if (e != cudaSuccess) return e;
  }
  *out = &s;
  return cudaSuccess;
}

pkv_status from_cuda(cudaError_t e) { return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA; }

}  // namespace

namespace pkv {

uint32_t *device_error_word(cudaError_t *status) {
  int dev = 0;
  *status = cudaGetDevice(&dev);
  if (*status != cudaSuccess) return nullptr;
  if (dev < 0 || dev >= kMaxDevices) {
    *status = cudaErrorInvalidDevice;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_err_ptr[dev] == nullptr) {
    void *p = nullptr;
    *status = cudaGetSymbolAddress(&p, g_device_errors);
    if (*status != cudaSuccess) return nullptr;
    g_err_ptr[dev] = static_cast<uint32_t *>(p);
  }
  return g_err_ptr[dev];
}

int sm_count(int device) {
  if (device < 0 || device >= kMaxDevices) return 0;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_sms[device] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, device) == cudaSuccess)
      g_sms[device] = n;
  }
  return g_sms[device];
}

}  // namespace pkv

extern "C" {

pkv_status pkv_store_kvcache(const void *key, const void *value, void *k_cache, void *v_cache,
                             const int32_t *slot_mapping, int32_t num_tokens,
                             int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                             int32_t num_blocks, int64_t key_token_stride,
                             int64_t value_token_stride, pkv_dtype dtype, void *stream) {
  if (dtype != PKV_BF16) return PKV_ERR_DTYPE;
  if (num_tokens < 0 || num_kv_heads < 1 || head_dim < 1 || block_size < 1 || num_blocks < 1)
    return PKV_ERR_ARG;
  const int64_t row = int64_t(num_kv_heads) * head_dim;
  if (row % 8 != 0) return PKV_ERR_SHAPE;
  if (num_tokens == 0) return PKV_OK;
  if (!key || !value || !k_cache || !v_cache || !slot_mapping) return PKV_ERR_ARG;
  if (!aligned16(key) || !aligned16(value) || !aligned16(k_cache) || !aligned16(v_cache))
    return PKV_ERR_ARG;
  if (key_token_stride < row || value_token_stride < row || key_token_stride % 8 != 0 ||
      value_token_stride % 8 != 0)
    return PKV_ERR_ARG;
  cudaError_t e;
  uint32_t *err = pkv::device_error_word(&e);
  if (!err) return PKV_ERR_CUDA;
  e = pkv::launch_store_kvcache(key, value, k_cache, v_cache, slot_mapping, num_tokens,
                                static_cast<int32_t>(row), key_token_stride, value_token_stride,
                                int64_t(num_blocks) * block_size, err,
                                static_cast<cudaStream_t>(stream));
  return from_cuda(e);
}

pkv_status pkv_copy_blocks(void *k_cache, void *v_cache, const int32_t *src_block_ids,
                           const int32_t *dst_block_ids, const int32_t *num_rows,
                           int32_t num_pairs, int32_t num_kv_heads, int32_t head_dim,
                           int32_t block_size, int32_t num_blocks, pkv_dtype dtype, void *stream) {
  if (dtype != PKV_BF16) return PKV_ERR_DTYPE;
  if (num_pairs < 0 || num_pairs > 65535 || num_kv_heads < 1 || head_dim < 1 || block_size < 1 ||
      num_blocks < 1)
    return PKV_ERR_ARG;
  const int64_t row = int64_t(num_kv_heads) * head_dim;
  if (row % 8 != 0) return PKV_ERR_SHAPE;
  if (num_pairs == 0) return PKV_OK;
  if (!k_cache || !v_cache || !src_block_ids || !dst_block_ids) return PKV_ERR_ARG;
  if (!aligned16(k_cache) || !aligned16(v_cache)) return PKV_ERR_ARG;
  cudaError_t e;
  uint32_t *err = pkv::device_error_word(&e);
  if (!err) return PKV_ERR_CUDA;
  return from_cuda(pkv::launch_copy_blocks(k_cache, v_cache, src_block_ids, dst_block_ids,
                                           num_rows, num_pairs, block_size, num_blocks,
                                           static_cast<int32_t>(row), err,
                                           static_cast<cudaStream_t>(stream)));
}

pkv_status pkv_store_kvcache_fp8(const void *key, const void *value, void *k_cache, void *v_cache,
                                 float *k_scales, float *v_scales, const int32_t *slot_mapping,
                                 int32_t num_tokens, int32_t num_kv_heads, int32_t head_dim,
                                 int32_t block_size, int32_t num_blocks, int64_t key_token_stride,
                                 int64_t value_token_stride, void *stream) {
  if (num_tokens < 0 || num_kv_heads < 1 || block_size < 1 || num_blocks < 1) return PKV_ERR_ARG;
  if (head_dim != 128) return PKV_ERR_SHAPE;
  const int64_t row = int64_t(num_kv_heads) * head_dim;
  if (num_tokens == 0) return PKV_OK;
  if (!key || !value || !k_cache || !v_cache || !k_scales || !v_scales || !slot_mapping)
    return PKV_ERR_ARG;
  if (!aligned16(key) || !aligned16(value) || !aligned16(k_cache) || !aligned16(v_cache) ||
      !aligned16(k_scales) || !aligned16(v_scales))
    return PKV_ERR_ARG;
  if (key_token_stride < row || value_token_stride < row || key_token_stride % 8 != 0 ||
      value_token_stride % 8 != 0)
    return PKV_ERR_ARG;
  cudaError_t e;
  uint32_t *err = pkv::device_error_word(&e);
  if (!err) return PKV_ERR_CUDA;
  return from_cuda(pkv::launch_store_kvcache_fp8(key, value, k_cache, v_cache, k_scales, v_scales,
                                                 slot_mapping, num_tokens, num_kv_heads,
                                                 key_token_stride, value_token_stride,
                                                 int64_t(num_blocks) * block_size, err,
                                                 static_cast<cudaStream_t>(stream)));
}

size_t pkv_decode_workspace_size(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                                 int32_t head_dim) {
  if (num_seqs < 0 || num_q_heads < 1 || num_kv_heads < 1 || head_dim != 128 ||
      num_q_heads % num_kv_heads != 0)
    return 0;
  cudaError_t e;
  return pkv::decode_workspace_upper_bound(num_seqs, num_q_heads, num_kv_heads, &e);
}

}  // extern "C"

namespace {

// Shared body of pkv_paged_decode and pkv_decode_step (key_new == nullptr for the former).
pkv_status decode_call(void *out, const void *q, const void *key_new, const void *value_new,
                       int64_t key_stride, int64_t value_stride, const void *k_cache,
                       const void *v_cache, const int32_t *block_tables,
                       int32_t max_blocks_per_seq, const int32_t *context_lens, int32_t num_seqs,
                       int32_t max_context_len, int32_t num_q_heads, int32_t num_kv_heads,
                       int32_t head_dim, int32_t block_size, int32_t num_blocks, float scale,
                       void *workspace, size_t workspace_bytes, pkv_dtype dtype, void *stream,
                       const float *k_scales = nullptr, const float *v_scales = nullptr) {
  if (dtype != PKV_BF16) return PKV_ERR_DTYPE;
  const bool fp8 = k_scales != nullptr || v_scales != nullptr;
  if (fp8 && (!k_scales || !v_scales || !aligned16(k_scales) || !aligned16(v_scales)))
    return PKV_ERR_ARG;
  if (num_seqs < 0 || num_q_heads < 1 || num_kv_heads < 1 || block_size < 1 || num_blocks < 1 ||
      max_blocks_per_seq < 0 || max_context_len < 0 || !std::isfinite(scale))
    return PKV_ERR_ARG;
  if (head_dim != 128) return PKV_ERR_SHAPE;
  if (int64_t(max_context_len) > int64_t(max_blocks_per_seq) * block_size) return PKV_ERR_ARG;
  // the flat space the CTA ranges cut (int32 on the device): every token, once
  // per KV head on the per-head kernel, plus the per-segment units of the plan
  if (int64_t(num_seqs) * (int64_t(max_context_len) + pkv::kDecodeSegmentCost) * num_kv_heads >=
      (int64_t(1) << 31))
    return PKV_ERR_ARG;
  if (num_seqs == 0) return PKV_OK;
  if (!out || !q || !k_cache || !v_cache || !context_lens ||
      (!block_tables && max_blocks_per_seq > 0))
    return PKV_ERR_ARG;
  if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache))
    return PKV_ERR_ARG;
  if (key_new != nullptr || value_new != nullptr) {
    const int64_t row = int64_t(num_kv_heads) * head_dim;
    if (!key_new || !value_new || !aligned16(key_new) || !aligned16(value_new) ||
        key_stride < row || value_stride < row || key_stride % 8 != 0 || value_stride % 8 != 0)
      return PKV_ERR_ARG;
  }
  cudaError_t e;
  pkv::DecodePlan plan;
  if (num_q_heads % num_kv_heads != 0) return PKV_ERR_SHAPE;
  if (!pkv::choose_decode_plan(num_q_heads, num_kv_heads, block_size, &plan, &e, fp8))
    return e != cudaSuccess ? PKV_ERR_CUDA : PKV_ERR_SHAPE;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 ||
      workspace_bytes < pkv::decode_workspace_bytes(num_seqs, num_q_heads, num_kv_heads, plan))
    return PKV_ERR_WORKSPACE;
  uint32_t *err = pkv::device_error_word(&e);
  if (!err) return PKV_ERR_CUDA;
  pkv::DecodeArgs a;
  a.out = out;
  a.q = q;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.block_tables = block_tables;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.context_lens = context_lens;
  a.num_seqs = num_seqs;
  a.max_context_len = max_context_len;
  a.num_q_heads = num_q_heads;
  a.num_kv_heads = num_kv_heads;
  a.block_size = block_size;
  a.num_blocks = num_blocks;
  a.scale = scale;
  a.workspace = workspace;
  a.workspace_bytes = workspace_bytes;
  a.err = err;
  a.key_new = key_new;
  a.value_new = value_new;
  a.key_stride = key_stride;
  a.value_stride = value_stride;
  a.fp8 = fp8;
  a.k_scales = k_scales;
  a.v_scales = v_scales;
  return from_cuda(pkv::launch_paged_decode(a, plan, static_cast<cudaStream_t>(stream)));
}

}  // namespace

extern "C" {

pkv_status pkv_paged_decode(void *out, const void *q, const void *k_cache, const void *v_cache,
                            const int32_t *block_tables, int32_t max_blocks_per_seq,
                            const int32_t *context_lens, int32_t num_seqs,
                            int32_t max_context_len, int32_t num_q_heads, int32_t num_kv_heads,
                            int32_t head_dim, int32_t block_size, int32_t num_blocks, float scale,
                            void *workspace, size_t workspace_bytes, pkv_dtype dtype,
                            void *stream) {
  return decode_call(out, q, nullptr, nullptr, 0, 0, k_cache, v_cache, block_tables,
                     max_blocks_per_seq, context_lens, num_seqs, max_context_len, num_q_heads,
                     num_kv_heads, head_dim, block_size, num_blocks, scale, workspace,
                     workspace_bytes, dtype, stream);
}

pkv_status pkv_paged_decode_fp8(void *out, const void *q, const void *k_cache, const void *v_cache,
                                const float *k_scales, const float *v_scales,
                                const int32_t *block_tables, int32_t max_blocks_per_seq,
                                const int32_t *context_lens, int32_t num_seqs,
                                int32_t max_context_len, int32_t num_q_heads, int32_t num_kv_heads,
                                int32_t head_dim, int32_t block_size, int32_t num_blocks,
                                float scale, void *workspace, size_t workspace_bytes,
                                void *stream) {
  if (num_seqs > 0 && (!k_scales || !v_scales)) return PKV_ERR_ARG;
  return decode_call(out, q, nullptr, nullptr, 0, 0, k_cache, v_cache, block_tables,
                     max_blocks_per_seq, context_lens, num_seqs, max_context_len, num_q_heads,
                     num_kv_heads, head_dim, block_size, num_blocks, scale, workspace,
                     workspace_bytes, PKV_BF16, stream, k_scales, v_scales);
}

pkv_status pkv_decode_step(void *out, const void *q, const void *key_new, const void *value_new,
                           int64_t key_token_stride, int64_t value_token_stride, void *k_cache,
                           void *v_cache, const int32_t *block_tables, int32_t max_blocks_per_seq,
                           const int32_t *context_lens, int32_t num_seqs, int32_t max_context_len,
                           int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                           int32_t block_size, int32_t num_blocks, float scale, void *workspace,
                           size_t workspace_bytes, pkv_dtype dtype, void *stream) {
  if (num_seqs > 0 && (!key_new || !value_new)) return PKV_ERR_ARG;
  return decode_call(out, q, key_new, value_new, key_token_stride, value_token_stride, k_cache,
                     v_cache, block_tables, max_blocks_per_seq, context_lens, num_seqs,
                     max_context_len, num_q_heads, num_kv_heads, head_dim, block_size,
                     num_blocks, scale, workspace, workspace_bytes, dtype, stream);
}

pkv_status pkv_decode_step_fp8(void *out, const void *q, const void *key_new,
                               const void *value_new, int64_t key_token_stride,
                               int64_t value_token_stride, void *k_cache, void *v_cache,
                               float *k_scales, float *v_scales, const int32_t *block_tables,
                               int32_t max_blocks_per_seq, const int32_t *context_lens,
                               int32_t num_seqs, int32_t max_context_len, int32_t num_q_heads,
                               int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                               int32_t num_blocks, float scale, void *workspace,
                               size_t workspace_bytes, void *stream) {
  if (num_seqs > 0 && (!key_new || !value_new || !k_scales || !v_scales)) return PKV_ERR_ARG;
  return decode_call(out, q, key_new, value_new, key_token_stride, value_token_stride, k_cache,
                     v_cache, block_tables, max_blocks_per_seq, context_lens, num_seqs,
                     max_context_len, num_q_heads, num_kv_heads, head_dim, block_size,
                     num_blocks, scale, workspace, workspace_bytes, PKV_BF16, stream, k_scales,
                     v_scales);
}

size_t pkv_mixed_workspace_size(int32_t num_decode_seqs, int32_t num_q_heads,
                                int32_t num_kv_heads, int32_t head_dim) {
  if (num_decode_seqs < 0 || num_q_heads < 1 || num_kv_heads < 1 || head_dim != 128 ||
      num_q_heads % num_kv_heads != 0)
    return 0;
  const size_t lens = (sizeof(int32_t) * (size_t(num_decode_seqs) + 1) + 255) & ~size_t(255);
  if (num_decode_seqs == 0) return lens + pkv::kPrefillWorkspace;
  cudaError_t e;
  const size_t dec = pkv::decode_workspace_upper_bound(num_decode_seqs, num_q_heads, num_kv_heads, &e);
  return dec == 0 ? 0 : lens + dec + pkv::kPrefillWorkspace;
}

namespace {
// The persistent prefill kernel numbers its work items (a 128-row query tile
// of two heads, or two tiles of one head for an odd GQA group, per sequence)
// in 32 bits; shapes with more items than that are refused.
bool prefill_items_fit(int32_t max_seqlen_q, int32_t num_q_heads, int32_t num_kv_heads,
                       int32_t num_seqs) {
  const int64_t q_tiles = (int64_t(max_seqlen_q) + 127) / 128;
  const bool pair_tiles = (num_q_heads / num_kv_heads) % 2 != 0;
  const int64_t items = pair_tiles ? (q_tiles + 1) / 2 * num_q_heads * int64_t(num_seqs)
                                   : q_tiles * (num_q_heads / 2) * int64_t(num_seqs);
  return items < (int64_t(1) << 31);
}
}  // namespace

pkv_status pkv_mixed_step(void *out, const void *q, const void *key, const void *value,
                          const int32_t *slot_mapping, int64_t key_token_stride,
                          int64_t value_token_stride, void *k_cache, void *v_cache,
                          const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k,
                          int32_t max_seqlen_q, int32_t max_seqlen_k,
                          const int32_t *block_tables, int32_t max_blocks_per_seq,
                          int32_t num_seqs, int32_t num_decode_seqs, int32_t total_q,
                          int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                          int32_t block_size, int32_t num_blocks, float scale, void *workspace,
                          size_t workspace_bytes, pkv_dtype dtype, void *stream) {
  if (dtype != PKV_BF16) return PKV_ERR_DTYPE;
  if (num_seqs < 0 || num_decode_seqs < 0 || num_decode_seqs > num_seqs || total_q < 0 ||
      num_q_heads < 1 || num_kv_heads < 1 || block_size < 1 || num_blocks < 1 ||
      max_blocks_per_seq < 0 || max_seqlen_q < 0 || max_seqlen_k < 0 || !std::isfinite(scale))
    return PKV_ERR_ARG;
  if (head_dim != 128) return PKV_ERR_SHAPE;
  if (num_q_heads % num_kv_heads != 0) return PKV_ERR_SHAPE;
  if (int64_t(max_seqlen_k) > int64_t(max_blocks_per_seq) * block_size) return PKV_ERR_ARG;
  if (total_q < num_decode_seqs || num_seqs - num_decode_seqs > 65535) return PKV_ERR_ARG;
  if ((int64_t(max_seqlen_q) + 127) / 128 > 65535) return PKV_ERR_ARG;
  if (!prefill_items_fit(max_seqlen_q, num_q_heads, num_kv_heads, num_seqs - num_decode_seqs))
    return PKV_ERR_ARG;
  if (num_seqs == 0 || total_q == 0) return PKV_OK;
  if (!out || !q || !key || !value || !slot_mapping || !k_cache || !v_cache || !cu_seqlens_q ||
      !cu_seqlens_k || !block_tables || !workspace)
    return PKV_ERR_ARG;
  if (!aligned16(out) || !aligned16(q) || !aligned16(key) || !aligned16(value) ||
      !aligned16(k_cache) || !aligned16(v_cache) || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return PKV_ERR_ARG;
  const int64_t row = int64_t(num_kv_heads) * head_dim;
  if (key_token_stride < row || value_token_stride < row || key_token_stride % 8 != 0 ||
      value_token_stride % 8 != 0)
    return PKV_ERR_ARG;
  const int num_prefill = num_seqs - num_decode_seqs;
  if (num_prefill > 0 && !pkv::prefill_supported(num_q_heads, num_kv_heads, block_size))
    return PKV_ERR_SHAPE;
  cudaError_t e;
  pkv::DecodePlan plan{};
  if (num_decode_seqs > 0 &&
      !pkv::choose_decode_plan(num_q_heads, num_kv_heads, block_size, &plan, &e))
    return e != cudaSuccess ? PKV_ERR_CUDA : PKV_ERR_SHAPE;
  const size_t lens_bytes = (sizeof(int32_t) * (size_t(num_decode_seqs) + 1) + 255) & ~size_t(255);
  const size_t dec_bytes = num_decode_seqs > 0
      ? pkv::decode_workspace_bytes(num_decode_seqs, num_q_heads, num_kv_heads, plan) : 0;
  const size_t dec_aligned = (dec_bytes + 255) & ~size_t(255);
  if (workspace_bytes < lens_bytes + dec_aligned + pkv::kPrefillWorkspace) return PKV_ERR_WORKSPACE;
  uint32_t *err = pkv::device_error_word(&e);
  if (!err) return PKV_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // the prefill chunks D..S-1 (their query rows are absolute offsets in cu_seqlens_q)
  pkv::PrefillArgs pa;
  pa.out = out;
  pa.q = q;
  pa.k_cache = k_cache;
  pa.v_cache = v_cache;
  pa.cu_seqlens_q = cu_seqlens_q + num_decode_seqs;
  pa.cu_seqlens_k = cu_seqlens_k + num_decode_seqs;
  pa.max_seqlen_q = max_seqlen_q;
  pa.max_seqlen_k = max_seqlen_k;
  pa.block_tables = block_tables + static_cast<int64_t>(num_decode_seqs) * max_blocks_per_seq;
  pa.max_blocks_per_seq = max_blocks_per_seq;
  pa.num_seqs = num_prefill;
  pa.total_q = total_q;
  pa.num_q_heads = num_q_heads;
  pa.num_kv_heads = num_kv_heads;
  pa.block_size = block_size;
  pa.num_blocks = num_blocks;
  pa.scale = scale;
  pa.causal = 1;
  pa.err = err;
  pa.workspace = static_cast<uint8_t *>(workspace) + lens_bytes + dec_aligned;
  // With the all-heads decode kernel the prefill is launched between it and
  // the combine, overlapping its tail: it reads only the caches, which the
  // store below has finished writing before the decode's first kernel starts.
  const bool interleave = num_prefill > 0 && num_decode_seqs > 0 && plan.kind == 3 &&
                          pkv::prefill_pp_supported(num_q_heads, num_kv_heads, block_size);
  if (interleave) {
    if ((e = cudaMemsetAsync(pa.workspace, 0, sizeof(uint32_t), st)) != cudaSuccess) return PKV_ERR_CUDA;
    pa.ticket_zeroed = true;
    pa.overlap_previous = true;
  }
  // 1. every new token of the batch (decode tokens and chunk tokens) into the cache
  e = pkv::launch_store_kvcache(key, value, k_cache, v_cache, slot_mapping, total_q,
                                static_cast<int32_t>(row), key_token_stride, value_token_stride,
                                int64_t(num_blocks) * block_size, err, st);
  if (e != cudaSuccess) return PKV_ERR_CUDA;
  // With the prefill interleaved, part of it also runs beside the decode: a
  // launch on a share of the SMs (mixed_side_share) on the side stream, while
  // the decode kernel takes the others; the launch between the decode kernel
  // and its combine then takes the items left (both claim items from one ticket).
  // The side launch may start first: its CTA count, not the stream order,
  // keeps the decode kernel's SMs free.
  int dev = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PKV_ERR_CUDA;
  const int sms = pkv::sm_count(dev);
  const int side_ctas =
      interleave ? static_cast<int>(sms * mixed_side_share(num_decode_seqs, total_q - num_decode_seqs,
                                                           num_q_heads, num_kv_heads))
                 : 0;
  std::unique_lock<std::mutex> side_lock(g_side_mu, std::defer_lock);
  SideStream *side = nullptr;
  if (side_ctas > 0) {
    side_lock.lock();
    if ((e = side_stream_locked(dev, &side)) != cudaSuccess) return PKV_ERR_CUDA;
    pkv::PrefillArgs ps = pa;
    ps.overlap_previous = false;
    ps.max_ctas = side_ctas;
    if ((e = cudaEventRecord(side->fork, st)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(side->stream, side->fork, 0)) != cudaSuccess ||
        (e = pkv::launch_paged_prefill(ps, side->stream)) != cudaSuccess ||
        (e = cudaEventRecord(side->join, side->stream)) != cudaSuccess)
      return PKV_ERR_CUDA;
  }
  // 2. the decode sequences 0..D-1 (one query row each, rows 0..D-1)
  if (num_decode_seqs > 0) {
    int32_t *lens = static_cast<int32_t *>(workspace);
    if ((e = pkv::launch_mixed_decode_lens(cu_seqlens_q, cu_seqlens_k, num_decode_seqs, lens, err,
                                           st)) != cudaSuccess)
      return PKV_ERR_CUDA;
    pkv::DecodeArgs a;
    a.out = out;
    a.q = q;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.block_tables = block_tables;
    a.max_blocks_per_seq = max_blocks_per_seq;
    a.context_lens = lens;
    a.num_seqs = num_decode_seqs;
    a.max_context_len = max_seqlen_k;
    a.num_q_heads = num_q_heads;
    a.num_kv_heads = num_kv_heads;
    a.block_size = block_size;
    a.num_blocks = num_blocks;
    a.scale = scale;
    a.workspace = static_cast<uint8_t *>(workspace) + lens_bytes;
    a.workspace_bytes = dec_bytes;
    a.err = err;
    a.interleave = interleave ? &pa : nullptr;
    a.grid_override = side_ctas > 0 ? sms - side_ctas : 0;
    if ((e = pkv::launch_paged_decode(a, plan, st)) != cudaSuccess) return PKV_ERR_CUDA;
  }
  if (side != nullptr && (e = cudaStreamWaitEvent(st, side->join, 0)) != cudaSuccess)
    return PKV_ERR_CUDA;
  // 3. the prefill chunks, unless they ran between the decode kernels
  if (num_prefill > 0 && !interleave &&
      (e = pkv::launch_paged_prefill(pa, st)) != cudaSuccess)
    return PKV_ERR_CUDA;
  return PKV_OK;
}

size_t pkv_prefill_workspace_size(int32_t num_seqs, int32_t total_q, int32_t num_q_heads,
                                  int32_t head_dim) {
  (void)num_seqs;
  (void)total_q;
  (void)num_q_heads;
  (void)head_dim;
  return pkv::kPrefillWorkspace;
}

pkv_status pkv_paged_prefill(void *out, const void *q, const void *k_cache, const void *v_cache,
                             const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k,
                             int32_t max_seqlen_q, int32_t max_seqlen_k,
                             const int32_t *block_tables, int32_t max_blocks_per_seq,
                             int32_t num_seqs, int32_t total_q, int32_t num_q_heads,
                             int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                             int32_t num_blocks, float scale, int32_t causal, void *workspace,
                             size_t workspace_bytes, pkv_dtype dtype, void *stream) {
  if (dtype != PKV_BF16) return PKV_ERR_DTYPE;
  if (num_seqs < 0 || total_q < 0 || num_q_heads < 1 || num_kv_heads < 1 || block_size < 1 ||
      num_blocks < 1 || max_blocks_per_seq < 0 || max_seqlen_q < 0 || max_seqlen_k < 0 ||
      !std::isfinite(scale))
    return PKV_ERR_ARG;
  if (head_dim != 128) return PKV_ERR_SHAPE;
  if (int64_t(max_seqlen_k) > int64_t(max_blocks_per_seq) * block_size) return PKV_ERR_ARG;
  if (!pkv::prefill_supported(num_q_heads, num_kv_heads, block_size)) return PKV_ERR_SHAPE;
  if (num_seqs > 65535 || num_q_heads > 65535) return PKV_ERR_ARG;  // grid y / z limits
  if ((int64_t(max_seqlen_q) + 127) / 128 > 65535) return PKV_ERR_ARG;
  if (!prefill_items_fit(max_seqlen_q, num_q_heads, num_kv_heads, num_seqs)) return PKV_ERR_ARG;
  if (num_seqs == 0 || total_q == 0) return PKV_OK;
  if (!out || !q || !k_cache || !v_cache || !cu_seqlens_q || !cu_seqlens_k || !block_tables)
    return PKV_ERR_ARG;
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 ||
      workspace_bytes < pkv::kPrefillWorkspace)
    return PKV_ERR_WORKSPACE;
  if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache))
    return PKV_ERR_ARG;
  cudaError_t e;
  uint32_t *err = pkv::device_error_word(&e);
  if (!err) return PKV_ERR_CUDA;
  pkv::PrefillArgs a;
  a.out = out;
  a.q = q;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.cu_seqlens_q = cu_seqlens_q;
  a.cu_seqlens_k = cu_seqlens_k;
  a.max_seqlen_q = max_seqlen_q;
  a.max_seqlen_k = max_seqlen_k;
  a.block_tables = block_tables;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.num_seqs = num_seqs;
  a.total_q = total_q;
  a.num_q_heads = num_q_heads;
  a.num_kv_heads = num_kv_heads;
  a.block_size = block_size;
  a.num_blocks = num_blocks;
  a.scale = scale;
  a.causal = causal;
  a.err = err;
  a.workspace = workspace;
  return from_cuda(pkv::launch_paged_prefill(a, static_cast<cudaStream_t>(stream)));
}

pkv_status pkv_get_device_errors(void *stream, uint32_t *bits) {
  cudaError_t e;
  uint32_t *err = pkv::device_error_word(&e);
  if (!err) return PKV_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t host = 0;
  if (cudaMemcpyAsync(&host, err, sizeof host, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaMemsetAsync(err, 0, sizeof host, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return PKV_ERR_CUDA;
  if (bits) *bits = host;
  return host ? PKV_ERR_DEVICE : PKV_OK;
}

const char *pkv_status_string(pkv_status status) {
  switch (status) {
    case PKV_OK: return "ok";
    case PKV_ERR_ARG: return "invalid argument";
    case PKV_ERR_SHAPE: return "unsupported shape";
    case PKV_ERR_DTYPE: return "unsupported dtype";
    case PKV_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case PKV_ERR_CUDA: return "CUDA runtime error";
    case PKV_ERR_DEVICE: return "device-side range check fired";
  }
  return "unknown status";
}

int32_t pkv_version(void) { return 100; }

}  // extern "C"
