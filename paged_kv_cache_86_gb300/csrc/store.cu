// store.cu -- KV-cache write: scatter each new token's K and V rows into the
// cache slot named by slot_mapping (nano vllm代码详解 §2 context,
// `slot_mapping`; slot = block_id * block_size + offset).
//
// Pure data movement: one warp per token moves that token's K row and V row
// (num_kv_heads * head_dim bf16 each) with 16-byte vector loads and stores,
// so a warp touches 512 contiguous bytes per instruction on each side. The
// loads of a row are all issued before its stores to keep several 16-byte
// requests in flight per lane. Bound by HBM: 2 * row bytes read and written
// per token.
#include <cuda_runtime.h>

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr int kWarpsPerCta = 8;
constexpr int kVecsPerPass = 4;  // 16-byte vectors per lane per side before storing

__global__ void __launch_bounds__(kWarpsPerCta * 32)
store_kvcache_kernel(const uint4 *__restrict__ key, const uint4 *__restrict__ value,
                     uint4 *__restrict__ k_cache, uint4 *__restrict__ v_cache,
                     const int32_t *__restrict__ slot_mapping, int32_t num_tokens,
                     int32_t row_vecs, int64_t key_stride_vecs, int64_t value_stride_vecs,
                     int64_t num_slots, uint32_t *err) {
  const int lane = threadIdx.x & 31;
  const int64_t t = static_cast<int64_t>(blockIdx.x) * kWarpsPerCta + (threadIdx.x >> 5);
  if (t >= num_tokens) return;
  const int64_t slot = __ldg(slot_mapping + t);
  if (slot < 0) return;  // padded token
  if (slot >= num_slots) {
    if (lane == 0) raise_error(err, PKV_DEVERR_SLOT);
    return;
  }
  const uint4 *ks = key + t * key_stride_vecs;
  const uint4 *vs = value + t * value_stride_vecs;
  uint4 *kd = k_cache + slot * row_vecs;
  uint4 *vd = v_cache + slot * row_vecs;
  for (int base = 0; base < row_vecs; base += 32 * kVecsPerPass) {
    uint4 kr[kVecsPerPass], vr[kVecsPerPass];
#pragma unroll
    for (int j = 0; j < kVecsPerPass; ++j) {
      const int v = base + j * 32 + lane;
      if (v < row_vecs) {
        kr[j] = __ldg(ks + v);
        vr[j] = __ldg(vs + v);
      }
    }
#pragma unroll
    for (int j = 0; j < kVecsPerPass; ++j) {
      const int v = base + j * 32 + lane;
      if (v < row_vecs) {
        kd[v] = kr[j];
        vd[v] = vr[j];
      }
    }
  }
}

// fp8 E4M3 store: one warp per (token, KV head) row; the quantizer
// (quantize_row_e4m3) is in pkv_device.cuh, shared with the decode step.
__global__ void __launch_bounds__(kWarpsPerCta * 32)
store_kvcache_fp8_kernel(const __nv_bfloat16 *__restrict__ key,
                         const __nv_bfloat16 *__restrict__ value, uint8_t *__restrict__ k_cache,
                         uint8_t *__restrict__ v_cache, float *__restrict__ k_scales,
                         float *__restrict__ v_scales, const int32_t *__restrict__ slot_mapping,
                         int32_t num_tokens, int32_t num_kv_heads, int64_t key_stride,
                         int64_t value_stride, int64_t num_slots, uint32_t *err) {
  // one warp per (token, KV head): its K row and its V row, both loads first
  const int lane = threadIdx.x & 31;
  const int64_t gw = static_cast<int64_t>(blockIdx.x) * kWarpsPerCta + (threadIdx.x >> 5);
  const int64_t t = gw / num_kv_heads;
  const int h = static_cast<int>(gw - t * num_kv_heads);
  if (t >= num_tokens) return;
  const int64_t slot = __ldg(slot_mapping + t);
  if (slot < 0) return;  // padded token
  if (slot >= num_slots) {
    if (lane == 0 && h == 0) raise_error(err, PKV_DEVERR_SLOT);
    return;
  }
  const int64_t row = slot * num_kv_heads + h;
  const uint2 kb = __ldg(reinterpret_cast<const uint2 *>(key + t * key_stride + h * 128) + lane);
  const uint2 vb = __ldg(reinterpret_cast<const uint2 *>(value + t * value_stride + h * 128) + lane);
  quantize_row_e4m3(kb, reinterpret_cast<uint32_t *>(k_cache + row * 128), k_scales + row, lane);
  quantize_row_e4m3(vb, reinterpret_cast<uint32_t *>(v_cache + row * 128), v_scales + row, lane);
}

}  // namespace

cudaError_t launch_store_kvcache_fp8(const void *key, const void *value, void *k_cache,
                                     void *v_cache, float *k_scales, float *v_scales,
                                     const int32_t *slot_mapping, int32_t num_tokens,
                                     int32_t num_kv_heads, int64_t key_stride, int64_t value_stride,
                                     int64_t num_slots, uint32_t *err, cudaStream_t stream) {
  if (num_tokens == 0) return cudaSuccess;
  const int64_t warps = static_cast<int64_t>(num_tokens) * num_kv_heads;
  const unsigned grid = static_cast<unsigned>((warps + kWarpsPerCta - 1) / kWarpsPerCta);
  store_kvcache_fp8_kernel<<<grid, kWarpsPerCta * 32, 0, stream>>>(
      static_cast<const __nv_bfloat16 *>(key), static_cast<const __nv_bfloat16 *>(value),
      static_cast<uint8_t *>(k_cache), static_cast<uint8_t *>(v_cache), k_scales, v_scales,
      slot_mapping, num_tokens, num_kv_heads, key_stride, value_stride, num_slots, err);
  return cudaGetLastError();
}

cudaError_t launch_store_kvcache(const void *key, const void *value, void *k_cache, void *v_cache,
                                 const int32_t *slot_mapping, int32_t num_tokens,
                                 int32_t row_elems, int64_t key_stride, int64_t value_stride,
                                 int64_t num_slots, uint32_t *err, cudaStream_t stream) {
  if (num_tokens == 0) return cudaSuccess;
  const int32_t row_vecs = row_elems / 8;  // 8 bf16 per 16-byte vector
  const unsigned grid = static_cast<unsigned>((num_tokens + kWarpsPerCta - 1) / kWarpsPerCta);
  store_kvcache_kernel<<<grid, kWarpsPerCta * 32, 0, stream>>>(
      static_cast<const uint4 *>(key), static_cast<const uint4 *>(value),
      static_cast<uint4 *>(k_cache), static_cast<uint4 *>(v_cache), slot_mapping, num_tokens,
      row_vecs, key_stride / 8, value_stride / 8, num_slots, err);
  return cudaGetLastError();
}

}  // namespace pkv
