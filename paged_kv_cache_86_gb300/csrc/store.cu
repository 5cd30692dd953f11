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

// fp8 E4M3 store: each (token, KV head) row of 128 values is quantized with
// its own fp32 scale, amax / 448, and codes E4M3(x * (448 / amax)) rounded to
// nearest even with saturation (cvt.rn.satfinite); a zero row gives zero codes
// and scale 0 (LLM Infra 101 v0.2, KV Quantization: the cache stores low-bit
// values instead of bf16). One warp per token; lane l holds dims 4l..4l+3.
__device__ __forceinline__ uint32_t quantize4_e4m3(uint2 bits, float inv) {
  const float2 lo = bf16x2_to_float2(bits.x), hi = bf16x2_to_float2(bits.y);
  uint16_t c01, c23;
  // cvt packs its first operand into the upper byte
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(c01) : "f"(__fmul_rn(lo.y, inv)), "f"(__fmul_rn(lo.x, inv)));
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(c23) : "f"(__fmul_rn(hi.y, inv)), "f"(__fmul_rn(hi.x, inv)));
  return static_cast<uint32_t>(c01) | (static_cast<uint32_t>(c23) << 16);
}

// One 128-element row per warp, four elements per lane (`bits`, already loaded).
__device__ __forceinline__ void quantize_row_e4m3(const uint2 bits, uint32_t *codes, float *scale,
                                                  int lane) {
  const float2 lo = bf16x2_to_float2(bits.x), hi = bf16x2_to_float2(bits.y);
  float amax = fmaxf(fmaxf(fabsf(lo.x), fabsf(lo.y)), fmaxf(fabsf(hi.x), fabsf(hi.y)));
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  uint32_t c = 0u;
  float sc = 0.f;
  if (amax > 0.f) {
    const float inv = __fdiv_rn(448.f, amax);
    sc = __fdiv_rn(amax, 448.f);
    c = quantize4_e4m3(bits, inv);
  }
  codes[lane] = c;
  if (lane == 0) *scale = sc;
}

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
