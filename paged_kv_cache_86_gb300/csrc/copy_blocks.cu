// copy_blocks.cu -- block copy for copy-on-write of shared KV-cache blocks.
//
// When requests share read-only blocks (a common prefix, a forked branch) and
// the last shared block is not yet full, a branch that is about to write into
// it must first get its own copy, or it would change another request's history
// (推理运行时 §Prefix cache 与 copy-on-write). This kernel performs the copies
// a host block manager decides on: for pair p, rows [0, rows[p]) of block
// src[p] -> block dst[p], in both the K and the V cache ([NB, bs, Hkv, D]).
//
// Pure data movement, HBM-bound: 2 (K, V) x 2 (read, write) x rows x Hkv x D x
// 2 bytes per pair. Grid: (chunks of a block side, pairs, K/V); each thread
// moves kUnroll 16-byte vectors with all loads issued before the stores.
#include <cuda_runtime.h>

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 4;
constexpr int kVecsPerCta = kThreads * kUnroll;

__global__ void __launch_bounds__(kThreads)
copy_blocks_kernel(uint4 *__restrict__ k_cache, uint4 *__restrict__ v_cache,
                   const int32_t *__restrict__ src, const int32_t *__restrict__ dst,
                   const int32_t *__restrict__ rows, int32_t block_size, int32_t num_blocks,
                   int32_t row_vecs, uint32_t *err) {
  const int p = blockIdx.y;
  const int s = __ldg(src + p), d = __ldg(dst + p);
  if (s < 0 || s >= num_blocks || d < 0 || d >= num_blocks) {
    if (threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.z == 0) raise_error(err, PKV_DEVERR_BLOCK_ID);
    return;
  }
  int n = rows != nullptr ? __ldg(rows + p) : block_size;
  if (n < 0 || n > block_size) {
    if (threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.z == 0) raise_error(err, PKV_DEVERR_LENGTH);
    n = n < 0 ? 0 : block_size;
  }
  const int64_t vecs = static_cast<int64_t>(n) * row_vecs;     // of this block side
  const int64_t block_vecs = static_cast<int64_t>(block_size) * row_vecs;
  uint4 *cache = blockIdx.z == 0 ? k_cache : v_cache;
  const uint4 *from = cache + s * block_vecs;
  uint4 *to = cache + d * block_vecs;
  const int64_t v0 = static_cast<int64_t>(blockIdx.x) * kVecsPerCta + threadIdx.x;
  uint4 r[kUnroll];
#pragma unroll
  for (int u = 0; u < kUnroll; ++u) {
    const int64_t v = v0 + u * kThreads;
    if (v < vecs) r[u] = from[v];
  }
#pragma unroll
  for (int u = 0; u < kUnroll; ++u) {
    const int64_t v = v0 + u * kThreads;
    if (v < vecs) to[v] = r[u];
  }
}

}  // namespace

cudaError_t launch_copy_blocks(void *k_cache, void *v_cache, const int32_t *src,
                               const int32_t *dst, const int32_t *rows, int32_t num_pairs,
                               int32_t block_size, int32_t num_blocks, int32_t row_elems,
                               uint32_t *err, cudaStream_t stream) {
  if (num_pairs == 0) return cudaSuccess;
  const int32_t row_vecs = row_elems / 8;
  const int64_t block_vecs = static_cast<int64_t>(block_size) * row_vecs;
  const dim3 grid(static_cast<unsigned>((block_vecs + kVecsPerCta - 1) / kVecsPerCta),
                  static_cast<unsigned>(num_pairs), 2);
  copy_blocks_kernel<<<grid, kThreads, 0, stream>>>(static_cast<uint4 *>(k_cache),
                                                    static_cast<uint4 *>(v_cache), src, dst, rows,
                                                    block_size, num_blocks, row_vecs, err);
  return cudaGetLastError();
}

}  // namespace pkv
