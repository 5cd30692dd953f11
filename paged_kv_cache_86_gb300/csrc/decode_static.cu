// decode_static.cu -- pkv_paged_decode_static_ws: the paged decode of
// pkv_paged_decode, with its scratch space taken from a fixed array compiled
// into this library instead of a caller-provided workspace.
//
// Why it exists: some callers cannot hand the library extra device memory.
// A plug-in running inside a host framework whose allocator owns the whole
// device, a runtime that is given only its input and output buffers, or a
// latency-critical loop where a cudaMalloc (and the implicit synchronisation
// it may bring) is not allowed, all need a decode call that allocates nothing.
// This entry point allocates nothing: no cudaMalloc, no cudaFree, no
// allocating library routine. The caller still passes q, out, the caches and
// the metadata as device buffers.
//
// The cost: every GPU that loads the library reserves kStaticScratchBytes
// (16 MiB) of device memory for the array until the process exits, and all
// calls share that one array.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "pkv.h"

namespace {

constexpr size_t kStaticScratchBytes = size_t(16) << 20;  // 16 MiB

// Scratch of the split-decode kernels: the plan header, the per-sequence
// prefix sums and the partial (o, m, l) records of sequences cut by a CTA
// range. In host code this name is only a stand-in for the device array; its
// device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_decode_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device, resolved once per
// device (with that device current) and cached.
pkv_status scratch_for_current_device(void **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PKV_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr)
      return PKV_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return PKV_OK;
}

}  // namespace

extern "C" {

pkv_status pkv_paged_decode_static_ws(void *out, const void *q, const void *k_cache,
                                      const void *v_cache, const int32_t *block_tables,
                                      int32_t max_blocks_per_seq, const int32_t *context_lens,
                                      int32_t num_seqs, int32_t max_context_len,
                                      int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                      int32_t block_size, int32_t num_blocks, float scale,
                                      pkv_dtype dtype, void *stream) {
  if (num_seqs == 0) {
    return pkv_paged_decode(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq,
                            context_lens, num_seqs, max_context_len, num_q_heads, num_kv_heads,
                            head_dim, block_size, num_blocks, scale, nullptr, 0, dtype, stream);
  }
  const size_t need = pkv_decode_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim);
  if (need == 0) {
    // unsupported shape or bad counts: let the full check report which
    return pkv_paged_decode(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq,
                            context_lens, num_seqs, max_context_len, num_q_heads, num_kv_heads,
                            head_dim, block_size, num_blocks, scale, nullptr, 0, dtype, stream);
  }
  if (need > kStaticScratchBytes) return PKV_ERR_WORKSPACE;  // batch too large for the array
  void *scratch = nullptr;
  const pkv_status st = scratch_for_current_device(&scratch);
  if (st != PKV_OK) return st;
  return pkv_paged_decode(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                          num_seqs, max_context_len, num_q_heads, num_kv_heads, head_dim,
                          block_size, num_blocks, scale, scratch, kStaticScratchBytes, dtype,
                          stream);
}

}  // extern "C"
