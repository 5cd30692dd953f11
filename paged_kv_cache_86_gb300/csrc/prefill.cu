// prefill.cu -- paged varlen chunked-prefill attention on the tcgen05 tensor
// cores of GB300 (sm_103a).
//
// Sequence i owns query rows cu_seqlens_q[i] .. cu_seqlens_q[i+1]-1 and keys
// 0 .. k_len-1 of its block table (nano vllm代码详解 §2 context: cu_seqlens_q/k,
// max_seqlen_q/k, block_tables). With the causal mask, query row r of a chunk
// sits at absolute position prefix + r, prefix = k_len - q_len, and sees keys
// 0 .. prefix + r: the chunk continues its cached prefix (推理运行时 §Prefill
// 与 decode 输入; Mini-SGLang 源码解析（二）§6.6 chunked prefill). Prefill is
// compute-bound (Mini-SGLang 源码解析（二）§8.3), so the two dense contractions
// per tile, S = Q K^T and O += P V, run on tcgen05.mma with fp32 accumulators
// in tensor memory; only the softmax runs on the CUDA cores.
//
// The kernel is prefill_pp.cu's persistent ping-pong kernel: a work item is
// a 128-row query tile of two query heads of one KV head, or, for an odd GQA
// group, two consecutive query tiles of one head, so every supported shape
// runs on it. This file holds the entry's shape check and its dispatch.
#include <cuda_runtime.h>

#include "pkv_internal.h"

namespace pkv {

bool prefill_supported(int num_q_heads, int num_kv_heads, int block_size) {
  return prefill_pp_supported(num_q_heads, num_kv_heads, block_size);
}

cudaError_t launch_paged_prefill(const PrefillArgs &a, cudaStream_t stream) {
  if (a.num_seqs == 0 || a.total_q == 0 || a.max_seqlen_q == 0) return cudaSuccess;
  if (!prefill_supported(a.num_q_heads, a.num_kv_heads, a.block_size)) return cudaErrorInvalidValue;
  return launch_prefill_pp(a, stream);
}

}  // namespace pkv
