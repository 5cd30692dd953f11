/*
 * pkv.h -- C ABI of libpkv: attention over a block-paged KV cache on one
 * GB300 GPU (sm_103a).
 *
 * Three operations, whose arguments are the per-batch metadata fields that
 * nano-vllm's attention Context carries (nano vllm代码详解, §2 context:
 * is_prefill, cu_seqlens_q/k, max_seqlen_q/k, slot_mapping, context_lens,
 * block_tables):
 *
 *   pkv_store_kvcache  write each new token's K and V into the cache slot
 *                      named by slot_mapping;
 *   pkv_paged_decode   one query per sequence over its context_lens[i] cached
 *                      tokens, found through its block_tables row
 *                      (pkv_decode_step: the store of each sequence's newest
 *                      token and the decode in one call);
 *   pkv_paged_prefill  varlen query chunks (cu_seqlens_q) over their cached
 *                      prefix plus themselves (cu_seqlens_k), causal;
 *   pkv_copy_blocks    copy-on-write of shared cache blocks;
 *   *_fp8              the store, the decode and the decode step over an fp8
 *                      E4M3 cache;
 *   pkv_mixed_step     a batch of decode requests and prefill chunks.
 *
 * Cache layout. One layer's K cache and V cache are two separate arrays of
 * shape [num_blocks, block_size, num_kv_heads, head_dim], row-major, bf16.
 * Logical block j of a sequence lives in physical block block_tables[i][j]
 * (推理运行时, §分页 KV). Token p of a sequence is row p % block_size of
 * physical block block_tables[i][p / block_size], and a flat slot is
 * block_id * block_size + offset (the row-major index of a [num_blocks,
 * block_size] table, as in Mini-SGLang 源码解析（二）§6.8).
 *
 * Index arrays are int32 (Mini-SGLang 源码解析（二）§7.8 keeps its page table
 * in int32). Query head g reads KV head g / (num_q_heads / num_kv_heads).
 *
 * Ownership. The caller owns every buffer; all pointers except `stream` and
 * host scalars are DEVICE pointers. The library allocates no device memory.
 * Buffers that a call needs beyond its inputs and outputs (partial results of
 * split sequences) come from a caller-provided workspace whose size the
 * matching *_workspace_size function returns.
 *
 * Execution. Every call is asynchronous on `stream` (a cudaStream_t; NULL is
 * the legacy default stream) and never synchronises the host. A store must be
 * ordered before the decode/prefill that reads the stored tokens, e.g. by
 * issuing both on one stream.
 *
 * Errors. Arguments are validated on the host before anything is launched; a
 * failed check returns a negative pkv_status and launches nothing. Device data
 * (slots, block ids, lengths) is range-checked inside the kernels: an entry
 * that is out of range is skipped (never dereferenced), its output is
 * unspecified, and a bit is set in a per-device error word that
 * pkv_get_device_errors() returns and clears.
 *
 * Device state. The library keeps two pieces of state per device: the error
 * word and, for pkv_paged_decode_static_ws, the address of its scratch array.
 * Both are `__device__` variables of the library's module; their addresses are
 * looked up once per device (first use, with that device current) and kept.
 * Destroying the device's primary context while the library is loaded
 * (cudaDeviceReset, or the driver API's primary-context reset) invalidates
 * them: do not reset a device between calls into this library.
 */
#ifndef PKV_H_
#define PKV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    PKV_OK = 0,
    PKV_ERR_ARG = -1,       /* null pointer, negative size, misaligned pointer or stride */
    PKV_ERR_SHAPE = -2,     /* head_dim / head counts / block size the kernels do not support */
    PKV_ERR_DTYPE = -3,     /* dtype other than PKV_BF16 */
    PKV_ERR_WORKSPACE = -4, /* workspace missing or smaller than *_workspace_size() */
    PKV_ERR_CUDA = -5,      /* a CUDA runtime call failed (launch, attribute, copy) */
    PKV_ERR_DEVICE = -6     /* a device-side range check fired (see pkv_get_device_errors) */
} pkv_status;

typedef enum { PKV_BF16 = 0 } pkv_dtype;

/* Bits of the device error word. */
#define PKV_DEVERR_SLOT 0x1u        /* slot_mapping entry >= num_blocks * block_size */
#define PKV_DEVERR_BLOCK_ID 0x2u    /* block_tables entry outside [0, num_blocks) */
#define PKV_DEVERR_LENGTH 0x4u      /* a length beyond its table row or max_* bound, or negative */
#define PKV_DEVERR_TIMEOUT 0x8u     /* an on-chip wait hit its iteration limit */

/* ----------------------------------------------------------------- store --
 * For t < num_tokens: slot = slot_mapping[t]; slot < 0 marks a padded token
 * and writes nothing; otherwise block = slot / block_size, offset = slot %
 * block_size, and key[t] (num_kv_heads * head_dim elements) is copied bit for
 * bit to k_cache[block][offset], value[t] to v_cache[block][offset].
 * (nano vllm代码详解 §2 context: slot_mapping; Mini-SGLang 源码解析（二）
 * §6.7 writes each new token's page into the page table.)
 *
 *   key, value        token t's row starts at key + t * key_token_stride
 *                     (elements), so K and V may be views into a fused QKV
 *                     tensor; each row is num_kv_heads * head_dim contiguous
 *                     elements. Rows and strides must be 16-byte aligned.
 *   k_cache, v_cache  [num_blocks, block_size, num_kv_heads, head_dim], 16-byte aligned.
 *   slot_mapping      [num_tokens] int32. Slots must be distinct (a duplicate
 *                     slot leaves which token wins unspecified).
 * head_dim * num_kv_heads must be a multiple of 8. num_tokens == 0 is a no-op.
 */
pkv_status pkv_store_kvcache(const void *key, const void *value,
                             void *k_cache, void *v_cache,
                             const int32_t *slot_mapping, int32_t num_tokens,
                             int32_t num_kv_heads, int32_t head_dim,
                             int32_t block_size, int32_t num_blocks,
                             int64_t key_token_stride, int64_t value_token_stride,
                             pkv_dtype dtype, void *stream);

/* ------------------------------------------------------------ mixed batch --
 * pkv_mixed_step: one scheduling round's batch of decode requests and prefill
 * chunks under one token budget, N_scheduled = N_decode + N_prefill_chunk
 * (推理运行时 §Chunked prefill; §Prefill 与 decode 输入: the tokens of all
 * requests are flattened into one array and per-sequence metadata gives each
 * query range, context length and block table -- decode requests have one
 * query, chunks several, with cached history).
 *   Layout: sequences 0 .. num_decode_seqs-1 are decode requests, one query
 *   row each, rows 0 .. num_decode_seqs-1 (the decode-first order of a batch
 *   builder that gives every decode request its token before filling the rest
 *   of the budget with prefill chunks); sequences num_decode_seqs .. num_seqs-1
 *   are chunks. cu_seqlens_q / cu_seqlens_k [num_seqs + 1] as for
 *   pkv_paged_prefill (bottom-right causal); key / value [total_q, Hkv, D] are
 *   the K/V of every query row, written at slot_mapping [total_q] first.
 *   max_seqlen_q / max_seqlen_k bound the chunks' query rows and every
 *   sequence's keys.
 *   workspace: at least pkv_mixed_workspace_size(num_decode_seqs, ...) bytes,
 *   256-byte aligned.
 * The result equals pkv_store_kvcache followed by pkv_paged_prefill over the
 * whole batch; the decode sequences run on the split decode kernels instead of
 * occupying a 128-row query tile each. A decode sequence with other than one
 * query row sets PKV_DEVERR_LENGTH. Launches: the store, then the decode
 * (attention, combine) and the chunks' prefill. With the all-heads decode
 * kernel, part of the prefill runs beside it on a second stream of the
 * library (created on first use), forked from and joined back to `stream` by
 * events within the call, so work queued on `stream` afterwards follows all
 * of it and a CUDA graph captures the fork and the join; the rest of the
 * prefill takes the SMs the decode kernel frees. Otherwise the launches run
 * in stream order.
 */
size_t pkv_mixed_workspace_size(int32_t num_decode_seqs, int32_t num_q_heads,
                                int32_t num_kv_heads, int32_t head_dim);

pkv_status pkv_mixed_step(void *out, const void *q, const void *key, const void *value,
                          const int32_t *slot_mapping,
                          int64_t key_token_stride, int64_t value_token_stride,
                          void *k_cache, void *v_cache,
                          const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k,
                          int32_t max_seqlen_q, int32_t max_seqlen_k,
                          const int32_t *block_tables, int32_t max_blocks_per_seq,
                          int32_t num_seqs, int32_t num_decode_seqs, int32_t total_q,
                          int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                          int32_t block_size, int32_t num_blocks, float scale,
                          void *workspace, size_t workspace_bytes,
                          pkv_dtype dtype, void *stream);

/* ---------------------------------------------------------------- fp8 KV --
 * A quantized cache: the KV cache stores low-bit values instead of bf16, at
 * some loss of accuracy (LLM Infra 101 v0.2, KV Quantization). Format: OCP FP8
 * E4M3 codes (1 sign, 4 exponent bits with bias 7, 3 mantissa bits; largest
 * magnitude 448; 0x7F / 0xFF are NaN) with one fp32 scale per (token, KV head)
 * row of head_dim values, for K and V separately:
 *   k_cache, v_cache    [num_blocks, block_size, num_kv_heads, 128] uint8 codes
 *   k_scales, v_scales  [num_blocks * block_size, num_kv_heads] float, 16-byte
 *                       aligned; the scale of slot s, head h is element
 *                       s * num_kv_heads + h.
 * A row's value d is e4m3(code_d) * scale.
 *
 * pkv_store_kvcache_fp8: like pkv_store_kvcache, but each new bf16 row x is
 * quantized on the way: amax = max |x_d|; scale = amax / 448 and codes
 * E4M3(x_d * (448 / amax)), both fp32 operations rounded to nearest even, the
 * code rounded to the nearest finite E4M3 value (ties to even) and saturated
 * at 448; an all-zero row stores zero codes and scale 0. head_dim 128.
 */
pkv_status pkv_store_kvcache_fp8(const void *key, const void *value,
                                 void *k_cache, void *v_cache,
                                 float *k_scales, float *v_scales,
                                 const int32_t *slot_mapping, int32_t num_tokens,
                                 int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                 int32_t num_blocks,
                                 int64_t key_token_stride, int64_t value_token_stride,
                                 void *stream);

/* pkv_paged_decode_fp8: pkv_paged_decode over fp8 caches -- the attention of
 * each q row over the dequantized K/V rows. Same arguments, workspace and
 * errors as pkv_paged_decode, plus the scale arrays. q and out stay bf16. The
 * K codes enter the tensor core as E4M3, against each q row scaled by a power
 * of two and split into two E4M3 terms whose sum is the scaled row (exact for
 * bf16 q except for entries under about 2^-10 of the row's largest, off by at
 * most 2^-10 of the scaled unit there); V is expanded to f16 with its row
 * scales folded into the softmax weights. That kernel takes num_kv_heads 4
 * or 8 with block_size a multiple of 128 / num_kv_heads; other block sizes,
 * and 1 or 2 KV heads, run on the CUDA-core kernel, which expands the codes
 * to fp32 and applies the row scales to the scores and the weights.
 * Supported: head_dim 128, num_kv_heads in {1, 2, 4, 8}, num_q_heads /
 * num_kv_heads in {1, 2, 4, 8}, any block_size >= 1; other shapes return
 * PKV_ERR_SHAPE.
 */
pkv_status pkv_paged_decode_fp8(void *out, const void *q,
                                const void *k_cache, const void *v_cache,
                                const float *k_scales, const float *v_scales,
                                const int32_t *block_tables, int32_t max_blocks_per_seq,
                                const int32_t *context_lens, int32_t num_seqs,
                                int32_t max_context_len,
                                int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                int32_t block_size, int32_t num_blocks, float scale,
                                void *workspace, size_t workspace_bytes, void *stream);

/* pkv_decode_step_fp8: pkv_decode_step over fp8 caches -- each sequence's
 * newest bf16 K/V row (key_new / value_new, as in pkv_decode_step) is quantized
 * exactly as pkv_store_kvcache_fp8 quantizes it and written, codes and scales,
 * at logical position min(context_lens[i], max_context_len) - 1; then
 * pkv_paged_decode_fp8 runs. Equal, bit for bit, to pkv_store_kvcache_fp8 with
 * those slots followed by pkv_paged_decode_fp8, in one call (the quantizing
 * store runs inside the decode's first launch). Same shapes, workspace and
 * errors as pkv_paged_decode_fp8.
 */
pkv_status pkv_decode_step_fp8(void *out, const void *q,
                               const void *key_new, const void *value_new,
                               int64_t key_token_stride, int64_t value_token_stride,
                               void *k_cache, void *v_cache,
                               float *k_scales, float *v_scales,
                               const int32_t *block_tables, int32_t max_blocks_per_seq,
                               const int32_t *context_lens, int32_t num_seqs,
                               int32_t max_context_len,
                               int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                               int32_t block_size, int32_t num_blocks, float scale,
                               void *workspace, size_t workspace_bytes, void *stream);

/* ------------------------------------------------------------ block copy --
 * pkv_copy_blocks: for p < num_pairs, rows 0 .. num_rows[p]-1 of physical block
 * src_block_ids[p] are copied to the same rows of block dst_block_ids[p], in
 * both k_cache and v_cache (whole blocks when num_rows is NULL). This is the
 * copy-on-write step of prefix sharing: requests may point at the same
 * read-only blocks, and before a request writes into a shared block that is
 * not yet full it needs its own copy, or it would change another request's
 * history (推理运行时 §Prefix cache 与 copy-on-write; nano vllm代码详解 §3
 * Block / BlockManager keep shared blocks by reference count).
 *   src_block_ids, dst_block_ids, num_rows   [num_pairs] int32, device.
 *   num_pairs <= 65535. The dst blocks must be distinct and must not be
 *   the src of any pair in the same call (the copies run concurrently).
 * A block id outside [0, num_blocks) skips its pair and sets
 * PKV_DEVERR_BLOCK_ID; a row count outside [0, block_size] is clamped and sets
 * PKV_DEVERR_LENGTH.
 */
pkv_status pkv_copy_blocks(void *k_cache, void *v_cache,
                           const int32_t *src_block_ids, const int32_t *dst_block_ids,
                           const int32_t *num_rows, int32_t num_pairs,
                           int32_t num_kv_heads, int32_t head_dim,
                           int32_t block_size, int32_t num_blocks,
                           pkv_dtype dtype, void *stream);

/* ---------------------------------------------------------------- decode --
 * out[i, g, :] = softmax_p(scale * q[i, g, :] . K_i[p, g / G, :]) . V_i[p, g / G, :]
 * over p < context_lens[i], where K_i[p] is row p % block_size of physical
 * block block_tables[i * max_blocks_per_seq + p / block_size] and G =
 * num_q_heads / num_kv_heads. The new token of a decode step is stored first
 * and counts in context_lens[i]. A sequence with context_lens[i] == 0 gets a
 * zero row. (nano vllm代码详解 §2 context: context_lens, block_tables;
 * 推理运行时 §分页 KV: the kernel reads K/V through the mapping.)
 *
 *   out, q            [num_seqs, num_q_heads, head_dim] bf16, contiguous.
 *   block_tables      [num_seqs, max_blocks_per_seq] int32; entries past
 *                     ceil(context_lens[i] / block_size) are never read.
 *   context_lens      [num_seqs] int32, each in [0, max_context_len] and
 *                     max_context_len <= max_blocks_per_seq * block_size.
 *   workspace         device buffer of at least
 *                     pkv_decode_workspace_size(num_seqs, num_q_heads,
 *                     num_kv_heads, head_dim) bytes, 256-byte aligned. Its
 *                     contents need no initialisation and are scratch after
 *                     the call; two calls in flight at once need two workspaces.
 *   Supported: head_dim 128, num_q_heads a multiple of num_kv_heads, any
 *   scale, and either block_size a multiple of 8 with at most 16 query heads
 *   per KV head (tensor-core kernels), or any block_size >= 1 with
 *   num_kv_heads in {1, 2, 4, 8} and num_q_heads / num_kv_heads in {1, 2, 4,
 *   8}. Other shapes return PKV_ERR_SHAPE.
 * The work is split into equal token ranges over the GPU's SMs; a sequence that
 * spans several ranges is finished by a log-sum-exp combine pass.
 */
size_t pkv_decode_workspace_size(int32_t num_seqs, int32_t num_q_heads,
                                 int32_t num_kv_heads, int32_t head_dim);

pkv_status pkv_paged_decode(void *out, const void *q,
                            const void *k_cache, const void *v_cache,
                            const int32_t *block_tables, int32_t max_blocks_per_seq,
                            const int32_t *context_lens, int32_t num_seqs,
                            int32_t max_context_len,
                            int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                            int32_t block_size, int32_t num_blocks, float scale,
                            void *workspace, size_t workspace_bytes,
                            pkv_dtype dtype, void *stream);

/* ----------------------------------------------------------- decode step --
 * pkv_decode_step: one decode step of a batch in one call -- the store of each
 * sequence's newest token followed by pkv_paged_decode, with the same
 * arguments, supported shapes, workspace and errors as pkv_paged_decode, plus:
 *   key_new, value_new  [num_seqs, num_kv_heads, head_dim] bf16 rows (token
 *                       strides key_token_stride / value_token_stride in
 *                       elements, multiples of 8, 16-byte aligned): the K and V
 *                       of each sequence's newest token.
 * Row i is written to the cache at logical position n_i - 1 of sequence i,
 * n_i = context_lens[i] (which counts the new token), i.e. to slot
 * block_tables[i][(n_i - 1) / block_size] * block_size + (n_i - 1) % block_size,
 * the last filled row of the sequence's last block (nano vllm代码详解 §2
 * Sequence: last_block_num_tokens; §3.2.4 may_append: the last block is the
 * one being written), and then attended to. Sequences with n_i == 0 store
 * nothing and get a zero row. The result equals pkv_store_kvcache with those
 * slots followed by pkv_paged_decode, in the launches of pkv_paged_decode
 * alone: with bf16 caches on the all-heads tcgen05 kernel the attention kernel
 * writes each row just before it loads the stage that holds it; otherwise
 * the decode's planning launch writes the rows beside the range planning.
 * A block id outside [0, num_blocks) skips the write and sets
 * PKV_DEVERR_BLOCK_ID.
 * Graphs: the launches depend only on the host arguments, so a call can be
 * captured in a CUDA graph and replayed with new contents in the same buffers;
 * padding a batch up to a captured size with context_lens 0 rows is allowed.
 */
pkv_status pkv_decode_step(void *out, const void *q,
                           const void *key_new, const void *value_new,
                           int64_t key_token_stride, int64_t value_token_stride,
                           void *k_cache, void *v_cache,
                           const int32_t *block_tables, int32_t max_blocks_per_seq,
                           const int32_t *context_lens, int32_t num_seqs,
                           int32_t max_context_len,
                           int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                           int32_t block_size, int32_t num_blocks, float scale,
                           void *workspace, size_t workspace_bytes,
                           pkv_dtype dtype, void *stream);

/* ------------------------------------------------- decode, no allocation --
 * pkv_paged_decode_static_ws: the same computation, arguments and errors as
 * pkv_paged_decode, for callers that cannot give the library any device memory
 * of its own -- e.g. a plug-in inside a framework whose allocator owns the
 * device, or a runtime that only hands over its input and output buffers. The
 * call allocates nothing (no cudaMalloc, no cudaFree, no allocating library
 * routine): its scratch space is one fixed 16 MiB device array compiled into
 * the library, which every GPU that loads the library keeps until the process
 * exits. None of the source pages has a counterpart of this call; it exists
 * only for such callers.
 *   Limit: a batch whose pkv_decode_workspace_size(num_seqs, num_q_heads,
 *   num_kv_heads, head_dim) exceeds 16 MiB (16777216 bytes) is rejected with
 *   PKV_ERR_WORKSPACE before anything is launched.
 *   Set-up: the first call on each device looks up the array's device address
 *   (cudaGetSymbolAddress) with that device current and caches it; make that
 *   first call before any stream capture, and do not reset the device while
 *   the library is loaded (the cached address would be stale).
 *   Sharing: all calls share the one array and it keeps the last call's
 *   contents (nothing in it needs to start at zero). Calls whose kernels may
 *   overlap on the GPU (different streams without ordering) race on it; order
 *   them on one stream.
 */
pkv_status pkv_paged_decode_static_ws(void *out, const void *q,
                                      const void *k_cache, const void *v_cache,
                                      const int32_t *block_tables, int32_t max_blocks_per_seq,
                                      const int32_t *context_lens, int32_t num_seqs,
                                      int32_t max_context_len,
                                      int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                      int32_t block_size, int32_t num_blocks, float scale,
                                      pkv_dtype dtype, void *stream);

/* --------------------------------------------------------------- prefill --
 * Sequence i owns query rows cu_seqlens_q[i] .. cu_seqlens_q[i+1]-1 (q_len
 * rows) and keys 0 .. k_len-1 with k_len = cu_seqlens_k[i+1] - cu_seqlens_k[i],
 * read through its block_tables row. With causal != 0, query row r sits at
 * absolute position (k_len - q_len) + r and attends to keys 0 .. (k_len -
 * q_len) + r: a chunk follows its cached prefix (推理运行时 §Prefill 与
 * decode 输入; Mini-SGLang 源码解析（二）§6.6 chunked prefill). The chunk's own
 * K/V must already be stored (pkv_store_kvcache) before this call.
 *
 *   out, q            [total_q, num_q_heads, head_dim] bf16, contiguous,
 *                     total_q = cu_seqlens_q[num_seqs].
 *   cu_seqlens_q/k    [num_seqs + 1] int32, non-decreasing, starting at 0;
 *                     q_len <= max_seqlen_q, k_len <= max_seqlen_k <=
 *                     max_blocks_per_seq * block_size, and q_len <= k_len when causal.
 *   workspace         at least pkv_prefill_workspace_size(...) bytes (256),
 *                     256-byte aligned: the work ticket of the persistent
 *                     kernel, reset by the call itself; two calls in flight at
 *                     once need two workspaces.
 *   Supported: head_dim 128; num_q_heads a multiple of num_kv_heads; any
 *   block_size >= 1 (K/V tiles of a block size that is a multiple of 8 are
 *   loaded as TMA boxes, others are gathered row by row); num_seqs and
 *   ceil(max_seqlen_q / 128) at most 65535. Unsupported shapes return
 *   PKV_ERR_SHAPE.
 */
size_t pkv_prefill_workspace_size(int32_t num_seqs, int32_t total_q,
                                  int32_t num_q_heads, int32_t head_dim);

pkv_status pkv_paged_prefill(void *out, const void *q,
                             const void *k_cache, const void *v_cache,
                             const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k,
                             int32_t max_seqlen_q, int32_t max_seqlen_k,
                             const int32_t *block_tables, int32_t max_blocks_per_seq,
                             int32_t num_seqs, int32_t total_q,
                             int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                             int32_t block_size, int32_t num_blocks, float scale,
                             int32_t causal, void *workspace, size_t workspace_bytes,
                             pkv_dtype dtype, void *stream);

/* ------------------------------------------------------------- utilities --
 * pkv_get_device_errors: waits for `stream`, then returns (in *bits) and
 * clears the error word of the current device. Returns PKV_ERR_DEVICE when any
 * bit was set, PKV_OK otherwise, PKV_ERR_CUDA if the copy failed.
 */
pkv_status pkv_get_device_errors(void *stream, uint32_t *bits);

const char *pkv_status_string(pkv_status status);

/* pkv_selftest_bounded_wait: an on-GPU check of the failure path the kernels
 * rely on (no fault, trap or endless loop is involved). One CTA of two warps
 * runs eight steps and meets once per step on an OR-reducing hardware barrier;
 * in step fail_step warp 1 waits 5 ms on an mbarrier that nothing arrives on.
 * The wait must give up, raise PKV_DEVERR_TIMEOUT in the device error word,
 * and both warps must leave the loop in that step.
 *   result  device int32[4], zeroed by the caller: the step in which warp 0
 *           and warp 1 left, 1 if the timeout was reported, the number of
 *           steps both completed. fail_step >= 8: no wait runs out.
 * Asynchronous on `stream`; read result and pkv_get_device_errors after it.
 */
pkv_status pkv_selftest_bounded_wait(int32_t fail_step, int32_t *result, void *stream);

/* Library version: major * 10000 + minor * 100 + patch. */
int32_t pkv_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H_ */
