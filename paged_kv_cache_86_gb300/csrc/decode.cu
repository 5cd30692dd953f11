// decode.cu -- split-context paged decode attention for GB300 (sm_103a).
//
// One query token per sequence attends to its context_lens[i] cached tokens,
// read through its block_tables row (nano vllm代码详解 §2 context;
// 推理运行时 §分页 KV: logical block j -> physical block b_j). Decode is bound
// by reading the KV cache (Mini-SGLang 源码解析（二）§8.3: decode is
// memory-bound on KV cache reads), so the design goal is to stream every K/V
// byte exactly once at full HBM bandwidth with all SMs busy whatever the
// length mix.
//
// Three launches on the caller's stream (the all-heads tcgen05 kernel of
// decode_tcg.cu with bf16 caches plans the call itself: two launches):
//   1. plan     one CTA: prefix sums cu[i] of the (range-checked) context
//               lengths and the token-range size W = ceil(total / grid)
//               (rounded up to 16, at least 64).
//   2. split    a persistent grid of `grid` CTAs (every SM, as many CTAs as
//               fit). CTA b owns the flat token range [b*W, (b+1)*W) of the
//               concatenated contexts, so every CTA streams the same number
//               of bytes however long or short the sequences are. Inside a
//               CTA, one producer warp walks the range sequence by sequence
//               and block by block and moves each run of up to
//               16 KB / (Hkv * row bytes) tokens of one physical block into
//               a shared-memory stage with two bulk TMA copies (K and V; a
//               run of one block is contiguous across all KV heads in the
//               [NB, bs, Hkv, D] layout); a stage over blocks shorter than
//               it takes one such pair of copies per block it touches. Eight
//               consumer warps each take one KV head and an 8-token slice of
//               the stage (16 with fp8 codes, whose rows are half the
//               bytes and are expanded to fp32 as they are read): the G query heads
//               of the group are scored together (K is read from shared
//               memory once per group), scores are reduced across the 16
//               lanes of a half-warp with a reduce-scatter of shuffles, the
//               online softmax (base 2; q is pre-scaled by scale*log2 e) is
//               updated once per stage, and P*V is accumulated with packed
//               fp32x2 FMAs. A sequence wholly inside one range is
//               normalised and written as bf16 directly; a sequence cut by a
//               range boundary leaves a partial (o/l, m, l) for each of its
//               pieces.
//   3. combine  one warp per (sequence, query head) merges the partials of cut sequences
//               with the log-sum-exp rule  M = max m_s,
//               o = sum_s l_s 2^(m_s - M) o_s / sum_s l_s 2^(m_s - M),
//               and writes zero rows for empty sequences.
#include <cuda_runtime.h>
#include <math.h>

#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr int kHeadDim = 128;
constexpr int kHeadBytes = kHeadDim * 2;      // one token of one KV head, bf16
constexpr int kConsumerWarps = 8;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kStages = 3;
constexpr int kStageBytes = 32768;            // K half + V half
constexpr int kTokensPerWarp = 8;             // stage tokens per consumer warp (bf16; fp8 twice)
constexpr int kMinRange = 64;
constexpr float kLog2e = 1.4426950408889634f;
constexpr unsigned kFull = 0xffffffffu;

enum : int { kFirst = 1, kLast = 2, kEnd = 4, kSkip = 8 };

struct StageDesc {
  int seq, pos, ntok, flags, slot, pad0, pad1, pad2;
};

// Workspace: a 256-byte header, cu[S+1], then the partial results.
struct Header {
  int total;   // sum of clamped context lengths
  int range;   // tokens per CTA range (W)
};

__host__ __device__ inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

struct WsLayout {
  size_t cu, ml, o, total;
  int entries;  // partial (o, m, l) records per query head
};

__host__ __device__ inline WsLayout ws_layout(int num_seqs, int num_q_heads, int wph, int grid) {
  WsLayout l;
  l.cu = 256;
  const int entries = 2 * grid * wph + (wph > 1 ? num_seqs * wph : 0);
  l.entries = entries;
  l.ml = align256(l.cu + sizeof(int) * (size_t(num_seqs) + 1));
  l.o = align256(l.ml + sizeof(float2) * size_t(entries) * num_q_heads);
  l.total = align256(l.o + sizeof(float) * size_t(entries) * num_q_heads * kHeadDim);
  return l;
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ------------------------------------------------------------------ plan --

// units_per_token: 1 when a CTA range covers tokens of all KV heads (split
// kernel), num_kv_heads when it covers (KV head, token) pairs (tcgen05 kernel).
// Decode step: the newest token row of each sequence, written by the plan
// launch's CTAs 1.. while CTA 0 computes the prefix sums (key == nullptr: none).
constexpr int kStoreSeqsPerCta = 8;   // decode step: new rows written by four warps per sequence

struct NewTokens {
  const uint4 *key;
  const uint4 *value;
  uint4 *k_cache;
  uint4 *v_cache;
  const int32_t *block_tables;
  int max_blocks_per_seq;
  int block_size;
  int num_blocks;
  int row_vecs;              // 16-byte vectors per token row (Hkv * 128 bf16)
  int64_t key_stride_vecs;
  int64_t value_stride_vecs;
  // fp8 E4M3 caches: each (token, KV head) row is quantized on the way in, its
  // codes to k_cache / v_cache ([slots, Hkv, 128] bytes) and its scale to
  // k_scales / v_scales ([slots, Hkv])
  int fp8;
  int num_kv_heads;
  float *k_scales;
  float *v_scales;
};

__global__ void __launch_bounds__(1024)
decode_plan_kernel(const int32_t *__restrict__ context_lens, int num_seqs, int max_context_len,
                   int grid, int units_per_token, int min_range, int seg_cost, uint8_t *ws,
                   uint32_t *err, NewTokens nt) {
  __shared__ int warp_sums[32];
  __shared__ int base;
  int *cu = reinterpret_cast<int *>(ws + 256);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  // the attention kernel is launched as a programmatic dependent of this one:
  // it may start its prologue now and waits for this grid before reading
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (blockIdx.x > 0) {
    // Decode step: four warps per sequence (eight sequences per CTA, so the
    // rows spread over many SMs) write its newest token at logical position
    // n - 1, n = context_lens[i] clamped to [0, max_context_len] as below
    // (n = 0 writes nothing): row (n-1) % bs of block block_tables[i][(n-1) / bs].
    // Over fp8 caches each (token, KV head) row is quantized on the way in, as
    // the fp8 store does it. The decode kernel that reads the cache is the next
    // launch on the stream.
    const int i = (blockIdx.x - 1) * kStoreSeqsPerCta + (warp >> 2);
    const int part = warp & 3;
    if (i >= num_seqs) return;
    int n = context_lens[i];
    n = n < 0 ? 0 : (n > max_context_len ? max_context_len : n);
    if (n == 0) return;
    const int pos = n - 1;
    const int blk = nt.block_tables[static_cast<int64_t>(i) * nt.max_blocks_per_seq + pos / nt.block_size];
    if (blk < 0 || blk >= nt.num_blocks) {
      if (lane == 0) raise_error(err, PKV_DEVERR_BLOCK_ID);
      return;
    }
    const int64_t row = static_cast<int64_t>(blk) * nt.block_size + pos % nt.block_size;
    if (nt.fp8) {
      const uint2 *kin = reinterpret_cast<const uint2 *>(nt.key) + i * nt.key_stride_vecs * 2;
      const uint2 *vin = reinterpret_cast<const uint2 *>(nt.value) + i * nt.value_stride_vecs * 2;
      for (int h = part; h < nt.num_kv_heads; h += 4) {
        const int64_t r8 = row * nt.num_kv_heads + h;
        const uint2 kb = __ldg(kin + h * 32 + lane);
        const uint2 vb = __ldg(vin + h * 32 + lane);
        quantize_row_e4m3(kb, reinterpret_cast<uint32_t *>(nt.k_cache) + r8 * 32, nt.k_scales + r8, lane);
        quantize_row_e4m3(vb, reinterpret_cast<uint32_t *>(nt.v_cache) + r8 * 32, nt.v_scales + r8, lane);
      }
      return;
    }
    for (int v = part * 32 + lane; v < nt.row_vecs; v += 128) {
      const uint4 kv = __ldg(nt.key + i * nt.key_stride_vecs + v);
      const uint4 vv = __ldg(nt.value + i * nt.value_stride_vecs + v);
      nt.k_cache[row * nt.row_vecs + v] = kv;
      nt.v_cache[row * nt.row_vecs + v] = vv;
    }
    return;
  }
  if (threadIdx.x == 0) {
    base = 0;
    cu[0] = 0;
  }
  __syncthreads();
  for (int start = 0; start < num_seqs; start += 1024) {
    const int i = start + threadIdx.x;
    int x = 0;
    if (i < num_seqs) {
      x = context_lens[i];
      if (x < 0 || x > max_context_len) {
        raise_error(err, PKV_DEVERR_LENGTH);
        x = x < 0 ? 0 : max_context_len;
      }
    }
    // a non-empty sequence takes seg_cost units of the flat space in front of
    // its tokens (the fixed cost of a segment, so ranges balance time)
    int v = x > 0 ? x + seg_cost : 0;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(kFull, v, off);
      if (lane >= off) v += y;
    }
    if (lane == 31) warp_sums[warp] = v;
    __syncthreads();
    if (warp == 0) {
      int w = warp_sums[lane];
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(kFull, w, off);
        if (lane >= off) w += y;
      }
      warp_sums[lane] = w;
    }
    __syncthreads();
    const int incl = v + (warp > 0 ? warp_sums[warp - 1] : 0);
    if (i < num_seqs) cu[i + 1] = base + incl;
    __syncthreads();
    if (threadIdx.x == 1023) base += incl;
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    Header *h = reinterpret_cast<Header *>(ws);
    const int total = base;
    const long long units = static_cast<long long>(total) * units_per_token;
    long long range = (units + grid - 1) / grid;
    range = (range + 15) / 16 * 16;
    h->total = total;
    h->range = static_cast<int>(range < min_range ? min_range : range);
  }
}

// ----------------------------------------------------------------- split --

struct SplitParams {
  __nv_bfloat16 *out;
  const __nv_bfloat16 *q;
  const uint8_t *k_cache;
  const uint8_t *v_cache;
  const int32_t *block_tables;
  int max_blocks_per_seq;
  int num_seqs;
  int num_q_heads;
  int num_kv_heads;
  int block_size;
  int num_blocks;
  float qscale;  // scale * log2(e)
  const uint8_t *ws;
  float2 *ml;    // partial (m, l) records
  float *po;     // partial normalised outputs
  uint32_t *err;
  const float *k_scales;  // fp8 caches: [NB * bs, Hkv] row scales
  const float *v_scales;
};

// A consumer warp takes kTokensPerWarp tokens of a stage (fp8 caches, whose
// rows are half the bytes: twice as many), so a stage holds
// kConsumerWarps * tokens-per-warp / Hkv tokens of all KV heads; with fp8 caches
// their row scales (token-major, one per KV head) sit beside it. Shared memory
// is laid out for the larger fp8 counts.
constexpr int kTokensPerWarpMax = 2 * kTokensPerWarp;
constexpr int kScaleEntriesMax = kConsumerWarps * kTokensPerWarpMax;

// Two E4M3 codes (the first in the low byte) -> two floats, exactly.
__device__ __forceinline__ float2 e4m3x2_to_float2(uint32_t codes) {
  uint32_t h;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"(static_cast<unsigned short>(codes & 0xffffu)));
  return __half22float2(*reinterpret_cast<const __half2 *>(&h));
}

__device__ __forceinline__ uint2 lds64(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}

template <int G>
struct GroupTraits {
  static constexpr int kLogG = G == 1 ? 0 : G == 2 ? 1 : G == 4 ? 2 : 3;
  static constexpr int kScatterShift = 4 - kLogG;  // head of a lane after the reduce-scatter
};

// F8: the caches hold E4M3 codes with a scale per (token, KV head) row; the
// codes are expanded on the CUDA cores and the scales applied to the scores
// (K) and to the softmax weights (V).
template <int G, bool F8>
__global__ void __launch_bounds__(kThreads, G <= 4 ? 2 : 1)
decode_split_kernel(const SplitParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t *stage_base = smem;
  uint64_t *full_bar = reinterpret_cast<uint64_t *>(smem + kStages * kStageBytes);
  uint64_t *empty_bar = full_bar + kStages;
  StageDesc *desc = reinterpret_cast<StageDesc *>(empty_bar + kStages);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(desc + kStages);
  constexpr int kTPW = F8 ? kTokensPerWarpMax : kTokensPerWarp;  // tokens per consumer warp
  constexpr int kEntries = kConsumerWarps * kTPW;  // (token, KV head) entries of a stage
  constexpr int kRowsPerLane = kEntries / 32;      // token rows a lane copies (one KV head)
  float *scale_buf = reinterpret_cast<float *>(desc + kStages) + 32;  // [stage][K, V][entry]
  float *score_buf = scale_buf + kStages * 2 * kScaleEntriesMax;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const Header hdr = *reinterpret_cast<const Header *>(p.ws);
  const int *cu = reinterpret_cast<const int *>(p.ws + 256);
  const int lo = static_cast<int>(blockIdx.x) * hdr.range;
  const int hi = min(lo + hdr.range, hdr.total);
  constexpr int head_bytes = F8 ? kHeadDim : kHeadBytes;  // one token of one KV head
  const int row_bytes = p.num_kv_heads * head_bytes;
  const int wph = kConsumerWarps / p.num_kv_heads;  // consumer warps per KV head

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_addr(&full_bar[s]), 1);
      mbar_init(smem_addr(&empty_bar[s]), kConsumerWarps);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();

  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------ producer
    // tokens a stage's consumer warps take (bf16: the whole K half of a stage)
    const int stage_tokens = kEntries / p.num_kv_heads;
    const uint64_t policy = l2_policy_evict_first();
    int issued = 0;
    bool ok = true;

    // Arms one stage; returns false (and arms nothing) once waiting for a free
    // stage has given up.
    auto issue = [&](int seq, int pos, int ntok, int flags, int slot, int blk, int off) {
      const int s = issued % kStages;
      const uint32_t round = static_cast<uint32_t>(issued / kStages);
      int good = 1;
      if (lane == 0 && round > 0 && !mbar_wait(smem_addr(&empty_bar[s]), (round - 1) & 1, abort_flag)) {
        good = 0;
        *abort_flag = 1;
        raise_error(p.err, PKV_DEVERR_TIMEOUT);
      }
      if constexpr (F8) {  // the rows' scales, written before the stage is armed
        good = __shfl_sync(kFull, good, 0);
        if (good && (flags & kEnd) == 0 && blk >= 0 && blk < p.num_blocks) {
          float *sk = scale_buf + s * 2 * kEntries;
          const int64_t r0 = (static_cast<int64_t>(blk) * p.block_size + off) * p.num_kv_heads;
          for (int e = lane; e < ntok * p.num_kv_heads; e += 32) {
            sk[e] = __ldg(p.k_scales + r0 + e);
            sk[kEntries + e] = __ldg(p.v_scales + r0 + e);
          }
        }
        __syncwarp();
      }
      if (lane == 0) {
        if (good) {
          const bool valid = (flags & kEnd) == 0 && blk >= 0 && blk < p.num_blocks;
          if ((flags & kEnd) == 0 && !valid) {
            flags |= kSkip;
            raise_error(p.err, PKV_DEVERR_BLOCK_ID);
          }
          StageDesc d;
          d.seq = seq; d.pos = pos; d.ntok = ntok; d.flags = flags; d.slot = slot;
          d.pad0 = d.pad1 = d.pad2 = 0;
          desc[s] = d;
          const uint32_t fb = smem_addr(&full_bar[s]);
          if (valid) {
            const uint32_t bytes = static_cast<uint32_t>(ntok * row_bytes);
            mbar_arrive_expect_tx(fb, 2 * bytes);
            const size_t src = (static_cast<size_t>(blk) * p.block_size + off) * row_bytes;
            const uint32_t dst = smem_addr(stage_base + s * kStageBytes);
            bulk_g2s(dst, p.k_cache + src, bytes, fb, policy);
            bulk_g2s(dst + kStageBytes / 2, p.v_cache + src, bytes, fb, policy);
          } else {
            mbar_arrive(fb);
          }
        }
      }
      good = __shfl_sync(kFull, good, 0);
      if (good) ++issued;
      return good != 0;
    };

    // Blocks shorter than a stage: one stage takes ntok consecutive tokens of
    // the sequence over several blocks. Lane c copies the run of the stage's
    // tokens that lies in the c-th block it touches (and runs c + 32, ...
    // when there are more than 32), K and V, as one copy each. A block id out
    // of range skips the whole stage.
    auto issue_rows = [&](int seq, int pos, int ntok, int flags, int slot, const int32_t *row) {
      const int s = issued % kStages;
      const uint32_t round = static_cast<uint32_t>(issued / kStages);
      const int lb0 = pos / p.block_size;
      const int nruns = (pos + ntok - 1) / p.block_size - lb0 + 1;  // <= ntok
      int blk[kRowsPerLane];
      bool bad = false;
#pragma unroll
      for (int u = 0; u < kRowsPerLane; ++u) {
        blk[u] = 0;
        const int c = lane + 32 * u;
        if (c < nruns) {
          blk[u] = __ldg(row + lb0 + c);
          bad |= blk[u] < 0 || blk[u] >= p.num_blocks;
        }
      }
      bad = __any_sync(kFull, bad);
      const uint32_t fb = smem_addr(&full_bar[s]);
      int good = 1;
      if (lane == 0 && round > 0 && !mbar_wait(smem_addr(&empty_bar[s]), (round - 1) & 1, abort_flag)) {
        good = 0;
        *abort_flag = 1;
        raise_error(p.err, PKV_DEVERR_TIMEOUT);
      }
      if constexpr (F8) {  // the rows' scales, written before the stage is armed
        good = __shfl_sync(kFull, good, 0);
        float *sk = scale_buf + s * 2 * kEntries;
        for (int e = lane; e < kEntries && good && !bad; e += 32) {
          // entry e: token e / Hkv, in run c (its block held by lane c & 31 in blk[c >> 5])
          const int t = e / p.num_kv_heads;
          const int c = (pos + t) / p.block_size - lb0;
          int b = 0;
#pragma unroll
          for (int u = 0; u < kRowsPerLane; ++u) {
            const int bu = __shfl_sync(kFull, blk[u], c & 31);
            if ((c >> 5) == u) b = bu;
          }
          if (e < ntok * p.num_kv_heads) {
            const int64_t rr = (static_cast<int64_t>(b) * p.block_size + (pos + t) % p.block_size) *
                                   p.num_kv_heads + e % p.num_kv_heads;
            sk[e] = __ldg(p.k_scales + rr);
            sk[kEntries + e] = __ldg(p.v_scales + rr);
          }
        }
        __syncwarp();
      }
      if (lane == 0) {
        if (good) {
          if (bad) {
            flags |= kSkip;
            raise_error(p.err, PKV_DEVERR_BLOCK_ID);
          }
          StageDesc d;
          d.seq = seq; d.pos = pos; d.ntok = ntok; d.flags = flags; d.slot = slot;
          d.pad0 = d.pad1 = d.pad2 = 0;
          desc[s] = d;
          if (bad) mbar_arrive(fb);
          else mbar_arrive_expect_tx(fb, static_cast<uint32_t>(2 * ntok * row_bytes));
        }
      }
      good = __shfl_sync(kFull, good, 0);  // (also orders lane 0's expect_tx before the copies)
      if (good && !bad) {
        const uint64_t policy_rows = l2_policy_evict_first();
        const uint32_t dst0 = smem_addr(stage_base + s * kStageBytes);
#pragma unroll
        for (int u = 0; u < kRowsPerLane; ++u) {
          const int c = lane + 32 * u;
          if (c < nruns) {
            const int a = max(pos, (lb0 + c) * p.block_size);            // first token of the run
            const int e = min(pos + ntok, (lb0 + c + 1) * p.block_size);  // one past its last
            const size_t src = (static_cast<size_t>(blk[u]) * p.block_size + a % p.block_size) *
                               row_bytes;
            const uint32_t dst = dst0 + (a - pos) * row_bytes;
            const uint32_t bytes = static_cast<uint32_t>((e - a) * row_bytes);
            bulk_g2s(dst, p.k_cache + src, bytes, fb, policy_rows);
            bulk_g2s(dst + kStageBytes / 2, p.v_cache + src, bytes, fb, policy_rows);
          }
        }
      }
      if (good) ++issued;
      return good != 0;
    };

    if (lo < hi) {
      // first sequence whose tokens reach past lo
      int a = 0, b = p.num_seqs - 1;
      while (a < b) {
        const int m = (a + b) >> 1;
        if (cu[m + 1] > lo) b = m; else a = m + 1;
      }
      for (int i = a; ok && i < p.num_seqs; ++i) {
        const int c0 = cu[i], c1 = cu[i + 1];
        if (c0 >= hi) break;
        if (c1 == c0) continue;
        const int seg_lo = max(lo, c0) - c0;
        const int seg_hi = min(hi, c1) - c0;
        const bool complete = c0 >= lo && c1 <= hi;
        const int slot = complete ? -1 : (c0 <= lo ? 2 * int(blockIdx.x) : 2 * int(blockIdx.x) + 1);
        const int32_t *row = p.block_tables + static_cast<size_t>(i) * p.max_blocks_per_seq;
        int cached = -1 << 30, my_id = -1;
        bool first = true;
        for (int pos = seg_lo; ok && pos < seg_hi && p.block_size < stage_tokens;) {
          const int ntok = min(stage_tokens, seg_hi - pos);
          const int flags = (first ? kFirst : 0) | (pos + ntok == seg_hi ? kLast : 0);
          first = false;
          ok = issue_rows(i, pos, ntok, flags, slot, row);
          pos += ntok;
        }
        for (int pos = seg_lo; ok && pos < seg_hi && p.block_size >= stage_tokens;) {
          const int lb = pos / p.block_size;
          const int off = pos - lb * p.block_size;
          const int ntok = min(min(stage_tokens, p.block_size - off), seg_hi - pos);
          if (lb < cached || lb >= cached + 32) {  // refill the window of 32 block ids
            cached = lb;
            my_id = lb + lane < p.max_blocks_per_seq ? __ldg(row + lb + lane) : -1;
          }
          const int blk = __shfl_sync(kFull, my_id, lb - cached);
          const int flags = (first ? kFirst : 0) | (pos + ntok == seg_hi ? kLast : 0);
          first = false;
          ok = issue(i, pos, ntok, flags, slot, blk, off);
          pos += ntok;
        }
      }
    }
    if (ok) ok = issue(0, 0, 0, kEnd, -1, 0, 0);
    // Drain: every copy this CTA issued must land before its shared memory goes away.
    if (lane == 0) {
      const int first = issued > kStages ? issued - kStages : 0;
      for (int k = first; k < issued; ++k)
        mbar_wait(smem_addr(&full_bar[k % kStages]), (k / kStages) & 1, nullptr);
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  using Tr = GroupTraits<G>;
  const int head = warp % p.num_kv_heads;
  const int sub = warp / p.num_kv_heads;
  const int hf = lane >> 4;
  const int l16 = lane & 15;
  const int my_head_after_scatter = l16 >> Tr::kScatterShift;
  const bool score_writer = (l16 & ((16 / G) - 1)) == 0;
  const int own_g = lane & (G - 1);  // head whose score sum this lane keeps
  float *sc = score_buf + warp * kTPW * G;

  float2 q2[G][4];
  float2 acc[G][4];
  float m_run[G];
  float l_part = 0.f;

  for (int k = 0;; ++k) {
    const int s = k % kStages;
    if (!__all_sync(kFull, mbar_wait(smem_addr(&full_bar[s]), (k / kStages) & 1, abort_flag))) {
      if (lane == 0) {
        *abort_flag = 1;
        raise_error(p.err, PKV_DEVERR_TIMEOUT);
      }
      break;
    }
    const StageDesc d = desc[s];
    if (d.flags & kEnd) break;

    if (d.flags & kFirst) {
      const uint4 *qrow = reinterpret_cast<const uint4 *>(
          p.q + (static_cast<size_t>(d.seq) * p.num_q_heads + head * G) * kHeadDim);
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const uint4 raw = __ldg(qrow + g * (kHeadDim / 8) + l16);
        const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const float2 f = bf16x2_to_float2(w[c]);
          q2[g][c] = make_float2(f.x * p.qscale, f.y * p.qscale);
          acc[g][c] = make_float2(0.f, 0.f);
        }
        m_run[g] = -INFINITY;
      }
      l_part = 0.f;
    }

    const int t0 = sub * kTPW;
    const int nw = (d.flags & kSkip) ? 0 : min(max(d.ntok - t0, 0), kTPW);
    if (nw > 0) {
      // lane l16 of each half-warp holds dims 8 l16 .. 8 l16 + 7 of a row
      const uint32_t kb = smem_addr(stage_base + s * kStageBytes) + t0 * row_bytes +
                          head * head_bytes + l16 * (head_bytes / 16);
      const uint32_t vb = kb + kStageBytes / 2;
      // fp8: row scales of this warp's tokens, entry (token, KV head)
      const float *sks = scale_buf + s * 2 * kEntries + t0 * p.num_kv_heads + head;

      // scores of this warp's tokens, two tokens (one per half-warp) at a time
      for (int it = 0; it < (nw + 1) >> 1; ++it) {
        const int j = 2 * it + hf;
        float2 k0, k1, k2, k3;
        if constexpr (F8) {
          const uint2 kr = lds64(kb + j * row_bytes);
          k0 = e4m3x2_to_float2(kr.x); k1 = e4m3x2_to_float2(kr.x >> 16);
          k2 = e4m3x2_to_float2(kr.y); k3 = e4m3x2_to_float2(kr.y >> 16);
        } else {
          const uint4 kr = lds128(kb + j * row_bytes);
          k0 = bf16x2_to_float2(kr.x); k1 = bf16x2_to_float2(kr.y);
          k2 = bf16x2_to_float2(kr.z); k3 = bf16x2_to_float2(kr.w);
        }
        // (fp8: the K row's scale multiplies the dot product; j past nw reads
        // an unused entry of the stage)
        const float kscale = F8 ? sks[j * p.num_kv_heads] : 1.f;
        float sv[G];
#pragma unroll
        for (int g = 0; g < G; ++g) {
          float2 a2 = fmul2(q2[g][0], k0);
          a2 = ffma2(q2[g][1], k1, a2);
          a2 = ffma2(q2[g][2], k2, a2);
          a2 = ffma2(q2[g][3], k3, a2);
          sv[g] = (a2.x + a2.y) * kscale;
        }
        // reduce-scatter over the 16 lanes of the half-warp: each level halves
        // the heads a lane keeps and adds its partner's copy of them
#pragma unroll
        for (int n = G, off = 8; n > 1; n >>= 1, off >>= 1) {
          const bool up = (lane & off) != 0;
#pragma unroll
          for (int i2 = 0; i2 < n / 2; ++i2) {
            const float send = up ? sv[i2] : sv[i2 + n / 2];
            const float keep = up ? sv[i2 + n / 2] : sv[i2];
            sv[i2] = keep + __shfl_xor_sync(kFull, send, off);
          }
        }
#pragma unroll
        for (int off = 8 >> Tr::kLogG; off >= 1; off >>= 1)
          sv[0] += __shfl_xor_sync(kFull, sv[0], off);
        if (j < nw && score_writer) sc[j * G + my_head_after_scatter] = sv[0];
      }
      __syncwarp();

      // online softmax update, once per stage: entry e = token * G + head, lane
      // l holding entries l, l + 32, ... (all of head l % G)
      constexpr int kVals = (kTPW * G + 31) / 32;
      const int ne = nw * G;
      float vals[kVals];
      float mx = -INFINITY;
#pragma unroll
      for (int u = 0; u < kVals; ++u) {
        vals[u] = lane + 32 * u < ne ? sc[lane + 32 * u] : -INFINITY;
        mx = fmaxf(mx, vals[u]);
      }
#pragma unroll
      for (int off = 16; off >= G; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, off));
      float alpha[G];
      float m_own = 0.f, alpha_own = 1.f;
      bool rescale = false;
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float stage_max = __shfl_sync(kFull, mx, g);
        const float m_new = fmaxf(m_run[g], stage_max);
        alpha[g] = fast_exp2(m_run[g] - m_new);
        rescale |= alpha[g] != 1.f;
        m_run[g] = m_new;
        if (own_g == g) {
          m_own = m_new;
          alpha_own = alpha[g];
        }
      }
      float psum = 0.f;
#pragma unroll
      for (int u = 0; u < kVals; ++u) {
        if (lane + 32 * u < ne) {
          const float pu = fast_exp2(vals[u] - m_own);
          sc[lane + 32 * u] = pu;
          psum += pu;
        }
      }
      l_part = l_part * alpha_own + psum;
      if (rescale) {
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float2 a2 = make_float2(alpha[g], alpha[g]);
#pragma unroll
          for (int c = 0; c < 4; ++c) acc[g][c] = fmul2(acc[g][c], a2);
        }
      }
      __syncwarp();

      // P * V (fp8: the V row's scale multiplies the softmax weights)
      for (int j = hf; j < nw; j += 2) {
        float2 v0f, v1f, v2f, v3f;
        if constexpr (F8) {
          const uint2 vr = lds64(vb + j * row_bytes);
          v0f = e4m3x2_to_float2(vr.x); v1f = e4m3x2_to_float2(vr.x >> 16);
          v2f = e4m3x2_to_float2(vr.y); v3f = e4m3x2_to_float2(vr.y >> 16);
        } else {
          const uint4 vr = lds128(vb + j * row_bytes);
          v0f = bf16x2_to_float2(vr.x); v1f = bf16x2_to_float2(vr.y);
          v2f = bf16x2_to_float2(vr.z); v3f = bf16x2_to_float2(vr.w);
        }
        const float vscale = F8 ? sks[kEntries + j * p.num_kv_heads] : 1.f;
        float pj[G];
        if constexpr (G == 1) {
          pj[0] = sc[j];
        } else if constexpr (G == 2) {
          const float2 t = *reinterpret_cast<const float2 *>(sc + j * 2);
          pj[0] = t.x; pj[1] = t.y;
        } else {
#pragma unroll
          for (int g4 = 0; g4 < G; g4 += 4) {
            const float4 t = *reinterpret_cast<const float4 *>(sc + j * G + g4);
            pj[g4] = t.x; pj[g4 + 1] = t.y; pj[g4 + 2] = t.z; pj[g4 + 3] = t.w;
          }
        }
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float2 pp = make_float2(pj[g] * vscale, pj[g] * vscale);
          acc[g][0] = ffma2(pp, v0f, acc[g][0]);
          acc[g][1] = ffma2(pp, v1f, acc[g][1]);
          acc[g][2] = ffma2(pp, v2f, acc[g][2]);
          acc[g][3] = ffma2(pp, v3f, acc[g][3]);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_addr(&empty_bar[s]));

    if (d.flags & kLast) {
      // fold the two half-warps and the per-lane softmax sums
#pragma unroll
      for (int g = 0; g < G; ++g)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          acc[g][c].x += __shfl_xor_sync(kFull, acc[g][c].x, 16);
          acc[g][c].y += __shfl_xor_sync(kFull, acc[g][c].y, 16);
        }
      float lt = l_part;
#pragma unroll
      for (int off = 16; off >= G; off >>= 1) lt += __shfl_xor_sync(kFull, lt, off);
      float l_sum[G];
#pragma unroll
      for (int g = 0; g < G; ++g) l_sum[g] = __shfl_sync(kFull, lt, g);

      if (wph == 1 && d.slot < 0) {
        if (hf == 0) {
#pragma unroll
          for (int g = 0; g < G; ++g) {
            const float inv = l_sum[g] > 0.f ? 1.f / l_sum[g] : 0.f;
            uint4 o;
            o.x = float2_to_bf16x2(acc[g][0].x * inv, acc[g][0].y * inv);
            o.y = float2_to_bf16x2(acc[g][1].x * inv, acc[g][1].y * inv);
            o.z = float2_to_bf16x2(acc[g][2].x * inv, acc[g][2].y * inv);
            o.w = float2_to_bf16x2(acc[g][3].x * inv, acc[g][3].y * inv);
            uint4 *dst = reinterpret_cast<uint4 *>(
                p.out + (static_cast<size_t>(d.seq) * p.num_q_heads + head * G + g) * kHeadDim);
            dst[l16] = o;
          }
        }
      } else {
        const int entry = d.slot >= 0 ? d.slot * wph + sub
                                      : 2 * int(gridDim.x) * wph + d.seq * wph + sub;
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const int qh = head * G + g;
          const size_t rec = static_cast<size_t>(entry) * p.num_q_heads + qh;
          const float inv = l_sum[g] > 0.f ? 1.f / l_sum[g] : 0.f;
          if (hf == 0) {
            float4 *dst = reinterpret_cast<float4 *>(p.po + rec * kHeadDim) + l16 * 2;
            dst[0] = make_float4(acc[g][0].x * inv, acc[g][0].y * inv, acc[g][1].x * inv,
                                 acc[g][1].y * inv);
            dst[1] = make_float4(acc[g][2].x * inv, acc[g][2].y * inv, acc[g][3].x * inv,
                                 acc[g][3].y * inv);
          }
          if (lane == 0) p.ml[rec] = make_float2(m_run[g], l_sum[g]);
        }
      }
    }
  }
}

// --------------------------------------------------------------- combine --

struct CombineParams {
  __nv_bfloat16 *out;
  const uint8_t *ws;
  const float2 *ml;
  const float *po;
  int num_seqs;
  int num_q_heads;
  int wph;
  int grid;
  int tc;      // records of the tcgen05 kernel: one row per (slot, query head of the group)
  int group;
  int seg_cost;  // units in front of each non-empty sequence in the flat space (see the plan)
};

// One warp per (sequence, query head); lane l owns dims 4l .. 4l+3. The
// partial records of the sequence are enumerated in order; lanes first load
// (m, l) of records lane, lane+32, ... so every load of a pass is independent.
// Returns the record row: ml[row], po[row * 128 ..].
__device__ __forceinline__ long long combine_row(const CombineParams &p, int i, int qh,
                                                 long long start, int range, long long b_first,
                                                 bool complete, int k) {
  if (p.tc) {
    const long long b = b_first + k;
    const long long slot = (b == b_first && start > b * range) ? 2 * b + 1 : 2 * b;
    return slot * p.group + qh % p.group;
  }
  long long rec;
  if (complete) {
    rec = 2LL * p.grid * p.wph + static_cast<long long>(i) * p.wph + k;
  } else {
    const long long b = b_first + k / p.wph;
    const long long slot = (b == b_first && start > b * range) ? 2 * b + 1 : 2 * b;
    rec = slot * p.wph + k % p.wph;
  }
  return rec * p.num_q_heads + qh;
}

constexpr int kCombineWarps = 8;

__global__ void __launch_bounds__(kCombineWarps * 32) decode_combine_kernel(const CombineParams p) {
  // launched as a programmatic dependent of the attention kernel (a no-op otherwise)
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int lane = threadIdx.x & 31;
  const int gw = blockIdx.x * kCombineWarps + (threadIdx.x >> 5);
  if (gw >= p.num_seqs * p.num_q_heads) return;
  const int i = gw / p.num_q_heads;
  const int qh = gw - i * p.num_q_heads;
  const Header hdr = *reinterpret_cast<const Header *>(p.ws);
  const int *cu = reinterpret_cast<const int *>(p.ws + 256);
  const int v0 = cu[i], c1 = cu[i + 1];
  uint2 *orow = reinterpret_cast<uint2 *>(p.out + (static_cast<size_t>(i) * p.num_q_heads + qh) * kHeadDim);
  if (c1 == v0) {  // empty context: zero row
    orow[lane] = make_uint2(0u, 0u);
    return;
  }
  const int c0 = v0 + p.seg_cost;  // first token of the sequence in the flat space
  // position of this (head, sequence) in the flat space the CTA ranges cut
  const long long start = p.tc ? static_cast<long long>(qh / p.group) * hdr.total + c0 : c0;
  const long long b_first = start / hdr.range;
  const long long b_last = (start + (c1 - c0) - 1) / hdr.range;
  const bool complete = b_first == b_last;
  if ((p.tc || p.wph == 1) && complete) return;  // written directly by the attention kernel
  const int n = p.tc ? static_cast<int>(b_last - b_first + 1)
                     : (complete ? p.wph : static_cast<int>(b_last - b_first + 1) * p.wph);

  float m_max = -INFINITY;
  for (int k = lane; k < n; k += 32) {
    const long long row = combine_row(p, i, qh, start, hdr.range, b_first, complete, k);
    m_max = fmaxf(m_max, p.ml[row].x);
  }
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) m_max = fmaxf(m_max, __shfl_xor_sync(kFull, m_max, off));

  float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
  float l_tot = 0.f;
  if (m_max != -INFINITY) {
    for (int base = 0; base < n; base += 32) {
      float wk = 0.f;
      long long row_k = 0;
      if (base + lane < n) {
        row_k = combine_row(p, i, qh, start, hdr.range, b_first, complete, base + lane);
        const float2 ml = p.ml[row_k];
        wk = ml.y * fast_exp2(ml.x - m_max);
      }
      const int cnt = min(32, n - base);
      // eight records per pass, all eight loads issued before the sums (the
      // partials sit in L2; the latency of one load per record would add up)
      for (int k0 = 0; k0 < cnt; k0 += 8) {
        float4 v[8];
        float wgt[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int k = min(k0 + u, cnt - 1);  // past the end: a valid row, weight 0
          wgt[u] = __shfl_sync(kFull, wk, k);
          const long long row = __shfl_sync(kFull, row_k, k);
          v[u] = reinterpret_cast<const float4 *>(p.po + row * kHeadDim)[lane];
          if (k0 + u >= cnt) wgt[u] = 0.f;
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          o.x += wgt[u] * v[u].x; o.y += wgt[u] * v[u].y;
          o.z += wgt[u] * v[u].z; o.w += wgt[u] * v[u].w;
          l_tot += wgt[u];
        }
      }
    }
  }
  const float inv = l_tot > 0.f ? 1.f / l_tot : 0.f;
  uint2 packed;
  packed.x = float2_to_bf16x2(o.x * inv, o.y * inv);
  packed.y = float2_to_bf16x2(o.z * inv, o.w * inv);
  orow[lane] = packed;
}

size_t split_smem_bytes(int group) {
  return size_t(kStages) * kStageBytes + 2 * kStages * sizeof(uint64_t) +
         kStages * sizeof(StageDesc) + 32 * sizeof(float) +
         size_t(kStages) * 2 * kScaleEntriesMax * sizeof(float) +
         size_t(kConsumerWarps) * kTokensPerWarpMax * group * sizeof(float);
}

// both instances (bf16, fp8) of a group; the grid follows the bf16 one's
// occupancy (the CTAs wait on none of each other, so more CTAs than fit at
// once only queue)
template <int G>
cudaError_t prepare_split(int *ctas_per_sm) {
  const size_t smem = split_smem_bytes(G);
  cudaError_t e = cudaFuncSetAttribute(decode_split_kernel<G, true>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(decode_split_kernel<G, false>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  if (e != cudaSuccess) return e;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas_per_sm, decode_split_kernel<G, false>,
                                                       kThreads, smem);
}

bool supported_heads(int num_q_heads, int num_kv_heads) {
  if (num_kv_heads != 1 && num_kv_heads != 2 && num_kv_heads != 4 && num_kv_heads != 8) return false;
  if (num_q_heads % num_kv_heads != 0) return false;
  const int g = num_q_heads / num_kv_heads;
  return g == 1 || g == 2 || g == 4 || g == 8;
}

}  // namespace

int split_grid(int num_q_heads, int num_kv_heads, cudaError_t *status) {
  *status = cudaSuccess;
  if (!supported_heads(num_q_heads, num_kv_heads)) return 0;
  int dev = 0;
  if ((*status = cudaGetDevice(&dev)) != cudaSuccess) return 0;
  int per_sm = 0;
  switch (num_q_heads / num_kv_heads) {
    case 1: *status = prepare_split<1>(&per_sm); break;
    case 2: *status = prepare_split<2>(&per_sm); break;
    case 4: *status = prepare_split<4>(&per_sm); break;
    default: *status = prepare_split<8>(&per_sm); break;
  }
  if (*status != cudaSuccess || per_sm < 1) return 0;
  return per_sm * sm_count(dev);
}

// Mixed batch: sequences 0..D-1 are decode sequences (one query row each, rows
// 0..D-1); their context lengths are the differences of cu_seqlens_k. A layout
// that breaks this (a decode sequence with other than one query row) is
// reported as PKV_DEVERR_LENGTH.
__global__ void mixed_decode_lens_kernel(const int32_t *__restrict__ cu_q,
                                         const int32_t *__restrict__ cu_k, int num_decode,
                                         int32_t *__restrict__ lens, uint32_t *err) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= num_decode) return;
  lens[i] = cu_k[i + 1] - cu_k[i];
  if (cu_q[i] != i || cu_q[i + 1] != i + 1) raise_error(err, PKV_DEVERR_LENGTH);
}

cudaError_t launch_mixed_decode_lens(const int32_t *cu_q, const int32_t *cu_k, int num_decode,
                                     int32_t *lens, uint32_t *err, cudaStream_t stream) {
  if (num_decode == 0) return cudaSuccess;
  mixed_decode_lens_kernel<<<(num_decode + 255) / 256, 256, 0, stream>>>(cu_q, cu_k, num_decode,
                                                                         lens, err);
  return cudaGetLastError();
}

// The plan launch: CTA 0 plans the ranges; with new tokens (decode step), CTAs
// 1.. write them, 32 sequences per CTA.
cudaError_t launch_plan(const DecodeArgs &a, int grid, int units_per_token, int min_range,
                        int seg_cost, uint8_t *ws, cudaStream_t stream) {
  NewTokens nt{};
  unsigned ctas = 1;
  if (a.key_new != nullptr) {
    nt.key = static_cast<const uint4 *>(a.key_new);
    nt.value = static_cast<const uint4 *>(a.value_new);
    nt.k_cache = static_cast<uint4 *>(const_cast<void *>(a.k_cache));
    nt.v_cache = static_cast<uint4 *>(const_cast<void *>(a.v_cache));
    nt.block_tables = a.block_tables;
    nt.max_blocks_per_seq = a.max_blocks_per_seq;
    nt.block_size = a.block_size;
    nt.num_blocks = a.num_blocks;
    nt.row_vecs = a.num_kv_heads * (kHeadDim / 8);
    nt.key_stride_vecs = a.key_stride / 8;
    nt.value_stride_vecs = a.value_stride / 8;
    nt.fp8 = a.fp8 ? 1 : 0;
    nt.num_kv_heads = a.num_kv_heads;
    nt.k_scales = const_cast<float *>(a.k_scales);
    nt.v_scales = const_cast<float *>(a.v_scales);
    ctas += static_cast<unsigned>((a.num_seqs + kStoreSeqsPerCta - 1) / kStoreSeqsPerCta);
  }
  decode_plan_kernel<<<ctas, 1024, 0, stream>>>(a.context_lens, a.num_seqs, a.max_context_len,
                                                grid, units_per_token, min_range, seg_cost, ws,
                                                a.err, nt);
  return cudaGetLastError();
}

size_t tc_workspace(int num_seqs, int group, int grid) {
  const size_t rows = size_t(2) * grid * group;
  const size_t ml = align256(256 + sizeof(int) * (size_t(num_seqs) + 1));
  const size_t o = align256(ml + sizeof(float2) * rows);
  return align256(o + sizeof(float) * rows * kHeadDim);
}

bool choose_decode_plan(int num_q_heads, int num_kv_heads, int block_size, DecodePlan *plan,
                        cudaError_t *status, bool fp8) {
  *status = cudaSuccess;
  // fp8 caches: the all-heads tcgen05 kernel where its fp8 instance applies,
  // else the CUDA-core kernel
  if (decode_tcg_supported(num_q_heads, num_kv_heads, block_size, fp8)) {
    plan->kind = 3;
    plan->tc = false;
    plan->grid = decode_tc_grid();
    return plan->grid > 0;
  }
  // the CUDA-core kernel spreads 8 consumer warps evenly over the KV heads and
  // is instantiated for groups of 1, 2, 4 and 8 query heads
  const int group = num_q_heads / num_kv_heads;
  const bool split_ok =
      kConsumerWarps % num_kv_heads == 0 && (group == 1 || group == 2 || group == 4 || group == 8);
  // The per-head tcgen05 kernel loads block-sized TMA boxes: from 16 rows up it
  // is the faster one, at 8-row boxes the CUDA-core kernel, whose stages take
  // whole token rows over several blocks, measured faster (512 sequences,
  // 8 KV heads, block 8: 0.51 against 0.71 ms; 4 KV heads: 0.24 against 0.37)
  if (!fp8 && decode_tc_supported(num_q_heads, num_kv_heads, block_size) &&
      (block_size % 16 == 0 || !split_ok)) {
    plan->kind = 2;
    plan->tc = true;
    plan->grid = decode_tc_grid();
    return plan->grid > 0;
  }
  if (!split_ok) return false;
  plan->kind = 1;
  plan->tc = false;
  plan->grid = split_grid(num_q_heads, num_kv_heads, status);
  return plan->grid > 0;
}

size_t decode_workspace_bytes(int num_seqs, int num_q_heads, int num_kv_heads,
                              const DecodePlan &plan) {
  if (plan.kind == 2) return tc_workspace(num_seqs, num_q_heads / num_kv_heads, plan.grid);
  if (plan.kind == 3)  // + the prefix sums of CTAs 1.. (each CTA plans the call itself)
    return ws_layout(num_seqs, num_q_heads, 1, plan.grid).total +
           align256(sizeof(int) * size_t(plan.grid - 1) * tcg_cu_stride(num_seqs));
  const int wph = plan.kind == 1 ? kConsumerWarps / num_kv_heads : 1;
  return ws_layout(num_seqs, num_q_heads, wph, plan.grid).total;
}

size_t decode_workspace_upper_bound(int num_seqs, int num_q_heads, int num_kv_heads,
                                    cudaError_t *status) {
  size_t need = 0;
  DecodePlan plan;
  // the kernel depends on the block size: try one of each kind
  for (int bs : {128, 8, 1}) {
    if (choose_decode_plan(num_q_heads, num_kv_heads, bs, &plan, status)) {
      const size_t s = decode_workspace_bytes(num_seqs, num_q_heads, num_kv_heads, plan);
      if (s > need) need = s;
    }
  }
  *status = cudaSuccess;
  return need;
}

cudaError_t launch_paged_decode(const DecodeArgs &a, const DecodePlan &plan, cudaStream_t stream) {
  if (a.num_seqs == 0) return cudaSuccess;
  const int grid = (plan.kind == 3 && a.grid_override > 0 && a.grid_override < plan.grid)
                       ? a.grid_override : plan.grid;
  const int wph = kConsumerWarps / a.num_kv_heads;
  const int group = a.num_q_heads / a.num_kv_heads;
  uint8_t *ws = static_cast<uint8_t *>(a.workspace);
  cudaError_t e;

  CombineParams cp;
  cp.out = static_cast<__nv_bfloat16 *>(a.out);
  cp.ws = ws;
  cp.num_seqs = a.num_seqs;
  cp.num_q_heads = a.num_q_heads;
  cp.wph = wph;
  cp.grid = grid;
  cp.group = group;
  cp.tc = plan.tc ? 1 : 0;
  cp.seg_cost = 0;

  if (plan.kind == 3) {
    // bf16 caches: no plan launch, the attention kernel plans the call itself
    // and writes a decode step's new rows. fp8 caches: the plan launch plans
    // the call and quantizes the new rows first, which measured faster.
    const WsLayout lay = ws_layout(a.num_seqs, a.num_q_heads, 1, grid);
    DecodeArgs at = a;
    if (a.fp8) {
      if ((e = launch_plan(a, grid, 1, 128, kDecodeSegmentCost, ws, stream)) != cudaSuccess) return e;
      at.key_new = at.value_new = nullptr;
    }
    cp.wph = 1;
    cp.seg_cost = kDecodeSegmentCost;
    cp.ml = reinterpret_cast<float2 *>(ws + lay.ml);
    cp.po = reinterpret_cast<float *>(ws + lay.o);
    if ((e = launch_decode_tcg(at, grid, reinterpret_cast<float2 *>(ws + lay.ml),
                               reinterpret_cast<float *>(ws + lay.o), kDecodeSegmentCost,
                               reinterpret_cast<int *>(ws + lay.total), tcg_cu_stride(a.num_seqs),
                               stream)) != cudaSuccess)
      return e;
    // mixed batch: the prefill runs on the SMs the attention kernel leaves as
    // its CTAs finish; the combine below waits for the prefill, which waits
    // for the attention kernel before it exits
    if (a.interleave != nullptr && (e = launch_paged_prefill(*a.interleave, stream)) != cudaSuccess)
      return e;
  } else if (plan.kind == 2) {
    if ((e = launch_plan(a, grid, a.num_kv_heads, 128, 0, ws, stream)) != cudaSuccess) return e;
    const size_t ml = align256(256 + sizeof(int) * (size_t(a.num_seqs) + 1));
    const size_t o = align256(ml + sizeof(float2) * size_t(2) * grid * group);
    cp.ml = reinterpret_cast<float2 *>(ws + ml);
    cp.po = reinterpret_cast<float *>(ws + o);
    if ((e = launch_decode_tc(a, grid, reinterpret_cast<float2 *>(ws + ml),
                              reinterpret_cast<float *>(ws + o), stream)) != cudaSuccess)
      return e;
  } else {
    const WsLayout lay = ws_layout(a.num_seqs, a.num_q_heads, wph, grid);
    if ((e = launch_plan(a, grid, 1, kMinRange, 0, ws, stream)) != cudaSuccess) return e;
    SplitParams sp;
    sp.out = static_cast<__nv_bfloat16 *>(a.out);
    sp.q = static_cast<const __nv_bfloat16 *>(a.q);
    sp.k_cache = static_cast<const uint8_t *>(a.k_cache);
    sp.v_cache = static_cast<const uint8_t *>(a.v_cache);
    sp.block_tables = a.block_tables;
    sp.max_blocks_per_seq = a.max_blocks_per_seq;
    sp.num_seqs = a.num_seqs;
    sp.num_q_heads = a.num_q_heads;
    sp.num_kv_heads = a.num_kv_heads;
    sp.block_size = a.block_size;
    sp.num_blocks = a.num_blocks;
    sp.qscale = a.scale * kLog2e;
    sp.ws = ws;
    sp.ml = reinterpret_cast<float2 *>(ws + lay.ml);
    sp.po = reinterpret_cast<float *>(ws + lay.o);
    sp.err = a.err;
    cp.ml = sp.ml;
    cp.po = sp.po;
    const size_t smem = split_smem_bytes(group);
    sp.k_scales = a.k_scales;
    sp.v_scales = a.v_scales;
    if (a.fp8) {
      switch (group) {
        case 1: decode_split_kernel<1, true><<<grid, kThreads, smem, stream>>>(sp); break;
        case 2: decode_split_kernel<2, true><<<grid, kThreads, smem, stream>>>(sp); break;
        case 4: decode_split_kernel<4, true><<<grid, kThreads, smem, stream>>>(sp); break;
        default: decode_split_kernel<8, true><<<grid, kThreads, smem, stream>>>(sp); break;
      }
    } else {
      switch (group) {
        case 1: decode_split_kernel<1, false><<<grid, kThreads, smem, stream>>>(sp); break;
        case 2: decode_split_kernel<2, false><<<grid, kThreads, smem, stream>>>(sp); break;
        case 4: decode_split_kernel<4, false><<<grid, kThreads, smem, stream>>>(sp); break;
        default: decode_split_kernel<8, false><<<grid, kThreads, smem, stream>>>(sp); break;
      }
    }
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  const int warps = a.num_seqs * a.num_q_heads;
  const unsigned ctas = static_cast<unsigned>((warps + kCombineWarps - 1) / kCombineWarps);
  if (plan.kind == 1) {
    decode_combine_kernel<<<ctas, kCombineWarps * 32, 0, stream>>>(cp);
    return cudaGetLastError();
  }
  // behind a tcgen05 attention kernel: a programmatic dependent launch hides
  // the launch latency (the kernel waits for the attention grid first)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ctas);
  cfg.blockDim = dim3(kCombineWarps * 32);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_combine_kernel, cp);
}

}  // namespace pkv
