// decode_tc.cu -- paged decode attention with the two contractions on the
// tcgen05 tensor cores (sm_103a): tokens are the MMA's M dimension.
//
// What is computed is the same as decode.cu (one query per sequence over its
// context_lens[i] tokens, read through block_tables; nano vllm代码详解 §2
// context; 推理运行时 §分页 KV). Decode reads every K/V byte once and is bound
// by HBM (Mini-SGLang 源码解析（二）§8.3), so the aim is to spend almost no
// instructions per byte: per 128 cached tokens of one KV head the CTA issues
// 16 MMAs and each softmax thread handles one token.
//
// Work split: the flat space of (KV head, token) pairs -- head-major, each
// head's part being the concatenated contexts -- is cut into equal ranges of
// W pairs, one per CTA (grid = SMs); every CTA streams the same bytes whatever
// the length mix. A range is walked as segments (one head, one sequence, a
// token interval); a segment is walked in stages of 128 tokens.
//
// Per CTA (192 threads):
//   warp 0    producer: for each stage, tiled TMA loads of the K and V rows of
//             the stage's tokens for one KV head, block by block (box = 64
//             dims x 1 head x R rows, R = largest power of two <= 128 dividing
//             the block size; 128-byte swizzle), plus the G query rows of the
//             head group when a segment starts. Three stages of 64 KB.
//   warp 1    TMEM owner and MMA issuer:
//               S^T[128 tok x 16] = K[128 tok x 128 d] . Q^T  (Q: 16 rows, G real)
//               O^T[128 d x 16]  += V^T[128 d x 128 tok] . P^T (V as MN-major A)
//             S^T is double-buffered in TMEM; O^T accumulates over a segment.
//   warps 2-5 softmax, one thread per token (TMEM lane): scale to base 2,
//             mask tokens outside the segment, exchange the per-head stage max
//             across the four warps, rescale O^T when the max grows, write P^T
//             as bf16, zero the V rows of masked tokens (so stale or unwritten
//             cache rows never meet the PV MMA), and at a segment's end divide
//             O^T by the summed l and store bf16 rows (or a partial record
//             (o/l, m, l) for a segment cut by a range boundary, merged by the
//             combine kernel in decode.cu's log-sum-exp rule).
// All waits are bounded; a timeout sets PKV_DEVERR_TIMEOUT and the CTA drains
// its copies and MMAs, frees TMEM and exits.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "pkv_device.cuh"
#include "pkv_internal.h"
#include "pkv_tc.cuh"

namespace pkv {

// shared with decode.cu's plan/combine kernels
struct TcHeader {
  int total;   // sum of clamped context lengths
  int range;   // (KV head, token) pairs per CTA
};

namespace {

constexpr int kTok = 128;             // tokens per stage (= MMA M for S^T)
constexpr int kHD = 128;
constexpr int kN = 16;                // MMA N: query heads of the group, padded
constexpr int kRegion = 16384;        // 128 rows x 128 B
constexpr int kKVBytes = 2 * kRegion;
constexpr int kStages = 3;
constexpr int kThreads = 192;
constexpr int kTmemCols = 64;         // S^T x2 (16 each), O^T (16)
constexpr int kSmallRegion = kN * 128;  // 16 rows x 128 B
constexpr float kLog2e = 1.4426950408889634f;

constexpr int kOffK = 0;
constexpr int kOffV = kStages * kKVBytes;
constexpr int kOffQ = 2 * kStages * kKVBytes;          // Q^T x2, 4 KB each
constexpr int kOffP = kOffQ + 2 * 2 * kSmallRegion;    // P^T, 4 KB
constexpr int kOffRed = kOffP + 2 * kSmallRegion;      // max exchange [2][4][16] + sums [4][16]
constexpr int kOffDesc = kOffRed + (2 * 4 * kN + 4 * kN) * 4;
constexpr int kOffBar = kOffDesc + kStages * 32;
constexpr int kNumBars = 2 * kStages + 2 + 2 + 1 + 1 + 1 + 1;  // kv_full/empty, s_full/free, p_full, pv_done, mx, lsum
constexpr int kSmemBytes = kOffBar + kNumBars * 8 + 16 + 1024;

enum : int { kFirst = 1, kLast = 2, kEnd = 4 };

struct TcDesc {
  int seq, head, pa, p0, p1, flags, slot, qbuf;
};

struct TcParams {
  __nv_bfloat16 *out;
  const int32_t *block_tables;
  int max_blocks_per_seq;
  int num_seqs;
  int num_q_heads;
  int num_kv_heads;
  int group;
  int block_size;
  int num_blocks;
  int box_rows;
  float scale_log2;
  const uint8_t *ws;
  float2 *ml;
  float *po;
  uint32_t *err;
};

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};"
      :: "r"(taddr), "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])),
         "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])),
         "r"(__float_as_uint(v[5])), "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])),
         "r"(__float_as_uint(v[8])), "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])),
         "r"(__float_as_uint(v[11])), "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])),
         "r"(__float_as_uint(v[14])), "r"(__float_as_uint(v[15]))
      : "memory");
}

// K-major, 128-byte swizzled operand of 128 rows (K tile) or 16 rows (Q^T, P^T):
// K step kk (16 elements) = column region kk/4 (region stride `region`), 32 B inside.
__device__ __forceinline__ uint64_t desc_k(uint32_t base, int kk, uint32_t region) {
  return smem_desc_sw128(base + (kk >> 2) * region + (kk & 3) * 32, 16, 1024);
}

// V tile as the MN-major A operand: M = 128 dims (two 64-dim regions), K = tokens.
__device__ __forceinline__ uint64_t desc_v(uint32_t base, int kk) {
  return smem_desc_sw128(base + kk * 2048, kRegion, 1024);
}

__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, const volatile int *abort) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort));
}

__global__ void __launch_bounds__(kThreads, 1)
decode_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                 const __grid_constant__ CUtensorMap tm_v, const TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_addr(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  uint8_t *smem = smem_raw + (base - raw_addr);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // launched as a programmatic dependent of the plan launch: let the combine
  // behind this kernel be scheduled early too (it waits for this grid)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  const uint32_t bar0 = base + kOffBar;
  auto kv_full = [&](int s) { return bar0 + 8u * s; };
  auto kv_empty = [&](int s) { return bar0 + 8u * (kStages + s); };
  auto s_full = [&](int b) { return bar0 + 8u * (2 * kStages + b); };
  auto s_free = [&](int b) { return bar0 + 8u * (2 * kStages + 2 + b); };
  const uint32_t p_full = bar0 + 8u * (2 * kStages + 4);
  const uint32_t pv_done = bar0 + 8u * (2 * kStages + 5);
  const uint32_t mx_bar = bar0 + 8u * (2 * kStages + 6);
  const uint32_t ls_bar = bar0 + 8u * (2 * kStages + 7);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + kOffBar + kNumBars * 8);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  TcDesc *desc = reinterpret_cast<TcDesc *>(smem + kOffDesc);
  float *red_max = reinterpret_cast<float *>(smem + kOffRed);  // [2][4][16]
  float *red_sum = red_max + 2 * 4 * kN;                         // [4][16]

  const uint32_t sK = base + kOffK, sV = base + kOffV, sQ = base + kOffQ, sP = base + kOffP;

  // zero Q^T (both buffers) and P^T: rows >= G stay zero for the whole kernel
  for (int i = threadIdx.x; i < (4 * kSmallRegion + 2 * kSmallRegion) / 16; i += kThreads)
    reinterpret_cast<uint4 *>(smem + kOffQ)[i] = make_uint4(0u, 0u, 0u, 0u);
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(kv_full(s), 1);
      mbar_init(kv_empty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(s_full(b), 1);
      mbar_init(s_free(b), 4);
    }
    mbar_init(p_full, 4);
    mbar_init(pv_done, 1);
    mbar_init(mx_bar, 4);
    mbar_init(ls_bar, 4);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  fence_proxy_async_smem();  // zeroed operand rows are read by the tensor core
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // everything above may overlap the plan launch; the plan and the inputs
  // are read only after this wait
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const TcHeader hdr = *reinterpret_cast<const TcHeader *>(p.ws);
  const int *cu = reinterpret_cast<const int *>(p.ws + 256);
  const long long units = static_cast<long long>(hdr.total) * p.num_kv_heads;
  const long long lo = static_cast<long long>(blockIdx.x) * hdr.range;
  const long long hi = min(lo + hdr.range, units);
  auto fail = [&]() {
    *abort_flag = 1;
    raise_error(p.err, PKV_DEVERR_TIMEOUT);
  };

  if (warp == 0) {
    // --------------------------------------------------------------- producer
    const int R = p.box_rows;
    const int pieces = kTok / R;
    const int oob_row = p.num_blocks * p.block_size;
    int issued = 0, segs = 0;
    bool ok = true;
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
    }
    // one stage: returns false once waiting for a free slot gave up
    auto stage = [&](const TcDesc &d, bool with_q) -> bool {
      const int s = issued % kStages;
      const int round = issued / kStages;
      int row = oob_row;
      bool loaded = false;
      if (!(d.flags & kEnd) && lane < pieces) {
        const int tok = d.pa + lane * R;
        loaded = tok < d.p1 && tok + R > d.p0;
        if (loaded) {
          const int blk = __ldg(p.block_tables + static_cast<size_t>(d.seq) * p.max_blocks_per_seq +
                                tok / p.block_size);
          if (blk >= 0 && blk < p.num_blocks) {
            row = blk * p.block_size + tok % p.block_size;
          } else {
            raise_error(p.err, PKV_DEVERR_BLOCK_ID);
            loaded = false;
          }
        }
      }
      const unsigned mask = __ballot_sync(0xffffffffu, loaded);
      int good = 1;
      if (lane == 0) {
        if (round > 0 && !mbar_wait(kv_empty(s), (round - 1) & 1, abort_flag)) {
          good = 0;
          fail();
        } else {
          desc[s] = d;
          const uint32_t bytes = __popc(mask) * R * 128 * 4 + (with_q ? 2 * p.group * 128 : 0);
          if (bytes) mbar_arrive_expect_tx(kv_full(s), bytes);
          else mbar_arrive(kv_full(s));
          if (with_q) {
            const uint32_t qdst = sQ + d.qbuf * 2 * kSmallRegion;
            const int qrow = d.seq * p.num_q_heads + d.head * p.group;
            tma_load_3d(qdst, &tm_q, 0, qrow, 0, kv_full(s));
            tma_load_3d(qdst + kSmallRegion, &tm_q, 64, qrow, 0, kv_full(s));
          }
        }
      }
      good = __shfl_sync(0xffffffffu, good, 0);
      if (!good) return false;
      if (loaded) {
        const uint32_t kd = sK + s * kKVBytes + lane * R * 128;
        const uint32_t vd = sV + s * kKVBytes + lane * R * 128;
        tma_load_3d(kd, &tm_k, 0, d.head, row, kv_full(s));
        tma_load_3d(kd + kRegion, &tm_k, 64, d.head, row, kv_full(s));
        tma_load_3d(vd, &tm_v, 0, d.head, row, kv_full(s));
        tma_load_3d(vd + kRegion, &tm_v, 64, d.head, row, kv_full(s));
      }
      ++issued;
      return true;
    };

    if (lo < hi) {
      const int total = hdr.total;
      long long u = lo;
      while (ok && u < hi) {
        const int head = static_cast<int>(u / total);
        const int off = static_cast<int>(u - static_cast<long long>(head) * total);
        // sequence containing flat token `off` (first with cu[i+1] > off)
        int a = 0, b = p.num_seqs - 1;
        while (a < b) {
          const int m = (a + b) >> 1;
          if (cu[m + 1] > off) b = m; else a = m + 1;
        }
        const int i = a;
        const int c0 = cu[i], c1 = cu[i + 1];
        const long long seg_end_u = min(hi, static_cast<long long>(head) * total + c1);
        TcDesc d;
        d.seq = i;
        d.head = head;
        d.p0 = off - c0;
        d.p1 = static_cast<int>(seg_end_u - static_cast<long long>(head) * total) - c0;
        const long long seg_lo = static_cast<long long>(head) * total + c0;
        const bool complete = seg_lo >= lo && seg_lo + (c1 - c0) <= hi;
        d.slot = complete ? -1 : (seg_lo <= lo ? 2 * int(blockIdx.x) : 2 * int(blockIdx.x) + 1);
        d.qbuf = segs & 1;
        bool first = true;
        for (int pa = d.p0 - d.p0 % R; ok && pa < d.p1; pa += kTok) {
          d.pa = pa;
          d.flags = (first ? kFirst : 0) | (pa + kTok >= d.p1 ? kLast : 0);
          ok = stage(d, first);
          first = false;
        }
        ++segs;
        u = seg_end_u;
      }
    }
    if (ok) {
      TcDesc e;
      e.seq = e.head = e.pa = e.p0 = e.p1 = e.slot = e.qbuf = 0;
      e.flags = kEnd;
      ok = stage(e, false);
    }
    if (lane == 0) {  // drain: the last copies must land before the CTA exits
      for (int j = max(0, issued - kStages); j < issued; ++j)
        mbar_wait(kv_full(j % kStages), (j / kStages) & 1, nullptr);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = umma_idesc_bf16(kTok, kN, false);
      constexpr uint32_t idesc_pv = umma_idesc_bf16(kHD, kN, false) | (1u << 15);  // A MN-major
      bool ok = true;
      int pv_issued = 0, s_issued = 0;
      int prev_s = -1, prev_first = 0;
      auto issue_pv = [&](int t, int s, int first) -> bool {
        if (!mbar_wait(p_full, t & 1, abort_flag)) return false;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kTok / 16; ++kk)
          umma_bf16(tmem + 32, desc_v(sV + s * kKVBytes, kk), desc_k(sP, kk, kSmallRegion),
                    idesc_pv, (first && kk == 0) ? 0u : 1u);
        umma_commit(pv_done);
        umma_commit(kv_empty(s));
        ++pv_issued;
        return true;
      };
      for (int j = 0;; ++j) {
        const int s = j % kStages;
        if (!mbar_wait(kv_full(s), (j / kStages) & 1, abort_flag)) { ok = false; break; }
        const TcDesc d = desc[s];
        if (d.flags & kEnd) break;
        const int buf = j & 1;
        if (j >= 2 && !mbar_wait(s_free(buf), ((j - 2) >> 1) & 1, abort_flag)) { ok = false; break; }
        tc_fence_after();
        const uint32_t q = sQ + d.qbuf * 2 * kSmallRegion;
#pragma unroll
        for (int kk = 0; kk < kHD / 16; ++kk)
          umma_bf16(tmem + buf * 16, desc_k(sK + s * kKVBytes, kk, kRegion),
                    desc_k(q, kk, kSmallRegion), idesc_s, kk > 0 ? 1u : 0u);
        umma_commit(s_full(buf));
        ++s_issued;
        if (j > 0 && !issue_pv(j - 1, prev_s, prev_first)) { ok = false; break; }
        prev_s = s;
        prev_first = (d.flags & kFirst) ? 1 : 0;
      }
      if (ok && s_issued > pv_issued) ok = issue_pv(s_issued - 1, prev_s, prev_first);
      if (!ok) fail();
      if (s_issued > 0) mbar_wait(s_full((s_issued - 1) & 1), ((s_issued - 1) >> 1) & 1, nullptr);
      if (pv_issued > 0) mbar_wait(pv_done, (pv_issued - 1) & 1, nullptr);
    }
    __syncwarp();
  } else {
    // --------------------------------------------------------------- softmax
    const int sw = warp - 2;                    // softmax warp 0..3
    const int quad = warp & 3;                  // TMEM lane quadrant this warp may access
    const int t = quad * 32 + lane;             // token (S^T lane) and dim (O^T lane)
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const int G = p.group;
    float m_run[kN], l_part[kN];
#pragma unroll
    for (int g = 0; g < kN; ++g) {
      m_run[g] = -INFINITY;
      l_part[g] = 0.f;
    }
    int segs_done = 0;
    bool ok = true;
    for (int j = 0;; ++j) {
      const int s = j % kStages;
      if (!warp_wait(kv_full(s), (j / kStages) & 1, abort_flag)) { ok = false; break; }
      const TcDesc d = desc[s];
      if (d.flags & kEnd) break;
      const int buf = j & 1;
      if (!warp_wait(s_full(buf), (j >> 1) & 1, abort_flag)) { ok = false; break; }
      tc_fence_after();
      float sc[kN];
      tmem_ld16(tmem + lane_off + buf * 16, sc);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(s_free(buf));

      const int tok = d.pa + t;
      const bool valid = tok >= d.p0 && tok < d.p1;
      const bool first = (d.flags & kFirst) != 0;
      // per-head maximum of the stage across the 128 tokens
      float wm[kN];
#pragma unroll
      for (int g = 0; g < kN; ++g) {
        sc[g] = valid ? sc[g] * p.scale_log2 : -INFINITY;
        float v = g < G ? sc[g] : -INFINITY;
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
        wm[g] = v;
      }
      float *rm = red_max + (j & 1) * 4 * kN + sw * kN;
      if (lane < kN) {
        float mine = -INFINITY;
#pragma unroll
        for (int g = 0; g < kN; ++g) if (lane == g) mine = wm[g];
        rm[lane] = mine;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(mx_bar);
      if (!warp_wait(mx_bar, j & 1, abort_flag)) { ok = false; break; }
      const float *rmj = red_max + (j & 1) * 4 * kN;
      float alpha[kN];
      bool grow = false;
#pragma unroll
      for (int g = 0; g < kN; ++g) {
        const float sm = fmaxf(fmaxf(rmj[g], rmj[kN + g]), fmaxf(rmj[2 * kN + g], rmj[3 * kN + g]));
        const float m_prev = first ? -INFINITY : m_run[g];
        const float m_new = fmaxf(m_prev, sm);
        alpha[g] = (first || g >= G) ? (g >= G ? 1.f : 0.f) : ex2(m_prev - m_new);
        grow |= (!first && g < G && alpha[g] != 1.f);
        m_run[g] = m_new;
      }
      // the previous stage's PV must be done before O^T is rescaled or P^T rewritten
      if (j > 0) {
        if (!warp_wait(pv_done, (j - 1) & 1, abort_flag)) { ok = false; break; }
        tc_fence_after();
      }
      if (grow) {
        float o[kN];
        tmem_ld16(tmem + lane_off + 32, o);
        tmem_wait_ld();
#pragma unroll
        for (int g = 0; g < kN; ++g) o[g] *= alpha[g];
        tmem_st16(tmem + lane_off + 32, o);
        tmem_wait_st();
      }
      // P^T[g][tok] (bf16), K-major 128-byte swizzled: 16 rows x 128 tokens
      const uint32_t prow_base = sP + (t >> 6) * kSmallRegion;
      const int tc = t & 63;
#pragma unroll
      for (int g = 0; g < kN; ++g) {
        if (g < G) {
          // the weight is rounded to bf16 before it enters the row sum, so the
          // sum matches the weights the PV MMA multiplies
          const __nv_bfloat16 hb = __float2bfloat16_rn(valid ? ex2(sc[g] - m_run[g]) : 0.f);
          const float pv = __bfloat162float(hb);
          l_part[g] = (first ? 0.f : l_part[g] * alpha[g]) + pv;
          const uint32_t addr = prow_base + (g >> 3) * 1024 + (g & 7) * 128 +
                                ((((tc >> 3) ^ (g & 7)) << 4) | ((tc & 7) << 1));
          asm volatile("st.shared.b16 [%0], %1;" :: "r"(addr),
                       "h"(*reinterpret_cast<const unsigned short *>(&hb)) : "memory");
        }
      }
      if (!valid) {  // masked token: its V row must be zero for the PV MMA
        const uint32_t vrow = sV + s * kKVBytes + (t >> 3) * 1024 + (t & 7) * 128;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" :: "r"(vrow + c * 16), "r"(0u) : "memory");
          asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" :: "r"(vrow + kRegion + c * 16), "r"(0u) : "memory");
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full);

      if (d.flags & kLast) {
        // l of each head: sum over the 128 tokens
        float ws_[kN];
#pragma unroll
        for (int g = 0; g < kN; ++g) {
          float v = l_part[g];
#pragma unroll
          for (int off = 16; off >= 1; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
          ws_[g] = v;
        }
        if (lane < kN) {
          float mine = 0.f;
#pragma unroll
          for (int g = 0; g < kN; ++g) if (lane == g) mine = ws_[g];
          red_sum[sw * kN + lane] = mine;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(ls_bar);
        if (!warp_wait(ls_bar, segs_done & 1, abort_flag)) { ok = false; break; }
        if (!warp_wait(pv_done, j & 1, abort_flag)) { ok = false; break; }
        tc_fence_after();
        float o[kN];
        tmem_ld16(tmem + lane_off + 32, o);
        tmem_wait_ld();
        float l_sum[kN];
#pragma unroll
        for (int g = 0; g < kN; ++g)
          l_sum[g] = red_sum[g] + red_sum[kN + g] + red_sum[2 * kN + g] + red_sum[3 * kN + g];
        if (d.slot < 0) {
          __nv_bfloat16 *orow = p.out + (static_cast<size_t>(d.seq) * p.num_q_heads +
                                         static_cast<size_t>(d.head) * G) * kHD + t;
#pragma unroll
          for (int g = 0; g < kN; ++g)
            if (g < G) orow[g * kHD] = __float2bfloat16_rn(l_sum[g] > 0.f ? o[g] / l_sum[g] : 0.f);
        } else {
          const size_t rec = static_cast<size_t>(d.slot) * G;
#pragma unroll
          for (int g = 0; g < kN; ++g) {
            if (g < G) {
              p.po[(rec + g) * kHD + t] = l_sum[g] > 0.f ? o[g] / l_sum[g] : 0.f;
              if (t == 0) p.ml[rec + g] = make_float2(m_run[g], l_sum[g]);
            }
          }
        }
        ++segs_done;
        // the next segment's first PV overwrites O^T only after p_full of its
        // first stage, which these threads arrive on after this read
      }
    }
    if (!ok) fail();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

bool make_map3(CUtensorMap *map, const void *ptr, uint64_t rows, uint64_t heads, uint32_t box_rows,
               uint32_t box_heads) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(kHD), heads, rows};
  cuuint64_t strides[2] = {kHD * 2, heads * kHD * 2};
  cuuint32_t box[3] = {64, box_heads, box_rows};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool decode_tc_supported(int num_q_heads, int num_kv_heads, int block_size) {
  return num_kv_heads >= 1 && num_q_heads % num_kv_heads == 0 &&
         num_q_heads / num_kv_heads <= kN && block_size % 8 == 0;
}

int decode_tc_grid() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  return sm_count(dev);
}

size_t decode_tc_smem_bytes() { return kSmemBytes; }

cudaError_t launch_decode_tc(const DecodeArgs &a, int grid, float2 *ml, float *po,
                             cudaStream_t stream) {
  static std::once_flag attr_once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(attr_once, [] {
    attr_err = cudaFuncSetAttribute(decode_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    kSmemBytes);
  });
  if (attr_err != cudaSuccess) return attr_err;
  int box_rows = a.block_size & -a.block_size;
  if (box_rows > kTok) box_rows = kTok;
  const int group = a.num_q_heads / a.num_kv_heads;
  CUtensorMap tq, tk, tv;
  const uint64_t cache_rows = static_cast<uint64_t>(a.num_blocks) * a.block_size;
  // q viewed as [1 row, num_seqs * Hq "heads", 128]: box = 64 dims x G heads
  if (!make_map3(&tq, a.q, 1, static_cast<uint64_t>(a.num_seqs) * a.num_q_heads, 1, group) ||
      !make_map3(&tk, a.k_cache, cache_rows, a.num_kv_heads, box_rows, 1) ||
      !make_map3(&tv, a.v_cache, cache_rows, a.num_kv_heads, box_rows, 1))
    return cudaErrorInvalidValue;
  TcParams p;
  p.out = static_cast<__nv_bfloat16 *>(a.out);
  p.block_tables = a.block_tables;
  p.max_blocks_per_seq = a.max_blocks_per_seq;
  p.num_seqs = a.num_seqs;
  p.num_q_heads = a.num_q_heads;
  p.num_kv_heads = a.num_kv_heads;
  p.group = group;
  p.block_size = a.block_size;
  p.num_blocks = a.num_blocks;
  p.box_rows = box_rows;
  p.scale_log2 = a.scale * kLog2e;
  p.ws = static_cast<const uint8_t *>(a.workspace);
  p.ml = ml;
  p.po = po;
  p.err = a.err;
  // programmatic dependent launch: the set-up (barriers, TMEM) runs while the
  // plan launch before it on the stream finishes
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_tc_kernel, tq, tk, tv, p);
}

}  // namespace pkv
