// decode_tcg.cu -- paged decode attention on tcgen05, all KV heads of a block
// per stage (sm_103a). This is the fast decode path for GQA shapes.
//
// Computes what decode.cu computes (one query per sequence over its
// context_lens[i] tokens, read through block_tables; nano vllm代码详解 §2
// context; 推理运行时 §分页 KV). Decode is HBM-bound (Mini-SGLang 源码解析（二）
// §8.3), and on GB300 the bytes only move at full speed when each copy covers
// whole token rows: in the [NB, bs, Hkv, D] cache a run of T tokens of one
// block is T * Hkv * 256 contiguous bytes. So a stage here is T = 128 / Hkv
// consecutive tokens of one block with ALL their KV heads: 128 rows, loaded by
// one tiled TMA box per 64-dim half through a (dim, token, head) view of the
// cache, which lands in shared memory ordered [head][token][dim] -- exactly the
// 128-row K-major operand the tensor core wants.
//
//   S^T[128 rows x N] = K[128 rows x 128 d] . Q^T[N x 128 d]     (N = Hq padded to 16)
//     row h*T + t is token t of KV head h; column n = h'*G + g is query head n.
//     Only the columns of the row's own head (h' = h) are used; the others are
//     spare tensor-core work, which costs nothing here.
//   O^T[128 d x N] += V^T[128 d x 128 rows] . P^T[128 rows x N]
//     P^T is block-diagonal: row h*T + t holds p only in the columns of head h,
//     so each query head accumulates only the V rows of its own KV head.
//
// Per CTA (one CTA per SM): warp 0 loads Q rows when a sequence segment starts
// and the K box of every stage, warp 6 the V box (separate K and V rings of up
// to three 32 KB stages each, so V never holds up the next S), warp 1 owns
// TMEM and issues the MMAs, warps 2-5 run the softmax with one thread per row:
// the T rows of a KV head sit in one warp. A segment's first stage fixes each
// head's reference maximum (warp shuffles); later stages only test whether a
// score exceeds it by more than 2^8, and the four softmax warps meet once per
// stage on one hardware barrier that ORs that test over their threads: only
// when it fires do they compute new maxima and rescale O^T together. Rows of
// tokens outside the segment are masked and their V rows zeroed, so unwritten
// cache slots never reach the PV MMA.
//
// A shared-memory access (a barrier probe, a load) that the MMA thread issues
// behind its own MMAs waits until the tensor core has taken them. With bf16
// caches (256 threads) warp 7 therefore does all the barrier polling and hands
// the MMA warp commands through a counting hardware barrier; with fp8 caches
// (480 threads: two converter warpgroups added) the MMA thread polls itself,
// reading every barrier of a round before issuing that round's MMAs.
//
// fp8 caches (E4M3 codes, one scale per token and KV head): the S MMA reads the
// raw K codes straight from the ring as E4M3 (kind::f8f6f4) against Q^T split
// into two E4M3 terms whose sum is Q^T (times a power of two per row), and the
// K scales multiply the scores; V is expanded to f16 by a converter warpgroup
// and its scales are folded into P, so the PV MMA stays f16.
//
// CTA b owns the flat token range [bW, (b+1)W) of the concatenated contexts
// (all heads), exactly like the split kernel in decode.cu, and leaves the same
// partial records (o/l, m, l) for sequences a range boundary cuts; decode.cu's
// combine kernel merges them.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "pkv_device.cuh"
#include "pkv_internal.h"
#include "pkv_tc.cuh"

namespace pkv {
namespace {

constexpr int kRows = 128;            // MMA M: rows of a stage (T tokens x Hkv heads)
constexpr int kHD = 128;
constexpr int kRegion = 16384;        // 128 rows x 128 B (one 64-dim half)
constexpr int kKVBytes = 2 * kRegion;
constexpr int kThreads = 256;  // K producer, MMA, 4 softmax warps, V producer, MMA scheduler
// fp8 caches add two converter warpgroups (warps 7-10: Q, 11-14: V); their MMA
// warp polls its barriers itself (no scheduler warp)
constexpr int kThreadsF8 = 480;
constexpr int kRawCodes = 16384;      // one fp8 stage: 128 rows x 128 one-byte codes
constexpr int kRawStage = 17408;      // codes + 128 fp32 row scales, padded to 1024 B
constexpr int kMaxN = 128;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleThreshold = 8.f;
constexpr int kSoftmaxBarrier = 1;    // named barrier of the four softmax warps (0 is __syncthreads)
constexpr int kIssueBarrier = 2;      // named barrier of the MMA warp and the MMA scheduler warp
// commands from the scheduler to the MMA warp (a count from 0 to 31)
enum : int { kCmdPV = 1, kCmdPVFirst = 2, kCmdS = 4, kCmdFinish = 8, kCmdAbort = 16 };

enum : int { kFirst = 1, kLast = 2, kEnd = 4 };

struct GDesc {
  int seq, pa, p0, p1, flags, slot, qbuf, pad;
};

struct GParams {
  __nv_bfloat16 *out;
  const int32_t *block_tables;
  int max_blocks_per_seq;
  int num_seqs;
  int num_q_heads;
  int num_kv_heads;
  int group;
  int n_cols;          // N: num_q_heads rounded up to 16
  int tokens;          // T = 128 / num_kv_heads
  int block_size;
  int num_blocks;
  int stages;
  int tmem_cols;
  float scale_log2;
  const uint8_t *ws;
  float2 *ml;
  float *po;
  uint32_t *err;
  const float *k_scales;  // fp8 caches: [NB * bs, Hkv] row scales
  const float *v_scales;
  int seg_cost;           // units in front of each non-empty sequence in the flat space
  // the plan: with bf16 caches computed by every CTA from the lengths and
  // their bound, the prefix sums going to the workspace's cu[] (CTA 0; the
  // combine reads them) or cu_copies + (b - 1) * cu_stride (CTA b > 0); with
  // fp8 caches (which measured faster so) read from the workspace, where the
  // plan launch before this kernel left it
  const int32_t *context_lens;
  int max_context_len;
  int *cu_copies;
  int cu_stride;
  // decode step over bf16 caches (key_new == nullptr otherwise): each
  // sequence's newest K/V row, [S, Hkv, 128] bf16 with these token strides in
  // elements, is written to the cache by the CTA that owns the sequence's last
  // position, before that stage is loaded
  const __nv_bfloat16 *key_new;
  const __nv_bfloat16 *value_new;
  int64_t key_stride;
  int64_t value_stride;
  uint8_t *k_cache;
  uint8_t *v_cache;
};

// shared-memory map, all offsets from a 1024-aligned base
struct GLayout {
  int k, v, q, p, alpha, lsum, msum, desc, bar, vflag, qs, kr, vr, total;
};

__host__ __device__ inline GLayout g_layout(int stages, int n_cols, bool f8 = false) {
  GLayout L;
  const int small = n_cols * 128;         // one 64-dim half of Q^T / P^T (N rows x 128 B)
  // fp8: the S MMA reads the raw K codes, so shared memory holds only the f16 V ring
  L.k = 0;
  L.v = f8 ? 0 : stages * kKVBytes;
  L.q = L.v + stages * kKVBytes;
  L.p = L.q + 2 * small;                  // one Q^T buffer (2 halves)
  L.alpha = L.p + 2 * 2 * small;          // two P^T buffers (2 halves over the 128 rows each)
  L.lsum = L.alpha + (2 * kMaxN + 4) * 4; // [kMaxN] row sums
  L.msum = L.lsum + kMaxN * 4;            // [kMaxN] maxima
  L.desc = L.msum + kMaxN * 4;
  L.bar = L.desc + 4 * 32;
  L.vflag = L.bar + 34 * 8 + 16;          // 34 barriers, TMEM slot + abort flag, then V stage flags
  L.total = L.vflag + 16;
  L.qs = L.kr = L.vr = 0;
  if (f8) {                               // raw fp8 rings, 1024-aligned for the 128-byte swizzle
    L.qs = L.total;                       // [kMaxN] 1 / scale of each Q^T row (below)
    L.kr = (L.qs + kMaxN * 4 + 1023) & ~1023;
    L.vr = L.kr + stages * kRawStage;
    L.total = L.vr + stages * kRawStage;
  }
  return L;
}

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

// C consecutive fp32 TMEM columns of this thread's lane (warp-collective), C in {1..32}.
template <int C>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, float (&v)[C]) {
  uint32_t r[C];
  if constexpr (C == 1) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];" : "=r"(r[0]) : "r"(taddr));
  } else if constexpr (C == 2) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x2.b32 {%0, %1}, [%2];"
                 : "=r"(r[0]), "=r"(r[1]) : "r"(taddr));
  } else if constexpr (C == 4) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(taddr));
  } else if constexpr (C == 8) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                   "=r"(r[6]), "=r"(r[7]) : "r"(taddr));
  } else if constexpr (C == 16) {
    float t[16];
    tmem_ld16(taddr, t);
#pragma unroll
    for (int i = 0; i < 16; ++i) r[i] = __float_as_uint(t[i]);
  } else {
    static_assert(C == 32, "unsupported column count");
    float t[16], u[16];
    tmem_ld16(taddr, t);
    tmem_ld16(taddr + 16, u);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      r[i] = __float_as_uint(t[i]);
      r[16 + i] = __float_as_uint(u[i]);
    }
  }
#pragma unroll
  for (int i = 0; i < C; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ uint64_t desc_k(uint32_t base, int kk, uint32_t region) {
  return smem_desc_sw128(base + (kk >> 2) * region + (kk & 3) * 32, 16, 1024);
}

// start-address increment (16-byte units, the descriptor's low field) of K
// step kk from step 0 of a K-major operand with 64-dim regions region16 * 16
// bytes apart: the issuing thread builds a descriptor once per group and steps it
__device__ __forceinline__ uint64_t kstep(int kk, uint32_t region16) {
  return static_cast<uint64_t>((kk >> 2) * region16 + (kk & 3) * 2);
}

__device__ __forceinline__ uint64_t desc_v(uint32_t base, int kk) {
  return smem_desc_sw128(base + kk * 2048, kRegion, 1024);
}

__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, const volatile int *abort) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort));
}

__device__ __forceinline__ void st_shared_f16(uint32_t addr, float v) {
  const __half h = __float2half_rn(v);
  asm volatile("st.shared.b16 [%0], %1;" :: "r"(addr), "h"(*reinterpret_cast<const unsigned short *>(&h))
               : "memory");
}

// Two E4M3 codes (low byte first in memory) -> two f16 (exact).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t codes) {
  uint32_t h;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"(codes));
  return h;
}

__device__ __forceinline__ uint4 e4m3x8_to_f16x8(uint2 c) {
  uint4 r;
  r.x = e4m3x2_to_f16x2(static_cast<uint16_t>(c.x & 0xffffu));
  r.y = e4m3x2_to_f16x2(static_cast<uint16_t>(c.x >> 16));
  r.z = e4m3x2_to_f16x2(static_cast<uint16_t>(c.y & 0xffffu));
  r.w = e4m3x2_to_f16x2(static_cast<uint16_t>(c.y >> 16));
  return r;
}

__device__ __forceinline__ void sts128(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};"
               :: "r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}

// Row r of a raw fp8 stage (128-byte rows, 128-byte swizzle: chunk c of row r
// sits at chunk c ^ (r & 7)) -> row r of the f16 operand stage (two 64-dim
// regions of 128-byte rows with the same swizzle), the layout the bf16 TMA
// boxes produce.
__device__ __forceinline__ void convert_row_e4m3(uint32_t raw, uint32_t cv, int r) {
  const uint32_t sw = static_cast<uint32_t>(r & 7);
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const uint4 w = lds128(raw + r * 128 + ((c ^ sw) << 4));       // dims 16c .. 16c+15
    const uint32_t row = cv + (c >> 2) * kRegion + r * 128;
    const uint32_t c2 = static_cast<uint32_t>((2 * c) & 7);
    sts128(row + ((c2 ^ sw) << 4), e4m3x8_to_f16x8(make_uint2(w.x, w.y)));
    sts128(row + (((c2 + 1) ^ sw) << 4), e4m3x8_to_f16x8(make_uint2(w.z, w.w)));
  }
}

// D[tmem] (+)= A[smem desc] * B[smem desc], both E4M3 (kind::f8f6f4; the
// operand formats come from idesc, 0 = E4M3), f32 accumulator.
__device__ __forceinline__ void umma_f8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                        uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}"
      :: "r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate) : "memory");
}

// Two floats -> two E4M3 codes (round to nearest even, saturating), the first
// in the low byte; and back, exactly.
__device__ __forceinline__ uint32_t f32x2_to_e4m3x2(float lo, float hi) {
  uint16_t c;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(c) : "f"(hi), "f"(lo));  // first operand -> upper byte
  return c;
}

__device__ __forceinline__ float2 e4m3x2_to_f32x2(uint32_t codes) {
  const uint32_t h = e4m3x2_to_f16x2(static_cast<uint16_t>(codes));
  return __half22float2(*reinterpret_cast<const __half2 *>(&h));
}

// Q^T for the fp8 S MMA, in place, by 128 threads (t = 0..127; four per row,
// in one warp): each bf16 row n (dims 0..63 in region 0, 64..127 in region 1,
// 128-byte rows, 128-byte swizzle) becomes two E4M3 rows hi (region 0) and lo
// (region 1), 128 codes each, with
//   q[d] * sq = hi[d] + lo[d],   sq = 2^e, max_d |q[d]| * sq in (224, 448],
// hi the nearest E4M3 value to q * sq and lo the nearest to what is left. A
// bf16 value has 8 significant bits and an E4M3 value 4, so hi + lo is q * sq
// exactly except where lo falls below the E4M3 subnormal step 2^-9 (values
// under 2^-2 after scaling, about 2^-10 of the row maximum); the error there
// is at most 2^-10 after scaling. qinv[n] = 1 / sq.
__device__ __forceinline__ void split_q_e4m3(uint32_t qbuf, uint32_t region, int n_rows, int t,
                                             float *qinv) {
  const int quarter = t & 3;                         // dims 32 * quarter .. +31
  for (int n0 = 0; n0 < n_rows; n0 += 32) {
    const int n = n0 + (t >> 2);
    const bool have = n < n_rows;
    const uint32_t sw = static_cast<uint32_t>(n & 7);
    uint32_t w[16];                                  // bf16 pairs, dims 32q + 2i, +1
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (have)
        v = lds128(qbuf + (quarter >> 1) * region + n * 128 +
                   (((4 * (quarter & 1) + c) ^ sw) << 4));
      w[4 * c + 0] = v.x;
      w[4 * c + 1] = v.y;
      w[4 * c + 2] = v.z;
      w[4 * c + 3] = v.w;
    }
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float2 f = bf16x2_to_float2(w[i]);
      amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
    }
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    int e = 0;                                       // sq = 2^e
    if (amax > 0.f && amax <= 3.0e38f) {
      e = static_cast<int>((__float_as_uint(448.f / amax) >> 23) & 0xffu) - 127;
      e = max(-126, min(126, e));
      if (amax * __uint_as_float(static_cast<uint32_t>(e + 127) << 23) > 448.f) --e;
      e = max(-126, e);
    }
    const float sq = __uint_as_float(static_cast<uint32_t>(e + 127) << 23);
    __syncwarp();                                    // the row is read before any lane rewrites it
#pragma unroll
    for (int cc = 0; cc < 2; ++cc) {                 // code chunk 2q + cc: dims 16 (2q + cc) .. +15
      uint32_t hi[4], lo[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        uint32_t hc = 0, lc = 0;
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const float2 f = bf16x2_to_float2(w[8 * cc + 2 * k + u]);
          const float x0 = f.x * sq, x1 = f.y * sq;  // exact (power of two)
          const uint32_t h2 = f32x2_to_e4m3x2(x0, x1);
          const float2 hv = e4m3x2_to_f32x2(h2);
          const uint32_t l2 = f32x2_to_e4m3x2(x0 - hv.x, x1 - hv.y);  // the differences are exact
          hc |= h2 << (16 * u);
          lc |= l2 << (16 * u);
        }
        hi[k] = hc;
        lo[k] = lc;
      }
      if (have) {
        const uint32_t off = n * 128 + ((static_cast<uint32_t>(2 * quarter + cc) ^ sw) << 4);
        sts128(qbuf + off, make_uint4(hi[0], hi[1], hi[2], hi[3]));
        sts128(qbuf + region + off, make_uint4(lo[0], lo[1], lo[2], lo[3]));
      }
    }
    if (have && quarter == 0) qinv[n] = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);
    __syncwarp();
  }
}

__device__ __forceinline__ void st_shared_b16(uint32_t addr, float v) {
  const __nv_bfloat16 h = __float2bfloat16_rn(v);
  asm volatile("st.shared.b16 [%0], %1;" :: "r"(addr), "h"(*reinterpret_cast<const unsigned short *>(&h))
               : "memory");
}

// T: tokens per stage (128 / Hkv); G: query heads per KV head; F8: the caches
// hold E4M3 codes with per-row scales (K read by the MMA as E4M3, V expanded
// to f16 on chip).
template <int T, int G, bool F8>
__global__ void __launch_bounds__(F8 ? kThreadsF8 : kThreads, 1)
decode_tcg_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const GParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_addr(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  uint8_t *smem = smem_raw + (base - raw_addr);
  constexpr int NT = F8 ? kThreadsF8 : kThreads;
  const GLayout L = g_layout(p.stages, p.n_cols, F8);
  const int N = p.n_cols;
  const int S = p.stages;
  const uint32_t small = N * 128;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // launched as a programmatic dependent of the previous kernel on the stream:
  // let the combine pass behind this kernel be scheduled early too (it waits
  // for this grid)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  const uint32_t bar0 = base + L.bar;
  // K and V have their own rings: a K slot is free once every softmax warp has
  // seen S computed from it (which also means its stage descriptor was read);
  // a V slot once the PV MMA that reads it has completed
  auto k_full = [&](int s) { return bar0 + 8u * s; };
  auto k_empty = [&](int s) { return bar0 + 8u * (4 + s); };
  auto v_full = [&](int s) { return bar0 + 8u * (16 + s); };
  auto v_empty = [&](int s) { return bar0 + 8u * (20 + s); };
  auto s_full = [&](int b) { return bar0 + 8u * (8 + b); };
  auto s_free = [&](int b) { return bar0 + 8u * (10 + b); };
  // P^T is double-buffered: stage j writes buffer j & 1, so the softmax of stage
  // j only waits for PV(j-2) before writing, not for PV(j-1)
  auto p_full = [&](int b) { return bar0 + 8u * (b ? 33 : 12); };
  auto pv_done = [&](int b) { return bar0 + 8u * (b ? 32 : 13); };
  const uint32_t l_bar = bar0 + 8u * 15;    // per-segment row-sum exchange
  // fp8: the loaders' copies land on kr_full / vr_full; the converters then
  // fill the f16 stage and arrive on k_full / v_full
  auto kr_full = [&](int s) { return bar0 + 8u * (24 + s); };
  auto vr_full = [&](int s) { return bar0 + 8u * (28 + s); };
  volatile int *vflag = reinterpret_cast<volatile int *>(smem + L.vflag);  // V stage flags
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L.bar + 34 * 8);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  GDesc *desc = reinterpret_cast<GDesc *>(smem + L.desc);
  float *alpha_buf = reinterpret_cast<float *>(smem + L.alpha);          // [2][kMaxN]
  volatile int *stop_flag = reinterpret_cast<volatile int *>(alpha_buf + 2 * kMaxN);  // softmax warps leave
  float *lsum_buf = reinterpret_cast<float *>(smem + L.lsum);
  float *msum_buf = reinterpret_cast<float *>(smem + L.msum);
  const uint32_t sK = base + L.k, sV = base + L.v, sQ = base + L.q, sP = base + L.p;

  // Q^T and P^T padding rows/columns must read as zeros for the whole kernel
  for (int i = threadIdx.x; i < (6 * static_cast<int>(small)) / 16; i += NT)
    reinterpret_cast<uint4 *>(smem + L.q)[i] = make_uint4(0u, 0u, 0u, 0u);
  if (threadIdx.x == 0) *stop_flag = 0;
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(k_full(s), F8 ? 4 : 1);
      mbar_init(k_empty(s), 4);
      mbar_init(v_full(s), F8 ? 4 : 1);
      mbar_init(v_empty(s), 1);
      if (F8) {
        mbar_init(kr_full(s), 1);
        mbar_init(vr_full(s), 1);
      }
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(s_full(b), 1);
      mbar_init(s_free(b), 4);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(p_full(b), 4);
      mbar_init(pv_done(b), 1);
    }
    mbar_init(l_bar, 4);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(tmem_slot), p.tmem_cols);
    tmem_relinquish();
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // everything above may overlap the previous kernel on the stream (launched
  // as its programmatic dependent); the inputs are read only after this wait
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // The plan, computed by every CTA: prefix sums cu of the clamped lengths in
  // the flat space (a non-empty sequence takes seg_cost units, then its
  // tokens), the total, and the range size W = ceil(total / grid) rounded up
  // to 16, at least 128. CTA 0 also leaves cu and (total, W) in the workspace
  // for the combine.
  constexpr bool kSelfPlan = !F8;
  int *cu_w = (blockIdx.x == 0 || !kSelfPlan)
                  ? reinterpret_cast<int *>(const_cast<uint8_t *>(p.ws) + 256)
                  : p.cu_copies + static_cast<size_t>(blockIdx.x - 1) * p.cu_stride;
  int total = 0;
  int range = 0;
  if (!kSelfPlan) {
    total = reinterpret_cast<const int *>(p.ws)[0];
    range = reinterpret_cast<const int *>(p.ws)[1];
  } else {
    int *wsum = reinterpret_cast<int *>(alpha_buf);  // scratch until the roles start
    constexpr int kWarps = NT / 32;
    for (int start = 0; start < p.num_seqs; start += NT) {
      const int i = start + static_cast<int>(threadIdx.x);
      int x = 0;
      if (i < p.num_seqs) {
        x = p.context_lens[i];
        if (x < 0 || x > p.max_context_len) {
          if (blockIdx.x == 0) raise_error(p.err, PKV_DEVERR_LENGTH);
          x = x < 0 ? 0 : p.max_context_len;
        }
      }
      int v = x > 0 ? x + p.seg_cost : 0;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, v, off);
        if (lane >= off) v += y;
      }
      if (lane == 31) wsum[warp] = v;
      __syncthreads();
      if (warp == 0) {
        int w = lane < kWarps ? wsum[lane] : 0;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, w, off);
          if (lane >= off) w += y;
        }
        if (lane < kWarps) wsum[lane] = w;
      }
      __syncthreads();
      if (i < p.num_seqs) cu_w[i + 1] = total + v + (warp > 0 ? wsum[warp - 1] : 0);
      total += wsum[kWarps - 1];
      __syncthreads();
    }
    long long range_ll = (static_cast<long long>(total) + gridDim.x - 1) / gridDim.x;
    range_ll = (range_ll + 15) / 16 * 16;
    range = static_cast<int>(range_ll < 128 ? 128 : range_ll);
    if (threadIdx.x == 0) {
      cu_w[0] = 0;
      if (blockIdx.x == 0) {
        int *hdr = reinterpret_cast<int *>(const_cast<uint8_t *>(p.ws));
        hdr[0] = total;
        hdr[1] = range;
      }
    }
    __syncthreads();  // the producers read cu_w
  }
  const int *cu = kSelfPlan ? cu_w : reinterpret_cast<const int *>(p.ws + 256);
  const int lo = static_cast<int>(blockIdx.x) * range;
  const int hi = min(lo + range, total);
  const uint32_t tmem_o = tmem;                       // O^T: columns [0, N)
  // S^T buffers; fp8: each 2N wide, the hi half of Q^T in columns [0, N) and
  // the lo half in [N, 2N)
  constexpr int kSWidth = F8 ? 2 : 1;
  auto tmem_s = [&](int b) { return tmem + N * (1 + kSWidth * b); };
  auto fail = [&]() {
    *abort_flag = 1;
    raise_error(p.err, PKV_DEVERR_TIMEOUT);
  };

  if (warp == 0 || warp == 6) {
    // -------------------------------------------------------------- producers
    // Both walk the same stages; warp 0 loads K (and Q, and writes the stage
    // descriptors), warp 6 loads V.
    const bool is_k = warp == 0;
    int issued = 0, segs = 0;
    int q_last[2] = {-1, -1};  // last stage whose S MMA reads each Q^T buffer
    bool ok = true;
    if (lane == 0) {
      if (is_k) {
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
      } else {
        tma_prefetch_desc(&tm_v);
      }
    }
    auto stage = [&](const GDesc &d, int blk_row, bool with_q) -> bool {
      const int s = issued % S;
      const int round = issued / S;
      int good = 1;
      if (lane == 0) {
        const uint32_t empty = is_k ? k_empty(s) : v_empty(s);
        const uint32_t full = F8 ? (is_k ? kr_full(s) : vr_full(s)) : (is_k ? k_full(s) : v_full(s));
        // a Q^T buffer may only be refilled once the S MMAs of the previous
        // segment that used it are done (the slot wait covers stage issued - S)
        const int prev_q = (is_k && with_q) ? q_last[d.qbuf] : -1;
        if (prev_q >= 0 && prev_q > issued - S &&
            !mbar_wait(k_empty(prev_q % S), (prev_q / S) & 1, abort_flag)) {
          good = 0;
          fail();
        } else if (round > 0 && !mbar_wait(empty, (round - 1) & 1, abort_flag)) {
          good = 0;
          fail();
        } else {
          const bool load = !(d.flags & kEnd) && blk_row >= 0;
          uint32_t bytes = load ? (F8 ? kRawCodes + kRows * 4 : 2 * kRegion) : 0;
          if (is_k) {
            desc[s] = d;
            if (with_q) bytes += 2 * p.num_q_heads * 128;
          } else if (F8) {
            vflag[s] = d.flags;
          }
          if (bytes) mbar_arrive_expect_tx(full, bytes);
          else mbar_arrive(full);
          if (is_k && with_q) {
            const uint32_t qdst = sQ + d.qbuf * 2 * small;
            tma_load_3d(qdst, &tm_q, 0, 0, d.seq, full);
            tma_load_3d(qdst + small, &tm_q, 64, 0, d.seq, full);
          }
          if (load && F8) {
            // 128 rows of 128 codes in one box, then the rows' 128 scales
            const uint32_t dst = base + (is_k ? L.kr : L.vr) + s * kRawStage;
            tma_load_3d(dst, is_k ? &tm_k : &tm_v, 0, blk_row, 0, full);
            const float *sc = (is_k ? p.k_scales : p.v_scales) +
                              static_cast<int64_t>(blk_row) * p.num_kv_heads;
            bulk_g2s(dst + kRawCodes, sc, kRows * 4, full, l2_policy_evict_first());
          } else if (load) {
            const uint32_t dst = (is_k ? sK : sV) + s * kKVBytes;
            const CUtensorMap *map = is_k ? &tm_k : &tm_v;
            tma_load_3d(dst, map, 0, blk_row, 0, full);
            tma_load_3d(dst + kRegion, map, 64, blk_row, 0, full);
          }
        }
      }
      good = __shfl_sync(0xffffffffu, good, 0);
      if (good) {
        if (!(d.flags & kEnd)) q_last[d.qbuf] = issued;
        ++issued;
      }
      return good != 0;
    };

    if (lo < hi) {
      int a = 0, b = p.num_seqs - 1;
      while (a < b) {
        const int m = (a + b) >> 1;
        if (cu[m + 1] > lo) b = m; else a = m + 1;
      }
      for (int i = a; ok && i < p.num_seqs; ++i) {
        // the sequence occupies [cu[i], cu[i+1]) of the flat space: seg_cost
        // units that stand for the fixed cost of a segment, then its tokens
        // [c0, c1); a range that ends before c0 has none of its tokens
        if (cu[i + 1] == cu[i]) continue;
        const int c0 = cu[i] + p.seg_cost, c1 = cu[i + 1];
        if (c0 >= hi) break;
        GDesc d;
        d.seq = i;
        d.p0 = max(lo, c0) - c0;
        d.p1 = min(hi, c1) - c0;
        const bool complete = c0 >= lo && c1 <= hi;
        d.slot = complete ? -1 : (c0 <= lo ? 2 * int(blockIdx.x) : 2 * int(blockIdx.x) + 1);
        d.qbuf = 0;  // one Q^T buffer: refilled once the previous segment's S MMAs are done
        d.pad = 0;
        // decode step (bf16 caches): if this CTA owns the sequence's last
        // position, its new row (the K warp the K row, the V warp the V row) is
        // loaded now, so the loads are done by the segment's last stage, where
        // it is written. (fp8 caches: the rows are quantized by a launch before
        // this kernel, which is faster than quantizing here.)
        const bool owns_new = !F8 && p.key_new != nullptr && c1 <= hi;
        uint4 nv[64 / T];   // this lane's 16-byte pieces of the row (Hkv * 256 B)
        if (owns_new) {
          const __nv_bfloat16 *src = (is_k ? p.key_new : p.value_new) +
                                     static_cast<int64_t>(i) * (is_k ? p.key_stride : p.value_stride);
#pragma unroll
          for (int u = 0; u < 64 / T; ++u) nv[u] = reinterpret_cast<const uint4 *>(src)[u * 32 + lane];
        }
        const int32_t *row = p.block_tables + static_cast<size_t>(i) * p.max_blocks_per_seq;
        int cached = -(1 << 30), my_id = -1;
        bool first = true;
        for (int pa = d.p0 - d.p0 % T; ok && pa < d.p1; pa += T) {
          const int lb = pa / p.block_size;
          if (lb < cached || lb >= cached + 32) {  // window of 32 block ids, one per lane
            cached = lb;
            my_id = lb + lane < p.max_blocks_per_seq ? __ldg(row + lb + lane) : -1;
          }
          const int blk = __shfl_sync(0xffffffffu, my_id, lb - cached);
          int blk_row = -1;
          if (blk >= 0 && blk < p.num_blocks) {
            blk_row = blk * p.block_size + (pa - lb * p.block_size);
          } else if (lane == 0 && is_k) {
            raise_error(p.err, PKV_DEVERR_BLOCK_ID);
          }
          d.pa = pa;
          d.flags = (first ? kFirst : 0) | (pa + T >= d.p1 ? kLast : 0);
          if (owns_new && pa + T >= d.p1 && blk_row >= 0) {
            // the sequence's last position is in this stage: write the new
            // row there first, then let the copy engine read it
            const int64_t slot = blk_row + (c1 - c0 - 1 - pa);
            uint4 *d4 = reinterpret_cast<uint4 *>(is_k ? p.k_cache : p.v_cache) + slot * (16 * (128 / T));
#pragma unroll
            for (int u = 0; u < 64 / T; ++u) d4[u * 32 + lane] = nv[u];
            asm volatile("fence.proxy.async.global;" ::: "memory");
            __syncwarp();
          }
          ok = stage(d, blk_row, first);
          first = false;
        }
        ++segs;
      }
    }
    if (ok) {
      GDesc e;
      e.seq = e.pa = e.p0 = e.p1 = e.slot = e.qbuf = e.pad = 0;
      e.flags = kEnd;
      ok = stage(e, -1, false);
    }
    if (lane == 0) {  // drain: the last copies must land before the CTA exits
      for (int j = max(0, issued - S); j < issued; ++j) {
        const int sj = j % S;
        mbar_wait(F8 ? (is_k ? kr_full(sj) : vr_full(sj)) : (is_k ? k_full(sj) : v_full(sj)),
                  (j / S) & 1, nullptr);
      }
    }
  } else if (F8 && warp == 1) {
    // ------------------------------------------- MMA issuer, fp8 (self-polling)
    // With 15 warps every SM sub-partition already runs three or four busy
    // warps, and a separate scheduler warp measured slower than this thread
    // polling its barriers itself (probes first, then the round's MMAs).
    if (lane == 0) {
      // S is E4M3 x E4M3 (kind::f8f6f4), PV f16 x f16: format field 0 means
      // E4M3 for the one and f16 for the other
      constexpr uint32_t kFmt = ~((1u << 7) | (1u << 10));
      const uint32_t idesc_s = umma_idesc_bf16(kRows, 2 * N, false) & kFmt;
      const uint32_t idesc_pv = (umma_idesc_bf16(kHD, N, false) | (1u << 15)) & kFmt;  // A (V) MN-major
      bool ok = true;
      int pv_issued = 0, s_issued = 0;
      // S(j) and PV(j-1) are independent (S^T is double-buffered, PV reads P^T and
      // V), so each is issued as soon as its own inputs are ready: S(j) when K(j)
      // has landed and S^T[j & 1] is free, PV(t) when P(t) and V(t) are ready.
      // The issuer polls both without blocking on either.
      uint32_t first_of = 0;      // bit t & 31: kFirst of stage t, kept from S(t) until PV(t)
      int end_at = -1;            // index of the stage that ends the walk
      unsigned long long idle_since = 0;
      for (uint32_t idle = 0;;) {
        bool did = false;
        // Probes first, MMAs after: a shared-memory access (a barrier probe, a
        // descriptor load) that this thread issues behind its own MMAs waits
        // until the tensor core has taken them, so each round reads everything
        // it needs before it issues anything.
        const int j = s_issued, sj = j % S, bj = j & 1;
        const int t = pv_issued, st = t % S;
        bool do_s = false, do_pv = false;
        int flags = 0;
        if (end_at < 0 && s_issued - pv_issued < 4) {
          const bool k_ready = mbar_test_wait(k_full(sj), (j / S) & 1);
          const bool s_ready = j < 2 || mbar_test_wait(s_free(bj), ((j - 2) >> 1) & 1);
          if (k_ready && s_ready) {
            flags = desc[sj].flags;  // the only field the issuer needs
            if (flags & kEnd) {
              end_at = j;
              did = true;
            } else {
              do_s = true;
            }
          }
        }
        if (pv_issued < s_issued) {
          const bool v_ready = mbar_test_wait(v_full(st), (t / S) & 1);
          const bool p_ready = mbar_test_wait(p_full(t & 1), (t >> 1) & 1);
          do_pv = v_ready && p_ready;
        }
        if (do_s) {
          tc_fence_after();
          // [S_hi | S_lo]^T = K . [Q_hi ; Q_lo]^T: the N hi rows and the N lo
          // rows of the split Q^T buffer are one 2N-row operand, so each
          // step (32 dims) reads the raw K codes once
          const uint64_t dkr = desc_k(base + L.kr + sj * kRawStage, 0, 0), dq = desc_k(sQ, 0, 0);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            umma_f8(tmem_s(bj), dkr + kstep(kk, 0), dq + kstep(kk, 0), idesc_s, kk > 0 ? 1u : 0u);
          umma_commit(s_full(bj));
          first_of = (first_of & ~(1u << (j & 31))) | ((flags & kFirst) ? 1u << (j & 31) : 0u);
          ++s_issued;
          did = true;
        }
        if (do_pv) {
          tc_fence_after();
          const bool first = (first_of >> (t & 31)) & 1u;
          const uint64_t dv = desc_v(sV + st * kKVBytes, 0), dp = desc_k(sP + (t & 1) * 2 * small, 0, small);
#pragma unroll
          for (int kk = 0; kk < kRows / 16; ++kk)
            umma_bf16(tmem_o, dv + static_cast<uint64_t>(kk * (2048 >> 4)), dp + kstep(kk, small >> 4),
                      idesc_pv, (first && kk == 0) ? 0u : 1u);
          umma_commit(pv_done(t & 1));
          umma_commit(v_empty(st));
          ++pv_issued;
          did = true;
        }
        if (end_at >= 0 && pv_issued == s_issued) break;
        // the clock is only read while idle: from the 256th empty poll on
        if (did) {
          idle = 0;
        } else if ((++idle & 255u) == 0) {
          const unsigned long long now = global_timer_ns();
          if (idle == 256u) {
            idle_since = now;
          } else if (*abort_flag || now - idle_since > kWaitTimeoutNs) {
            ok = false;
            break;
          }
        }
      }
      if (!ok) fail();
      if (s_issued > 0) mbar_wait(s_full((s_issued - 1) & 1), ((s_issued - 1) >> 1) & 1, nullptr);
      if (pv_issued > 0) mbar_wait(pv_done((pv_issued - 1) & 1), ((pv_issued - 1) >> 1) & 1, nullptr);
    }
    __syncwarp();
  } else if (!F8 && warp == 1) {
    // ------------------------------------------- MMA issuer, bf16 (commanded)
    // Issues what the scheduler warp tells it, in a fixed order: S(0), S(1),
    // then per stage t: PV(t) and S(t + 2). A shared-memory access this thread
    // issued behind its own MMAs would wait until the tensor core has taken
    // them, so it makes none: it learns each command at a hardware barrier
    // that sums a predicate over the scheduler's lanes.
    const uint32_t idesc_s = umma_idesc_bf16(kRows, N, false);
    const uint32_t idesc_pv = umma_idesc_bf16(kHD, N, false) | (1u << 15);  // A (V) MN-major
    int s_issued = 0, pv_issued = 0;
    for (;;) {
      const int cmd = bar_red_popc(kIssueBarrier, 64, false);
      if (cmd & (kCmdFinish | kCmdAbort)) break;
      if (lane == 0) {
        if (cmd & kCmdPV) {
          const int t = pv_issued, st = t % S;
          const bool first = (cmd & kCmdPVFirst) != 0;
          tc_fence_after();
          const uint64_t dv = desc_v(sV + st * kKVBytes, 0), dp = desc_k(sP + (t & 1) * 2 * small, 0, small);
#pragma unroll
          for (int kk = 0; kk < kRows / 16; ++kk)
            umma_bf16(tmem_o, dv + static_cast<uint64_t>(kk * (2048 >> 4)), dp + kstep(kk, small >> 4),
                      idesc_pv, (first && kk == 0) ? 0u : 1u);
          umma_commit(pv_done(t & 1));
          umma_commit(v_empty(st));
        }
        if (cmd & kCmdS) {
          const int j = s_issued, sj = j % S, bj = j & 1;
          tc_fence_after();
          const uint64_t dk = desc_k(sK + sj * kKVBytes, 0, kRegion), dq = desc_k(sQ, 0, small);
#pragma unroll
          for (int kk = 0; kk < kHD / 16; ++kk)
            umma_bf16(tmem_s(bj), dk + kstep(kk, kRegion >> 4), dq + kstep(kk, small >> 4), idesc_s,
                      kk > 0 ? 1u : 0u);
          umma_commit(s_full(bj));
        }
      }
      if (cmd & kCmdPV) ++pv_issued;
      if (cmd & kCmdS) ++s_issued;
    }
    // every MMA issued completes before TMEM is freed
    if (lane == 0) {
      if (s_issued > 0) mbar_wait(s_full((s_issued - 1) & 1), ((s_issued - 1) >> 1) & 1, nullptr);
      if (pv_issued > 0) mbar_wait(pv_done((pv_issued - 1) & 1), ((pv_issued - 1) >> 1) & 1, nullptr);
    }
    __syncwarp();
  } else if (!F8 && warp == NT / 32 - 1) {
    // --------------------------------------------------------- MMA scheduler
    // Polls the inputs of the MMA warp's next groups and hands them over as
    // commands: PV(t) once V(t) and P(t) are ready; S(j) once K(j) is ready
    // and the softmax warps have read S^T[j & 1] (S(j - 2)), which S(j)
    // overwrites. Both may go in one command, PV first.
    // The walk ends at the stage whose descriptor carries kEnd.
    auto send = [&](int cmd) { bar_red_popc(kIssueBarrier, 64, lane < cmd); };
    int t_pv = 0, j_s = 0;      // next PV, next S
    int n = -1;                 // number of stages, once the end has been seen
    uint32_t first_of = 0;      // bit t & 31: kFirst of stage t
    bool ok = true;
    unsigned long long idle_since = 0;
    for (uint32_t idle = 0;;) {
      int cmd = 0, done = 0;
      if (lane == 0) {
        bool pv = false;
        if (t_pv < j_s) {
          const bool v_ready = mbar_test_wait(v_full(t_pv % S), (t_pv / S) & 1);
          const bool p_ready = mbar_test_wait(p_full(t_pv & 1), (t_pv >> 1) & 1);
          pv = v_ready && p_ready;
        }
        const int pv_after = t_pv + (pv ? 1 : 0);
        bool sv = false;
        // at most two S ahead of the PVs: S(j) writes the S^T buffer of S(j - 2)
        if (n < 0 && j_s - pv_after < 3 && mbar_test_wait(k_full(j_s % S), (j_s / S) & 1) &&
            (j_s < 2 || mbar_test_wait(s_free(j_s & 1), ((j_s - 2) >> 1) & 1))) {
          const int flags = desc[j_s % S].flags;
          if (flags & kEnd) {
            n = j_s;
          } else {
            sv = true;
            first_of = (first_of & ~(1u << (j_s & 31))) | ((flags & kFirst) ? 1u << (j_s & 31) : 0u);
          }
        }
        if (pv) cmd |= kCmdPV | (((first_of >> (t_pv & 31)) & 1u) ? kCmdPVFirst : 0);
        if (sv) cmd |= kCmdS;
        done = (n >= 0 && pv_after == n) ? 1 : 0;
        // nothing to hand over: sleep on the barrier that usually completes
        // next (P of the oldest pending PV, else the next K stage) instead of
        // spinning, which would take issue slots from the warps sharing this
        // scheduler's SM sub-partition
        if (!cmd && !done) {
          if (t_pv < j_s) mbar_try_wait(p_full(t_pv & 1), (t_pv >> 1) & 1);
          else if (n < 0) mbar_try_wait(k_full(j_s % S), (j_s / S) & 1);
        }
      }
      cmd = __shfl_sync(0xffffffffu, cmd, 0);
      done = __shfl_sync(0xffffffffu, done, 0);
      n = __shfl_sync(0xffffffffu, n, 0);
      if (cmd) {
        send(cmd);
        if (cmd & kCmdPV) ++t_pv;
        if (cmd & kCmdS) ++j_s;
        idle = 0;
      }
      if (done) break;
      if (!cmd && (++idle & 255u) == 0) {
        int stop = 0;
        if (lane == 0) {
          const unsigned long long now = global_timer_ns();
          if (idle == 256u) idle_since = now;
          else if (*abort_flag || now - idle_since > kWaitTimeoutNs) stop = 1;
        }
        if (__shfl_sync(0xffffffffu, stop, 0)) {
          ok = false;
          break;
        }
      }
    }
    if (!ok) fail();
    send(ok ? kCmdFinish : kCmdAbort);
  } else if (F8 && warp >= 7 && warp < 15) {
    // ------------------------------------------------------------ converters
    // Warps 11-14 expand each raw V stage, one 128-code row per thread, from
    // E4M3 into the f16 operand layout. The S MMA reads the raw K codes as they
    // landed; warps 7-10 only turn, at a segment's first stage, the new Q^T
    // buffer into its two E4M3 terms (split_q_e4m3).
    const bool is_k = warp < 11;
    const int r = static_cast<int>(threadIdx.x) - (is_k ? 224 : 352);
    float *qinv = reinterpret_cast<float *>(smem + L.qs);
    for (int j = 0;; ++j) {
      const int s = j % S;
      if (!warp_wait(is_k ? kr_full(s) : vr_full(s), (j / S) & 1, abort_flag)) {
        fail();
        break;
      }
      const int flags = is_k ? desc[s].flags : vflag[s];
      if (flags & kEnd) {
        __syncwarp();
        if (is_k && lane == 0) mbar_arrive(k_full(s));  // lets the MMA and softmax see the end
        break;
      }
      if (!is_k) convert_row_e4m3(base + L.vr + s * kRawStage, sV + s * kKVBytes, r);
      if (is_k && (flags & kFirst)) split_q_e4m3(sQ + desc[s].qbuf * 2 * small, small, N, r, qinv);
      fence_proxy_async_smem();  // generic-proxy writes -> tensor-core reads
      __syncwarp();
      if (lane == 0) mbar_arrive(is_k ? k_full(s) : v_full(s));
    }
  } else {
    // --------------------------------------------------------------- softmax
    const int quad = warp & 3;                  // TMEM lane quadrant of this warp
    const int r = quad * 32 + lane;             // stage row (S^T lane) and dim (O^T lane)
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const int head = r / T;                     // KV head of this row
    const int t = r - head * T;                 // token of this row inside the stage
    constexpr int kHeadsInWarp = 32 / T;
    constexpr int kCols = kHeadsInWarp * G;   // S^T columns of the heads of this warp
    const int warp_head0 = (quad * 32) / T;
    const int my_slot = head - warp_head0;      // which of the warp's heads this lane's row is
    float m_used[G], l_part[G];
#pragma unroll
    for (int g = 0; g < G; ++g) {
      m_used[g] = -INFINITY;
      l_part[g] = 0.f;
    }
    int segs_done = 0;
    bool ok = true;
    // fp8: 1 / scale of the Q^T rows of this row's query heads (S^T column
    // h*G + g), set at each segment's first stage
    float qinv[G];
#pragma unroll
    for (int g = 0; g < G; ++g) qinv[g] = 1.f;
    // P^T (N rows x 128 stage rows, K-major, 128-byte swizzle): element (n, r)
    const uint32_t p_half = (r >> 6) * small;
    const int rc = r & 63;
    // The four softmax warps meet once per stage on a hardware barrier that
    // also ORs a flag over their threads. The flag is raised when the maximum
    // of a query head grew past the rescale threshold (rare: all four warps
    // then rescale O^T together) or when a warp gave up on a wait (all four
    // then leave the loop in the same stage, so none is left at the barrier).
    // Between those events the warps exchange nothing: the common stage has
    // no shared-memory round trip for the maximum and no shuffles.
    for (int j = 0;; ++j) {
      const int s = j % S;
      const int buf = j & 1;
      const uint32_t ring_parity = (j / S) & 1;
      // A stage's inputs are usually all in place when the softmax warps get
      // to it (the loaders run stages ahead, S(j) was issued as soon as S(j-2)
      // had been read), and each shared-memory round trip costs hundreds of
      // cycles while the copy engine, the converters and the tensor core
      // stream through shared memory. So the barriers of S(j), PV(j-2) and
      // (fp8) the raw V stage are probed together with the wait for the stage
      // descriptor, and the descriptor and the row scales are read together;
      // only a barrier that was not complete yet is waited on further below.
      bool vr_ready = !F8 || mbar_test_wait(vr_full(s), ring_parity);
      bool s_ready = mbar_test_wait(s_full(buf), (j >> 1) & 1);
      bool pv_ready = j < 2 || mbar_test_wait(pv_done(buf), ((j - 2) >> 1) & 1);
      GDesc d = {0, 0, 0, 0, kEnd, 0, 0, 0};
      float kscale = 1.f, vscale = 1.f;
      if (ok && !warp_wait(k_full(s), ring_parity, abort_flag)) ok = false;
      vr_ready = __all_sync(0xffffffffu, vr_ready);
      if (ok) {
        const int4 *dv = reinterpret_cast<const int4 *>(desc + s);
        const int4 d0 = dv[0], d1 = dv[1];
        d = {d0.x, d0.y, d0.z, d0.w, d1.x, d1.y, d1.z, d1.w};
        // fp8: the row scales sit in the raw stages, which the loaders may
        // refill once every softmax warp has arrived on k_empty (below) and
        // the PV MMA of this stage has completed. Read whatever the stage
        // holds (an end stage loads nothing, and its values go unused).
        if (F8) {
          kscale = reinterpret_cast<const float *>(smem + L.kr + s * kRawStage + kRawCodes)[t * p.num_kv_heads + head];
          if (vr_ready)
            vscale = reinterpret_cast<const float *>(smem + L.vr + s * kRawStage + kRawCodes)[t * p.num_kv_heads + head];
          if ((d.flags & (kFirst | kEnd)) == kFirst) {
#pragma unroll
            for (int g = 0; g < G; ++g) qinv[g] = reinterpret_cast<const float *>(smem + L.qs)[head * G + g];
          }
        }
      }
      s_ready = __all_sync(0xffffffffu, s_ready);
      pv_ready = __all_sync(0xffffffffu, pv_ready);
      const bool end = ok && (d.flags & kEnd);
      const bool work = ok && !end;
      const bool first = (d.flags & kFirst) != 0;
      const int tok = d.pa + t;
      const bool valid = work && tok >= d.p0 && tok < d.p1;
      const bool partial = d.pa < d.p0 || d.pa + T > d.p1;
      float sc[G];
      bool need = false;
      if (work && !s_ready && !warp_wait(s_full(buf), (j >> 1) & 1, abort_flag)) ok = false;
      if (ok && work) {
        tc_fence_after();
        // the S^T columns of all heads of this warp in one load (fp8: one
        // from each half, summed); keep this row's G
        float cols[kCols];
        tmem_ld_cols<kCols>(tmem_s(buf) + lane_off + warp_head0 * G, cols);
        if constexpr (F8) {
          float lo[kCols];
          tmem_ld_cols<kCols>(tmem_s(buf) + lane_off + N + warp_head0 * G, lo);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < kCols; ++i) {
            asm volatile("" : "+f"(cols[i]), "+f"(lo[i]));  // the sums stay behind the wait
            cols[i] += lo[i];
          }
        } else {
          tmem_wait_ld();
        }
        tc_fence_before();
        __syncwarp();
        // S^T[j & 1] has been read (S(j + 2) may overwrite it); S(j) has
        // completed, so K(j) is no longer read, and the descriptor and the K
        // scales of this stage have been read too: the K slot is free
        if (lane == 0) {
          mbar_arrive(s_free(buf));
          mbar_arrive(k_empty(s));
        }
#pragma unroll
        for (int g = 0; g < G; ++g) {
          float v = cols[g];
#pragma unroll
          for (int k = 1; k < kHeadsInWarp; ++k) v = (my_slot == k) ? cols[k * G + g] : v;
          sc[g] = valid ? v * (F8 ? p.scale_log2 * kscale * qinv[g] : p.scale_log2) : -INFINITY;
        }
        if (first) {
          // a segment's first stage fixes the reference maximum of each query
          // head: the maximum over the T rows of its KV head (one warp)
          float vmax[G];
#pragma unroll
          for (int g = 0; g < G; ++g) vmax[g] = sc[g];
#pragma unroll
          for (int off = T >> 1; off >= 1; off >>= 1)
#pragma unroll
            for (int g = 0; g < G; ++g) vmax[g] = fmaxf(vmax[g], __shfl_xor_sync(0xffffffffu, vmax[g], off));
#pragma unroll
          for (int g = 0; g < G; ++g) m_used[g] = vmax[g];
        } else {
#pragma unroll
          for (int g = 0; g < G; ++g) need |= sc[g] > m_used[g] + kRescaleThreshold;
        }
      }
      // PV(j-2) read this stage's P^T buffer: it must be done before the rewrite
      if (ok && work && j >= 2) {
        if (pv_ready || warp_wait(pv_done(buf), ((j - 2) >> 1) & 1, abort_flag)) tc_fence_after();
        else ok = false;
      }
      // a partial stage zeroes its masked rows of the converted V stage, so it
      // waits for the conversion (fp8) or the load (bf16)
      if (ok && work && partial && !warp_wait(v_full(s), ring_parity, abort_flag)) ok = false;
      // fp8: P^T rows carry the V row scale, read from the raw V stage once it
      // has landed (above, if it had by then; a partial stage's conversion
      // implies it)
      if (F8 && ok && work && !vr_ready) {
        if (partial || warp_wait(vr_full(s), ring_parity, abort_flag))
          vscale = reinterpret_cast<const float *>(smem + L.vr + s * kRawStage + kRawCodes)[t * p.num_kv_heads + head];
        else
          ok = false;
      }
      if (!ok && lane == 0) {
        *stop_flag = 1;
        *abort_flag = 1;  // the other roles give up their waits too
      }
      if (bar_red_or(kSoftmaxBarrier, 128, need || !ok)) {
        if (*stop_flag) {
          ok = false;
          break;
        }
        // some head's maximum grew (the flag is only raised in working stages,
        // so every warp is in one): new maxima of every head, O^T rescaled
        float vmax[G];
#pragma unroll
        for (int g = 0; g < G; ++g) vmax[g] = sc[g];
#pragma unroll
        for (int off = T >> 1; off >= 1; off >>= 1)
#pragma unroll
          for (int g = 0; g < G; ++g) vmax[g] = fmaxf(vmax[g], __shfl_xor_sync(0xffffffffu, vmax[g], off));
        float alpha[G];
#pragma unroll
        for (int g = 0; g < G; ++g) {
          alpha[g] = 1.f;
          if (vmax[g] > m_used[g] + kRescaleThreshold) {
            alpha[g] = ex2(m_used[g] - vmax[g]);
            m_used[g] = vmax[g];
          }
          l_part[g] *= alpha[g];
        }
        if (t == 0) {
#pragma unroll
          for (int g = 0; g < G; ++g) alpha_buf[head * G + g] = alpha[g];
        }
        bar_sync(kSoftmaxBarrier, 128);
        // O^T may only be rescaled once every earlier PV has landed in it
        if (j >= 1) {
          if (warp_wait(pv_done((j - 1) & 1), ((j - 1) >> 1) & 1, abort_flag)) tc_fence_after();
          else ok = false;
        }
        if (ok) {
          for (int c0 = 0; c0 < N; c0 += 16) {
            float o[16];
            tmem_ld16(tmem_o + lane_off + c0, o);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 16; ++e)
              if (c0 + e < p.num_q_heads) o[e] *= alpha_buf[c0 + e];
            asm volatile(
                "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
                "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};"
                :: "r"(tmem_o + lane_off + c0), "f"(o[0]), "f"(o[1]), "f"(o[2]), "f"(o[3]),
                   "f"(o[4]), "f"(o[5]), "f"(o[6]), "f"(o[7]), "f"(o[8]), "f"(o[9]), "f"(o[10]),
                   "f"(o[11]), "f"(o[12]), "f"(o[13]), "f"(o[14]), "f"(o[15])
                : "memory");
          }
          tmem_wait_st();
        }
      }
      if (end) break;
      if (!ok) continue;  // the next stage's barrier takes every warp out

      // P^T values and running row sums. bf16: each weight is rounded to bf16
      // before it is summed, so the row sum is the sum of exactly the weights
      // the PV MMA multiplies (the normalised output is then a convex
      // combination of the V rows whatever the rounding)
      float pr[G];
#pragma unroll
      for (int g = 0; g < G; ++g) {
        pr[g] = valid ? ex2(sc[g] - m_used[g]) : 0.f;
        if (!F8) pr[g] = __bfloat162float(__float2bfloat16_rn(pr[g]));
        l_part[g] = first ? pr[g] : l_part[g] + pr[g];
      }
      const uint32_t p_region = sP + buf * 2 * small + p_half;
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const int n = head * G + g;
        const uint32_t addr = p_region + (n >> 3) * 1024 + (n & 7) * 128 +
                              ((((rc >> 3) ^ (n & 7)) << 4) | ((rc & 7) << 1));
        if (F8) st_shared_f16(addr, pr[g] * vscale);
        else st_shared_b16(addr, pr[g]);
      }
      if (!valid) {  // masked row: its V row must be zero for the PV MMA
        const uint32_t vrow = sV + s * kKVBytes + (r >> 3) * 1024 + (r & 7) * 128;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" :: "r"(vrow + c * 16), "r"(0u) : "memory");
          asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" :: "r"(vrow + kRegion + c * 16), "r"(0u) : "memory");
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full(buf));

      if (d.flags & kLast) {
        // row sums of each query head: sum over the T rows of its KV head
        float ls[G];
#pragma unroll
        for (int g = 0; g < G; ++g) ls[g] = l_part[g];
#pragma unroll
        for (int off = T >> 1; off >= 1; off >>= 1)
#pragma unroll
          for (int g = 0; g < G; ++g) ls[g] += __shfl_xor_sync(0xffffffffu, ls[g], off);
        if (t == 0) {
#pragma unroll
          for (int g = 0; g < G; ++g) {
            lsum_buf[head * G + g] = ls[g];
            msum_buf[head * G + g] = m_used[g];
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(l_bar);
        if (!warp_wait(l_bar, segs_done & 1, abort_flag) ||
            !warp_wait(pv_done(buf), (j >> 1) & 1, abort_flag)) {
          ok = false;
          continue;
        }
        tc_fence_after();
        // O^T lane r is output dim r: write every query head's value of this dim
        for (int c0 = 0; c0 < N; c0 += 16) {
          float o[16];
          tmem_ld16(tmem_o + lane_off + c0, o);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const int n = c0 + e;
            if (n < p.num_q_heads) {
              const float l = lsum_buf[n];
              const float v = l > 0.f ? o[e] / l : 0.f;
              if (d.slot < 0) {
                p.out[(static_cast<size_t>(d.seq) * p.num_q_heads + n) * kHD + r] = __float2bfloat16_rn(v);
              } else {
                const size_t rec = static_cast<size_t>(d.slot) * p.num_q_heads + n;
                p.po[rec * kHD + r] = v;
                if (r == 0) p.ml[rec] = make_float2(msum_buf[n], l);
              }
            }
          }
        }
        ++segs_done;
      }
    }
    if (!ok) fail();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, p.tmem_cols);
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

bool encode(CUtensorMap *map, const void *ptr, const cuuint64_t (&dims)[3],
            const cuuint64_t (&strides)[2], const cuuint32_t (&box)[3],
            CUtensorMapDataType type = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, type, 3, const_cast<void *>(ptr), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

using TcgKernel = void (*)(const CUtensorMap, const CUtensorMap, const CUtensorMap, const GParams);

template <int T, bool F8>
TcgKernel tcg_kernel_for_g(int g) {
  switch (g) {
    case 1: return decode_tcg_kernel<T, 1, F8>;
    case 2: return decode_tcg_kernel<T, 2, F8>;
    case 4: return decode_tcg_kernel<T, 4, F8>;
    case 8: return decode_tcg_kernel<T, 8, F8>;
    default: return nullptr;
  }
}

// instantiated shapes: T in {8, 16, 32} (Hkv 16, 8, 4), G in {1, 2, 4, 8}; the
// fp8 variant for T 16 (Hkv 8) and 32 (Hkv 4)
TcgKernel tcg_kernel_for(int t, int g, bool f8) {
  if (f8) {
    switch (t) {
      case 16: return tcg_kernel_for_g<16, true>(g);
      case 32: return tcg_kernel_for_g<32, true>(g);
      default: return nullptr;
    }
  }
  switch (t) {
    case 8: return tcg_kernel_for_g<8, false>(g);
    case 16: return tcg_kernel_for_g<16, false>(g);
    case 32: return tcg_kernel_for_g<32, false>(g);
    default: return nullptr;
  }
}

int pick_stages(int n_cols, bool f8) {
  for (int s = 3; s >= 2; --s)
    if (g_layout(s, n_cols, f8).total + 1024 <= 227 * 1024) return s;
  return 0;
}

}  // namespace

bool decode_tcg_supported(int num_q_heads, int num_kv_heads, int block_size, bool fp8) {
  if (num_kv_heads != 4 && num_kv_heads != 8 && num_kv_heads != 16) return false;
  if (num_q_heads % num_kv_heads != 0) return false;
  if (tcg_kernel_for(kRows / num_kv_heads, num_q_heads / num_kv_heads, fp8) == nullptr) return false;
  const int n_cols = (num_q_heads + 15) / 16 * 16;
  // O^T + the S^T buffers in TMEM
  if (n_cols > kMaxN || (fp8 ? 5 : 3) * n_cols + 16 > 512) return false;
  const int T = kRows / num_kv_heads;
  return block_size % T == 0 && pick_stages(n_cols, fp8) > 0;
}

cudaError_t launch_decode_tcg(const DecodeArgs &a, int grid, float2 *ml, float *po, int seg_cost,
                              int *cu_copies, int cu_stride, cudaStream_t stream) {
  const int n_cols = (a.num_q_heads + 15) / 16 * 16;
  const bool f8 = a.fp8;
  const int stages = pick_stages(n_cols, f8);
  const size_t smem = g_layout(stages, n_cols, f8).total + 1024;
  cudaError_t e = cudaSuccess;
  const int T = kRows / a.num_kv_heads;
  CUtensorMap tq, tk, tv;
  const cuuint64_t cache_rows = static_cast<cuuint64_t>(a.num_blocks) * a.block_size;
  const cuuint64_t hkv = a.num_kv_heads;
  // q as (dim, head, sequence): one box = all query heads of a sequence, one 64-dim half
  const cuuint64_t qd[3] = {kHD, static_cast<cuuint64_t>(a.num_q_heads), static_cast<cuuint64_t>(a.num_seqs)};
  const cuuint64_t qs[2] = {kHD * 2, static_cast<cuuint64_t>(a.num_q_heads) * kHD * 2};
  const cuuint32_t qb[3] = {64, static_cast<cuuint32_t>(a.num_q_heads), 1};
  // cache as (dim, token row, head): one box = T tokens x all heads, one 64-dim half
  const cuuint64_t cd[3] = {kHD, cache_rows, hkv};
  const cuuint64_t cs[2] = {hkv * kHD * 2, kHD * 2};
  const cuuint32_t cb[3] = {64, static_cast<cuuint32_t>(T), static_cast<cuuint32_t>(hkv)};
  // fp8 cache: one-byte codes, a box of all 128 dims is one 128-byte swizzle row
  const cuuint64_t cs8[2] = {hkv * kHD, kHD};
  const cuuint32_t cb8[3] = {kHD, static_cast<cuuint32_t>(T), static_cast<cuuint32_t>(hkv)};
  const bool maps_ok =
      encode(&tq, a.q, qd, qs, qb) &&
      (f8 ? encode(&tk, a.k_cache, cd, cs8, cb8, CU_TENSOR_MAP_DATA_TYPE_UINT8) &&
                encode(&tv, a.v_cache, cd, cs8, cb8, CU_TENSOR_MAP_DATA_TYPE_UINT8)
          : encode(&tk, a.k_cache, cd, cs, cb) && encode(&tv, a.v_cache, cd, cs, cb));
  if (!maps_ok) return cudaErrorInvalidValue;
  int tmem_cols = 32;
  while (tmem_cols < (f8 ? 5 : 3) * n_cols + 16) tmem_cols <<= 1;
  GParams p;
  p.out = static_cast<__nv_bfloat16 *>(a.out);
  p.block_tables = a.block_tables;
  p.max_blocks_per_seq = a.max_blocks_per_seq;
  p.num_seqs = a.num_seqs;
  p.num_q_heads = a.num_q_heads;
  p.num_kv_heads = a.num_kv_heads;
  p.group = a.num_q_heads / a.num_kv_heads;
  p.n_cols = n_cols;
  p.tokens = T;
  p.block_size = a.block_size;
  p.num_blocks = a.num_blocks;
  p.stages = stages;
  p.tmem_cols = tmem_cols;
  p.scale_log2 = a.scale * kLog2e;
  p.ws = static_cast<const uint8_t *>(a.workspace);
  p.ml = ml;
  p.po = po;
  p.err = a.err;
  p.k_scales = a.k_scales;
  p.v_scales = a.v_scales;
  p.seg_cost = seg_cost;
  p.context_lens = a.context_lens;
  p.max_context_len = a.max_context_len;
  p.cu_copies = cu_copies;
  p.cu_stride = cu_stride;
  p.key_new = static_cast<const __nv_bfloat16 *>(a.key_new);
  p.value_new = static_cast<const __nv_bfloat16 *>(a.value_new);
  p.key_stride = a.key_stride;
  p.value_stride = a.value_stride;
  p.k_cache = static_cast<uint8_t *>(const_cast<void *>(a.k_cache));
  p.v_cache = static_cast<uint8_t *>(const_cast<void *>(a.v_cache));
  auto kern = tcg_kernel_for(T, p.group, f8);
  if (kern == nullptr) return cudaErrorInvalidValue;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  // programmatic dependent launch: the prologue (barriers, TMEM, descriptor
  // prefetch) runs while the previous kernel on the stream (the plan launch
  // with fp8 caches) finishes
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(f8 ? kThreadsF8 : kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, tq, tk, tv, p);
}

}  // namespace pkv
