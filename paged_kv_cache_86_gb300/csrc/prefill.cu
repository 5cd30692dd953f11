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
// One CTA = one 128-row query tile of one query head of one sequence. Warps:
//   0      TMA producer: the Q tile once, then per 128-key tile the K and V
//          tiles, gathered block by block from the paged cache with tiled
//          tensor loads (box = 64 dims x 1 KV head x R rows, R = the largest
//          power of two <= 128 dividing the block size), 128-byte swizzled,
//          two stages. Pieces past the sequence read zeros (out-of-range
//          coordinates), so stale shared memory never reaches the MMAs.
//   1      TMEM owner and MMA issuer (one lane): S(j) = Q K(j)^T into TMEM
//          columns 0..127, then O += P(j-1) V(j-1) into columns 128..255.
//   2..5   softmax + epilogue, one thread per query row (its TMEM lane):
//          load S(j), scale to base 2, mask, update the running max lazily
//          (O and l are rescaled only when the max grows by more than 2^8,
//          so P stays <= 256 and rescales are rare), write P as bf16 into a
//          swizzled shared-memory tile (the A operand of the PV MMA), and at
//          the end divide O by the row sum and store bf16 rows.
// Every wait is bounded; on a timeout the CTA records PKV_DEVERR_TIMEOUT,
// drains what it issued, frees its TMEM and exits.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "pkv_device.cuh"
#include "pkv_internal.h"
#include "pkv_tc.cuh"

namespace pkv {
namespace {

constexpr int kTile = 128;          // query rows per CTA, keys per KV tile
constexpr int kHD = 128;            // head dim
constexpr int kRegion = 16384;      // 128 rows x 64 bf16, one 128-byte swizzle column
constexpr int kTileBytes = 2 * kRegion;
constexpr int kStages = 2;
constexpr int kThreads = 192;
constexpr int kTmemCols = 256;      // S: 0..127, O: 128..255
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleThreshold = 8.f;  // log2 units

// shared memory map (offsets from a 1024-byte aligned base)
constexpr int kOffQ = 0;
constexpr int kOffK = kOffQ + kTileBytes;
constexpr int kOffV = kOffK + kStages * kTileBytes;
constexpr int kOffP = kOffV + kStages * kTileBytes;
constexpr int kOffBar = kOffP + kTileBytes;
constexpr int kNumBars = 1 + 4 * kStages + 4;  // q_full, k_full/v_full/k_empty/v_empty, s_full, s_free, p_full, pv_done
constexpr int kSmemBytes = kOffBar + kNumBars * 8 + 16 + 1024;  // + tmem slot, abort flag, alignment slack

struct PrefillParams {
  __nv_bfloat16 *out;
  const int32_t *cu_q;
  const int32_t *cu_k;
  const int32_t *block_tables;
  int max_blocks_per_seq;
  int num_seqs;
  int total_q;
  int num_q_heads;
  int group;
  int block_size;
  int num_blocks;
  int max_seqlen_q;
  int max_seqlen_k;
  int causal;
  int box_rows;   // R
  float scale_log2;
  uint32_t *err;
};

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint64_t desc_kmajor(uint32_t tile_base, int kk) {
  // K step kk (16 elements): column region kk/4, 32-byte step inside the swizzle row
  return smem_desc_sw128(tile_base + (kk >> 2) * kRegion + (kk & 3) * 32, 16, 1024);
}

// start-address increment (16-byte units, the descriptor's low field) of K
// step kk from step 0 of a K-major tile: the issuing thread builds each
// descriptor once per group and steps it
__device__ __forceinline__ uint64_t kmajor_step(int kk) {
  return static_cast<uint64_t>(((kk >> 2) * kRegion + (kk & 3) * 32) >> 4);
}

__device__ __forceinline__ uint64_t desc_v_mnmajor(uint32_t tile_base, int kk) {
  // 16 keys = two 8-row groups (1024 bytes each); N = 128 dims = two regions
  return smem_desc_sw128(tile_base + kk * 2048, kRegion, 1024);
}

__global__ void __launch_bounds__(kThreads, 1)
prefill_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const PrefillParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_addr(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  uint8_t *smem = smem_raw + (base - raw_addr);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int seq = blockIdx.z;
  const int qh = blockIdx.y;
  const int r0 = blockIdx.x * kTile;

  const int q_begin = p.cu_q[seq], q_end = p.cu_q[seq + 1];
  const int k_len = p.cu_k[seq + 1] - p.cu_k[seq];
  const int q_len = q_end - q_begin;
  if (q_len < 0 || q_len > p.max_seqlen_q || q_end > p.total_q || k_len < 0 ||
      k_len > p.max_seqlen_k || (p.causal && q_len > k_len)) {
    if (threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.y == 0) raise_error(p.err, PKV_DEVERR_LENGTH);
    return;
  }
  if (r0 >= q_len) return;
  const int prefix = p.causal ? k_len - q_len : 0;
  const int last_row = min(r0 + kTile - 1, q_len - 1);
  const int key_end = p.causal ? min(prefix + last_row + 1, k_len) : k_len;
  const int n_tiles = (key_end + kTile - 1) / kTile;
  const int kvh = qh / p.group;

  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kOffBar);
  const uint32_t bar0 = smem_addr(bars);
  auto bar = [&](int i) { return bar0 + 8u * i; };
  const uint32_t q_full = bar(0);
  auto k_full = [&](int s) { return bar(1 + s); };
  auto v_full = [&](int s) { return bar(1 + kStages + s); };
  auto k_empty = [&](int s) { return bar(1 + 2 * kStages + s); };
  auto v_empty = [&](int s) { return bar(1 + 3 * kStages + s); };
  const uint32_t s_full = bar(1 + 4 * kStages);
  const uint32_t s_free = bar(2 + 4 * kStages);
  const uint32_t p_full = bar(3 + 4 * kStages);
  const uint32_t pv_done = bar(4 + 4 * kStages);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + kOffBar + kNumBars * 8);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(k_full(s), 1);
      mbar_init(v_full(s), 1);
      mbar_init(k_empty(s), 1);
      mbar_init(v_empty(s), 1);
    }
    mbar_init(s_full, 1);
    mbar_init(s_free, 4);
    mbar_init(p_full, 4);
    mbar_init(pv_done, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tmem_s = tmem;
  const uint32_t tmem_o = tmem + kTile;

  const uint32_t sQ = base + kOffQ;
  auto sK = [&](int s) { return base + kOffK + s * kTileBytes; };
  auto sV = [&](int s) { return base + kOffV + s * kTileBytes; };
  const uint32_t sP = base + kOffP;

  auto fail = [&]() {
    *abort_flag = 1;
    raise_error(p.err, PKV_DEVERR_TIMEOUT);
  };

  if (warp == 0) {
    // ------------------------------------------------------------- producer
    int k_issued = 0, v_issued = 0;
    bool ok = true;
    if (n_tiles > 0) {
      if (lane == 0) {
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
        mbar_arrive_expect_tx(q_full, kTileBytes);
        tma_load_3d(sQ, &tm_q, 0, qh, q_begin + r0, q_full);
        tma_load_3d(sQ + kRegion, &tm_q, 64, qh, q_begin + r0, q_full);
      }
      const int R = p.box_rows;
      const int pieces = kTile / R;
      const int oob_row = p.num_blocks * p.block_size;  // past the cache: reads zeros
      const int32_t *bt = p.block_tables + static_cast<size_t>(seq) * p.max_blocks_per_seq;
      for (int j = 0; ok && j < n_tiles; ++j) {
        const int s = j % kStages;
        const int round = j / kStages;
        // this lane's piece of the tile: cache row of keys j*128 + lane*R ..
        int row = oob_row;
        if (lane < pieces) {
          const int key = j * kTile + lane * R;
          if (key < k_len) {
            const int blk = __ldg(bt + key / p.block_size);
            if (blk >= 0 && blk < p.num_blocks) row = blk * p.block_size + key % p.block_size;
            else raise_error(p.err, PKV_DEVERR_BLOCK_ID);
          }
        }
        for (int which = 0; which < 2 && ok; ++which) {  // 0: K, 1: V
          const uint32_t full = which ? v_full(s) : k_full(s);
          const uint32_t empty = which ? v_empty(s) : k_empty(s);
          const uint32_t dst = which ? sV(s) : sK(s);
          const CUtensorMap *map = which ? &tm_v : &tm_k;
          int good = 1;
          if (lane == 0) {
            if (round > 0 && !mbar_wait(empty, (round - 1) & 1, abort_flag)) {
              good = 0;
              fail();
            } else {
              mbar_arrive_expect_tx(full, kTileBytes);
            }
          }
          good = __shfl_sync(0xffffffffu, good, 0);
          if (!good) {
            ok = false;
            break;
          }
          if (lane < pieces) {
            tma_load_3d(dst + lane * R * 128, map, 0, kvh, row, full);
            tma_load_3d(dst + kRegion + lane * R * 128, map, 64, kvh, row, full);
          }
          if (which) ++v_issued; else ++k_issued;
        }
      }
      // drain: the last loads of each stage must land before the CTA exits
      if (lane == 0) {
        mbar_wait(q_full, 0, nullptr);
        for (int j = max(0, k_issued - kStages); j < k_issued; ++j)
          mbar_wait(k_full(j % kStages), (j / kStages) & 1, nullptr);
        for (int j = max(0, v_issued - kStages); j < v_issued; ++j)
          mbar_wait(v_full(j % kStages), (j / kStages) & 1, nullptr);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && n_tiles > 0) {
      constexpr uint32_t idesc_s = umma_idesc_bf16(kTile, kTile, false);
      constexpr uint32_t idesc_pv = umma_idesc_bf16(kTile, kHD, true);
      bool ok = mbar_wait(q_full, 0, abort_flag);
      int pv_issued = 0, s_issued = 0;
      auto issue_pv = [&](int t) -> bool {
        const int s = t % kStages;
        if (!mbar_wait(v_full(s), (t / kStages) & 1, abort_flag)) return false;
        if (!mbar_wait(p_full, t & 1, abort_flag)) return false;
        tc_fence_after();
        const uint64_t dp = desc_kmajor(sP, 0), dv = desc_v_mnmajor(sV(s), 0);
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk)
          umma_bf16(tmem_o, dp + kmajor_step(kk), dv + static_cast<uint64_t>(kk * (2048 >> 4)), idesc_pv,
                    (t > 0 || kk > 0) ? 1u : 0u);
        umma_commit(pv_done);
        umma_commit(v_empty(s));
        ++pv_issued;
        return true;
      };
      for (int j = 0; ok && j < n_tiles; ++j) {
        const int s = j % kStages;
        ok = mbar_wait(k_full(s), (j / kStages) & 1, abort_flag);
        if (ok && j > 0) ok = mbar_wait(s_free, (j - 1) & 1, abort_flag);
        if (!ok) break;
        tc_fence_after();
        const uint64_t dq = desc_kmajor(sQ, 0), dk = desc_kmajor(sK(s), 0);
#pragma unroll
        for (int kk = 0; kk < kHD / 16; ++kk)
          umma_bf16(tmem_s, dq + kmajor_step(kk), dk + kmajor_step(kk), idesc_s, kk > 0 ? 1u : 0u);
        umma_commit(s_full);
        umma_commit(k_empty(s));
        ++s_issued;
        if (j > 0) ok = issue_pv(j - 1);
      }
      if (ok) ok = issue_pv(n_tiles - 1);
      if (!ok) fail();
      // every MMA this thread issued has completed once its last commit lands
      if (s_issued > 0) mbar_wait(s_full, (s_issued - 1) & 1, nullptr);
      if (pv_issued > 0) mbar_wait(pv_done, (pv_issued - 1) & 1, nullptr);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------- softmax warps
    const int quad = warp & 3;                       // TMEM lanes 32*quad .. 32*quad+31
    const int r = quad * 32 + lane;                  // query row inside the tile
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const int qpos = prefix + r0 + r;                // absolute position of this row
    const int visible = p.causal ? min(qpos + 1, k_len) : k_len;
    float m_used = -INFINITY, l_sum = 0.f;
    bool ok = true;
    // P tile row address pieces (128-byte swizzle: 16-byte chunk c of row r at c ^ (r % 8))
    const uint32_t p_row = sP + (r >> 3) * 1024 + (r & 7) * 128;

    for (int j = 0; ok && j < n_tiles; ++j) {
      if (!__all_sync(0xffffffffu, mbar_wait(s_full, j & 1, abort_flag))) { ok = false; break; }
      tc_fence_after();
      float s[kTile];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(tmem_s + lane_off + c * 32, *reinterpret_cast<float(*)[32]>(s + c * 32));
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(s_free);

      const int key0 = j * kTile;
      float mt = -INFINITY;
      if (key0 + kTile <= visible) {
#pragma unroll
        for (int c = 0; c < kTile; ++c) {
          s[c] *= p.scale_log2;
          mt = fmaxf(mt, s[c]);
        }
      } else {
#pragma unroll
        for (int c = 0; c < kTile; ++c) {
          s[c] = (key0 + c < visible) ? s[c] * p.scale_log2 : -INFINITY;
          mt = fmaxf(mt, s[c]);
        }
      }
      float alpha = 1.f;
      const bool grow = mt > m_used + kRescaleThreshold;
      if (grow) {
        alpha = ex2(m_used - mt);
        m_used = mt;
        l_sum *= alpha;
      }
      // PV(j-1) must be done before O is rescaled or the P tile rewritten
      if (j > 0) {
        if (!__all_sync(0xffffffffu, mbar_wait(pv_done, (j - 1) & 1, abort_flag))) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (__any_sync(0xffffffffu, grow)) {
          const float a = grow ? alpha : 1.f;
#pragma unroll 1
          for (int c = 0; c < 4; ++c) {
            float o[32];
            tmem_ld32(tmem_o + lane_off + c * 32, o);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] *= a;
            tmem_st32(tmem_o + lane_off + c * 32, o);
          }
          tmem_wait_st();
        }
      }
      float rs = 0.f;
#pragma unroll
      for (int c8 = 0; c8 < kTile / 8; ++c8) {
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float a0 = ex2(s[c8 * 8 + 2 * e] - m_used);
          const float a1 = ex2(s[c8 * 8 + 2 * e + 1] - m_used);
          rs += a0 + a1;
          w[e] = float2_to_bf16x2(a0, a1);
        }
        const int chunk = c8 & 7;
        const uint32_t addr = p_row + (c8 >> 3) * kRegion + ((chunk ^ (r & 7)) << 4);
        asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};"
                     :: "r"(addr), "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]) : "memory");
      }
      l_sum += rs;
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full);
    }

    if (!ok) fail();
    // epilogue: O / l -> bf16 rows
    const bool have = n_tiles > 0;
    if (have && ok) {
      ok = __all_sync(0xffffffffu, mbar_wait(pv_done, (n_tiles - 1) & 1, abort_flag));
      tc_fence_after();
    }
    const bool store = (r0 + r) < q_len;
    __nv_bfloat16 *orow = p.out + (static_cast<size_t>(q_begin) + r0 + r) * p.num_q_heads * kHD +
                          static_cast<size_t>(qh) * kHD;
    const float inv = (l_sum > 0.f) ? 1.f / l_sum : 0.f;
#pragma unroll 1
    for (int c = 0; c < 4; ++c) {
      float o[32];
      if (have && ok) {
        tmem_ld32(tmem_o + lane_off + c * 32, o);
        tmem_wait_ld();
      } else {
#pragma unroll
        for (int e = 0; e < 32; ++e) o[e] = 0.f;
      }
      if (store) {
        uint4 *dst = reinterpret_cast<uint4 *>(orow + c * 32);
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          uint4 v;
          v.x = float2_to_bf16x2(o[q4 * 8 + 0] * inv, o[q4 * 8 + 1] * inv);
          v.y = float2_to_bf16x2(o[q4 * 8 + 2] * inv, o[q4 * 8 + 3] * inv);
          v.z = float2_to_bf16x2(o[q4 * 8 + 4] * inv, o[q4 * 8 + 5] * inv);
          v.w = float2_to_bf16x2(o[q4 * 8 + 6] * inv, o[q4 * 8 + 7] * inv);
          dst[q4] = v;
        }
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

// ------------------------------------------------------------ tensor maps --

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

// 3-D map over a [rows, heads, 128] bf16 array: box = 64 dims x 1 head x box_rows rows.
bool make_map(CUtensorMap *map, const void *base, uint64_t rows, uint64_t heads, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(kHD), heads, rows};
  cuuint64_t strides[2] = {kHD * 2, heads * kHD * 2};
  cuuint32_t box[3] = {64, 1, box_rows};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool prefill_supported(int num_q_heads, int num_kv_heads, int block_size) {
  return num_kv_heads >= 1 && num_q_heads % num_kv_heads == 0 && block_size % 8 == 0;
}

cudaError_t launch_paged_prefill(const PrefillArgs &a, cudaStream_t stream) {
  if (a.num_seqs == 0 || a.total_q == 0 || a.max_seqlen_q == 0) return cudaSuccess;
  if (prefill_pp_supported(a.num_q_heads, a.num_kv_heads, a.block_size))
    return launch_prefill_pp(a, stream);
  static std::once_flag attr_once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(attr_once, [] {
    attr_err = cudaFuncSetAttribute(prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    kSmemBytes);
  });
  if (attr_err != cudaSuccess) return attr_err;
  int box_rows = a.block_size & -a.block_size;
  if (box_rows > kTile) box_rows = kTile;
  CUtensorMap tq, tk, tv;
  const uint64_t cache_rows = static_cast<uint64_t>(a.num_blocks) * a.block_size;
  if (!make_map(&tq, a.q, a.total_q, a.num_q_heads, kTile) ||
      !make_map(&tk, a.k_cache, cache_rows, a.num_kv_heads, box_rows) ||
      !make_map(&tv, a.v_cache, cache_rows, a.num_kv_heads, box_rows))
    return cudaErrorInvalidValue;
  PrefillParams p;
  p.out = static_cast<__nv_bfloat16 *>(a.out);
  p.cu_q = a.cu_seqlens_q;
  p.cu_k = a.cu_seqlens_k;
  p.block_tables = a.block_tables;
  p.max_blocks_per_seq = a.max_blocks_per_seq;
  p.num_seqs = a.num_seqs;
  p.total_q = a.total_q;
  p.num_q_heads = a.num_q_heads;
  p.group = a.num_q_heads / a.num_kv_heads;
  p.block_size = a.block_size;
  p.num_blocks = a.num_blocks;
  p.max_seqlen_q = a.max_seqlen_q;
  p.max_seqlen_k = a.max_seqlen_k;
  p.causal = a.causal ? 1 : 0;
  p.box_rows = box_rows;
  p.scale_log2 = a.scale * kLog2e;
  p.err = a.err;
  dim3 grid((a.max_seqlen_q + kTile - 1) / kTile, a.num_q_heads, a.num_seqs);
  prefill_kernel<<<grid, kThreads, kSmemBytes, stream>>>(tq, tk, tv, p);
  return cudaGetLastError();
}

}  // namespace pkv
