// prefill_pp.cu -- paged chunked-prefill attention, two query heads per CTA in
// ping-pong on the tcgen05 tensor cores (sm_103a).
//
// Same computation as prefill.cu (varlen query chunks over their cached prefix
// plus themselves, bottom-right causal; nano vllm代码详解 §2 context;
// 推理运行时 §Prefill 与 decode 输入; Mini-SGLang 源码解析（二）§6.6), and the
// same compute-bound regime (Mini-SGLang 源码解析（二）§8.3). What changes is
// the schedule, so that the tensor core never waits for a softmax:
//
//   * One work item = one 128-row query tile of TWO query heads A and B of the
//     same KV head (GQA), or, when the GQA group is odd, two consecutive query
//     tiles A and B of one head: either way the K and V tiles are loaded once
//     for both.
//   * Two softmax warpgroups (warps 0-3 for A, 4-7 for B). While one computes
//     the softmax of its tile, the tensor core runs the other head's S and PV.
//     The third warpgroup holds the Q/K loader (warp 8), the MMA issuer (warp
//     9) and the V loader (warp 10); it gives up most of its registers
//     (setmaxnreg) so each softmax thread can keep a whole 128-score row live.
//     MMA issue order per KV tile j: PV_A(j-1), S_A(j), PV_B(j-1), S_B(j).
//   * All four accumulators live in TMEM (S_A, S_B, O_A, O_B: 4 x 128 columns,
//     the whole TMEM of the SM). P is written back as bf16 over the first 64
//     columns of its S and fed to the PV MMA as the A operand straight from
//     TMEM, so shared memory only holds Q_A, Q_B and two K and two V stages.
//   * The softmax works on raw scores (max of s, then exp2(s*c - m*c) with one
//     FFMA per element, c = scale * log2 e) and rescales O lazily: only when a
//     row's maximum grows by more than 2^8 (in units of c), so O stays valid
//     and P <= 256 fits bf16. A rescale needs no extra wait: S_X(j) completing
//     implies PV_X(j-1) completed (the tensor core runs one CTA's MMAs in order).
//
// Every wait is bounded; on a timeout the CTA records PKV_DEVERR_TIMEOUT,
// drains its copies and MMAs, frees its TMEM and exits.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "pkv_device.cuh"
#include "pkv_internal.h"
#include "pkv_tc.cuh"

namespace pkv {
namespace {

constexpr int kTile = 128;
constexpr int kHD = 128;
constexpr int kRegion = 16384;
constexpr int kTileBytes = 2 * kRegion;
constexpr int kKStages = 3;          // K is needed first (S), so it runs furthest ahead
constexpr int kVStages = 2;
constexpr int kThreads = 384;        // softmax A (warpgroup 0), softmax B (1), loaders + MMA (2)
constexpr int kWarpQK = 8, kWarpMma = 9, kWarpV = 10;
// Register split: launched at 168 per thread (384 x 168 = 64512); warpgroup 2
// drops to 104 and the two softmax warpgroups rise to 200, which adds back up
// to the launch total: 2 x 128 x 200 + 128 x 104 = 64512.
constexpr int kRegsLaunch = 168, kRegsLow = 104, kRegsHigh = 200;
static_assert(2 * 128 * kRegsHigh + 128 * kRegsLow == kThreads * kRegsLaunch,
              "setmaxnreg split must add up to the launch allocation");
constexpr int kTmemCols = 512;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleThreshold = 8.f;

constexpr int kOffQ = 0;                              // Q_A, Q_B
constexpr int kOffK = kOffQ + 2 * kTileBytes;
constexpr int kOffV = kOffK + kKStages * kTileBytes;
constexpr int kOffBar = kOffV + kVStages * kTileBytes;
constexpr int kItemRing = 4;         // work items handed from the Q/K loader to the other roles
// q, k/v full/empty, s/p/pv x2, q_empty, o_free x2, item full/empty x kItemRing
constexpr int kNumBars = 1 + 2 * kKStages + 2 * kVStages + 9 + 2 * kItemRing;
constexpr int kSmemBytes = kOffBar + kNumBars * 8 + 16 + 4 * kItemRing + 1024;
constexpr int kItemReaders = 1 + 1 + 8;   // V loader, MMA issuer, eight softmax warps

struct PPParams {
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
  int box_rows;
  // block sizes that are not a multiple of 8: the loaders gather K/V rows with
  // cp.async (a TMA box must fill whole 8-row swizzle atoms)
  const uint8_t *k_cache;
  const uint8_t *v_cache;
  int num_kv_heads;
  int q_tiles;       // 128-row query tiles of the longest chunk
  int pair_tiles;    // odd GQA group: A and B are two consecutive query tiles of one head
  uint32_t *ticket;  // next unclaimed work item (zeroed before the launch)
  float scale_log2;
  uint32_t *err;
};

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint64_t desc_kmajor(uint32_t tile_base, int kk) {
  return smem_desc_sw128(tile_base + (kk >> 2) * kRegion + (kk & 3) * 32, 16, 1024);
}

// start-address increment (16-byte units, the descriptor's low field) of K
// step kk from step 0 of a K-major tile
__device__ __forceinline__ uint32_t kmajor_step(int kk) {
  return static_cast<uint32_t>(((kk >> 2) * kRegion + (kk & 3) * 32) >> 4);
}

// descriptor d with its start address moved by `step` 16-byte units: a 32-bit
// add, since the 14-bit address field (shared memory is under 256 KB) never
// carries into the descriptor's upper word
__device__ __forceinline__ uint64_t desc_at(uint64_t d, uint32_t step) {
  return (d & 0xFFFFFFFF00000000ull) | static_cast<uint32_t>(static_cast<uint32_t>(d) + step);
}

__device__ __forceinline__ uint64_t desc_v_mnmajor(uint32_t tile_base, int kk) {
  return smem_desc_sw128(tile_base + kk * 2048, kRegion, 1024);
}

// D[tmem] (+)= A[tmem] * B[smem desc], bf16 inputs, fp32 accumulator.
__device__ __forceinline__ void umma_bf16_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                                 uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
      :: "r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate) : "memory");
}

__device__ __forceinline__ void tmem_st32_u(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
      "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};"
      :: "r"(taddr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]),
         "r"(v[7]), "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]),
         "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]),
         "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]),
         "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}

__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, const volatile int *abort) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort));
}

// kGather: the loaders gather K/V rows with cp.async (block sizes that are not
// a multiple of 8) instead of loading TMA boxes; a separate instance, so that
// the box path compiles as if the gather did not exist
template <bool kGather>
__global__ void __launch_bounds__(kThreads, 1)
prefill_pp_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const PPParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_addr(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  uint8_t *smem = smem_raw + (base - raw_addr);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // Persistent: each CTA claims work items from a global ticket (the Q/K loader
  // takes the next one when it starts an item and passes it to the other roles
  // through a small ring), so long and short items balance across SMs. Item w
  // is query tile (last first) w % n_xt of head pair (w / n_xt) % n_hp of
  // sequence w / (n_xt * n_hp): items claimed close in time read the K/V of a
  // few sequences (L2 reuse). All roles walk the same items, skip the same ones.
  // With an odd GQA group the two heads of a pair would read different K/V, so
  // A and B are instead two consecutive query tiles of one head (a "tile" of
  // the walk is then 256 rows): they still share every K/V tile, and A's rows
  // mask the last one, which only B needs.
  const int xt_rows = p.pair_tiles ? 2 * kTile : kTile;   // rows of the walk's tile
  const int n_xt = p.pair_tiles ? (p.q_tiles + 1) / 2 : p.q_tiles;
  const int n_hp = p.pair_tiles ? p.num_q_heads : p.num_q_heads / 2;
  const int head_step = p.pair_tiles ? 0 : 1;             // head of B = head of A + head_step
  const int row_step = p.pair_tiles ? kTile : 0;          // first row of B = first row of A + row_step
  const int n_items = n_xt * n_hp * p.num_seqs;
  struct Item {
    int seq, qh_a, r0, q_begin, q_len, k_len, prefix, n_tiles, kvh;
  };
  auto item_at = [&](int w, Item &it) -> bool {
    it.r0 = (n_xt - 1 - w % n_xt) * xt_rows;
    it.qh_a = (1 + head_step) * ((w / n_xt) % n_hp);
    it.seq = w / (n_xt * n_hp);
    it.q_begin = p.cu_q[it.seq];
    const int q_end = p.cu_q[it.seq + 1];
    it.k_len = p.cu_k[it.seq + 1] - p.cu_k[it.seq];
    it.q_len = q_end - it.q_begin;
    if (it.q_len < 0 || it.q_len > p.max_seqlen_q || q_end > p.total_q || it.k_len < 0 ||
        it.k_len > p.max_seqlen_k || (p.causal && it.q_len > it.k_len)) {
      if (threadIdx.x == 0 && it.qh_a == 0 && it.r0 == 0) raise_error(p.err, PKV_DEVERR_LENGTH);
      return false;
    }
    if (it.r0 >= it.q_len) return false;
    it.prefix = p.causal ? it.k_len - it.q_len : 0;
    const int last_row = min(it.r0 + xt_rows - 1, it.q_len - 1);
    const int key_end = p.causal ? min(it.prefix + last_row + 1, it.k_len) : it.k_len;
    it.n_tiles = (key_end + kTile - 1) / kTile;
    it.kvh = it.qh_a / p.group;
    return true;
  };

  const uint32_t bar0 = base + kOffBar;
  const uint32_t q_full = bar0;
  constexpr int kB = 1 + 2 * kKStages + 2 * kVStages;
  auto k_full = [&](int s) { return bar0 + 8u * (1 + s); };
  auto k_empty = [&](int s) { return bar0 + 8u * (1 + kKStages + s); };
  auto v_full = [&](int s) { return bar0 + 8u * (1 + 2 * kKStages + s); };
  auto v_empty = [&](int s) { return bar0 + 8u * (1 + 2 * kKStages + kVStages + s); };
  auto s_full = [&](int x) { return bar0 + 8u * (kB + x); };
  auto p_full = [&](int x) { return bar0 + 8u * (kB + 2 + x); };
  auto pv_done = [&](int x) { return bar0 + 8u * (kB + 4 + x); };
  const uint32_t q_empty = bar0 + 8u * (kB + 6);                         // last S of an item done
  auto o_free = [&](int x) { return bar0 + 8u * (kB + 7 + x); };         // O_X read out
  auto item_full = [&](int i) { return bar0 + 8u * (kB + 9 + i); };
  auto item_empty = [&](int i) { return bar0 + 8u * (kB + 9 + kItemRing + i); };
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + kOffBar + kNumBars * 8);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  volatile int *item_ring = reinterpret_cast<volatile int *>(smem + kOffBar + kNumBars * 8 + 16);

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    for (int s = 0; s < kKStages; ++s) {
      mbar_init(k_full(s), 1);
      mbar_init(k_empty(s), 1);
    }
    for (int s = 0; s < kVStages; ++s) {
      mbar_init(v_full(s), 1);
      mbar_init(v_empty(s), 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(s_full(x), 1);
      mbar_init(p_full(x), 4);
      mbar_init(pv_done(x), 1);
      mbar_init(o_free(x), 4);
    }
    for (int i = 0; i < kItemRing; ++i) {
      mbar_init(item_full(i), 1);
      mbar_init(item_empty(i), kItemReaders);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == kWarpMma) {
    tmem_alloc(smem_addr(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  auto tmem_s = [&](int x) { return tmem + x * kTile; };           // S_A, S_B (P over cols 0..63)
  auto tmem_o = [&](int x) { return tmem + (2 + x) * kTile; };     // O_A, O_B
  const uint32_t sQ = base + kOffQ;
  auto sK = [&](int s) { return base + kOffK + s * kTileBytes; };
  auto sV = [&](int s) { return base + kOffV + s * kTileBytes; };
  auto fail = [&]() {
    *abort_flag = 1;
    raise_error(p.err, PKV_DEVERR_TIMEOUT);
  };
  // The n-th item of this CTA for a reader role (a whole warp, or lane 0 of the
  // MMA warp alone): -1 on a timeout; n_items or more ends the walk.
  auto read_item = [&](int n, bool whole_warp) -> int {
    const int slot = n % kItemRing;
    const uint32_t par = (n / kItemRing) & 1;
    const bool got = whole_warp ? warp_wait(item_full(slot), par, abort_flag)
                                : mbar_wait(item_full(slot), par, abort_flag);
    if (!got) return -1;
    const int w = item_ring[slot];
    if (whole_warp) __syncwarp();
    if (!whole_warp || lane == 0) mbar_arrive(item_empty(slot));
    return w;
  };

  if (warp >= 8) {
    // The loader / MMA warpgroup hands registers to the softmax warpgroups;
    // each branch of the split holds exactly one setmaxnreg, executed by all
    // four warps of its warpgroup.
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" :: "n"(kRegsLow));
    if (warp == kWarpQK || warp == kWarpV) {
      // ------------------------------------------------------------ producers
      // one warp loads Q_A, Q_B and the K tiles, the other the V tiles; the
      // rings run on across items, so the next item's loads overlap the end of
      // the current one
      const bool is_k = warp == kWarpQK;
      const int stages = is_k ? kKStages : kVStages;
      int issued = 0, items = 0;
      bool ok = true;
      if (lane == 0) {
        if (is_k) {
          tma_prefetch_desc(&tm_q);
          tma_prefetch_desc(&tm_k);
        } else {
          tma_prefetch_desc(&tm_v);
        }
      }
      const int R = p.box_rows;
      const int pieces = kTile / R;
      const int oob_row = p.num_blocks * p.block_size;
      Item it;
      for (int n = 0; ok; ++n) {
        int w;
        if (is_k) {  // claim the next item and hand it to the readers
          w = -1;
          if (lane == 0) {
            const int slot = n % kItemRing;
            if (n >= kItemRing &&
                !mbar_wait(item_empty(slot), ((n / kItemRing) - 1) & 1, abort_flag)) {
              fail();
            } else {
              w = static_cast<int>(atomicAdd(p.ticket, 1u));
              item_ring[slot] = w;
              mbar_arrive(item_full(slot));
            }
          }
          w = __shfl_sync(0xffffffffu, w, 0);
        } else {
          w = read_item(n, true);
        }
        if (w < 0) {
          ok = false;
          break;
        }
        if (w >= n_items) break;
        if (!item_at(w, it) || it.n_tiles == 0) continue;
        if (is_k) {
          int good = 1;
          if (lane == 0) {
            // Q_A, Q_B are reloaded once the previous item's last S MMA is done
            if (items > 0 && !mbar_wait(q_empty, (items - 1) & 1, abort_flag)) {
              good = 0;
              fail();
            } else {
              mbar_arrive_expect_tx(q_full, 2 * kTileBytes);
              for (int x = 0; x < 2; ++x) {
                tma_load_3d(sQ + x * kTileBytes, &tm_q, 0, it.qh_a + x * head_step,
                            it.q_begin + it.r0 + x * row_step, q_full);
                tma_load_3d(sQ + x * kTileBytes + kRegion, &tm_q, 64, it.qh_a + x * head_step,
                            it.q_begin + it.r0 + x * row_step,
                            q_full);
              }
            }
          }
          if (!__shfl_sync(0xffffffffu, good, 0)) {
            ok = false;
            break;
          }
        }
        const int32_t *bt = p.block_tables + static_cast<size_t>(it.seq) * p.max_blocks_per_seq;
        if constexpr (kGather) {
          // Gather: the tile's 128 key rows (256 bytes each, one KV head) in
          // 16-byte pieces, a half-warp per row, into the 128-byte-swizzled
          // layout the TMA boxes produce; keys past k_len (or with a bad block
          // id) are zero-filled. cp.async writes through the generic proxy, so
          // a tile's full barrier is raised once its copies have landed and a
          // proxy fence has ordered them before the tensor core's reads. The
          // warp waits for that before it moves on: the ring's depth, not this
          // warp, keeps copies ahead of the MMAs (raising a tile only after the
          // next one was issued made each PV wait for the one before it).
          const uint8_t *cache = is_k ? p.k_cache : p.v_cache;
          const int half = lane >> 4, c = lane & 15;  // piece c: dims 8c .. 8c+7
          for (int j = 0; ok && j < it.n_tiles; ++j) {
            const int s = issued % stages;
            const int round = issued / stages;
            int good = 1;
            if (lane == 0 && round > 0 && !mbar_wait(is_k ? k_empty(s) : v_empty(s), (round - 1) & 1,
                                                     abort_flag)) {
              good = 0;
              fail();
            }
            if (!__shfl_sync(0xffffffffu, good, 0)) {
              ok = false;
              break;
            }
            const uint32_t dst = is_k ? sK(s) : sV(s);
#pragma unroll 1
            for (int u = 0; u < kTile / 32; ++u) {
              // cache row of key 32u + lane of the tile, -1 for none
              int my_row = -1;
              const int key_l = j * kTile + 32 * u + lane;
              if (key_l < it.k_len) {
                const int blk = __ldg(bt + key_l / p.block_size);
                if (blk >= 0 && blk < p.num_blocks) my_row = blk * p.block_size + key_l % p.block_size;
                else if (is_k) raise_error(p.err, PKV_DEVERR_BLOCK_ID);
              }
#pragma unroll
              for (int i = 0; i < 16; ++i) {  // keys 32u + 2i (lanes 0-15) and 32u + 2i + 1 (16-31)
                const int kk = 2 * i + half;
                const int row = __shfl_sync(0xffffffffu, my_row, kk);
                const int key = 32 * u + kk;
                const size_t src_row = static_cast<size_t>(row < 0 ? 0 : row) * p.num_kv_heads + it.kvh;
                cp_async16(dst + (c >> 3) * kRegion + key * 128 + ((((c & 7) ^ (key & 7))) << 4),
                           cache + src_row * (kHD * 2) + c * 16, row < 0 ? 0 : 16);
              }
            }
            cp_async_commit();
            cp_async_wait<0>();
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(is_k ? k_full(s) : v_full(s));
            ++issued;
          }
        } else {
          for (int j = 0; ok && j < it.n_tiles; ++j) {
            const int s = issued % stages;
            const int round = issued / stages;
            int row = oob_row;
            if (lane < pieces) {
              const int key = j * kTile + lane * R;
              if (key < it.k_len) {
                const int blk = __ldg(bt + key / p.block_size);
                if (blk >= 0 && blk < p.num_blocks) row = blk * p.block_size + key % p.block_size;
                else if (is_k) raise_error(p.err, PKV_DEVERR_BLOCK_ID);
              }
            }
            const uint32_t full = is_k ? k_full(s) : v_full(s);
            const uint32_t empty = is_k ? k_empty(s) : v_empty(s);
            const uint32_t dst = is_k ? sK(s) : sV(s);
            const CUtensorMap *map = is_k ? &tm_k : &tm_v;
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
              tma_load_3d(dst + lane * R * 128, map, 0, it.kvh, row, full);
              tma_load_3d(dst + kRegion + lane * R * 128, map, 64, it.kvh, row, full);
            }
            ++issued;
          }
        }
        ++items;
      }
      if (lane == 0) {  // drain: the last copies must land before the CTA exits
        if (is_k && items > 0) mbar_wait(q_full, (items - 1) & 1, nullptr);
        if constexpr (!kGather)  // (gathered rows have landed at each item's end)
          for (int j = max(0, issued - stages); j < issued; ++j)
            mbar_wait(is_k ? k_full(j % stages) : v_full(j % stages), (j / stages) & 1, nullptr);
      }
    } else if (warp == kWarpMma) {
      // ------------------------------------------------------------ MMA issuer
      if (lane == 0) {
        constexpr uint32_t idesc_s = umma_idesc_bf16(kTile, kTile, false);
        constexpr uint32_t idesc_pv = umma_idesc_bf16(kTile, kHD, true);  // B (V) MN-major
        bool ok = true;
        int s_commits[2] = {0, 0}, pv_commits[2] = {0, 0};
        int kbase = 0, vbase = 0, items = 0;
        auto issue_s = [&](int x, int kt, bool last_s) {
          const int s = kt % kKStages;
          // descriptors of step 0; later steps only move the start address
          const uint64_t dq = desc_kmajor(sQ + x * kTileBytes, 0), dk = desc_kmajor(sK(s), 0);
#pragma unroll
          for (int kk = 0; kk < kHD / 16; ++kk)
            umma_bf16(tmem_s(x), desc_at(dq, kmajor_step(kk)), desc_at(dk, kmajor_step(kk)), idesc_s,
                      kk > 0 ? 1u : 0u);
          umma_commit(s_full(x));
          ++s_commits[x];
          if (x == 1) {
            umma_commit(k_empty(s));             // K has fed both heads
            if (last_s) umma_commit(q_empty);    // the item's Q_A, Q_B are no longer read
          }
        };
        auto issue_pv = [&](int x, int j, int vt) -> bool {
          const int s = vt % kVStages;
          if (!mbar_wait(p_full(x), pv_commits[x] & 1, abort_flag)) return false;
          // the first PV of an item overwrites O_X: the previous item's epilogue
          // must have read it out
          if (j == 0 && items > 0 && !mbar_wait(o_free(x), (items - 1) & 1, abort_flag)) return false;
          tc_fence_after();
          const uint64_t dv = desc_v_mnmajor(sV(s), 0);
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk)
            umma_bf16_tmem_a(tmem_o(x), tmem_s(x) + kk * 8, desc_at(dv, kk * (2048 >> 4)), idesc_pv,
                             (j > 0 || kk > 0) ? 1u : 0u);
          umma_commit(pv_done(x));
          ++pv_commits[x];
          if (x == 1) umma_commit(v_empty(s));   // V has fed both heads
          return true;
        };
        Item it;
        for (int n = 0; ok; ++n) {
          const int w = read_item(n, false);
          if (w < 0) {
            ok = false;
            break;
          }
          if (w >= n_items) break;
          if (!item_at(w, it) || it.n_tiles == 0) continue;
          const int nt = it.n_tiles;
          // S_A(0), S_B(0), then per tile: PV_A(j), S_A(j+1), PV_B(j), S_B(j+1)
          ok = mbar_wait(q_full, items & 1, abort_flag) &&
               mbar_wait(k_full(kbase % kKStages), (kbase / kKStages) & 1, abort_flag);
          if (!ok) break;
          tc_fence_after();
          issue_s(0, kbase, false);
          issue_s(1, kbase, nt == 1);
          for (int j = 0; ok && j < nt; ++j) {
            const int vt = vbase + j, kt1 = kbase + j + 1;
            if (!mbar_wait(v_full(vt % kVStages), (vt / kVStages) & 1, abort_flag)) { ok = false; break; }
            const bool more = j + 1 < nt;
            for (int x = 0; ok && x < 2; ++x) {
              if (!issue_pv(x, j, vt)) { ok = false; break; }
              if (more) {
                if (x == 0 && !mbar_wait(k_full(kt1 % kKStages), (kt1 / kKStages) & 1, abort_flag)) {
                  ok = false;
                  break;
                }
                tc_fence_after();
                issue_s(x, kt1, j + 2 == nt);
              }
            }
          }
          kbase += nt;
          vbase += nt;
          ++items;
        }
        if (!ok) fail();
        for (int x = 0; x < 2; ++x) {  // every issued MMA completes before TMEM is freed
          if (s_commits[x] > 0) mbar_wait(s_full(x), (s_commits[x] - 1) & 1, nullptr);
          if (pv_commits[x] > 0) mbar_wait(pv_done(x), (pv_commits[x] - 1) & 1, nullptr);
        }
      }
      __syncwarp();
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" :: "n"(kRegsHigh));
    // ------------------------------------------------------- softmax A / B
    const int x = warp >> 2;                         // 0: head A, 1: head B
    const int quad = warp & 3;                       // TMEM lanes 32*quad .. 32*quad+31
    const int r = quad * 32 + lane;                  // query row inside the tile
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const float c = p.scale_log2;
    bool ok = true;
    int tiles_done = 0;                              // S_X tiles consumed over all items
    Item it;
    for (int n = 0; ok; ++n) {
      const int w = read_item(n, true);
      if (w < 0) {
        ok = false;
        break;
      }
      if (w >= n_items) break;
      if (!item_at(w, it)) continue;
      const int r0x = it.r0 + x * row_step;            // first row of this warpgroup's tile
      const int qpos = it.prefix + r0x + r;
      const int visible = p.causal ? min(qpos + 1, it.k_len) : it.k_len;
      float m_used = -INFINITY, l_sum = 0.f;         // running max of raw scores, row sum

      for (int j = 0; ok && j < it.n_tiles; ++j) {
        if (!warp_wait(s_full(x), (tiles_done + j) & 1, abort_flag)) { ok = false; break; }
        tc_fence_after();
        float s[kTile];
#pragma unroll
        for (int cc = 0; cc < 4; ++cc)
          tmem_ld32(tmem_s(x) + lane_off + cc * 32, *reinterpret_cast<float(*)[32]>(s + cc * 32));
        tmem_wait_ld();

        const int key0 = j * kTile;
        if (key0 + kTile > visible) {
#pragma unroll
          for (int e = 0; e < kTile; ++e) s[e] = (key0 + e < visible) ? s[e] : -INFINITY;
        }
        const float mt = max128(s);
        // lazy rescale: only when the maximum grows by more than 2^8 after scaling
        const bool grow = mt != -INFINITY && (m_used == -INFINITY || (mt - m_used) * c > kRescaleThreshold);
        float alpha = 1.f;
        if (grow) {
          if (m_used != -INFINITY) {
            alpha = ex2((m_used - mt) * c);
            l_sum *= alpha;
          }
          m_used = mt;
        }
        // O_X holds PV_X(0..j-1), complete because S_X(j) completed after it; the
        // TMEM loads and stores are warp-collective, so the whole warp takes part
        if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
          for (int cc = 0; cc < 4; ++cc) {
            float o[32];
            tmem_ld32(tmem_o(x) + lane_off + cc * 32, o);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] *= alpha;
            tmem_st32(tmem_o(x) + lane_off + cc * 32, o);
          }
          tmem_wait_st();
        }
        // P = exp2(s*c - m*c) as bf16 pairs over TMEM columns 0..63 of S_X; the
        // scaling and the row sum run two lanes per instruction (FFMA2 / FADD2).
        const float mc = m_used * c;
        float2 rs2[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) rs2[i] = make_float2(0.f, 0.f);
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t pk[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const float2 xx = ffma2(make_float2(s[half * 64 + 2 * e], s[half * 64 + 2 * e + 1]),
                                    make_float2(c, c), make_float2(-mc, -mc));
            const float2 pp = make_float2(ex2(xx.x), ex2(xx.y));
            rs2[e & 3] = fadd2(rs2[e & 3], pp);
            pk[e] = float2_to_bf16x2(pp.x, pp.y);
          }
          tmem_st32_u(tmem_s(x) + lane_off + half * 32, pk);
        }
        const float2 rs01 = fadd2(rs2[0], rs2[1]), rs23 = fadd2(rs2[2], rs2[3]);
        l_sum += (rs01.x + rs01.y) + (rs23.x + rs23.y);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(p_full(x));
      }
      if (!ok) break;
      // epilogue: O / l -> bf16 rows, then O_X is handed back for the next item
      const bool have = it.n_tiles > 0;
      if (have) {
        ok = warp_wait(pv_done(x), (tiles_done + it.n_tiles - 1) & 1, abort_flag);
        tc_fence_after();
      }
      const bool store = (r0x + r) < it.q_len;
      __nv_bfloat16 *orow = p.out + (static_cast<size_t>(it.q_begin) + r0x + r) * p.num_q_heads * kHD +
                            static_cast<size_t>(it.qh_a + x * head_step) * kHD;
      const float inv = (l_sum > 0.f) ? 1.f / l_sum : 0.f;
#pragma unroll 1
      for (int cc = 0; cc < 4; ++cc) {
        float o[32];
        if (have && ok) {
          tmem_ld32(tmem_o(x) + lane_off + cc * 32, o);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = 0.f;
        }
        if (store) {
          uint4 *dst = reinterpret_cast<uint4 *>(orow + cc * 32);
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
      if (have) {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(o_free(x));
      }
      tiles_done += it.n_tiles;
    }
    if (!ok) fail();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  // launched as a programmatic dependent that overlaps the previous kernel:
  // finish only after it has, so that the next dependent sees both done (a
  // no-op for an ordinary launch)
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

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

bool prefill_pp_supported(int num_q_heads, int num_kv_heads, int block_size) {
  return num_kv_heads >= 1 && num_q_heads % num_kv_heads == 0 && block_size >= 1;
}

cudaError_t launch_prefill_pp(const PrefillArgs &a, cudaStream_t stream) {
  static std::once_flag attr_once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(attr_once, [] {
    for (auto kern : {prefill_pp_kernel<false>, prefill_pp_kernel<true>}) {
      if (attr_err == cudaSuccess)
        attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
      // setmaxnreg.inc waits until the registers it asks for are free; the split
      // only adds up if the kernel was built with exactly kRegsLaunch per thread,
      // so refuse to launch any other build rather than risk a wait that never ends.
      cudaFuncAttributes fa;
      if (attr_err == cudaSuccess) attr_err = cudaFuncGetAttributes(&fa, kern);
      if (attr_err == cudaSuccess && fa.numRegs != kRegsLaunch) attr_err = cudaErrorInvalidConfiguration;
    }
  });
  if (attr_err != cudaSuccess) return attr_err;
  auto kern = (a.block_size % 8 != 0) ? prefill_pp_kernel<true> : prefill_pp_kernel<false>;
  int box_rows = a.block_size & -a.block_size;
  if (box_rows > kTile) box_rows = kTile;
  CUtensorMap tq, tk, tv;
  const uint64_t cache_rows = static_cast<uint64_t>(a.num_blocks) * a.block_size;
  if (!make_map(&tq, a.q, a.total_q, a.num_q_heads, kTile) ||
      !make_map(&tk, a.k_cache, cache_rows, a.num_kv_heads, box_rows) ||
      !make_map(&tv, a.v_cache, cache_rows, a.num_kv_heads, box_rows))
    return cudaErrorInvalidValue;
  PPParams p;
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
  p.k_cache = static_cast<const uint8_t *>(a.k_cache);
  p.v_cache = static_cast<const uint8_t *>(a.v_cache);
  p.num_kv_heads = a.num_kv_heads;
  p.scale_log2 = a.scale * kLog2e;
  p.err = a.err;
  p.q_tiles = (a.max_seqlen_q + kTile - 1) / kTile;
  p.pair_tiles = (p.group % 2 != 0) ? 1 : 0;
  p.ticket = static_cast<uint32_t *>(a.workspace);
  if (p.ticket == nullptr) return cudaErrorInvalidValue;
  if (!a.ticket_zeroed)
    if (cudaError_t me = cudaMemsetAsync(p.ticket, 0, sizeof(uint32_t), stream)) return me;
  const long long n_items =
      p.pair_tiles ? static_cast<long long>((p.q_tiles + 1) / 2) * a.num_q_heads * a.num_seqs
                   : static_cast<long long>(p.q_tiles) * (a.num_q_heads / 2) * a.num_seqs;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const int sms = sm_count(dev);
  if (sms <= 0) return cudaErrorInvalidValue;
  long long ctas = n_items < sms ? n_items : sms;
  if (a.max_ctas > 0 && a.max_ctas < ctas) ctas = a.max_ctas;
  const dim3 grid(static_cast<unsigned>(ctas));
  if (!a.overlap_previous) {
    kern<<<grid, kThreads, kSmemBytes, stream>>>(tq, tk, tv, p);
    return cudaGetLastError();
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, tq, tk, tv, p);
}

}  // namespace pkv
