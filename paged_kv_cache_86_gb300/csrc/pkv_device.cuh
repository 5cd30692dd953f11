// pkv_device.cuh -- small device helpers shared by the libpkv kernels:
// bf16 unpacking, packed fp32x2 FMA, mbarrier and bulk-copy (TMA) wrappers
// written as inline PTX for sm_103a, bounded waits and the device error word.
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

#include "pkv.h"

namespace pkv {

// ------------------------------------------------------------ error word --

// Waits that can only stall on a bug give up after this many nanoseconds of
// %globaltimer (or this many polls), record PKV_DEVERR_TIMEOUT and return.
constexpr unsigned long long kWaitTimeoutNs = 2000000000ull;  // 2 s
constexpr uint32_t kWaitMaxPolls = 1u << 28;

__device__ __forceinline__ void raise_error(uint32_t *err, uint32_t bits) {
  if (err != nullptr) atomicOr(err, bits);
}

__device__ __forceinline__ unsigned long long global_timer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// --------------------------------------------------------------- numbers --

// A 32-bit word holding two bf16 values: the low half is the element at the
// lower address. bf16 -> fp32 is exact: the bf16 bits are the high half.
__device__ __forceinline__ float2 bf16x2_to_float2(uint32_t w) {
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

__device__ __forceinline__ uint32_t float2_to_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);  // round to nearest even
  return *reinterpret_cast<uint32_t *>(&h);
}

// d = a * b + c on two fp32 lanes at once (one FFMA2 on sm_100+).
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  unsigned long long ra, rb, rc, rd;
  ra = *reinterpret_cast<unsigned long long *>(&a);
  rb = *reinterpret_cast<unsigned long long *>(&b);
  rc = *reinterpret_cast<unsigned long long *>(&c);
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(rd) : "l"(ra), "l"(rb), "l"(rc));
  return *reinterpret_cast<float2 *>(&rd);
}

__device__ __forceinline__ float2 fmul2(float2 a, float2 b) {
  unsigned long long ra, rb, rd;
  ra = *reinterpret_cast<unsigned long long *>(&a);
  rb = *reinterpret_cast<unsigned long long *>(&b);
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(rd) : "l"(ra), "l"(rb));
  return *reinterpret_cast<float2 *>(&rd);
}

__device__ __forceinline__ float2 fadd2(float2 a, float2 b) {
  unsigned long long ra, rb, rd;
  ra = *reinterpret_cast<unsigned long long *>(&a);
  rb = *reinterpret_cast<unsigned long long *>(&b);
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(rd) : "l"(ra), "l"(rb));
  return *reinterpret_cast<float2 *>(&rd);
}

// max(a, b, c) in one instruction (three-operand max.f32, sm_100+); like
// fmaxf, a NaN operand is ignored.
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Maximum of 128 values as eight independent chains of three-operand maxima
// (68 instructions, dependency depth 10) instead of one serial chain of 127.
__device__ __forceinline__ float max128(const float (&v)[128]) {
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = fmaxf(v[i], v[i + 8]);
#pragma unroll
  for (int e = 16; e < 128; e += 16) {
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = fmax3(acc[i], v[e + i], v[e + 8 + i]);
  }
  return fmax3(fmax3(acc[0], acc[1], acc[2]), fmax3(acc[3], acc[4], acc[5]), fmaxf(acc[6], acc[7]));
}

// ------------------------------------------------------------ shared mem --

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}

// -------------------------------------------------------------- mbarrier --

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(bar), "r"(count) : "memory");
}

// Make barrier initialisation visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
               :: "r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
  return ok != 0;
}

// Non-blocking probe: has the phase with the given parity completed?
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
  return ok != 0;
}

// Wait until the phase with the given parity has completed. Gives up (returns
// false) when *abort becomes non-zero or after limit_ns; never spins forever.
__device__ __forceinline__ bool mbar_wait_for(uint32_t bar, uint32_t parity, const volatile int *abort,
                                              unsigned long long limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_timer_ns();
  for (uint32_t polls = 1; polls < kWaitMaxPolls; ++polls) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((polls & 63u) == 0) {
      if (abort != nullptr && *abort) return false;
      if (global_timer_ns() - t0 > limit_ns) return false;
    }
  }
  return false;
}

__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity,
                                          const volatile int *abort) {
  return mbar_wait_for(bar, parity, abort, kWaitTimeoutNs);
}

// ------------------------------------------------------- fp8 E4M3 rows --

// fp8 E4M3 store: each (token, KV head) row of 128 values is quantized with
// its own fp32 scale, amax / 448, and codes E4M3(x * (448 / amax)) rounded to
// nearest even with saturation (cvt.rn.satfinite); a zero row gives zero codes
// and scale 0 (LLM Infra 101 v0.2, KV Quantization: the cache stores low-bit
// values instead of bf16). One warp per row; lane l holds dims 4l..4l+3.
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

// ------------------------------------------------------ named barriers --

// Hardware barrier `id` over `nthreads` threads (whole warps) that also ORs
// `v` over them; every participating warp must reach it the same number of
// times. Orders the participants' shared-memory accesses like __syncthreads.
__device__ __forceinline__ bool bar_red_or(int id, int nthreads, bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 q, %1, 0;\n\t"
      "barrier.cta.red.or.pred p, %2, %3, q;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(r) : "r"(static_cast<uint32_t>(v)), "r"(id), "r"(nthreads) : "memory");
  return r != 0;
}

// Hardware barrier that returns how many participating threads passed true.
__device__ __forceinline__ int bar_red_popc(int id, int nthreads, bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred q;\n\t"
      "setp.ne.u32 q, %1, 0;\n\t"
      "barrier.cta.red.popc.u32 %0, %2, %3, q;\n\t}"
      : "=r"(r) : "r"(static_cast<uint32_t>(v)), "r"(id), "r"(nthreads) : "memory");
  return static_cast<int>(r);
}

__device__ __forceinline__ void bar_sync(int id, int nthreads) {
  asm volatile("barrier.cta.sync.aligned %0, %1;" :: "r"(id), "r"(nthreads) : "memory");
}

// ------------------------------------------------------------ bulk copy --

__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// One non-tensor TMA copy of `bytes` (multiple of 16, both addresses 16-byte
// aligned) from global to this CTA's shared memory, completing on `bar`.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes,
                                         uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1], %2, [%3], %4;"
      :: "r"(dst), "l"(src), "r"(bytes), "r"(bar), "l"(policy) : "memory");
}

// cp.async: 16 bytes global -> shared, asynchronously (src_bytes 0 zero-fills
// them); the copies of a thread are grouped by commit and waited for by group.
// They write through the generic proxy: a fence.proxy.async is needed before
// the tensor core reads what they wrote.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" :: "r"(dst), "l"(src), "r"(src_bytes)
               : "memory");
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }

template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" :: "n"(N) : "memory"); }

// Named barrier over a subset of the CTA's warps.
__device__ __forceinline__ void named_barrier(uint32_t id, uint32_t threads) {
  asm volatile("bar.sync %0, %1;" :: "r"(id), "r"(threads) : "memory");
}

}  // namespace pkv
