// selftest.cu -- an on-GPU check of the failure path that every kernel here
// relies on: a bounded mbarrier wait that runs out reports instead of hanging,
// and two warps that meet once per step on an OR-reducing hardware barrier
// leave their loop in the same step when one of them gives up (the protocol of
// the decode kernel's softmax warps). The wait runs out on a barrier that
// nothing arrives on; no fault, trap or endless loop is involved.
#include <cuda_runtime.h>

#include "pkv.h"
#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr int kSteps = 8;
constexpr unsigned long long kShortLimitNs = 5000000ull;  // 5 ms

// res[0], res[1]: the step in which warp 0 / warp 1 left the loop;
// res[2]: 1 if warp 1's wait reported the timeout; res[3]: steps both completed.
__global__ void __launch_bounds__(64) selftest_wait_kernel(int fail_step, int32_t *res, uint32_t *err) {
  __shared__ __align__(8) uint64_t never;  // no thread ever arrives on it
  __shared__ int stop;
  __shared__ int done;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t bar = smem_addr(&never);
  if (threadIdx.x == 0) {
    mbar_init(bar, 1);
    fence_barrier_init();
    stop = 0;
    done = 0;
  }
  __syncthreads();
  int step = 0;
  for (; step < kSteps; ++step) {
    bool ok = true;
    if (warp == 1 && step == fail_step) {
      ok = __all_sync(0xffffffffu, mbar_wait_for(bar, 0, nullptr, kShortLimitNs));
      if (!ok && lane == 0) {
        stop = 1;
        res[2] = 1;
        raise_error(err, PKV_DEVERR_TIMEOUT);
      }
    }
    if (bar_red_or(1, 64, !ok)) {
      if (stop) break;
    }
    if (threadIdx.x == 0) ++done;
  }
  if (lane == 0) res[warp] = step;
  __syncthreads();
  if (threadIdx.x == 0) res[3] = done;
}

}  // namespace
}  // namespace pkv

extern "C" pkv_status pkv_selftest_bounded_wait(int32_t fail_step, int32_t *result, void *stream) {
  if (result == nullptr || fail_step < 0) return PKV_ERR_ARG;
  cudaError_t e;
  uint32_t *err = pkv::device_error_word(&e);
  if (!err) return PKV_ERR_CUDA;
  pkv::selftest_wait_kernel<<<1, 64, 0, static_cast<cudaStream_t>(stream)>>>(fail_step, result, err);
  return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}
