// prefill.cu -- paged varlen chunked-prefill attention (tcgen05 path: pending).
#include <cuda_runtime.h>

#include "pkv_internal.h"

namespace pkv {

bool prefill_supported(int, int, int) { return false; }

cudaError_t launch_paged_prefill(const PrefillArgs &, cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace pkv
