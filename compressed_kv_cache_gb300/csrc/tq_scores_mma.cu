// bf16 tensor-core scorer (TQ_PATH_BF16_MMA).  Not built yet: the path reports
// itself unavailable and TQ_PATH_AUTO resolves to the fp32 path.
#include "tq_internal.cuh"

namespace tq {

bool mma_path_available() { return false; }

cudaError_t launch_scores_mma(const float*, const float*, const uint8_t*, const void*,
                              const void*, const float*, float*, int, int, int, int, int, bool,
                              cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace tq
