// The failure path of the library's bounded waits, run on purpose and without a fault:
// one warp waits on an mbarrier that nothing arrives on.  wait_parity_bounded gives up
// after the library's budget (kWaitBudgetNs of the GPU's global timer), sets this
// unit's fault bit and the kernel returns, so the context stays usable.
#include "tq_internal.cuh"

namespace tq {
namespace {

constexpr unsigned int kFaultCheck = 16u;   // the bit tq_device_faults reports for it

__global__ void wait_expiry_kernel() {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(&bar));
  if (threadIdx.x == 0) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(a) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncwarp();
  wait_parity_bounded(a, 0, kFaultCheck);
}

}  // namespace

cudaError_t launch_wait_expiry(cudaStream_t st) {
  wait_expiry_kernel<<<1, 32, 0, st>>>();
  return cudaGetLastError();
}

cudaError_t take_faults_check(unsigned int* bits) { return take_unit_faults(bits); }

}  // namespace tq
