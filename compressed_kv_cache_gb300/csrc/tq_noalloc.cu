// tq_solve_packed_noalloc: the fused query transform + packed scoring call for
// callers that must not allocate device memory.
//
// Who needs it: a plugin inside an inference engine is usually handed only its
// input and output buffers, while the engine owns every device allocation; a
// service that reserves all of its device memory at start-up treats any later
// cudaMalloc as a failure, because an allocation can fail under memory pressure
// or synchronise the device in the middle of serving.  Such callers cannot
// provide the A/T workspace that tq_solve_packed takes.
//
// Instead the two transformed-query arrays live in one file-scope device array of
// fixed size, kNoAllocBytes (1 MiB).  Every GPU that loads libtq holds this array
// until the process exits.  Host code never dereferences the array's name (on the
// host it is only a stand-in for the symbol): the device address is looked up with
// cudaGetSymbolAddress once per device, on the first call made while that device is
// current, and cached.  Nothing in the array has to start at zero: the query
// transform writes every element of A and T before the scorer reads it, so the
// contents a previous call left behind are never used.  All calls on a device share
// the one array, so calls whose work can overlap on the GPU (different streams,
// different host threads) race on it and must be serialised by the caller.
#include <mutex>

#include "tq_internal.cuh"

namespace {

constexpr size_t kNoAllocBytes = size_t(1) << 20;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char tq_noalloc_scratch[kNoAllocBytes];

std::mutex g_scratch_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up once per device).
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (g_scratch_addr[dev] == nullptr) {
    void* addr = nullptr;
    e = cudaGetSymbolAddress(&addr, tq_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = addr;
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" {

tq_status tq_solve_packed_noalloc(const void* Q, tq_qtype qtype, const uint8_t* idx_plane,
                                  const uint8_t* sign_plane, const uint16_t* gamma_f16,
                                  const float* Pi, const float* S_mat, const float* codebook,
                                  float* scores, int P, int H, int B, int S, int D, int idx_bits,
                                  tq_path path, cudaStream_t stream) {
  if (P < 1 || B < 1 || D < 1) return TQ_ERR_INVALID_VALUE;
  const size_t need = tq_workspace_bytes(P, B, D);
  if (need == 0) return TQ_ERR_INVALID_VALUE;
  if (need > kNoAllocBytes) return TQ_ERR_WORKSPACE;   // P*B*D too large for the fixed scratch
  void* scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess) return TQ_ERR_LAUNCH;
  return tq_solve_packed(Q, qtype, idx_plane, sign_plane, gamma_f16, Pi, S_mat, codebook, scores,
                         P, H, B, S, D, idx_bits, scratch, kNoAllocBytes, path, stream);
}

}  // extern "C"
