// Internal declarations shared by the libtq translation units (not part of the ABI).
#pragma once

#include <atomic>

#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "tq.h"

namespace tq {

// sqrt(pi/2) rounded to float32: the QJL scale numerator of the TurboQuant_prod
// estimator (kanthi.in §3, TurboQuantProd.dequantize; riteshyadav.xyz epilogue).
constexpr float kSqrtHalfPi = 1.25331413731550025f;

inline float qjl_scale(int D) { return kSqrtHalfPi / static_cast<float>(D); }

// ---- launchers (return the CUDA error of the launch, cudaSuccess otherwise) ----

// Query tile of the tensor-core path: NT = min(B, 128) rounded up to 16, ceil(B/NT) tiles.
// A kernel launched as a programmatic dependent shares SMs with the grid before it only
// when both run under the same L1 / shared-memory split, so every kernel of such a pair
// asks for the largest shared-memory carveout.  Set once per device and kernel.
template <typename Kernel>
inline cudaError_t prefer_max_shared(Kernel kernel, std::atomic<uint64_t>& done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (done.load(std::memory_order_acquire) & bit) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
  if (e != cudaSuccess) return e;
  done.fetch_or(bit, std::memory_order_acq_rel);
  return cudaSuccess;
}

inline int mma_query_tile(int B) { const int n = B < 128 ? B : 128; return (n + 15) / 16 * 16; }
inline int mma_query_tiles(int B) { const int nt = mma_query_tile(B); return (B + nt - 1) / nt; }
// Bytes of the bf16 query operand of the tensor-core path for P problems (D = 128):
// per (problem, query tile) NT rows x 256 K in the no-swizzle core-matrix layout.
inline size_t mma_y_bytes(int P, int B) {
  return static_cast<size_t>(P) * mma_query_tiles(B) * mma_query_tile(B) * 512;
}

// Ybf (optional, D == 128 only): also write A and T as the tensor-core query operand.
// hsigns (optional, [H][D] +-1, D a power of two): A = H diag(s) q by a fast
// Walsh-Hadamard transform instead of the dense rows of Pi (Pi is then unused).
// share_sm: the scorer launched next shares SMs with the transform (the two-CTA tensor-core
// configuration, mma_shares_sm).
cudaError_t launch_prepare(const void* Q, tq_qtype qtype, const float* Pi, const float* S_mat,
                           float* A, float* T, int P, int H, int B, int D, cudaStream_t st,
                           uint16_t* Ybf = nullptr, const float* hsigns = nullptr,
                           bool share_sm = false);

cudaError_t launch_scores_unpacked_fp32(const float* A, const float* T, const uint8_t* K_idx,
                                        const int8_t* signs, const float* gamma,
                                        const float* codebook, float* scores, int P, int B,
                                        int S, int D, int C, cudaStream_t st);

// after_prepare: launched right behind this call's query transform on the same
// stream (programmatic dependent launch; A and T are read after that grid completes).
cudaError_t launch_scores_packed_fp32(const float* A, const float* T, const uint8_t* idx_plane,
                                      const uint8_t* sign_plane, const uint16_t* gamma_f16,
                                      const float* codebook, float* scores, int P, int B, int S,
                                      int D, int idx_bits, bool after_prepare, cudaStream_t st);

// Fused query transform + packed fp32 scoring (one kernel): D == 128, B <= 8 and
// fewer problems than half the SMs of the current device.
bool fused_packed_supported(int P, int B, int D);
cudaError_t launch_solve_packed_fused(const void* Q, tq_qtype qtype, const float* Pi,
                                      const float* S_mat, int H, const uint8_t* idx_plane,
                                      const uint8_t* sign_plane, const uint16_t* gamma_f16,
                                      const float* codebook, float* scores, int P, int B, int S,
                                      int idx_bits, cudaStream_t st);

// bf16 tensor-core path (D == 128). `packed` selects the cache layout; for the
// unpacked layout idx_bits is ignored and C is the codebook size.  `after_prepare`:
// the launch directly follows this call's query transform on the same stream and may
// start early (programmatic dependent launch); A and T are read only after the
// transform grid has completed.  Ybf: the query operand prepared by that transform
// (one bulk copy per CTA instead of converting A and T).
bool mma_path_available();
// Whether the tensor-core scorer runs in its two-CTA-per-SM configuration for this shape
// (and so can share SMs with the query transform launched before it).
bool mma_shares_sm(int P, int B, int S);

cudaError_t launch_scores_mma(const float* A, const float* T, const uint8_t* idx,
                              const void* signs, const void* gamma, const float* codebook,
                              float* scores, int P, int B, int S, int C, int idx_bits,
                              bool packed, bool after_prepare, cudaStream_t st,
                              const uint16_t* Ybf = nullptr);

// MSE-only scores from A = Pi q, packed codes and fp16 norms (D % 32 == 0, 1-4 bits).
cudaError_t launch_scores_mse(const float* A, const uint8_t* idx_plane, const uint16_t* norm_f16,
                              const float* codebook, float* scores, int P, int B, int S, int D,
                              int idx_bits, bool norm_correction, cudaStream_t st);

// Fused decode over MSE keys and values (D = 128, 1-3 bit codes): split-KV partials in
// `part` (decode_part_floats(P, B, S) floats), then the combine and Pi_v^T.
size_t decode_part_floats(int P, int B, int S);
cudaError_t launch_decode_mse(const float* A, const uint8_t* k_plane, const uint16_t* k_norm,
                              const float* k_cb, int k_bits, const uint8_t* v_plane,
                              const uint16_t* v_norm, const float* v_cb, int v_bits,
                              const float* Pi_v, float* out, float* part, int P, int H, int B, int S,
                              float scale, cudaStream_t st);
// The same over a TurboQuant_prod key cache: code plane, sign plane and fp16 gamma.
cudaError_t launch_decode_prod(const float* A, const float* T, const uint8_t* k_plane,
                               const uint8_t* k_sign, const uint16_t* k_gamma, const float* k_cb,
                               int k_bits, const uint8_t* v_plane, const uint16_t* v_norm,
                               const float* v_cb, int v_bits, const float* Pi_v, float* out,
                               float* part, int P, int H, int B, int S, float scale, cudaStream_t st);

cudaError_t launch_pack_indices(const uint8_t* K_idx, uint8_t* plane, int64_t n, int D, int bits,
                                cudaStream_t st);
cudaError_t launch_unpack_indices(const uint8_t* plane, uint8_t* K_idx, int64_t n, int D,
                                  int bits, cudaStream_t st);
cudaError_t launch_pack_signs(const int8_t* signs, uint8_t* plane, int64_t n, int D,
                              cudaStream_t st);
cudaError_t launch_unpack_signs(const uint8_t* plane, int8_t* signs, int64_t n, int D,
                                cudaStream_t st);

inline int ceil_div(int64_t a, int64_t b) { return static_cast<int>((a + b - 1) / b); }

// ---- bounded waits ----------------------------------------------------------
// Every spin on an mbarrier in this library gives up after kWaitBudgetNs of the GPU's
// global timer, records the failure in its translation unit's fault word and lets the
// kernel finish (its outputs are then NaN); tq_device_faults reads and clears the words.
constexpr uint64_t kWaitBudgetNs = 1000000000ull;   // 1 s

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// L2 prefetch of [p, p + bytes), trimmed to whole 16-byte blocks inside the range.  A
// hint only: what it brings into L2 is read by later loads, so it may be issued before
// griddepcontrol.wait whatever the grid before this one writes.
__device__ __forceinline__ void prefetch_l2(const void* p, size_t bytes) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(p);
  const uintptr_t lo = (a + 15) & ~static_cast<uintptr_t>(15);
  const uintptr_t hi = (a + bytes) & ~static_cast<uintptr_t>(15);
  if (hi > lo)
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(lo), "r"(static_cast<uint32_t>(hi - lo))
                 : "memory");
}

// Fault bits, one per kernel family.
enum : unsigned int { kFaultLut = 1u, kFaultMma = 2u, kFaultDecode = 4u, kFaultCompress = 8u };

// Reads and clears the fault word of each translation unit that has bounded waits
// (synchronous: a cudaMemcpyFromSymbol per unit); ORs the bits into *bits.
cudaError_t take_faults_simt(unsigned int* bits);
cudaError_t take_faults_mma(unsigned int* bits);
cudaError_t take_faults_decode(unsigned int* bits);
cudaError_t take_faults_compress(unsigned int* bits);

namespace {
// This translation unit's fault word (internal linkage: one per unit).
__device__ unsigned int g_wait_fault = 0;

__device__ __forceinline__ bool mbar_poll(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile("{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
               : "=r"(ok)
               : "r"(bar), "r"(parity)
               : "memory");
  return ok != 0;
}

// Wait for the given phase parity of a local mbarrier for at most kWaitBudgetNs; on
// running out, set `fault` in this unit's fault word and return false.
__device__ __forceinline__ bool wait_parity_bounded(uint32_t bar, uint32_t parity, unsigned int fault) {
  if (mbar_poll(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (;;) {
    for (int i = 0; i < 64; ++i)
      if (mbar_poll(bar, parity)) return true;
    if (global_ns() - t0 > kWaitBudgetNs) {
      atomicOr(&g_wait_fault, fault);
      return false;
    }
  }
}

// Host side of this unit's fault word.
inline cudaError_t take_unit_faults(unsigned int* bits) {
  unsigned int v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_wait_fault, sizeof v);
  if (e != cudaSuccess) return e;
  if (v != 0) {
    const unsigned int z = 0;
    e = cudaMemcpyToSymbol(g_wait_fault, &z, sizeof z);
  }
  *bits |= v;
  return e;
}
}  // namespace

}  // namespace tq
