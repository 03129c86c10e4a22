// Lookup-table shape shared by the fp32 packed scorers (D = 128): each query turns
// into tables of partial sums over G consecutive codes, indexed by the G codes'
// bits together (the byte-level table of "Implementing TurboQuant on NVIDIA's AGX
// Thor", zededa.com, "Dead End: Byte-Level Lookup Table", cut to 4- and 6-bit keys
// and moved to shared memory).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace tq {

template <int BITS>
struct LutShape {
  static constexpr int G = BITS == 1 ? 4 : 2;            // codes per lookup
  static constexpr int KB = G * BITS;                    // key bits per lookup
  static constexpr int NV = 1 << KB;                     // entries per code table
  static constexpr int NPI = 128 / G;                    // code tables per query
  static constexpr int NPS = 32;                         // sign tables per query (4 signs each)
  static constexpr int PER_Q = NPI * NV + NPS * 16;      // floats per query (codes and signs)
};

// The codebook (2^BITS centroids) copied into shared memory, one load per centroid
// per CTA: the first 2^BITS threads of the calling group (from `first` on) each copy
// one, and the caller orders the copy before any read with a barrier.  Every thread of
// every CTA reading the codebook from global memory would send all those requests to
// the one L2 slice that holds it.  The load goes through L2 (ld.global.cg): kernels
// launched as programmatic dependents run beside the grid before them, so nothing they
// read after griddepcontrol.wait may go through the read-only path, which assumes the
// data stays unchanged for the kernel's lifetime.
template <int BITS>
__device__ __forceinline__ void stage_codebook(const float* __restrict__ codebook, float* sCb, int first) {
  const int i = static_cast<int>(threadIdx.x) - first;
  if (i >= 0 && i < (1 << BITS)) sCb[i] = __ldcg(codebook + i);
}

// Centroids of the table value this thread keeps fixed while it builds tables
// (value v = thread % NV; code i of v is bits BITS*i .. BITS*i+BITS-1), from the
// shared copy stage_codebook made.
template <int BITS>
__device__ __forceinline__ void table_centroids(const float* sCb, float (&cv)[LutShape<BITS>::G]) {
  using L = LutShape<BITS>;
  const int v = threadIdx.x % L::NV;
#pragma unroll
  for (int k = 0; k < L::G; ++k) cv[k] = sCb[(v >> (BITS * k)) & ((1 << BITS) - 1)];
}

// Two fp32 additions in one instruction (sm_100 packed f32x2): acc.lo += a, acc.hi += b.
__device__ __forceinline__ void add2(unsigned long long& acc, float a, float b) {
  asm("{\n\t.reg .b64 t;\n\tmov.b64 t, {%1, %2};\n\tadd.rn.f32x2 %0, %0, t;\n\t}" : "+l"(acc) : "f"(a), "f"(b));
}
__device__ __forceinline__ float sum2(unsigned long long acc) {
  return __uint_as_float(static_cast<uint32_t>(acc)) + __uint_as_float(static_cast<uint32_t>(acc >> 32));
}

// Eight lookups, one per 4-bit field of w, in the 16-entry tables g0 .. g0+7 (table g
// at tab + 16 g; field f of w is bits 4f .. 4f+3, field 2j the low and 2j+1 the high
// nibble of byte j).  The byte offsets 4 * field come from two masked shifts of w and
// one byte permute per field; each pair of lookups is one packed add per query.
template <int QB, int PER_Q>
__device__ __forceinline__ void lut_nibbles(const float* tab, uint32_t w, int g0,
                                            unsigned long long (&acc)[QB][2]) {
  const uint32_t lo = (w << 2) & 0x3C3C3C3Cu;
  const uint32_t hi = (w >> 2) & 0x3C3C3C3Cu;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint32_t ol = __byte_perm(lo, 0u, 0x4440u + j);
    const uint32_t oh = __byte_perm(hi, 0u, 0x4440u + j);
#pragma unroll
    for (int q = 0; q < QB; ++q) {
      const char* t = reinterpret_cast<const char*>(tab + q * PER_Q + (g0 + 2 * j) * 16);
      add2(acc[q][j & 1], *reinterpret_cast<const float*>(t + ol), *reinterpret_cast<const float*>(t + 64 + oh));
    }
  }
}

}  // namespace tq
