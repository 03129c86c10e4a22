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

// Centroids of the table value this thread keeps fixed while it builds tables
// (value v = thread % NV; code i of v is bits BITS*i .. BITS*i+BITS-1).
template <int BITS>
__device__ __forceinline__ void table_centroids(const float* __restrict__ codebook,
                                                float (&cv)[LutShape<BITS>::G]) {
  using L = LutShape<BITS>;
  const int v = threadIdx.x % L::NV;
#pragma unroll
  for (int k = 0; k < L::G; ++k) cv[k] = __ldg(codebook + ((v >> (BITS * k)) & ((1 << BITS) - 1)));
}

}  // namespace tq
