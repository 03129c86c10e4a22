// Bit packing of the cache format (little-endian bit stream per key):
// bit t of coordinate d is stream bit bits*d + t, stream bit i is bit (i % 8)
// of byte i / 8; the sign plane has bit d set exactly when sigma_d = +1.
// ("TurboQuant: Rotate-then-Quantize KV Caches at 3 Bits", kanthi.in, §8 slot
// sizes and §11 item 4: pack then unpack is the identity.)
//
// One thread per output byte (pack) or per output coordinate (unpack), over a
// grid-stride loop; the row of a key is a few dozen bytes, so the input reads
// of neighbouring threads fall in the same sectors.
#include "tq_internal.cuh"

namespace tq {
namespace {

constexpr int kThreads = 256;

inline int grid_for(int64_t n) {
  const int64_t blocks = (n + kThreads - 1) / kThreads;
  return static_cast<int>(blocks < 65536 ? (blocks > 0 ? blocks : 1) : 65536);
}

__global__ void pack_indices_kernel(const uint8_t* __restrict__ K_idx, uint8_t* __restrict__ plane,
                                    int64_t n_keys, int D, int bits) {
  const int row_bytes = D * bits / 8;
  const int64_t total = n_keys * row_bytes;
  for (int64_t e = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; e < total;
       e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t key = e / row_bytes;
    const int j = static_cast<int>(e % row_bytes);
    const uint8_t* row = K_idx + key * D;
    uint32_t byte = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int pos = 8 * j + i;
      const int d = pos / bits, t = pos % bits;
      byte |= ((static_cast<uint32_t>(row[d]) >> t) & 1u) << i;
    }
    plane[e] = static_cast<uint8_t>(byte);
  }
}

__global__ void unpack_indices_kernel(const uint8_t* __restrict__ plane, uint8_t* __restrict__ K_idx,
                                      int64_t n_keys, int D, int bits) {
  const int row_bytes = D * bits / 8;
  const int64_t total = n_keys * D;
  for (int64_t e = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; e < total;
       e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t key = e / D;
    const int d = static_cast<int>(e % D);
    const uint8_t* row = plane + key * row_bytes;
    uint32_t code = 0;
    for (int t = 0; t < bits; ++t) {
      const int pos = bits * d + t;
      code |= ((static_cast<uint32_t>(row[pos >> 3]) >> (pos & 7)) & 1u) << t;
    }
    K_idx[e] = static_cast<uint8_t>(code);
  }
}

__global__ void pack_signs_kernel(const int8_t* __restrict__ signs, uint8_t* __restrict__ plane,
                                  int64_t n_keys, int D) {
  const int row_bytes = D / 8;
  const int64_t total = n_keys * row_bytes;
  for (int64_t e = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; e < total;
       e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t key = e / row_bytes;
    const int j = static_cast<int>(e % row_bytes);
    const int8_t* row = signs + key * D + 8 * j;
    uint32_t byte = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) byte |= (row[i] > 0 ? 1u : 0u) << i;
    plane[e] = static_cast<uint8_t>(byte);
  }
}

__global__ void unpack_signs_kernel(const uint8_t* __restrict__ plane, int8_t* __restrict__ signs,
                                    int64_t n_keys, int D) {
  const int row_bytes = D / 8;
  const int64_t total = n_keys * D;
  for (int64_t e = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; e < total;
       e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t key = e / D;
    const int d = static_cast<int>(e % D);
    const uint32_t bit = (plane[key * row_bytes + (d >> 3)] >> (d & 7)) & 1u;
    signs[e] = bit ? int8_t(1) : int8_t(-1);
  }
}

}  // namespace

cudaError_t launch_pack_indices(const uint8_t* K_idx, uint8_t* plane, int64_t n, int D, int bits,
                                cudaStream_t st) {
  pack_indices_kernel<<<grid_for(n * D * bits / 8), kThreads, 0, st>>>(K_idx, plane, n, D, bits);
  return cudaGetLastError();
}

cudaError_t launch_unpack_indices(const uint8_t* plane, uint8_t* K_idx, int64_t n, int D,
                                  int bits, cudaStream_t st) {
  unpack_indices_kernel<<<grid_for(n * D), kThreads, 0, st>>>(plane, K_idx, n, D, bits);
  return cudaGetLastError();
}

cudaError_t launch_pack_signs(const int8_t* signs, uint8_t* plane, int64_t n, int D,
                              cudaStream_t st) {
  pack_signs_kernel<<<grid_for(n * D / 8), kThreads, 0, st>>>(signs, plane, n, D);
  return cudaGetLastError();
}

cudaError_t launch_unpack_signs(const uint8_t* plane, int8_t* signs, int64_t n, int D,
                                cudaStream_t st) {
  unpack_signs_kernel<<<grid_for(n * D), kThreads, 0, st>>>(plane, signs, n, D);
  return cudaGetLastError();
}

}  // namespace tq
