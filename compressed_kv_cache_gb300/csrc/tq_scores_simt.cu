// CUDA-core fp32 scorers (TQ_PATH_FP32).
//
// score[b,s] = sum_d A[b,d] c[idx[s,d]] + (sqrt(pi/2)/D) gamma[s] sum_d T[b,d] sigma[s,d]
// ("TurboQuant Attention in CUDA", riteshyadav.xyz, "Two kernels, two jobs":
// the scoring loop and its epilogue; zededa.com v6 for the packed unpack rule).
//
// Work decomposition (both kernels): one thread owns one cached key and a tile
// of QB queries of one problem, so every key byte is read from HBM once per
// query tile and decoded once for QB queries.  A and T of the tile sit in shared
// memory as [D][QB] (query-minor, so the QB values of one coordinate are one
// vector broadcast); the codebook sits in shared memory (unpacked) or in
// registers (packed, at most 8 centroids).  Each score has exactly one owner
// thread and one summation order (d ascending), so results are deterministic.
#include <atomic>

#include "tq_internal.cuh"

namespace tq {
namespace {

constexpr int kThreads = 128;

// QB consecutive floats starting at a 16-byte (QB % 4 == 0) / 8-byte aligned
// shared-memory address, loaded as vectors.
template <int QB>
__device__ __forceinline__ void load_row(const float* src, float (&dst)[QB]) {
  if constexpr (QB % 4 == 0) {
#pragma unroll
    for (int i = 0; i < QB; i += 4) {
      const float4 v = *reinterpret_cast<const float4*>(src + i);
      dst[i] = v.x; dst[i + 1] = v.y; dst[i + 2] = v.z; dst[i + 3] = v.w;
    }
  } else if constexpr (QB == 2) {
    const float2 v = *reinterpret_cast<const float2*>(src);
    dst[0] = v.x; dst[1] = v.y;
  } else {
    dst[0] = src[0];
  }
}

// Stage A and T of queries b0 .. b0+QB-1 of problem p as [D][QB]; rows past B are zero.
template <int QB>
__device__ __forceinline__ void stage_queries(const float* __restrict__ A,
                                              const float* __restrict__ T, float* sA, float* sT,
                                              int p, int b0, int B, int D) {
  for (int e = threadIdx.x; e < QB * D; e += blockDim.x) {
    const int q = e / D, d = e % D;
    float a = 0.f, t = 0.f;
    if (b0 + q < B) {
      const size_t o = (static_cast<size_t>(p) * B + b0 + q) * D + d;
      a = A[o];
      t = T[o];
    }
    sA[d * QB + q] = a;
    sT[d * QB + q] = t;
  }
}

// +1 / -1 as the sign bit to XOR into T: 0 when sigma = +1, 0x80000000 when -1.
__device__ __forceinline__ uint32_t flip_from_int8_byte(uint32_t byte) {
  return (byte & 0x80u) << 24;
}

template <int QB>
__device__ __forceinline__ void accumulate(const float* sA, const float* sT, int d, float c,
                                           uint32_t flip, float (&m)[QB], float (&r)[QB]) {
  float a[QB], t[QB];
  load_row<QB>(sA + d * QB, a);
  load_row<QB>(sT + d * QB, t);
#pragma unroll
  for (int q = 0; q < QB; ++q) {
    m[q] = fmaf(a[q], c, m[q]);
    r[q] += __int_as_float(__float_as_int(t[q]) ^ flip);
  }
}

template <int QB>
__device__ __forceinline__ void store_scores(float* __restrict__ scores, const float (&m)[QB],
                                             const float (&r)[QB], float kg, int p, int b0,
                                             int B, int S, int s) {
#pragma unroll
  for (int q = 0; q < QB; ++q) {
    if (b0 + q < B) scores[(static_cast<size_t>(p) * B + b0 + q) * S + s] = fmaf(kg, r[q], m[q]);
  }
}

// ---------------------------------------------------------------------------
// Unpacked cache: uint8 codes and int8 signs, one byte per coordinate.
// VEC16: D % 16 == 0, rows read as 16-byte vectors; otherwise byte by byte.
// ---------------------------------------------------------------------------
template <int QB, bool VEC16>
__global__ void __launch_bounds__(kThreads)
scores_unpacked_kernel(const float* __restrict__ A, const float* __restrict__ T,
                       const uint8_t* __restrict__ K_idx, const int8_t* __restrict__ signs,
                       const float* __restrict__ gamma, const float* __restrict__ codebook,
                       float* __restrict__ scores, int B, int S, int D, int C, float kappa) {
  extern __shared__ __align__(16) float smem[];
  float* sA = smem;
  float* sT = sA + QB * D;
  float* sC = sT + QB * D;
  const int p = blockIdx.z;
  const int b0 = blockIdx.y * QB;
  stage_queries<QB>(A, T, sA, sT, p, b0, B, D);
  for (int e = threadIdx.x; e < C; e += blockDim.x) sC[e] = codebook[e];
  __syncthreads();

  const int s = blockIdx.x * kThreads + threadIdx.x;
  if (s >= S) return;
  const size_t key = static_cast<size_t>(p) * S + s;
  const uint8_t* ki = K_idx + key * D;
  const uint8_t* ks = reinterpret_cast<const uint8_t*>(signs) + key * D;

  float m[QB], r[QB];
#pragma unroll
  for (int q = 0; q < QB; ++q) { m[q] = 0.f; r[q] = 0.f; }

  if constexpr (VEC16) {
    for (int d0 = 0; d0 < D; d0 += 16) {
      const uint4 vi = __ldg(reinterpret_cast<const uint4*>(ki + d0));
      const uint4 vs = __ldg(reinterpret_cast<const uint4*>(ks + d0));
      const uint32_t wi[4] = {vi.x, vi.y, vi.z, vi.w};
      const uint32_t wsg[4] = {vs.x, vs.y, vs.z, vs.w};
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const uint32_t code = (wi[u >> 2] >> (8 * (u & 3))) & 0xFFu;
        const uint32_t flip = flip_from_int8_byte(wsg[u >> 2] >> (8 * (u & 3)));
        accumulate<QB>(sA, sT, d0 + u, sC[code], flip, m, r);
      }
    }
  } else {
    for (int d = 0; d < D; ++d) {
      const uint32_t flip = flip_from_int8_byte(__ldg(ks + d));
      accumulate<QB>(sA, sT, d, sC[__ldg(ki + d)], flip, m, r);
    }
  }
  store_scores<QB>(scores, m, r, kappa * gamma[key], p, b0, B, S, s);
}

// ---------------------------------------------------------------------------
// Bit-packed cache: BITS-bit codes in a little-endian stream, one sign bit per
// coordinate, fp16 gamma.  D % 32 == 0: each 32-coordinate chunk is BITS words
// of codes and one word of signs, so every field position is a compile-time
// constant inside the unrolled chunk (3-bit fields that straddle a word are
// read with a funnel shift).
// ---------------------------------------------------------------------------
template <int BITS>
__device__ __forceinline__ float pick_centroid(const float (&c)[1 << BITS], uint32_t code) {
  if constexpr (BITS == 1) {
    return (code & 1u) ? c[1] : c[0];
  } else if constexpr (BITS == 2) {
    const float lo = (code & 1u) ? c[1] : c[0];
    const float hi = (code & 1u) ? c[3] : c[2];
    return (code & 2u) ? hi : lo;
  } else {
    const float c01 = (code & 1u) ? c[1] : c[0];
    const float c23 = (code & 1u) ? c[3] : c[2];
    const float c45 = (code & 1u) ? c[5] : c[4];
    const float c67 = (code & 1u) ? c[7] : c[6];
    const float lo = (code & 2u) ? c23 : c01;
    const float hi = (code & 2u) ? c67 : c45;
    return (code & 4u) ? hi : lo;
  }
}

template <int BITS, int QB>
__global__ void __launch_bounds__(kThreads)
scores_packed_kernel(const float* __restrict__ A, const float* __restrict__ T,
                     const uint8_t* __restrict__ idx_plane, const uint8_t* __restrict__ sign_plane,
                     const uint16_t* __restrict__ gamma_f16, const float* __restrict__ codebook,
                     float* __restrict__ scores, int B, int S, int D, float kappa) {
  constexpr int kC = 1 << BITS;
  extern __shared__ __align__(16) float smem[];
  float* sA = smem;
  float* sT = sA + QB * D;
  const int p = blockIdx.z;
  const int b0 = blockIdx.y * QB;
  stage_queries<QB>(A, T, sA, sT, p, b0, B, D);
  float cb[kC];
#pragma unroll
  for (int k = 0; k < kC; ++k) cb[k] = __ldg(codebook + k);
  __syncthreads();

  const int s = blockIdx.x * kThreads + threadIdx.x;
  if (s >= S) return;
  const size_t key = static_cast<size_t>(p) * S + s;
  const int chunks = D >> 5;
  const uint32_t* wi = reinterpret_cast<const uint32_t*>(idx_plane) + key * (chunks * BITS);
  const uint32_t* wsg = reinterpret_cast<const uint32_t*>(sign_plane) + key * chunks;

  float m[QB], r[QB];
#pragma unroll
  for (int q = 0; q < QB; ++q) { m[q] = 0.f; r[q] = 0.f; }

  for (int ch = 0; ch < chunks; ++ch) {
    uint32_t w[BITS + 1];
#pragma unroll
    for (int i = 0; i < BITS; ++i) w[i] = __ldg(wi + ch * BITS + i);
    w[BITS] = 0u;
    const uint32_t sw = __ldg(wsg + ch);
#pragma unroll
    for (int u = 0; u < 32; ++u) {
      constexpr int kMask = kC - 1;
      const int pos = BITS * u;
      const int wd = pos >> 5, sh = pos & 31;
      uint32_t code;
      if (sh + BITS <= 32) {
        code = (w[wd] >> sh) & kMask;
      } else {
        code = __funnelshift_r(w[wd], w[wd + 1], sh) & kMask;
      }
      const uint32_t flip = (~sw << (31 - u)) & 0x80000000u;
      accumulate<QB>(sA, sT, ch * 32 + u, pick_centroid<BITS>(cb, code), flip, m, r);
    }
  }
  const float g = __half2float(__ushort_as_half(__ldg(gamma_f16 + key)));
  store_scores<QB>(scores, m, r, kappa * g, p, b0, B, S, s);
}


// ---------------------------------------------------------------------------
// Bit-packed cache, D = 128, few queries: per-byte-group lookup tables.
//
// Each query's A and T turn into small tables of partial sums in shared memory
// (the byte-level table of zededa.com's "Dead End: Byte-Level Lookup Table",
// moved from global to shared memory and cut to 4/6-bit keys so that a warp's
// 32 lookups into one table never conflict on a bank):
//   code table  (position g, value v) = sum_{i<G} A[g*G+i] * c[(v >> BITS*i) & (C-1)]
//   sign table  (position g, value v) = sum_{i<4} T[4g+i] * (bit i of v ? +1 : -1)
// with G = 2 codes per lookup for 2- and 3-bit codes and 4 for 1-bit codes.  A
// key then costs 64 (1-bit: 32) code lookups and 32 sign lookups per query.
// ---------------------------------------------------------------------------
template <int BITS>
struct LutShape {
  static constexpr int G = BITS == 1 ? 4 : 2;            // codes per lookup
  static constexpr int KB = G * BITS;                    // key bits per lookup
  static constexpr int NV = 1 << KB;                     // entries per code table
  static constexpr int NPI = 128 / G;                    // code tables per query
  static constexpr int NPS = 32;                         // sign tables per query (4 signs each)
  static constexpr int PER_Q = NPI * NV + NPS * 16;      // floats per query
};

template <int BITS, int QB>
__global__ void __launch_bounds__(256)
scores_packed_lut_kernel(const float* __restrict__ A, const float* __restrict__ T,
                         const uint8_t* __restrict__ idx_plane,
                         const uint8_t* __restrict__ sign_plane,
                         const uint16_t* __restrict__ gamma_f16,
                         const float* __restrict__ codebook, float* __restrict__ scores, int B,
                         int S, float kappa) {
  using L = LutShape<BITS>;
  constexpr int D = 128;
  constexpr int kC = 1 << BITS;
  extern __shared__ __align__(16) float smem[];
  float* lut = smem;                      // [QB][NPI*NV + NPS*16]
  float* sAT = lut + QB * L::PER_Q;       // [QB][2][D] staging of A and T
  const int p = blockIdx.z;
  const int b0 = blockIdx.y * QB;
  const int stride = gridDim.x * blockDim.x;

  // Rows of the first key are requested before the tables are built, and every
  // iteration requests the next key's rows before it reduces the current key.
  uint4 nxt_i[BITS], nxt_s;
  uint16_t nxt_g = 0;
  auto fetch = [&](int s) {
    if (s < S) {
      const size_t key = static_cast<size_t>(p) * S + s;
      const uint4* ip = reinterpret_cast<const uint4*>(idx_plane + key * (16 * BITS));
#pragma unroll
      for (int i = 0; i < BITS; ++i) nxt_i[i] = __ldg(ip + i);
      nxt_s = __ldg(reinterpret_cast<const uint4*>(sign_plane + key * 16));
      nxt_g = __ldg(gamma_f16 + key);
    }
  };
  fetch(blockIdx.x * blockDim.x + threadIdx.x);
  for (int e = threadIdx.x; e < QB * 2 * D; e += blockDim.x) {
    const int q = e / (2 * D), k = e % (2 * D);
    float v = 0.f;
    if (b0 + q < B) {
      const size_t o = (static_cast<size_t>(p) * B + b0 + q) * D + (k % D);
      v = k < D ? A[o] : T[o];
    }
    sAT[e] = v;
  }
  float cb[kC];
#pragma unroll
  for (int k = 0; k < kC; ++k) cb[k] = __ldg(codebook + k);
  __syncthreads();
  for (int e = threadIdx.x; e < QB * L::PER_Q; e += blockDim.x) {
    const int q = e / L::PER_Q, r = e % L::PER_Q;
    const float* a = sAT + q * 2 * D;
    float v = 0.f;
    if (r < L::NPI * L::NV) {
      const int g = r / L::NV, val = r % L::NV;
#pragma unroll
      for (int i = 0; i < L::G; ++i) {
        const int code = (val >> (BITS * i)) & (kC - 1);
        float c = cb[0];
#pragma unroll
        for (int k = 1; k < kC; ++k) c = code == k ? cb[k] : c;
        v = fmaf(a[g * L::G + i], c, v);
      }
    } else {
      const int rr = r - L::NPI * L::NV;
      const int g = rr / 16, val = rr % 16;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float t = a[D + 4 * g + i];
        v += ((val >> i) & 1) ? t : -t;
      }
    }
    lut[e] = v;
  }
  __syncthreads();

  for (int s = blockIdx.x * blockDim.x + threadIdx.x; s < S; s += stride) {
    uint32_t w[4 * BITS + 1];
#pragma unroll
    for (int i = 0; i < BITS; ++i) {
      w[4 * i] = nxt_i[i].x; w[4 * i + 1] = nxt_i[i].y; w[4 * i + 2] = nxt_i[i].z; w[4 * i + 3] = nxt_i[i].w;
    }
    w[4 * BITS] = 0u;
    const uint32_t ws[4] = {nxt_s.x, nxt_s.y, nxt_s.z, nxt_s.w};
    const float g = __half2float(__ushort_as_half(nxt_g));
    fetch(s + stride);

    float m[QB], r[QB];
#pragma unroll
    for (int q = 0; q < QB; ++q) { m[q] = 0.f; r[q] = 0.f; }
#pragma unroll
    for (int gi = 0; gi < L::NPI; ++gi) {
      const int off = L::KB * gi;
      const int wd = off >> 5, sh = off & 31;
      uint32_t v;
      if (sh + L::KB <= 32) {
        v = (w[wd] >> sh) & (L::NV - 1);
      } else {
        v = __funnelshift_r(w[wd], w[wd + 1], sh) & (L::NV - 1);
      }
#pragma unroll
      for (int q = 0; q < QB; ++q) m[q] += lut[q * L::PER_Q + gi * L::NV + v];
    }
#pragma unroll
    for (int gi = 0; gi < L::NPS; ++gi) {
      const uint32_t v = (ws[gi >> 3] >> (4 * (gi & 7))) & 15u;
#pragma unroll
      for (int q = 0; q < QB; ++q) r[q] += lut[q * L::PER_Q + L::NPI * L::NV + gi * 16 + v];
    }
    store_scores<QB>(scores, m, r, kappa * g, p, b0, B, S, s);
  }
}

template <int BITS, int QB>
cudaError_t launch_lut_qb(const float* A, const float* T, const uint8_t* idx_plane,
                          const uint8_t* sign_plane, const uint16_t* gamma_f16,
                          const float* codebook, float* scores, int P, int B, int S,
                          cudaStream_t st) {
  using L = LutShape<BITS>;
  const size_t smem = (static_cast<size_t>(QB) * L::PER_Q + QB * 2 * 128) * sizeof(float);
  static std::atomic<uint64_t> configured{0};
  int dev = 0, sms = 148;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (smem > 48 * 1024 && !(configured.load(std::memory_order_acquire) & bit)) {
    e = cudaFuncSetAttribute(scores_packed_lut_kernel<BITS, QB>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    configured.fetch_or(bit, std::memory_order_acq_rel);
  }
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int qtiles = ceil_div(B, QB);
  const int tiles = ceil_div(S, 256);
  const int want = ceil_div(8LL * sms, static_cast<int64_t>(P) * qtiles);
  dim3 grid(tiles < want ? tiles : (want < 1 ? 1 : want), qtiles, P);
  scores_packed_lut_kernel<BITS, QB><<<grid, 256, smem, st>>>(
      A, T, idx_plane, sign_plane, gamma_f16, codebook, scores, B, S, qjl_scale(128));
  return cudaGetLastError();
}

template <int BITS>
cudaError_t launch_lut_bits(const float* A, const float* T, const uint8_t* idx_plane,
                            const uint8_t* sign_plane, const uint16_t* gamma_f16,
                            const float* codebook, float* scores, int P, int B, int S,
                            cudaStream_t st) {
  if (B <= 1) return launch_lut_qb<BITS, 1>(A, T, idx_plane, sign_plane, gamma_f16, codebook, scores, P, B, S, st);
  if (B <= 2) return launch_lut_qb<BITS, 2>(A, T, idx_plane, sign_plane, gamma_f16, codebook, scores, P, B, S, st);
  if (B <= 4 || BITS == 3) return launch_lut_qb<BITS, 4>(A, T, idx_plane, sign_plane, gamma_f16, codebook, scores, P, B, S, st);
  return launch_lut_qb<BITS, 8>(A, T, idx_plane, sign_plane, gamma_f16, codebook, scores, P, B, S, st);
}

template <int QB>
cudaError_t launch_unpacked_qb(const float* A, const float* T, const uint8_t* K_idx,
                               const int8_t* signs, const float* gamma, const float* codebook,
                               float* scores, int P, int B, int S, int D, int C, cudaStream_t st) {
  dim3 grid(ceil_div(S, kThreads), ceil_div(B, QB), P);
  const size_t sm = (2 * QB * D + C) * sizeof(float);
  const float kappa = qjl_scale(D);
  if (D % 16 == 0) {
    scores_unpacked_kernel<QB, true><<<grid, kThreads, sm, st>>>(A, T, K_idx, signs, gamma,
                                                                 codebook, scores, B, S, D, C,
                                                                 kappa);
  } else {
    scores_unpacked_kernel<QB, false><<<grid, kThreads, sm, st>>>(A, T, K_idx, signs, gamma,
                                                                  codebook, scores, B, S, D, C,
                                                                  kappa);
  }
  return cudaGetLastError();
}

template <int BITS, int QB>
cudaError_t launch_packed_qb(const float* A, const float* T, const uint8_t* idx_plane,
                             const uint8_t* sign_plane, const uint16_t* gamma_f16,
                             const float* codebook, float* scores, int P, int B, int S, int D,
                             cudaStream_t st) {
  dim3 grid(ceil_div(S, kThreads), ceil_div(B, QB), P);
  const size_t sm = 2 * QB * D * sizeof(float);
  scores_packed_kernel<BITS, QB><<<grid, kThreads, sm, st>>>(
      A, T, idx_plane, sign_plane, gamma_f16, codebook, scores, B, S, D, qjl_scale(D));
  return cudaGetLastError();
}

template <int BITS>
cudaError_t launch_packed_bits(const float* A, const float* T, const uint8_t* idx_plane,
                               const uint8_t* sign_plane, const uint16_t* gamma_f16,
                               const float* codebook, float* scores, int P, int B, int S, int D,
                               cudaStream_t st) {
  if (B <= 1) return launch_packed_qb<BITS, 1>(A, T, idx_plane, sign_plane, gamma_f16, codebook, scores, P, B, S, D, st);
  if (B <= 2) return launch_packed_qb<BITS, 2>(A, T, idx_plane, sign_plane, gamma_f16, codebook, scores, P, B, S, D, st);
  if (B <= 4) return launch_packed_qb<BITS, 4>(A, T, idx_plane, sign_plane, gamma_f16, codebook, scores, P, B, S, D, st);
  return launch_packed_qb<BITS, 8>(A, T, idx_plane, sign_plane, gamma_f16, codebook, scores, P, B, S, D, st);
}

}  // namespace

cudaError_t launch_scores_unpacked_fp32(const float* A, const float* T, const uint8_t* K_idx,
                                        const int8_t* signs, const float* gamma,
                                        const float* codebook, float* scores, int P, int B,
                                        int S, int D, int C, cudaStream_t st) {
  if (B <= 1) return launch_unpacked_qb<1>(A, T, K_idx, signs, gamma, codebook, scores, P, B, S, D, C, st);
  if (B <= 2) return launch_unpacked_qb<2>(A, T, K_idx, signs, gamma, codebook, scores, P, B, S, D, C, st);
  if (B <= 4) return launch_unpacked_qb<4>(A, T, K_idx, signs, gamma, codebook, scores, P, B, S, D, C, st);
  if (B <= 8) return launch_unpacked_qb<8>(A, T, K_idx, signs, gamma, codebook, scores, P, B, S, D, C, st);
  return launch_unpacked_qb<16>(A, T, K_idx, signs, gamma, codebook, scores, P, B, S, D, C, st);
}

cudaError_t launch_scores_packed_fp32(const float* A, const float* T, const uint8_t* idx_plane,
                                      const uint8_t* sign_plane, const uint16_t* gamma_f16,
                                      const float* codebook, float* scores, int P, int B, int S,
                                      int D, int idx_bits, cudaStream_t st) {
  if (D == 128) {
    switch (idx_bits) {
      case 1: return launch_lut_bits<1>(A, T, idx_plane, sign_plane, gamma_f16, codebook, scores, P, B, S, st);
      case 2: return launch_lut_bits<2>(A, T, idx_plane, sign_plane, gamma_f16, codebook, scores, P, B, S, st);
      default: return launch_lut_bits<3>(A, T, idx_plane, sign_plane, gamma_f16, codebook, scores, P, B, S, st);
    }
  }
  switch (idx_bits) {
    case 1: return launch_packed_bits<1>(A, T, idx_plane, sign_plane, gamma_f16, codebook, scores, P, B, S, D, st);
    case 2: return launch_packed_bits<2>(A, T, idx_plane, sign_plane, gamma_f16, codebook, scores, P, B, S, D, st);
    default: return launch_packed_bits<3>(A, T, idx_plane, sign_plane, gamma_f16, codebook, scores, P, B, S, D, st);
  }
}

}  // namespace tq
