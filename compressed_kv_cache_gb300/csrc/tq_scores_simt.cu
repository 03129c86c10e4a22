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

  // Table build.  Thread t keeps one table value v fixed (so its centroids, or its
  // signs, are fixed) and walks the table positions; A and T are read through L1.
  static_assert(256 % L::NV == 0, "code tables must tile the CTA");
  {
    const int v = threadIdx.x % L::NV;
    float cv[L::G];
#pragma unroll
    for (int k = 0; k < L::G; ++k) {
      const int code = (v >> (BITS * k)) & (kC - 1);
      cv[k] = __ldg(codebook + code);
    }
    const int vs = threadIdx.x & 15;
    for (int q = 0; q < QB; ++q) {
      const bool live = b0 + q < B;
      const size_t row = (static_cast<size_t>(p) * B + (live ? b0 + q : b0)) * D;
      float* tq = lut + q * L::PER_Q;
      for (int g = threadIdx.x / L::NV; g < L::NPI; g += 256 / L::NV) {
        float acc = 0.f;
#pragma unroll
        for (int k = 0; k < L::G; ++k) acc = fmaf(__ldg(A + row + g * L::G + k), cv[k], acc);
        tq[g * L::NV + v] = live ? acc : 0.f;
      }
      for (int g = threadIdx.x >> 4; g < L::NPS; g += 16) {
        float acc = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float t = __ldg(T + row + 4 * g + i);
          acc += ((vs >> i) & 1) ? t : -t;
        }
        tq[L::NPI * L::NV + g * 16 + vs] = live ? acc : 0.f;
      }
    }
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
  const size_t smem = static_cast<size_t>(QB) * L::PER_Q * sizeof(float);
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


// ---------------------------------------------------------------------------
// Fused query transform + packed scoring for few queries (D = 128): one
// persistent CTA per SM stages Pi and S_mat of its problem's head in shared
// memory (rows padded to 129 floats, so "thread d reads row d" is free of bank
// conflicts), computes A = Pi q and T = S_mat q for its query tile there
// ("TurboQuant Attention in CUDA", "Two kernels, two jobs": the first kernel,
// here inside the second), builds the same lookup tables as
// scores_packed_lut_kernel and scores its share of the keys.  The first keys'
// rows are in flight during the whole prologue.  One kernel per call, nothing
// written to a workspace.
// ---------------------------------------------------------------------------
template <int BITS, int QB>
constexpr size_t fused_smem_bytes() {
  return 2 * 128 * 128 * sizeof(float) + 16 + (QB * 128 + QB * 256 + QB * LutShape<BITS>::PER_Q) * sizeof(float);
}
template <int QB>
__host__ __device__ constexpr int fused_threads() { return QB <= 2 ? 512 : 256; }

__device__ __forceinline__ float load_query(const float* q, size_t i) { return q[i]; }
__device__ __forceinline__ float load_query(const __nv_bfloat16* q, size_t i) {
  return __bfloat162float(q[i]);
}

template <int BITS, int QB, typename QT>
__global__ void __launch_bounds__(fused_threads<QB>(), 1)
solve_packed_lut_kernel(const QT* __restrict__ Q, const float* __restrict__ Pi,
                        const float* __restrict__ Sm, int H, const uint8_t* __restrict__ idx_plane,
                        const uint8_t* __restrict__ sign_plane,
                        const uint16_t* __restrict__ gamma_f16,
                        const float* __restrict__ codebook, float* __restrict__ scores, int B,
                        int S, float kappa) {
  using L = LutShape<BITS>;
  constexpr int D = 128;
  constexpr int kC = 1 << BITS;
  constexpr int kT = fused_threads<QB>();
  extern __shared__ __align__(16) float smem[];
  float* sM = smem;                                       // [2][128][128]: Pi, then S_mat
  uint64_t* bar = reinterpret_cast<uint64_t*>(sM + 2 * 128 * 128);
  float* sQ = reinterpret_cast<float*>(bar + 2);          // [QB][128]
  float* sAT = sQ + QB * 128;                             // [QB][256]: A then T
  float* lut = sAT + QB * 256;                            // [QB][PER_Q]
  const int p = blockIdx.z;
  const int h = p % H;
  const int b0 = blockIdx.y * QB;
  const int stride = gridDim.x * kT;
  const int tid = threadIdx.x;

  // Pi and S_mat of head h arrive by two bulk copies on one mbarrier.  The barrier is
  // initialised and made visible to every thread before anyone issues or polls it.
  const uint32_t bar_a = static_cast<uint32_t>(__cvta_generic_to_shared(bar));
  if (tid == 0) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bar_a) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (tid == 0) {
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(bar_a),
                 "r"(2u * D * D * 4u)
                 : "memory");
    const uint32_t dst = static_cast<uint32_t>(__cvta_generic_to_shared(sM));
    const float* src0 = Pi + static_cast<size_t>(h) * D * D;
    const float* src1 = Sm + static_cast<size_t>(h) * D * D;
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(src0), "r"(D * D * 4u), "r"(bar_a)
                 : "memory");
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst + D * D * 4u),
                 "l"(src1), "r"(D * D * 4u), "r"(bar_a)
                 : "memory");
  }

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
  fetch(blockIdx.x * kT + tid);

  for (int e = tid; e < QB * D; e += kT) {
    const int q = e / D;
    sQ[e] = b0 + q < B ? load_query(Q, (static_cast<size_t>(p) * B + b0) * D + e) : 0.f;
  }
  // bounded wait for the two copies (about a second at most)
  bool landed = false;
  for (uint32_t it = 0; it < (1u << 22) && !landed; ++it) {
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], 0;\n\tselp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok) : "r"(bar_a) : "memory");
    landed = ok != 0;
  }
  __syncthreads();
  // thread t < 256: output coordinate d = t % 128 of A (t < 128) or of T; row d is walked in
  // the column order j = (jj + d) mod 128, so the 32 lanes of a warp read 32 banks
  if (tid < 256) {
    const int d = tid & 127;
    const float* row = sM + (tid >> 7) * D * D + d * D;
    float acc[QB];
#pragma unroll
    for (int q = 0; q < QB; ++q) acc[q] = 0.f;
#pragma unroll 8
    for (int jj = 0; jj < D; ++jj) {
      const int j = (jj + d) & (D - 1);
      const float m = row[j];
#pragma unroll
      for (int q = 0; q < QB; ++q) acc[q] = fmaf(m, sQ[q * D + j], acc[q]);
    }
#pragma unroll
    for (int q = 0; q < QB; ++q) sAT[q * 256 + tid] = landed ? acc[q] : __int_as_float(0x7fc00000);
  }
  __syncthreads();
  // lookup tables from A and T (thread keeps one table value fixed)
  {
    const int v = tid % L::NV;
    float cv[L::G];
#pragma unroll
    for (int k = 0; k < L::G; ++k) cv[k] = __ldg(codebook + ((v >> (BITS * k)) & (kC - 1)));
    const int vs = tid & 15;
    for (int q = 0; q < QB; ++q) {
      const float* a = sAT + q * 256;
      float* tq = lut + q * L::PER_Q;
      for (int g = tid / L::NV; g < L::NPI; g += kT / L::NV) {
        float acc = 0.f;
#pragma unroll
        for (int k = 0; k < L::G; ++k) acc = fmaf(a[g * L::G + k], cv[k], acc);
        tq[g * L::NV + v] = acc;
      }
      for (int g = tid >> 4; g < L::NPS; g += kT / 16) {
        float acc = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float t = a[D + 4 * g + i];
          acc += ((vs >> i) & 1) ? t : -t;
        }
        tq[L::NPI * L::NV + g * 16 + vs] = acc;
      }
    }
  }
  __syncthreads();

  for (int s = blockIdx.x * kT + tid; s < S; s += stride) {
    uint32_t w[4 * BITS + 1];
#pragma unroll
    for (int i = 0; i < BITS; ++i) {
      w[4 * i] = nxt_i[i].x; w[4 * i + 1] = nxt_i[i].y; w[4 * i + 2] = nxt_i[i].z; w[4 * i + 3] = nxt_i[i].w;
    }
    w[4 * BITS] = 0u;
    const uint32_t ws[4] = {nxt_s.x, nxt_s.y, nxt_s.z, nxt_s.w};
    const float g = __half2float(__ushort_as_half(nxt_g));
    fetch(s + stride);
    // two partial sums per query and part, for two independent add chains
    float m[2][QB], r[2][QB];
#pragma unroll
    for (int q = 0; q < QB; ++q) { m[0][q] = m[1][q] = 0.f; r[0][q] = r[1][q] = 0.f; }
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
      for (int q = 0; q < QB; ++q) m[gi & 1][q] += lut[q * L::PER_Q + gi * L::NV + v];
    }
#pragma unroll
    for (int gi = 0; gi < L::NPS; ++gi) {
      const uint32_t v = (ws[gi >> 3] >> (4 * (gi & 7))) & 15u;
#pragma unroll
      for (int q = 0; q < QB; ++q) r[gi & 1][q] += lut[q * L::PER_Q + L::NPI * L::NV + gi * 16 + v];
    }
    float mm[QB], rr[QB];
#pragma unroll
    for (int q = 0; q < QB; ++q) { mm[q] = m[0][q] + m[1][q]; rr[q] = r[0][q] + r[1][q]; }
    store_scores<QB>(scores, mm, rr, kappa * g, p, b0, B, S, s);
  }
}

template <int BITS, int QB, typename QT>
cudaError_t launch_fused_qb(const QT* Q, const float* Pi, const float* S_mat, int H,
                            const uint8_t* idx_plane, const uint8_t* sign_plane,
                            const uint16_t* gamma_f16, const float* codebook, float* scores,
                            int P, int B, int S, cudaStream_t st) {
  constexpr size_t smem = fused_smem_bytes<BITS, QB>();
  static std::atomic<uint64_t> configured{0};
  int dev = 0, sms = 148;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (!(configured.load(std::memory_order_acquire) & bit)) {
    e = cudaFuncSetAttribute(solve_packed_lut_kernel<BITS, QB, QT>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    configured.fetch_or(bit, std::memory_order_acq_rel);
  }
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int qtiles = ceil_div(B, QB);
  const int tiles = ceil_div(S, fused_threads<QB>());
  const int want = ceil_div(static_cast<int64_t>(sms), static_cast<int64_t>(P) * qtiles);
  dim3 grid(tiles < want ? tiles : (want < 1 ? 1 : want), qtiles, P);
  solve_packed_lut_kernel<BITS, QB, QT><<<grid, fused_threads<QB>(), smem, st>>>(
      Q, Pi, S_mat, H, idx_plane, sign_plane, gamma_f16, codebook, scores, B, S, qjl_scale(128));
  return cudaGetLastError();
}

template <int BITS, typename QT>
cudaError_t launch_fused_bits(const QT* Q, const float* Pi, const float* S_mat, int H,
                              const uint8_t* idx_plane, const uint8_t* sign_plane,
                              const uint16_t* gamma_f16, const float* codebook, float* scores,
                              int P, int B, int S, cudaStream_t st) {
  if (B <= 1) return launch_fused_qb<BITS, 1>(Q, Pi, S_mat, H, idx_plane, sign_plane, gamma_f16, codebook, scores, P, B, S, st);
  if (B <= 2) return launch_fused_qb<BITS, 2>(Q, Pi, S_mat, H, idx_plane, sign_plane, gamma_f16, codebook, scores, P, B, S, st);
  if (B <= 4 || BITS == 3) return launch_fused_qb<BITS, 4>(Q, Pi, S_mat, H, idx_plane, sign_plane, gamma_f16, codebook, scores, P, B, S, st);
  return launch_fused_qb<BITS, 8>(Q, Pi, S_mat, H, idx_plane, sign_plane, gamma_f16, codebook, scores, P, B, S, st);
}

template <typename QT>
cudaError_t launch_fused_typed(const QT* Q, const float* Pi, const float* S_mat, int H,
                               const uint8_t* idx_plane, const uint8_t* sign_plane,
                               const uint16_t* gamma_f16, const float* codebook, float* scores,
                               int P, int B, int S, int idx_bits, cudaStream_t st) {
  switch (idx_bits) {
    case 1: return launch_fused_bits<1>(Q, Pi, S_mat, H, idx_plane, sign_plane, gamma_f16, codebook, scores, P, B, S, st);
    case 2: return launch_fused_bits<2>(Q, Pi, S_mat, H, idx_plane, sign_plane, gamma_f16, codebook, scores, P, B, S, st);
    default: return launch_fused_bits<3>(Q, Pi, S_mat, H, idx_plane, sign_plane, gamma_f16, codebook, scores, P, B, S, st);
  }
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

namespace tq {

bool fused_packed_supported(int B, int D) { return D == 128 && B >= 1 && B <= 8; }

cudaError_t launch_solve_packed_fused(const void* Q, tq_qtype qtype, const float* Pi,
                                      const float* S_mat, int H, const uint8_t* idx_plane,
                                      const uint8_t* sign_plane, const uint16_t* gamma_f16,
                                      const float* codebook, float* scores, int P, int B, int S,
                                      int idx_bits, cudaStream_t st) {
  if (qtype == TQ_Q_BF16)
    return launch_fused_typed(static_cast<const __nv_bfloat16*>(Q), Pi, S_mat, H, idx_plane,
                              sign_plane, gamma_f16, codebook, scores, P, B, S, idx_bits, st);
  return launch_fused_typed(static_cast<const float*>(Q), Pi, S_mat, H, idx_plane, sign_plane,
                            gamma_f16, codebook, scores, P, B, S, idx_bits, st);
}

}  // namespace tq
