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
#include "tq_lut.cuh"

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
// moved from global to shared memory and cut to 4-bit keys, whose 16-entry
// tables take a warp's 32 lookups without a bank conflict; the 6-bit keys of
// 3-bit codes index 64-entry tables, at most two-way conflicts):
//   code table  (position g, value v) = sum_{i<G} A[g*G+i] * c[(v >> BITS*i) & (C-1)]
//   sign table  (position g, value v) = sum_{i<4} T[4g+i] * (bit i of v ? +1 : -1)
// with G = 2 codes per lookup for 2- and 3-bit codes and 4 for 1-bit codes.  A
// key then costs 64 (1-bit: 32) code lookups and 32 sign lookups per query.
// ---------------------------------------------------------------------------

// One key of the packed cache in registers: BITS 16-byte rows of codes, the
// 16-byte row of signs and the fp16 gamma.
template <int BITS>
struct PackedKey {
  uint4 idx[BITS];
  uint4 sg;
  uint16_t g;
};

template <int BITS>
__device__ __forceinline__ void load_packed_key(PackedKey<BITS>& k,
                                                const uint8_t* __restrict__ idx_plane,
                                                const uint8_t* __restrict__ sign_plane,
                                                const uint16_t* __restrict__ gamma_f16,
                                                size_t key) {
  const uint4* ip = reinterpret_cast<const uint4*>(idx_plane + key * (16 * BITS));
#pragma unroll
  for (int i = 0; i < BITS; ++i) k.idx[i] = __ldg(ip + i);
  k.sg = __ldg(reinterpret_cast<const uint4*>(sign_plane + key * 16));
  k.g = __ldg(gamma_f16 + key);
}

// Code and sign sums of one key for QB queries, read from the tables [QB][PER_Q]
// (code tables first, then the 32 sign tables).
template <int BITS, int QB>
__device__ __forceinline__ void lut_key_sums(const float* lut, const PackedKey<BITS>& k,
                                             float (&mm)[QB], float (&rr)[QB]) {
  using L = LutShape<BITS>;
  const uint32_t ws[4] = {k.sg.x, k.sg.y, k.sg.z, k.sg.w};
  unsigned long long r2[QB][2];
#pragma unroll
  for (int q = 0; q < QB; ++q) r2[q][0] = r2[q][1] = 0ull;
#pragma unroll
  for (int i = 0; i < 4; ++i) lut_nibbles<QB, L::PER_Q>(lut + L::NPI * L::NV, ws[i], 8 * i, r2);
  if constexpr (L::KB == 4) {
    // 1- and 2-bit codes: 4-bit fields, as the signs
    unsigned long long m2[QB][2];
#pragma unroll
    for (int q = 0; q < QB; ++q) m2[q][0] = m2[q][1] = 0ull;
#pragma unroll
    for (int i = 0; i < BITS; ++i) {
      lut_nibbles<QB, L::PER_Q>(lut, k.idx[i].x, 32 * i, m2);
      lut_nibbles<QB, L::PER_Q>(lut, k.idx[i].y, 32 * i + 8, m2);
      lut_nibbles<QB, L::PER_Q>(lut, k.idx[i].z, 32 * i + 16, m2);
      lut_nibbles<QB, L::PER_Q>(lut, k.idx[i].w, 32 * i + 24, m2);
    }
#pragma unroll
    for (int q = 0; q < QB; ++q) mm[q] = sum2(m2[q][0]) + sum2(m2[q][1]);
  } else {
    // 3-bit codes: 6-bit fields (pairs of codes), some straddling two words
    uint32_t w[4 * BITS + 1];
#pragma unroll
    for (int i = 0; i < BITS; ++i) {
      w[4 * i] = k.idx[i].x; w[4 * i + 1] = k.idx[i].y; w[4 * i + 2] = k.idx[i].z; w[4 * i + 3] = k.idx[i].w;
    }
    w[4 * BITS] = 0u;
    float m[2][QB];
#pragma unroll
    for (int q = 0; q < QB; ++q) m[0][q] = m[1][q] = 0.f;
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
    for (int q = 0; q < QB; ++q) mm[q] = m[0][q] + m[1][q];
  }
#pragma unroll
  for (int q = 0; q < QB; ++q) rr[q] = sum2(r2[q][0]) + sum2(r2[q][1]);
}

// Tables of QB queries from A (a[0..127]) and T (a[128..255]) of each query,
// a = at(q).  NT threads; thread t keeps one table value fixed and walks positions.
template <int BITS, int QB, int NT, typename At>
__device__ __forceinline__ void build_luts(At at, float* lut, const float (&cv)[LutShape<BITS>::G]) {
  using L = LutShape<BITS>;
  static_assert(NT % L::NV == 0, "code tables must tile the CTA");
  const int v = threadIdx.x % L::NV;
  const int vs = threadIdx.x & 15;
  for (int q = 0; q < QB; ++q) {
    float* tq = lut + q * L::PER_Q;
    for (int g = threadIdx.x / L::NV; g < L::NPI; g += NT / L::NV) {
      float acc = 0.f;
#pragma unroll
      for (int k = 0; k < L::G; ++k) acc = fmaf(at(q, g * L::G + k), cv[k], acc);
      tq[g * L::NV + v] = acc;
    }
    for (int g = threadIdx.x >> 4; g < L::NPS; g += NT / 16) {
      float acc = 0.f;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float t = at(q, 128 + 4 * g + i);
        acc += ((vs >> i) & 1) ? t : -t;
      }
      tq[L::NPI * L::NV + g * 16 + vs] = acc;
    }
  }
}

// Keys first, first + stride, ... below end (end <= S): two keys are always in
// flight ahead of the one being reduced.
template <int BITS, int QB>
__device__ __forceinline__ void lut_score_keys(const float* lut, const uint8_t* __restrict__ idx_plane,
                                               const uint8_t* __restrict__ sign_plane,
                                               const uint16_t* __restrict__ gamma_f16,
                                               float* __restrict__ scores, PackedKey<BITS>& k0,
                                               PackedKey<BITS>& k1, int first, int stride, int end,
                                               int p, int b0, int B, int S, float kappa) {
  const size_t base = static_cast<size_t>(p) * S;
  for (int64_t s = first; s < end; s += stride) {
    const PackedKey<BITS> cur = k0;
    k0 = k1;
    if (s + 2 * static_cast<int64_t>(stride) < end)
      load_packed_key<BITS>(k1, idx_plane, sign_plane, gamma_f16, base + s + 2 * static_cast<int64_t>(stride));
    float mm[QB], rr[QB];
    lut_key_sums<BITS, QB>(lut, cur, mm, rr);
    store_scores<QB>(scores, mm, rr, kappa * __half2float(__ushort_as_half(cur.g)), p, b0, B, S,
                     static_cast<int>(s));
  }
}

template <int BITS>
__device__ __forceinline__ void prefetch_two_keys(PackedKey<BITS>& k0, PackedKey<BITS>& k1,
                                                  const uint8_t* __restrict__ idx_plane,
                                                  const uint8_t* __restrict__ sign_plane,
                                                  const uint16_t* __restrict__ gamma_f16, int p,
                                                  int first, int stride, int end, int S) {
  const size_t base = static_cast<size_t>(p) * S;
  if (first < end) load_packed_key<BITS>(k0, idx_plane, sign_plane, gamma_f16, base + first);
  if (first + static_cast<int64_t>(stride) < end)
    load_packed_key<BITS>(k1, idx_plane, sign_plane, gamma_f16, base + first + stride);
}

// Stream-K scorer over many (problem, query tile) units: the keys of all units, laid
// end to end (unit-major), are cut into one equal contiguous range per CTA, so every
// SM gets the same number of keys however the units divide.  A range crosses unit
// boundaries at most a few times; at each one the CTA rebuilds its tables from that
// unit's A and T (staged in shared memory).  When launched right behind the query transform
// (programmatic dependent launch), the first keys and the codebook are requested
// before griddepcontrol.wait and A and T after it.
template <int BITS, int QB>
__global__ void __launch_bounds__(256, 2)
scores_packed_lut_kernel(const float* __restrict__ A, const float* __restrict__ T,
                         const uint8_t* __restrict__ idx_plane,
                         const uint8_t* __restrict__ sign_plane,
                         const uint16_t* __restrict__ gamma_f16,
                         const float* __restrict__ codebook, float* __restrict__ scores, int B,
                         int S, int qtiles, int64_t total, float kappa) {
  extern __shared__ __align__(16) float smem[];
  float* lut = smem;                      // [QB][NPI*NV + NPS*16]
  float* sAT = lut + QB * LutShape<BITS>::PER_Q;   // [QB][256]: the unit's A, then T
  const int64_t per = (total + gridDim.x - 1) / gridDim.x;
  int64_t w = min(static_cast<int64_t>(blockIdx.x) * per, total);
  const int64_t wend = min(w + per, total);
  __shared__ float sCb[1 << BITS];
  // every kernel before the query transform has completed when this grid starts, and
  // the transform does not write the codebook, so it may be read before the wait; the
  // barriers in the loop order the copy before the first table build
  stage_codebook<BITS>(codebook, sCb, 0);
  bool waited = false;
  while (w < wend) {
    const int u = static_cast<int>(w / S);
    const int sb = static_cast<int>(w - static_cast<int64_t>(u) * S);
    const int se = static_cast<int>(min(static_cast<int64_t>(S), sb + (wend - w)));
    const int p = u / qtiles;
    const int b0 = (u - p * qtiles) * QB;
    const int first = sb + static_cast<int>(threadIdx.x);
    // the segment's first two keys are requested before its tables are built
    PackedKey<BITS> k0, k1;
    prefetch_two_keys<BITS>(k0, k1, idx_plane, sign_plane, gamma_f16, p, first, 256, se, S);
    if (!waited) {
      asm volatile("griddepcontrol.wait;" ::: "memory");
      waited = true;
    }
    // the unit's A and T rows: one load round trip (QB values a thread), staged in
    // shared memory for the table build; queries past B read as zero
    float at[QB];
#pragma unroll
    for (int j = 0; j < QB; ++j) {
      const int e = static_cast<int>(threadIdx.x) + 256 * j, q = e >> 8, x = e & 255;
      const size_t row = (static_cast<size_t>(p) * B + b0 + q) * 128;
      at[j] = b0 + q < B ? (x < 128 ? __ldcg(A + row + x) : __ldcg(T + row + x - 128)) : 0.f;
    }
    __syncthreads();                      // the previous segment's tables are no longer read
#pragma unroll
    for (int j = 0; j < QB; ++j) sAT[threadIdx.x + 256 * j] = at[j];
    __syncthreads();
    float cv[LutShape<BITS>::G];
    table_centroids<BITS>(sCb, cv);
    build_luts<BITS, QB, 256>([&](int q, int e) { return sAT[q * 256 + e]; }, lut, cv);
    __syncthreads();
    lut_score_keys<BITS, QB>(lut, idx_plane, sign_plane, gamma_f16, scores, k0, k1, first, 256, se,
                             p, b0, B, S, kappa);
    w += se - sb;
  }
}

template <int BITS, int QB>
cudaError_t launch_lut_qb(const float* A, const float* T, const uint8_t* idx_plane,
                          const uint8_t* sign_plane, const uint16_t* gamma_f16,
                          const float* codebook, float* scores, int P, int B, int S,
                          bool after_prepare, cudaStream_t st) {
  using L = LutShape<BITS>;
  const size_t smem = static_cast<size_t>(QB) * (L::PER_Q + 256) * sizeof(float);
  auto kernel = scores_packed_lut_kernel<BITS, QB>;
  static std::atomic<int> slots[64];      // co-resident CTAs per device
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  int n = slots[dev & 63].load(std::memory_order_acquire);
  if (n == 0) {
    if (smem > 48 * 1024) {
      e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
      if (e != cudaSuccess) return e;
    }
    int sms = 0, per_sm = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, 256, smem);
    if (e != cudaSuccess) return e;
    n = sms * (per_sm > 0 ? per_sm : 1);
    slots[dev & 63].store(n, std::memory_order_release);
  }
  const int qtiles = ceil_div(B, QB);
  const int64_t total = static_cast<int64_t>(P) * qtiles * S;
  const int64_t want = (total + 255) / 256;             // at least a key per thread
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(want < n ? want : n));
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = after_prepare ? 1 : 0;
  e = cudaLaunchKernelEx(&cfg, kernel, A, T, idx_plane, sign_plane, gamma_f16, codebook, scores, B, S,
                         qtiles, total, qjl_scale(128));
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Bit-packed cache, D = 128, 2-bit codes, 2-4 queries: byte tables, skewed by lane.
//
// Per query tile, tables of partial sums indexed by a whole byte: a code byte (4 codes)
// at each of its 32 positions, and a sign byte (8 signs) at each of its 16 positions.
// An entry holds the QB queries' values side by side (QB floats), entry (e, p) of a
// table set sitting at ((e * NP + p) * QB) floats.  A key then costs 32 + 16 lookups
// of QB floats instead of 64 + 32.  Lane l walks a key's positions starting at l (its
// code row rotated left by l bytes, its sign row by l mod 16, in registers), so the
// lanes of one shared-memory phase (8 for 16-byte entries, 16 for 8-byte entries) read
// distinct positions, that is distinct bank groups, whatever their byte values.
// Tables are built from 16-entry tables of two codes / four signs:
//   byte entry (e, p) = pair/nibble entry (e & 15, 2p) + pair/nibble entry (e >> 4, 2p+1)
// ---------------------------------------------------------------------------
template <int QB>
struct Lut8 {
  static constexpr int kCode = 256 * 32 * QB;            // floats of the code byte tables
  static constexpr int kSign = 256 * 16 * QB;            // floats of the sign byte tables
  static constexpr int kPair = 64 * 16 * QB;             // 2-code tables, [e4][pos 0..63][q]
  static constexpr int kNib = 32 * 16 * QB;              // 4-sign tables, [e4][pos 0..31][q]
  static constexpr int kFloats = kCode + kSign + kPair + kNib + 256 * QB;   // + A/T staging
  static constexpr int kThreads = 512;
};

// rotate the 8 words left by r words (r in 0..7) and then by b bytes (b in 0..3)
__device__ __forceinline__ void rotate8(uint32_t (&w)[8], int r, int b) {
  uint32_t t[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) t[j] = (r & 1) ? w[(j + 1) & 7] : w[j];
#pragma unroll
  for (int j = 0; j < 8; ++j) w[j] = (r & 2) ? t[(j + 2) & 7] : t[j];
#pragma unroll
  for (int j = 0; j < 8; ++j) t[j] = (r & 4) ? w[(j + 4) & 7] : w[j];
#pragma unroll
  for (int j = 0; j < 8; ++j) w[j] = __funnelshift_r(t[j], t[(j + 1) & 7], 8 * b);
}
__device__ __forceinline__ void rotate4(uint32_t (&w)[4], int r, int b) {
  uint32_t t[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) t[j] = (r & 1) ? w[(j + 1) & 3] : w[j];
#pragma unroll
  for (int j = 0; j < 4; ++j) w[j] = (r & 2) ? t[(j + 2) & 3] : t[j];
#pragma unroll
  for (int j = 0; j < 4; ++j) t[j] = __funnelshift_r(w[j], w[(j + 1) & 3], 8 * b);
#pragma unroll
  for (int j = 0; j < 4; ++j) w[j] = t[j];
}

// one lookup of QB floats at byte offset off from tab, added to the pair accumulators
template <int QB>
__device__ __forceinline__ void lut8_add(const char* tab, uint32_t off, unsigned long long (&acc)[2]) {
  if constexpr (QB == 4) {
    const float4 v = *reinterpret_cast<const float4*>(tab + off);
    add2(acc[0], v.x, v.y);
    add2(acc[1], v.z, v.w);
  } else {
    const float2 v = *reinterpret_cast<const float2*>(tab + off);
    add2(acc[0], v.x, v.y);
  }
}

// The 8 partial sums (code and sign parts, QB queries) of one key from the byte tables.
template <int QB>
__device__ __forceinline__ void lut8_key_sums(const float* code8, const float* sign8, const PackedKey<2>& k,
                                              int lane, float (&mm)[QB], float (&rr)[QB]) {
  constexpr uint32_t kC = 4 * QB;                         // bytes of one entry
  constexpr int kEC = 32 * kC;                            // bytes per code byte value (32 positions)
  constexpr int kES = 16 * kC;                            // bytes per sign byte value (16 positions)
  uint32_t w[8] = {k.idx[0].x, k.idx[0].y, k.idx[0].z, k.idx[0].w, k.idx[1].x, k.idx[1].y, k.idx[1].z, k.idx[1].w};
  uint32_t ws[4] = {k.sg.x, k.sg.y, k.sg.z, k.sg.w};
  rotate8(w, lane >> 2, lane & 3);
  rotate4(ws, (lane >> 2) & 3, lane & 3);
  unsigned long long m2[2][2] = {{0ull, 0ull}, {0ull, 0ull}}, r2[2][2] = {{0ull, 0ull}, {0ull, 0ull}};
  const char* ct = reinterpret_cast<const char*>(code8);
  const char* st = reinterpret_cast<const char*>(sign8);
  // column of step i: ((i + lane) mod 32) entries for codes, ((i + lane) mod 16) for signs
  uint32_t col = static_cast<uint32_t>(lane) * kC;
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const uint32_t byte = (w[i >> 2] >> (8 * (i & 3))) & 0xffu;
    lut8_add<QB>(ct, byte * kEC + col, m2[i & 1]);
    if (i < 16) {
      const uint32_t sb = (ws[i >> 2] >> (8 * (i & 3))) & 0xffu;
      lut8_add<QB>(st, sb * kES + (col & (15u * kC)), r2[i & 1]);
    }
    col = (col + kC) & (31u * kC);
  }
#pragma unroll
  for (int q = 0; q < QB; ++q) {
    const int a = q >> 1;
    const bool hi = q & 1;
    const float m0 = hi ? __uint_as_float(static_cast<uint32_t>(m2[0][a] >> 32)) : __uint_as_float(static_cast<uint32_t>(m2[0][a]));
    const float m1 = hi ? __uint_as_float(static_cast<uint32_t>(m2[1][a] >> 32)) : __uint_as_float(static_cast<uint32_t>(m2[1][a]));
    const float r0 = hi ? __uint_as_float(static_cast<uint32_t>(r2[0][a] >> 32)) : __uint_as_float(static_cast<uint32_t>(r2[0][a]));
    const float r1 = hi ? __uint_as_float(static_cast<uint32_t>(r2[1][a] >> 32)) : __uint_as_float(static_cast<uint32_t>(r2[1][a]));
    mm[q] = m0 + m1;
    rr[q] = r0 + r1;
  }
}

// Tables of one unit from its A and T rows staged as sAT [256][QB]: first the 2-code and
// 4-sign tables, then the byte tables as sums of two of them.
template <int QB>
__device__ __forceinline__ void build_lut8(const float* sAT, float* code8, float* sign8, float* pair, float* nib,
                                           const float* cb4) {
  constexpr int NT = Lut8<QB>::kThreads;
  const int tid = threadIdx.x;
  // 2-code tables: pair[(e4 * 64 + g) * QB + q] = A[2g] c[e4 & 3] + A[2g+1] c[e4 >> 2]
  for (int e = tid; e < 64 * 16 * QB; e += NT) {
    const int q = e % QB, g = (e / QB) % 64, e4 = e / (QB * 64);
    pair[e] = fmaf(sAT[(2 * g) * QB + q], cb4[e4 & 3], sAT[(2 * g + 1) * QB + q] * cb4[e4 >> 2]);
  }
  // 4-sign tables: nib[(e4 * 32 + g) * QB + q] = sum_i T[4g+i] (bit i of e4 ? +1 : -1)
  for (int e = tid; e < 32 * 16 * QB; e += NT) {
    const int q = e % QB, g = (e / QB) % 32, e4 = e / (QB * 32);
    float acc = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float t = sAT[(128 + 4 * g + i) * QB + q];
      acc += ((e4 >> i) & 1) ? t : -t;
    }
    nib[e] = acc;
  }
  __syncthreads();
  // code byte tables: code8[(e * 32 + p) * QB + q] = pair(e & 15, 2p) + pair(e >> 4, 2p + 1)
  for (int e = tid; e < 256 * 32 * QB; e += NT) {
    const int q = e % QB, p = (e / QB) % 32, v = e / (QB * 32);
    code8[e] = pair[((v & 15) * 64 + 2 * p) * QB + q] + pair[((v >> 4) * 64 + 2 * p + 1) * QB + q];
  }
  // sign byte tables: sign8[(e * 16 + p) * QB + q] = nib(e & 15, 2p) + nib(e >> 4, 2p + 1)
  for (int e = tid; e < 256 * 16 * QB; e += NT) {
    const int q = e % QB, p = (e / QB) % 16, v = e / (QB * 16);
    sign8[e] = nib[((v & 15) * 32 + 2 * p) * QB + q] + nib[((v >> 4) * 32 + 2 * p + 1) * QB + q];
  }
}

// Stream-K scorer with byte tables (2-bit codes, QB = 2 or 4); the unit boundaries,
// staging and programmatic-dependent-launch protocol of scores_packed_lut_kernel.
template <int QB>
__global__ void __launch_bounds__(Lut8<QB>::kThreads, 1)
scores_packed_lut8_kernel(const float* __restrict__ A, const float* __restrict__ T,
                          const uint8_t* __restrict__ idx_plane, const uint8_t* __restrict__ sign_plane,
                          const uint16_t* __restrict__ gamma_f16, const float* __restrict__ codebook,
                          float* __restrict__ scores, int B, int S, int qtiles, int64_t total, float kappa) {
  using L = Lut8<QB>;
  constexpr int NT = L::kThreads;
  extern __shared__ __align__(16) float smem[];
  float* code8 = smem;
  float* sign8 = code8 + L::kCode;
  float* pair = sign8 + L::kSign;
  float* nib = pair + L::kPair;
  float* sAT = nib + L::kNib;                             // [256][QB]: the unit's A, then T
  __shared__ float cb4[4];
  const int tid = threadIdx.x, lane = tid & 31;
  const int64_t per = (total + gridDim.x - 1) / gridDim.x;
  int64_t w = min(static_cast<int64_t>(blockIdx.x) * per, total);
  const int64_t wend = min(w + per, total);
  bool waited = false;
  while (w < wend) {
    const int u = static_cast<int>(w / S);
    const int sb = static_cast<int>(w - static_cast<int64_t>(u) * S);
    const int se = static_cast<int>(min(static_cast<int64_t>(S), sb + (wend - w)));
    const int p = u / qtiles;
    const int b0 = (u - p * qtiles) * QB;
    const int first = sb + tid;
    // the segment's first two keys are requested before its tables are built
    PackedKey<2> k0, k1;
    prefetch_two_keys<2>(k0, k1, idx_plane, sign_plane, gamma_f16, p, first, NT, se, S);
    if (!waited) {
      asm volatile("griddepcontrol.wait;" ::: "memory");
      waited = true;
    }
    // the unit's A and T rows: one load round trip (QB values a thread before the
    // barrier), queries past B read as zero
    float at[(256 * QB + NT - 1) / NT];
#pragma unroll
    for (int j = 0; j < (256 * QB + NT - 1) / NT; ++j) {
      const int e = tid + NT * j, x = e / QB, q = e % QB;
      const size_t row = (static_cast<size_t>(p) * B + b0 + q) * 128;
      at[j] = e < 256 * QB && b0 + q < B ? (x < 128 ? __ldcg(A + row + x) : __ldcg(T + row + x - 128)) : 0.f;
    }
    const float cbv = tid < 4 ? __ldcg(codebook + tid) : 0.f;
    __syncthreads();                      // the previous segment's tables are no longer read
#pragma unroll
    for (int j = 0; j < (256 * QB + NT - 1) / NT; ++j) {
      const int e = tid + NT * j;
      if (e < 256 * QB) sAT[e] = at[j];
    }
    if (tid < 4) cb4[tid] = cbv;
    __syncthreads();
    build_lut8<QB>(sAT, code8, sign8, pair, nib, cb4);
    __syncthreads();
    const size_t base = static_cast<size_t>(p) * S;
    for (int64_t s = first; s < se; s += NT) {
      const PackedKey<2> cur = k0;
      k0 = k1;
      if (s + 2 * NT < se) load_packed_key<2>(k1, idx_plane, sign_plane, gamma_f16, base + s + 2 * NT);
      float mm[QB], rr[QB];
      lut8_key_sums<QB>(code8, sign8, cur, lane, mm, rr);
      store_scores<QB>(scores, mm, rr, kappa * __half2float(__ushort_as_half(cur.g)), p, b0, B, S,
                       static_cast<int>(s));
    }
    w += se - sb;
  }
}

template <int QB>
cudaError_t launch_lut8_qb(const float* A, const float* T, const uint8_t* idx_plane,
                           const uint8_t* sign_plane, const uint16_t* gamma_f16, const float* codebook,
                           float* scores, int P, int B, int S, bool after_prepare, cudaStream_t st) {
  using L = Lut8<QB>;
  const size_t smem = static_cast<size_t>(L::kFloats) * sizeof(float);
  auto kernel = scores_packed_lut8_kernel<QB>;
  static std::atomic<int> slots[64];      // co-resident CTAs per device
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  int n = slots[dev & 63].load(std::memory_order_acquire);
  if (n == 0) {
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    int sms = 0, per_sm = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, L::kThreads, smem);
    if (e != cudaSuccess) return e;
    n = sms * (per_sm > 0 ? per_sm : 1);
    slots[dev & 63].store(n, std::memory_order_release);
  }
  const int qtiles = ceil_div(B, QB);
  const int64_t total = static_cast<int64_t>(P) * qtiles * S;
  const int64_t want = (total + L::kThreads - 1) / L::kThreads;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(want < n ? want : n));
  cfg.blockDim = dim3(L::kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = after_prepare ? 1 : 0;
  e = cudaLaunchKernelEx(&cfg, kernel, A, T, idx_plane, sign_plane, gamma_f16, codebook, scores, B, S, qtiles,
                         total, qjl_scale(128));
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <int BITS>
cudaError_t launch_lut_bits(const float* A, const float* T, const uint8_t* idx_plane,
                            const uint8_t* sign_plane, const uint16_t* gamma_f16,
                            const float* codebook, float* scores, int P, int B, int S,
                            bool after_prepare, cudaStream_t st) {
  if (B <= 1) return launch_lut_qb<BITS, 1>(A, T, idx_plane, sign_plane, gamma_f16, codebook, scores, P, B, S, after_prepare, st);
  if constexpr (BITS == 2) {
    // 2-bit codes with 2-4 queries: byte tables (half the lookups)
    if (B <= 2) return launch_lut8_qb<2>(A, T, idx_plane, sign_plane, gamma_f16, codebook, scores, P, B, S, after_prepare, st);
    if (B <= 4) return launch_lut8_qb<4>(A, T, idx_plane, sign_plane, gamma_f16, codebook, scores, P, B, S, after_prepare, st);
  }
  if (B <= 2) return launch_lut_qb<BITS, 2>(A, T, idx_plane, sign_plane, gamma_f16, codebook, scores, P, B, S, after_prepare, st);
  if (B <= 4 || BITS == 3) return launch_lut_qb<BITS, 4>(A, T, idx_plane, sign_plane, gamma_f16, codebook, scores, P, B, S, after_prepare, st);
  return launch_lut_qb<BITS, 8>(A, T, idx_plane, sign_plane, gamma_f16, codebook, scores, P, B, S, after_prepare, st);
}


// ---------------------------------------------------------------------------
// Fused query transform + packed scoring for few queries (D = 128), one kernel
// per call with nothing written to a workspace ("TurboQuant Attention in CUDA",
// "Two kernels, two jobs": the first kernel, here inside the second).
//
// A cluster of CS CTAs serves one (problem, query tile); each CTA scores one
// contiguous range of the keys.  The stacked matrix [Pi; S_mat] of the problem's
// head has 256 rows; CTA rank r brings rows r*R .. r*R+R-1 (R = 256/CS) into its
// shared memory with one bulk copy and the query tile with another, forms those rows
// of A = Pi q and T = S_mat q for its QB queries (a warp per 8 rows), and sends each group
// of 8 rows to every CTA of the cluster by a shared-to-shared bulk copy that
// completes bytes on the receiver's mbarrier.  Once that mbarrier has seen all 256
// rows a CTA holds all of A and T, builds the lookup tables and scores its keys.
//
// Keys stream through a ring of kFusedStages shared-memory tiles of kFusedThreads
// keys (one key per thread per tile), each filled by two bulk copies (code rows, sign
// rows) that complete on the tile's mbarrier.  Registers hold the kernel to two CTAs
// a SM, so the clusters spread evenly.  The kernel is launched as a programmatic
// dependent and triggers its own dependents at entry: the next call's CTAs take each
// SM as this call's leave it.  Before griddepcontrol.wait a CTA only asks L2 to
// prefetch what it will read (its key range, its rows of [Pi; S_mat], the query
// tile), a hint that changes no result whatever the kernel before it writes.  Every
// read of global memory into registers or shared memory follows the wait; the rows
// of [Pi; S_mat] are requested before the key tiles, which queue behind them.
// ---------------------------------------------------------------------------
constexpr int kFusedThreads = 512;
constexpr int kFusedStages = 3;
// Dynamic shared memory of one CTA: the tables, the CTA's rows of [Pi; S_mat] and the
// key-tile ring (A/T and the barriers are static).
template <int BITS, int QB, int CS>
constexpr size_t fused_dyn_smem_bytes() {
  return static_cast<size_t>(QB) * LutShape<BITS>::PER_Q * sizeof(float) + (256 / CS) * 128 * sizeof(float) +
         static_cast<size_t>(kFusedStages) * kFusedThreads * (16 * BITS + 16);
}
// Keys of a range asked of L2 before the dependency wait, at most.
constexpr int kFusedPrefetchKeys = 2048;

__device__ __forceinline__ void expect_bytes(uint32_t bar, uint32_t bytes) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(bar),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}

// Coordinates 4*lane .. 4*lane+3 of one query row of 128, from the CTA's shared copy.
__device__ __forceinline__ float4 query4(const float* q, int lane) {
  return reinterpret_cast<const float4*>(q)[lane];
}
__device__ __forceinline__ float4 query4(const __nv_bfloat16* q, int lane) {
  const uint2 v = reinterpret_cast<const uint2*>(q)[lane];
  return make_float4(__uint_as_float(v.x << 16), __uint_as_float(v.x & 0xffff0000u),
                     __uint_as_float(v.y << 16), __uint_as_float(v.y & 0xffff0000u));
}

// Sums over the 32 lanes of 8 per-lane values v[0..7] at once (a transposing
// butterfly): afterwards lane l holds the full sum of value
// 4*bit4(l) + 2*bit3(l) + bit2(l), in v[0].  Nine shuffles instead of forty.
__device__ __forceinline__ float warp_sum8(float (&v)[8], int lane) {
  const bool h4 = (lane >> 4) & 1, h3 = (lane >> 3) & 1, h2 = (lane >> 2) & 1;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float send = h4 ? v[i] : v[i + 4];
    const float keep = h4 ? v[i + 4] : v[i];
    v[i] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const float send = h3 ? v[i] : v[i + 2];
    const float keep = h3 ? v[i + 2] : v[i];
    v[i] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
  }
  {
    const float send = h2 ? v[0] : v[1];
    const float keep = h2 ? v[1] : v[0];
    v[0] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
  }
  v[0] += __shfl_xor_sync(0xffffffffu, v[0], 2);
  v[0] += __shfl_xor_sync(0xffffffffu, v[0], 1);
  return v[0];
}

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t map_to_rank(uint32_t local_addr, uint32_t rank) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local_addr), "r"(rank));
  return remote;
}

template <int BITS, int QB, int CS, typename QT>
__global__ void __launch_bounds__(kFusedThreads, QB <= 2 ? 2 : 1)
solve_packed_lut_kernel(const QT* __restrict__ Q, const float* __restrict__ Pi,
                        const float* __restrict__ Sm, int H, const uint8_t* __restrict__ idx_plane,
                        const uint8_t* __restrict__ sign_plane,
                        const uint16_t* __restrict__ gamma_f16,
                        const float* __restrict__ codebook, float* __restrict__ scores, int B,
                        int S, float kappa) {
  using L = LutShape<BITS>;
  constexpr int D = 128;
  constexpr int kT = kFusedThreads;
  constexpr int R = 256 / CS;                             // rows of [Pi; S_mat] per CTA
  constexpr int kRowBytes = 16 * BITS;                    // code bytes of one key
  constexpr int kTile = kT * (kRowBytes + 16);            // bytes of one key tile
  static_assert(R % 8 == 0 && CS <= 32 && R / 8 <= kT / 32, "transform split");
  __shared__ __align__(16) float sAT[256 * QB];           // [256][QB]: rows of A, then of T
  __shared__ __align__(16) float sMine[R * QB];           // [R][QB]: this CTA's rows of A/T
  __shared__ __align__(8) uint64_t bars[2 + kFusedStages];   // rows, A/T, key tiles
  __shared__ float sCb[1 << BITS];
  __shared__ __align__(16) QT sQ[QB * D];                 // the query tile (rows up to B)
  extern __shared__ __align__(128) float dsm[];
  float* lut = dsm;                                       // [QB][PER_Q]
  float* sRows = lut + QB * L::PER_Q;                     // [R][128]
  uint8_t* sTiles = reinterpret_cast<uint8_t*>(sRows + R * D);   // [stage][kT code rows | kT sign rows]
  const int p = blockIdx.z;
  const int h = p % H;
  const int b0 = blockIdx.y * QB;
  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  // this CTA's keys: one contiguous range of whole tiles of 8 keys
  const int64_t per = ((static_cast<int64_t>(S) + gridDim.x - 1) / gridDim.x + 7) / 8 * 8;
  const int k_begin = static_cast<int>(min(static_cast<int64_t>(blockIdx.x) * per, static_cast<int64_t>(S)));
  const int k_end = static_cast<int>(min(static_cast<int64_t>(k_begin) + per, static_cast<int64_t>(S)));
  const int ntiles = (k_end - k_begin + kT - 1) / kT;
  const size_t key0 = static_cast<size_t>(p) * S + k_begin;
  const uint32_t rank = cluster_ctarank();
  const int row0 = static_cast<int>(rank) * R;
  const float* rows_src = (row0 < D ? Pi : Sm) + (static_cast<size_t>(h) * D + (row0 & (D - 1))) * D;
  const uint32_t bar_rows = static_cast<uint32_t>(__cvta_generic_to_shared(bars));
  const uint32_t bar_at = bar_rows + 8;
  const uint32_t bar_tile = bar_rows + 16;

  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (tid == 0) {
#pragma unroll
    for (int i = 0; i < 2 + kFusedStages; ++i)
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bar_rows + 8 * i) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    expect_bytes(bar_at, 256 * QB * 4);
    // hints only: whatever lands in L2 now is still read after the wait below
    prefetch_l2(rows_src, R * D * sizeof(float));
    const int npre = min(k_end - k_begin, kFusedPrefetchKeys);
    if (npre > 0) {
      prefetch_l2(idx_plane + key0 * kRowBytes, static_cast<size_t>(npre) * kRowBytes);
      prefetch_l2(sign_plane + key0 * 16, static_cast<size_t>(npre) * 16);
      prefetch_l2(gamma_f16 + key0, static_cast<size_t>(npre) * 2);
    }
    const int nq = min(QB, B - b0);
    prefetch_l2(Q + (static_cast<size_t>(p) * B + b0) * D, static_cast<size_t>(nq) * D * sizeof(QT));
  }
  // the barriers are initialised before any thread of the cluster uses them, and
  // every CTA of the cluster runs before anyone copies into a peer
  __syncthreads();
  cluster_arrive_relaxed();
  cluster_wait();
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int nq = min(QB, B - b0);                          // >= 1
  if (tid == 0) {
    // the query tile comes with the rows: one request per CTA rather than one per warp
    // that uses it (every CTA of the unit reads the same lines)
    const uint32_t qbytes = static_cast<uint32_t>(nq * D * sizeof(QT));
    expect_bytes(bar_rows, R * D * 4 + qbytes);
    bulk_g2s(sRows, rows_src, R * D * 4, bar_rows);
    bulk_g2s(sQ, Q + (static_cast<size_t>(p) * B + b0) * D, qbytes, bar_rows);
    for (int t = 0; t < kFusedStages && t < ntiles; ++t) {
      const int nk = min(kT, k_end - k_begin - t * kT);
      uint8_t* st = sTiles + t * kTile;
      expect_bytes(bar_tile + 8 * t, static_cast<uint32_t>(nk * (kRowBytes + 16)));
      bulk_g2s(st, idx_plane + (key0 + t * kT) * kRowBytes, nk * kRowBytes, bar_tile + 8 * t);
      bulk_g2s(st + kT * kRowBytes, sign_plane + (key0 + t * kT) * 16, nk * 16, bar_tile + 8 * t);
    }
  }
  // warps R/8 and up compute no rows of A/T, so the last one copies the codebook; the
  // barrier before the table build orders its copy before any read
  stage_codebook<BITS>(codebook, sCb, kT - 32);
  // gamma of this thread's key in the first tile (later tiles: one tile ahead)
  float g_next = k_begin + tid < k_end ? __half2float(__ushort_as_half(__ldcg(gamma_f16 + key0 + tid))) : 0.f;
  // rows of A/T: warp w takes groups of 8 rows; lane l reads coordinates 4l .. 4l+3
  // of each row (one conflict-free 512-byte row a warp) and the warp sums them.  Each
  // group goes to every CTA of the cluster by its own bulk copies, completing bytes
  // on the receiver's mbarrier, so no warp waits for another here.
  if (warp < R / 8) {
    const bool landed = wait_parity_bounded(bar_rows, 0, kFaultLut);
    float4 qx[QB];                                        // the query tile; rows past B are zero
#pragma unroll
    for (int q = 0; q < QB; ++q) qx[q] = q < nq ? query4(sQ + q * D, lane) : make_float4(0.f, 0.f, 0.f, 0.f);
    const int g = warp;
    float part[QB][8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float4 m = *reinterpret_cast<const float4*>(sRows + (g * 8 + i) * D + 4 * lane);
#pragma unroll
      for (int q = 0; q < QB; ++q)
        part[q][i] = fmaf(m.w, qx[q].w, fmaf(m.z, qx[q].z, fmaf(m.y, qx[q].y, m.x * qx[q].x)));
    }
    const int r = g * 8 + ((lane >> 4) & 1) * 4 + ((lane >> 3) & 1) * 2 + ((lane >> 2) & 1);
#pragma unroll
    for (int q = 0; q < QB; ++q) {
      const float v = warp_sum8(part[q], lane);
      if ((lane & 3) == 0) sMine[r * QB + q] = landed ? v : __int_as_float(0x7fc00000);
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncwarp();
    if (lane < CS) {
      const uint32_t src = static_cast<uint32_t>(__cvta_generic_to_shared(sMine + g * 8 * QB));
      const uint32_t dst = map_to_rank(
          static_cast<uint32_t>(__cvta_generic_to_shared(sAT + (row0 + g * 8) * QB)), static_cast<uint32_t>(lane));
      asm volatile("cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                   "r"(src), "r"(static_cast<uint32_t>(8 * QB * 4)),
                   "r"(map_to_rank(bar_at, static_cast<uint32_t>(lane)))
                   : "memory");
    }
  }
  // every copy into this CTA has completed (so every peer is done reading the slices
  // it sent here); the cluster barrier at the end keeps each CTA alive until all have
  const bool have_at = wait_parity_bounded(bar_at, 0, kFaultLut);
  cluster_arrive_relaxed();
  __syncthreads();
  float cv[L::G];
  table_centroids<BITS>(sCb, cv);
  build_luts<BITS, QB, kT>(
      [&](int q, int e) { return have_at ? sAT[e * QB + q] : __int_as_float(0x7fc00000); }, lut, cv);
  __syncthreads();
  for (int t = 0; t < ntiles; ++t) {
    const int stage = t % kFusedStages;
    const uint8_t* st = sTiles + stage * kTile;
    const bool have_keys = wait_parity_bounded(bar_tile + 8 * stage, (t / kFusedStages) & 1, kFaultLut);
    const int s = k_begin + t * kT + tid;
    const float g = g_next;
    if (t + 1 < ntiles)
      g_next = s + kT < k_end ? __half2float(__ushort_as_half(__ldcg(gamma_f16 + key0 + (t + 1) * kT + tid))) : 0.f;
    if (s < k_end) {
      PackedKey<BITS> k;
#pragma unroll
      for (int r = 0; r < BITS; ++r) k.idx[r] = *reinterpret_cast<const uint4*>(st + tid * kRowBytes + 16 * r);
      k.sg = *reinterpret_cast<const uint4*>(st + kT * kRowBytes + tid * 16);
      float mm[QB], rr[QB];
      lut_key_sums<BITS, QB>(lut, k, mm, rr);
      if (!have_keys) {
#pragma unroll
        for (int q = 0; q < QB; ++q) mm[q] = __int_as_float(0x7fc00000);
      }
      store_scores<QB>(scores, mm, rr, kappa * g, p, b0, B, S, s);
    }
    if (t + kFusedStages < ntiles) {
      __syncthreads();                    // every thread is done with this stage
      if (tid == 0) {
        const int tn = t + kFusedStages;
        const int nk = min(kT, k_end - k_begin - tn * kT);
        uint8_t* sd = sTiles + stage * kTile;
        expect_bytes(bar_tile + 8 * stage, static_cast<uint32_t>(nk * (kRowBytes + 16)));
        bulk_g2s(sd, idx_plane + (key0 + static_cast<size_t>(tn) * kT) * kRowBytes, nk * kRowBytes, bar_tile + 8 * stage);
        bulk_g2s(sd + kT * kRowBytes, sign_plane + (key0 + static_cast<size_t>(tn) * kT) * 16, nk * 16,
                 bar_tile + 8 * stage);
      }
    }
  }
  cluster_wait();
}

// One launch of the fused kernel with clusters of CS CTAs.  The grid gets as many
// clusters per (problem, query tile) unit as are co-resident for every unit at once
// (at least one), and no more than leave a CTA 64 keys.  For short calls (at most two
// key tiles a CTA) it keeps 1/9 of the co-resident clusters free: back-to-back calls
// overlap (programmatic dependent launch), and with every slot planned some clusters
// of the next call find no whole group of free SMs and start a wave late.  Measured on
// GB300 at B = 1: 131072 keys took 5.35 us a call at 36 clusters, 4.66 us at 32; from
// 524288 keys on the full grid is faster (3-9 %).
template <int BITS, int QB, int CS, typename QT>
cudaError_t launch_fused_cs(const QT* Q, const float* Pi, const float* S_mat, int H,
                            const uint8_t* idx_plane, const uint8_t* sign_plane,
                            const uint16_t* gamma_f16, const float* codebook, float* scores,
                            int P, int B, int S, cudaStream_t st) {
  constexpr size_t smem = fused_dyn_smem_bytes<BITS, QB, CS>();
  auto kernel = solve_packed_lut_kernel<BITS, QB, CS, QT>;
  static std::atomic<uint64_t> configured{0};
  static std::atomic<int> capacity[64];                   // co-resident clusters per device
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CS;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.blockDim = dim3(kFusedThreads);
  cfg.stream = st;
  cfg.attrs = attr;
  if (!(configured.load(std::memory_order_acquire) & bit)) {
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    int n = 0;
    cfg.gridDim = dim3(CS);
    cfg.numAttrs = 1;
    cfg.dynamicSmemBytes = smem;
    e = cudaOccupancyMaxActiveClusters(&n, kernel, &cfg);
    if (e != cudaSuccess) return e;
    capacity[dev & 63].store(n > 0 ? n : 1, std::memory_order_relaxed);
    configured.fetch_or(bit, std::memory_order_acq_rel);
  }
  const int qtiles = ceil_div(B, QB);
  const int64_t units = static_cast<int64_t>(P) * qtiles;
  int cap = capacity[dev & 63].load(std::memory_order_relaxed);
  if (static_cast<int64_t>(S) * units <= static_cast<int64_t>(cap) * CS * 2 * kFusedThreads) cap = cap * 8 / 9;
  const int fill = static_cast<int>(cap / units);
  const int most = ceil_div(S, 64 * CS);                  // at least 64 keys a CTA on average
  const int clusters = fill < most ? fill : most;
  const int gx = (clusters < 1 ? 1 : clusters) * CS;
  cfg.gridDim = dim3(gx, qtiles, P);
  cfg.numAttrs = 2;
  cfg.dynamicSmemBytes = smem;
  e = cudaLaunchKernelEx(&cfg, kernel, Q, Pi, S_mat, H, idx_plane, sign_plane, gamma_f16, codebook,
                         scores, B, S, qjl_scale(128));
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <int BITS, int QB, typename QT>
cudaError_t launch_fused_qb(const QT* Q, const float* Pi, const float* S_mat, int H,
                            const uint8_t* idx_plane, const uint8_t* sign_plane,
                            const uint16_t* gamma_f16, const float* codebook, float* scores,
                            int P, int B, int S, cudaStream_t st) {
  return launch_fused_cs<BITS, QB, 8, QT>(Q, Pi, S_mat, H, idx_plane, sign_plane, gamma_f16, codebook,
                                          scores, P, B, S, st);
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
                                      int D, int idx_bits, bool after_prepare, cudaStream_t st) {
  if (D == 128) {
    switch (idx_bits) {
      case 1: return launch_lut_bits<1>(A, T, idx_plane, sign_plane, gamma_f16, codebook, scores, P, B, S, after_prepare, st);
      case 2: return launch_lut_bits<2>(A, T, idx_plane, sign_plane, gamma_f16, codebook, scores, P, B, S, after_prepare, st);
      default: return launch_lut_bits<3>(A, T, idx_plane, sign_plane, gamma_f16, codebook, scores, P, B, S, after_prepare, st);
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

// The fused kernel gives every (problem, query tile) unit a cluster of 8 CTAs; with
// problems enough to fill half the SMs, the transform kernel followed by the
// stream-K scorer balances the SMs better.
bool fused_packed_supported(int P, int B, int D) {
  if (D != 128 || B < 1 || B > 8) return false;
  static std::atomic<int> sms_cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  int sms = sms_cache[dev & 63].load(std::memory_order_relaxed);
  if (sms == 0) {
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return false;
    sms_cache[dev & 63].store(sms, std::memory_order_relaxed);
  }
  return 2 * static_cast<int64_t>(P) < sms;
}

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

namespace tq {
cudaError_t take_faults_simt(unsigned int* bits) { return take_unit_faults(bits); }
}  // namespace tq
