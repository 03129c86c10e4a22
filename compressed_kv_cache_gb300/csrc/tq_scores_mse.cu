// MSE-only scorer (the TurboQuant-MSE variant: no residual sketch, one stored norm
// per key).  With A = Pi q from the query transform:
//
//   score[b,s] = n_s * sum_d A[b,d] c[idx[s,d]]                          (plain)
//   score[b,s] = n_s * sum_d A[b,d] c[idx[s,d]] / sqrt(sum_d c[idx[s,d]]^2)   (norm correction)
//
// ("TurboQuant: Rotate-then-Quantize KV Caches at 3 Bits", kanthi.in: §3
// TurboQuantMSE.dequantize, §8 "Kernel view: never un-rotate a key").  The cache is
// the packed code plane of tq_scores_packed (no sign plane) and an IEEE fp16 norm
// per key.
//
// Two kernels:
//   scores_mse_lut_kernel   D = 128, 1-3 bit codes: the lookup tables of the packed
//                           scorer (code tables only) plus one query-independent table
//                           of squared centroid sums for the correction; stream-K over
//                           the keys of all (problem, query tile) units.
//   scores_mse_kernel       any D % 32 == 0, 1-4 bit codes: thread per key, codebook
//                           and the query tile in shared memory.
// Each score has one owner thread and one summation order, so results are
// deterministic.
#include <atomic>

#include "tq_internal.cuh"
#include "tq_lut.cuh"

namespace tq {
namespace {

// One key in registers: BITS 16-byte rows of codes and the fp16 norm.
template <int BITS>
struct MseKey {
  uint4 idx[BITS];
  uint16_t n;
};

template <int BITS>
__device__ __forceinline__ void load_mse_key(MseKey<BITS>& k, const uint8_t* __restrict__ idx_plane,
                                             const uint16_t* __restrict__ norm_f16, size_t key) {
  const uint4* ip = reinterpret_cast<const uint4*>(idx_plane + key * (16 * BITS));
#pragma unroll
  for (int i = 0; i < BITS; ++i) k.idx[i] = __ldcg(ip + i);
  k.n = __ldcg(norm_f16 + key);
}

template <int QB>
__device__ __forceinline__ void store_mse(float* __restrict__ scores, const float (&m)[QB], float scale,
                                          int p, int b0, int B, int S, int s) {
#pragma unroll
  for (int q = 0; q < QB; ++q) {
    if (b0 + q < B) scores[(static_cast<size_t>(p) * B + b0 + q) * S + s] = m[q] * scale;
  }
}

// D = 128.  lut: [QB][NPI][NV] code tables; sq: [NV] sums of squared centroids of a
// table value (the same for every position and query); sA: [QB][128] the segment's
// rotated queries (one load round trip, requested ahead of the segment's keys).
template <int BITS, int QB>
__global__ void __launch_bounds__(256, 2)
scores_mse_lut_kernel(const float* __restrict__ A, const uint8_t* __restrict__ idx_plane,
                      const uint16_t* __restrict__ norm_f16, const float* __restrict__ codebook,
                      float* __restrict__ scores, int B, int S, int qtiles, int64_t total, int corr) {
  using L = LutShape<BITS>;
  extern __shared__ __align__(16) float smem[];
  float* lut = smem;
  float* sq = lut + QB * L::NPI * L::NV;
  float* sA = sq + L::NV;
  const int tid = threadIdx.x;
  // Launched as a programmatic dependent of whatever ran before it on the stream (the
  // query transform, typically): every global read follows this wait, so the launch
  // overlaps that kernel's tail and nothing else.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int v = tid % L::NV;
  __shared__ float sCb[1 << BITS];
  stage_codebook<BITS>(codebook, sCb, 0);   // read after the loop's first barrier
  const int64_t per = (total + gridDim.x - 1) / gridDim.x;
  int64_t w = min(static_cast<int64_t>(blockIdx.x) * per, total);
  const int64_t wend = min(w + per, total);
  while (w < wend) {
    const int u = static_cast<int>(w / S);
    const int sb = static_cast<int>(w - static_cast<int64_t>(u) * S);
    const int se = static_cast<int>(min(static_cast<int64_t>(S), sb + (wend - w)));
    const int p = u / qtiles;
    const int b0 = (u - p * qtiles) * QB;
    const size_t base = static_cast<size_t>(p) * S;
    // the segment's rotated queries, then its first two keys, are requested before its
    // tables are built (queries past B read as zero)
    constexpr int kAP = (QB * 128 + 255) / 256;
    float av[kAP];
#pragma unroll
    for (int j = 0; j < kAP; ++j) {
      const int e = tid + 256 * j, q = e >> 7;
      av[j] = e < QB * 128 && b0 + q < B ? __ldcg(A + (static_cast<size_t>(p) * B + b0 + q) * 128 + (e & 127)) : 0.f;
    }
    MseKey<BITS> k0, k1;
    const int first = sb + tid;
    if (first < se) load_mse_key<BITS>(k0, idx_plane, norm_f16, base + first);
    if (first + 256 < se) load_mse_key<BITS>(k1, idx_plane, norm_f16, base + first + 256);
    __syncthreads();                      // the previous segment's tables are no longer read
#pragma unroll
    for (int j = 0; j < kAP; ++j) {
      const int e = tid + 256 * j;
      if (e < QB * 128) sA[e] = av[j];
    }
    float cv[L::G];
    table_centroids<BITS>(sCb, cv);
    if (tid < L::NV) {
      float acc = 0.f;
#pragma unroll
      for (int k = 0; k < L::G; ++k) acc = fmaf(cv[k], cv[k], acc);
      sq[tid] = acc;
    }
    __syncthreads();
    for (int q = 0; q < QB; ++q) {
      const float* a = sA + q * 128;
      float* tq = lut + q * L::NPI * L::NV;
      for (int g = tid / L::NV; g < L::NPI; g += 256 / L::NV) {
        float acc = 0.f;
#pragma unroll
        for (int k = 0; k < L::G; ++k) acc = fmaf(a[g * L::G + k], cv[k], acc);
        tq[g * L::NV + v] = acc;
      }
    }
    __syncthreads();
    for (int s = first; s < se; s += 256) {
      const MseKey<BITS> cur = k0;
      k0 = k1;
      if (s + 512 < se) load_mse_key<BITS>(k1, idx_plane, norm_f16, base + s + 512);
      uint32_t wd[4 * BITS + 1];
#pragma unroll
      for (int i = 0; i < BITS; ++i) {
        wd[4 * i] = cur.idx[i].x; wd[4 * i + 1] = cur.idx[i].y; wd[4 * i + 2] = cur.idx[i].z; wd[4 * i + 3] = cur.idx[i].w;
      }
      wd[4 * BITS] = 0u;
      float m[2][QB], n2[2] = {0.f, 0.f};
#pragma unroll
      for (int q = 0; q < QB; ++q) m[0][q] = m[1][q] = 0.f;
#pragma unroll
      for (int gi = 0; gi < L::NPI; ++gi) {
        const int off = L::KB * gi;
        const int wi = off >> 5, sh = off & 31;
        const uint32_t val = (sh + L::KB <= 32) ? (wd[wi] >> sh) & (L::NV - 1)
                                                : __funnelshift_r(wd[wi], wd[wi + 1], sh) & (L::NV - 1);
#pragma unroll
        for (int q = 0; q < QB; ++q) m[gi & 1][q] += lut[(q * L::NPI + gi) * L::NV + val];
        if (corr) n2[gi & 1] += sq[val];
      }
      float mm[QB];
#pragma unroll
      for (int q = 0; q < QB; ++q) mm[q] = m[0][q] + m[1][q];
      const float nk = __half2float(__ushort_as_half(cur.n));
      store_mse<QB>(scores, mm, corr ? nk / sqrtf(n2[0] + n2[1]) : nk, p, b0, B, S, s);
    }
    w += se - sb;
  }
}

// Any D % 32 == 0 and 1-4 bit codes: thread per key, the query tile as [D][QB] and
// the codebook (at most 16 centroids, one bank each) in shared memory.
template <int BITS, int QB>
__global__ void __launch_bounds__(128)
scores_mse_kernel(const float* __restrict__ A, const uint8_t* __restrict__ idx_plane,
                  const uint16_t* __restrict__ norm_f16, const float* __restrict__ codebook,
                  float* __restrict__ scores, int B, int S, int D, int corr) {
  constexpr int kC = 1 << BITS;
  extern __shared__ __align__(16) float smem[];
  float* sA = smem;                       // [D][QB]
  float* sC = sA + QB * D;                // [kC]
  const int p = blockIdx.z;
  const int b0 = blockIdx.y * QB;
  for (int e = threadIdx.x; e < QB * D; e += blockDim.x) {
    const int q = e / D, d = e % D;
    sA[d * QB + q] = b0 + q < B ? A[(static_cast<size_t>(p) * B + b0 + q) * D + d] : 0.f;
  }
  if (threadIdx.x < kC) sC[threadIdx.x] = codebook[threadIdx.x];
  __syncthreads();
  const int s = blockIdx.x * blockDim.x + threadIdx.x;
  if (s >= S) return;
  const size_t key = static_cast<size_t>(p) * S + s;
  const int chunks = D >> 5;
  const uint32_t* wi = reinterpret_cast<const uint32_t*>(idx_plane) + key * (chunks * BITS);
  float m[QB], n2 = 0.f;
#pragma unroll
  for (int q = 0; q < QB; ++q) m[q] = 0.f;
  for (int ch = 0; ch < chunks; ++ch) {
    uint32_t w[BITS + 1];
#pragma unroll
    for (int i = 0; i < BITS; ++i) w[i] = __ldg(wi + ch * BITS + i);
    w[BITS] = 0u;
#pragma unroll
    for (int u = 0; u < 32; ++u) {
      const int pos = BITS * u;
      const int wd = pos >> 5, sh = pos & 31;
      const uint32_t code = (sh + BITS <= 32) ? (w[wd] >> sh) & (kC - 1)
                                              : __funnelshift_r(w[wd], w[wd + 1], sh) & (kC - 1);
      const float c = sC[code];
      const float* a = sA + (ch * 32 + u) * QB;
#pragma unroll
      for (int q = 0; q < QB; ++q) m[q] = fmaf(a[q], c, m[q]);
      n2 = fmaf(c, c, n2);
    }
  }
  const float nk = __half2float(__ushort_as_half(__ldg(norm_f16 + key)));
  store_mse<QB>(scores, m, corr ? nk / sqrtf(n2) : nk, p, b0, B, S, s);
}

template <int BITS, int QB>
cudaError_t launch_mse_lut_qb(const float* A, const uint8_t* idx_plane, const uint16_t* norm_f16,
                              const float* codebook, float* scores, int P, int B, int S, bool corr,
                              cudaStream_t st) {
  using L = LutShape<BITS>;
  const size_t smem = (static_cast<size_t>(QB) * L::NPI * L::NV + L::NV + QB * 128) * sizeof(float);
  auto kernel = scores_mse_lut_kernel<BITS, QB>;
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
  const int64_t want = (total + 255) / 256;
  const unsigned grid = static_cast<unsigned>(want < n ? want : n);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kernel, A, idx_plane, norm_f16, codebook, scores, B, S, qtiles, total,
                         corr ? 1 : 0);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <int BITS, int QB>
cudaError_t launch_mse_generic_qb(const float* A, const uint8_t* idx_plane, const uint16_t* norm_f16,
                                  const float* codebook, float* scores, int P, int B, int S, int D,
                                  bool corr, cudaStream_t st) {
  dim3 grid(ceil_div(S, 128), ceil_div(B, QB), P);
  const size_t smem = (static_cast<size_t>(QB) * D + (1 << BITS)) * sizeof(float);
  scores_mse_kernel<BITS, QB><<<grid, 128, smem, st>>>(A, idx_plane, norm_f16, codebook, scores, B, S, D,
                                                       corr ? 1 : 0);
  return cudaGetLastError();
}

template <int BITS>
cudaError_t launch_mse_bits(const float* A, const uint8_t* idx_plane, const uint16_t* norm_f16,
                            const float* codebook, float* scores, int P, int B, int S, int D, bool corr,
                            cudaStream_t st) {
  if constexpr (BITS <= 3) {
    if (D == 128) {
      if (B <= 1) return launch_mse_lut_qb<BITS, 1>(A, idx_plane, norm_f16, codebook, scores, P, B, S, corr, st);
      if (B <= 2) return launch_mse_lut_qb<BITS, 2>(A, idx_plane, norm_f16, codebook, scores, P, B, S, corr, st);
      if (B <= 4 || BITS == 3) return launch_mse_lut_qb<BITS, 4>(A, idx_plane, norm_f16, codebook, scores, P, B, S, corr, st);
      return launch_mse_lut_qb<BITS, 8>(A, idx_plane, norm_f16, codebook, scores, P, B, S, corr, st);
    }
  }
  if (B <= 1) return launch_mse_generic_qb<BITS, 1>(A, idx_plane, norm_f16, codebook, scores, P, B, S, D, corr, st);
  if (B <= 2) return launch_mse_generic_qb<BITS, 2>(A, idx_plane, norm_f16, codebook, scores, P, B, S, D, corr, st);
  if (B <= 4) return launch_mse_generic_qb<BITS, 4>(A, idx_plane, norm_f16, codebook, scores, P, B, S, D, corr, st);
  return launch_mse_generic_qb<BITS, 8>(A, idx_plane, norm_f16, codebook, scores, P, B, S, D, corr, st);
}

}  // namespace

cudaError_t launch_scores_mse(const float* A, const uint8_t* idx_plane, const uint16_t* norm_f16,
                              const float* codebook, float* scores, int P, int B, int S, int D,
                              int idx_bits, bool norm_correction, cudaStream_t st) {
  switch (idx_bits) {
    case 1: return launch_mse_bits<1>(A, idx_plane, norm_f16, codebook, scores, P, B, S, D, norm_correction, st);
    case 2: return launch_mse_bits<2>(A, idx_plane, norm_f16, codebook, scores, P, B, S, D, norm_correction, st);
    case 3: return launch_mse_bits<3>(A, idx_plane, norm_f16, codebook, scores, P, B, S, D, norm_correction, st);
    default: return launch_mse_bits<4>(A, idx_plane, norm_f16, codebook, scores, P, B, S, D, norm_correction, st);
  }
}

}  // namespace tq
