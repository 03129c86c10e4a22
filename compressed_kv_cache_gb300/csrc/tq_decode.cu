// Fused decode over an MSE-quantized key and value cache, in the rotated domain
// ("TurboQuant: Rotate-then-Quantize KV Caches at 3 Bits", kanthi.in, §8 "Kernel
// view: never un-rotate a key", the kernel form of tq_rotated_domain):
//
//   s[b,i]  = scale * nk_i * <A_b, ck[kidx_i]>          A_b = Pi_k q_b (rotated query)
//   p[b,:]  = softmax(s[b,:])
//   acc[b]  = sum_i p[b,i] nv_i cv[vidx_i]              accumulated in the rotated basis
//   out[b]  = Pi_v^T acc[b]                             one inverse rotation per query
//
// Split-KV (flash decoding): decode_split_kernel takes one chunk of keys and one tile
// of QB queries of a problem.  It builds the key lookup tables of the MSE scorer,
// scores its keys into shared memory (thread per key), reduces the chunk's maximum,
// turns the logits into exp(s - max) and their sum, then accumulates the weighted value
// codewords: a warp per key, lane l owning coordinates 4l .. 4l+3, so that each key's
// value row is read once per warp.  It writes (max, sum, acc[128]) per (query, chunk)
// to the workspace.  decode_combine_kernel merges the chunks of a query with the
// usual rescaling by exp(max_c - max) and applies Pi_v^T.  D = 128, 1-3 bit codes.
#include <atomic>

#include "tq_internal.cuh"
#include "tq_lut.cuh"

namespace tq {
namespace {

constexpr int kD = 128;
constexpr int kDecThreads = 256;
constexpr int kMaxChunk = 2048;          // keys per split CTA (shared-memory logits)
constexpr int kPart = 2 + kD;            // floats per (query, chunk): max, sum, acc

// The centroid of a 1-3 bit code from registers (no dynamic register indexing).
template <int BITS>
__device__ __forceinline__ float centroid_of(const float (&c)[1 << BITS], uint32_t code) {
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

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// Shared memory: lut [QB][NPI*NV] | logits [QB][chunk] | red [8 warps][QB][128]
template <int KBITS, int QB>
constexpr size_t split_smem_floats(int chunk) {
  return static_cast<size_t>(QB) * LutShape<KBITS>::NPI * LutShape<KBITS>::NV +
         static_cast<size_t>(QB) * chunk + static_cast<size_t>(kDecThreads / 32) * QB * kD;
}

template <int KBITS, int VBITS, int QB>
__global__ void __launch_bounds__(kDecThreads)
decode_split_kernel(const float* __restrict__ A, const uint8_t* __restrict__ k_plane,
                    const uint16_t* __restrict__ k_norm, const float* __restrict__ k_cb,
                    const uint8_t* __restrict__ v_plane, const uint16_t* __restrict__ v_norm,
                    const float* __restrict__ v_cb, float* __restrict__ part, int B, int S,
                    int chunk, int nchunks, float scale) {
  using L = LutShape<KBITS>;
  constexpr int kW = kDecThreads / 32;
  extern __shared__ __align__(16) float smem[];
  float* lut = smem;
  float* logit = lut + QB * L::NPI * L::NV;
  float* red = logit + QB * chunk;
  const int c = blockIdx.x, p = blockIdx.z, b0 = blockIdx.y * QB;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int k0 = c * chunk;
  const int n = min(chunk, S - k0);
  const size_t kbase = static_cast<size_t>(p) * S + k0;

  // key tables of the query tile (rows past B give zero tables)
  {
    float cv[L::G];
    table_centroids<KBITS>(k_cb, cv);
    const int v = tid % L::NV;
    for (int q = 0; q < QB; ++q) {
      const bool live = b0 + q < B;
      const float* a = A + (static_cast<size_t>(p) * B + (live ? b0 + q : b0)) * kD;
      float* tq = lut + q * L::NPI * L::NV;
      for (int g = tid / L::NV; g < L::NPI; g += kDecThreads / L::NV) {
        float acc = 0.f;
#pragma unroll
        for (int k = 0; k < L::G; ++k) acc = fmaf(__ldg(a + g * L::G + k), cv[k], acc);
        tq[g * L::NV + v] = live ? acc : 0.f;
      }
    }
  }
  __syncthreads();

  // logits, thread per key
  float mx[QB];
#pragma unroll
  for (int q = 0; q < QB; ++q) mx[q] = -INFINITY;
  for (int i = tid; i < n; i += kDecThreads) {
    const uint4* kp = reinterpret_cast<const uint4*>(k_plane + (kbase + i) * (16 * KBITS));
    uint32_t wd[4 * KBITS + 1];
#pragma unroll
    for (int r = 0; r < KBITS; ++r) {
      const uint4 x = __ldg(kp + r);
      wd[4 * r] = x.x; wd[4 * r + 1] = x.y; wd[4 * r + 2] = x.z; wd[4 * r + 3] = x.w;
    }
    wd[4 * KBITS] = 0u;
    const float nk = __half2float(__ushort_as_half(__ldg(k_norm + kbase + i)));
    float m[2][QB];
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
    }
#pragma unroll
    for (int q = 0; q < QB; ++q) {
      const float s = scale * nk * (m[0][q] + m[1][q]);
      logit[q * chunk + i] = s;
      mx[q] = fmaxf(mx[q], s);
    }
  }
  // chunk maximum per query
#pragma unroll
  for (int q = 0; q < QB; ++q) {
    mx[q] = warp_max(mx[q]);
    if (lane == 0) red[warp * QB + q] = mx[q];
  }
  __syncthreads();
  float M[QB];
#pragma unroll
  for (int q = 0; q < QB; ++q) {
    M[q] = red[q];
    for (int w = 1; w < kW; ++w) M[q] = fmaxf(M[q], red[w * QB + q]);
  }
  __syncthreads();
  // weights exp(s - max) in place, and their sum per query
  float sum[QB];
#pragma unroll
  for (int q = 0; q < QB; ++q) sum[q] = 0.f;
  for (int i = tid; i < n; i += kDecThreads) {
#pragma unroll
    for (int q = 0; q < QB; ++q) {
      const float e = expf(logit[q * chunk + i] - M[q]);
      logit[q * chunk + i] = e;
      sum[q] += e;
    }
  }
#pragma unroll
  for (int q = 0; q < QB; ++q) {
    sum[q] = warp_sum(sum[q]);
    if (lane == 0) red[warp * QB + q] = sum[q];
  }
  __syncthreads();
  float Ls[QB];
#pragma unroll
  for (int q = 0; q < QB; ++q) {
    Ls[q] = 0.f;
    for (int w = 0; w < kW; ++w) Ls[q] += red[w * QB + q];
  }
  __syncthreads();

  // weighted value codewords, warp per key; lane l owns coordinates 4l .. 4l+3, whose
  // codes are bits 4*VBITS*l .. 4*VBITS*l + 4*VBITS-1 of the key's value row
  float vc[1 << VBITS];
#pragma unroll
  for (int k = 0; k < (1 << VBITS); ++k) vc[k] = __ldg(v_cb + k);
  constexpr int kVW = 4 * VBITS;          // 32-bit words of one value row
  const int bit0 = 4 * VBITS * lane;
  const int wlo = bit0 >> 5, bsh = bit0 & 31;
  float acc[QB][4];
#pragma unroll
  for (int q = 0; q < QB; ++q) acc[q][0] = acc[q][1] = acc[q][2] = acc[q][3] = 0.f;
  for (int i = warp; i < n; i += kW) {
    const uint32_t* vr = reinterpret_cast<const uint32_t*>(v_plane + (kbase + i) * (16 * VBITS));
    const uint32_t word = lane < kVW ? __ldg(vr + lane) : 0u;
    const uint32_t lo = __shfl_sync(0xffffffffu, word, wlo);
    const uint32_t hi = __shfl_sync(0xffffffffu, word, wlo + 1);
    const uint32_t codes = __funnelshift_r(lo, hi, bsh);
    const float nv = __half2float(__ushort_as_half(__ldg(v_norm + kbase + i)));
    float cw[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) cw[j] = nv * centroid_of<VBITS>(vc, (codes >> (VBITS * j)) & ((1u << VBITS) - 1u));
#pragma unroll
    for (int q = 0; q < QB; ++q) {
      const float wq = logit[q * chunk + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[q][j] = fmaf(wq, cw[j], acc[q][j]);
    }
  }
#pragma unroll
  for (int q = 0; q < QB; ++q) {
#pragma unroll
    for (int j = 0; j < 4; ++j) red[(warp * QB + q) * kD + 4 * lane + j] = acc[q][j];
  }
  __syncthreads();
  for (int e = tid; e < QB * kD; e += kDecThreads) {
    const int q = e / kD, d = e % kD;
    if (b0 + q >= B) continue;
    float s = 0.f;
    for (int w = 0; w < kW; ++w) s += red[(w * QB + q) * kD + d];
    part[((static_cast<size_t>(p) * B + b0 + q) * nchunks + c) * kPart + 2 + d] = s;
  }
  if (tid < QB && b0 + tid < B) {
    float* pp = part + ((static_cast<size_t>(p) * B + b0 + tid) * nchunks + c) * kPart;
#pragma unroll
    for (int q = 0; q < QB; ++q) {
      if (q == tid) {
        pp[0] = M[q];
        pp[1] = Ls[q];
      }
    }
  }
}

// One query: merge the chunks (rescale by exp(max_c - max)), normalise, out = acc Pi_v.
__global__ void __launch_bounds__(kD)
decode_combine_kernel(const float* __restrict__ part, const float* __restrict__ Pi_v,
                      float* __restrict__ out, int H, int B, int nchunks) {
  __shared__ float sacc[kD];
  const int b = blockIdx.x, p = blockIdx.y, h = p % H, d = threadIdx.x;
  const float* pp = part + (static_cast<size_t>(p) * B + b) * nchunks * kPart;
  float M = -INFINITY;
  for (int c = 0; c < nchunks; ++c) M = fmaxf(M, pp[c * kPart]);
  float Lsum = 0.f, a = 0.f;
  for (int c = 0; c < nchunks; ++c) {
    const float e = expf(pp[c * kPart] - M);
    Lsum = fmaf(pp[c * kPart + 1], e, Lsum);
    a = fmaf(pp[c * kPart + 2 + d], e, a);
  }
  sacc[d] = a / Lsum;
  __syncthreads();
  const float* Pv = Pi_v + static_cast<size_t>(h) * kD * kD;
  float o = 0.f;
#pragma unroll 8
  for (int k = 0; k < kD; ++k) o = fmaf(sacc[k], __ldg(Pv + k * kD + d), o);
  out[(static_cast<size_t>(p) * B + b) * kD + d] = o;
}

template <int KBITS, int VBITS, int QB>
cudaError_t launch_decode_qb(const float* A, const uint8_t* k_plane, const uint16_t* k_norm,
                             const float* k_cb, const uint8_t* v_plane, const uint16_t* v_norm,
                             const float* v_cb, const float* Pi_v, float* out, float* part, int P,
                             int H, int B, int S, float scale, cudaStream_t st) {
  auto kernel = decode_split_kernel<KBITS, VBITS, QB>;
  static std::atomic<int> sms_cache[64];
  static std::atomic<uint64_t> configured{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  int sms = sms_cache[dev & 63].load(std::memory_order_relaxed);
  if (sms == 0) {
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    sms_cache[dev & 63].store(sms, std::memory_order_relaxed);
  }
  const uint64_t bit = 1ull << (dev & 63);
  if (!(configured.load(std::memory_order_acquire) & bit)) {
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(split_smem_floats<KBITS, QB>(kMaxChunk) * sizeof(float)));
    if (e != cudaSuccess) return e;
    configured.fetch_or(bit, std::memory_order_acq_rel);
  }
  // chunks of 256..2048 keys (a multiple of 256), enough of them for about two CTAs per SM
  const int qtiles = ceil_div(B, QB);
  const int64_t units = static_cast<int64_t>(P) * qtiles;
  const int64_t per_unit = (2LL * sms + units - 1) / units;
  int chunk = ceil_div(S, per_unit < 1 ? 1 : per_unit);
  chunk = (chunk + 255) / 256 * 256;
  chunk = chunk < 256 ? 256 : (chunk > kMaxChunk ? kMaxChunk : chunk);
  const int nchunks = ceil_div(S, chunk);
  const size_t smem = split_smem_floats<KBITS, QB>(chunk) * sizeof(float);
  dim3 grid(nchunks, qtiles, P);
  kernel<<<grid, kDecThreads, smem, st>>>(A, k_plane, k_norm, k_cb, v_plane, v_norm, v_cb, part, B, S,
                                          chunk, nchunks, scale);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  decode_combine_kernel<<<dim3(B, P), kD, 0, st>>>(part, Pi_v, out, H, B, nchunks);
  return cudaGetLastError();
}

template <int KBITS, int VBITS>
cudaError_t launch_decode_kv(const float* A, const uint8_t* k_plane, const uint16_t* k_norm,
                             const float* k_cb, const uint8_t* v_plane, const uint16_t* v_norm,
                             const float* v_cb, const float* Pi_v, float* out, float* part, int P,
                             int H, int B, int S, float scale, cudaStream_t st) {
  if (B <= 1) return launch_decode_qb<KBITS, VBITS, 1>(A, k_plane, k_norm, k_cb, v_plane, v_norm, v_cb, Pi_v, out, part, P, H, B, S, scale, st);
  if (B <= 2) return launch_decode_qb<KBITS, VBITS, 2>(A, k_plane, k_norm, k_cb, v_plane, v_norm, v_cb, Pi_v, out, part, P, H, B, S, scale, st);
  if (B <= 4 || KBITS == 3) return launch_decode_qb<KBITS, VBITS, 4>(A, k_plane, k_norm, k_cb, v_plane, v_norm, v_cb, Pi_v, out, part, P, H, B, S, scale, st);
  return launch_decode_qb<KBITS, VBITS, 8>(A, k_plane, k_norm, k_cb, v_plane, v_norm, v_cb, Pi_v, out, part, P, H, B, S, scale, st);
}

template <int KBITS>
cudaError_t launch_decode_k(const float* A, const uint8_t* k_plane, const uint16_t* k_norm,
                            const float* k_cb, const uint8_t* v_plane, const uint16_t* v_norm,
                            const float* v_cb, int v_bits, const float* Pi_v, float* out, float* part,
                            int P, int H, int B, int S, float scale, cudaStream_t st) {
  switch (v_bits) {
    case 1: return launch_decode_kv<KBITS, 1>(A, k_plane, k_norm, k_cb, v_plane, v_norm, v_cb, Pi_v, out, part, P, H, B, S, scale, st);
    case 2: return launch_decode_kv<KBITS, 2>(A, k_plane, k_norm, k_cb, v_plane, v_norm, v_cb, Pi_v, out, part, P, H, B, S, scale, st);
    default: return launch_decode_kv<KBITS, 3>(A, k_plane, k_norm, k_cb, v_plane, v_norm, v_cb, Pi_v, out, part, P, H, B, S, scale, st);
  }
}

}  // namespace

size_t decode_part_floats(int P, int B, int S) {
  // at most ceil(S / 256) chunks of (max, sum, acc[128]) per query
  return static_cast<size_t>(P) * B * ((static_cast<size_t>(S) + 255) / 256) * kPart;
}

cudaError_t launch_decode_mse(const float* A, const uint8_t* k_plane, const uint16_t* k_norm,
                              const float* k_cb, int k_bits, const uint8_t* v_plane,
                              const uint16_t* v_norm, const float* v_cb, int v_bits,
                              const float* Pi_v, float* out, float* part, int P, int H, int B, int S,
                              float scale, cudaStream_t st) {
  switch (k_bits) {
    case 1: return launch_decode_k<1>(A, k_plane, k_norm, k_cb, v_plane, v_norm, v_cb, v_bits, Pi_v, out, part, P, H, B, S, scale, st);
    case 2: return launch_decode_k<2>(A, k_plane, k_norm, k_cb, v_plane, v_norm, v_cb, v_bits, Pi_v, out, part, P, H, B, S, scale, st);
    default: return launch_decode_k<3>(A, k_plane, k_norm, k_cb, v_plane, v_norm, v_cb, v_bits, Pi_v, out, part, P, H, B, S, scale, st);
  }
}

}  // namespace tq
