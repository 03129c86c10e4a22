// TurboQuant_prod compressor: the write side of the cache.
//
// Host helpers (run once per head dimension / per KV head, not per token):
//   tq_lloyd_max_codebook  Lloyd-Max centroids for one coordinate of a uniform
//                          unit vector in R^D ("TurboQuant: Rotate-then-Quantize
//                          KV Caches at 3 Bits", kanthi.in, §2 fact 1 and §3).
//   tq_haar_rotation       Pi from the sign-fixed QR factor of a Gaussian matrix
//                          (same chapter, §3, HaarRotation).
// Device kernel:
//   tq_compress_keys       per key k: y = Pi k, idx = nearest centroid (midpoint
//                          search, ties to the lower index), r = k - Pi^T c[idx],
//                          sigma = sign(S_mat r) with sign(0) = +1, gamma = ||r||
//                          (same chapter §3 TurboQuantProd; zededa.com Theorem 2).
//
// The kernel computes in fp32: y, r and S_mat r carry fp32 rounding, so a
// coordinate within ~1e-6 of a cell edge (or an S_mat r entry within ~1e-6 of
// zero) may land on the other side than an exact evaluation would put it.
//
// One store pass (the chapter's §8 "Kernel checklist": rotate, search the midpoints,
// pack the bits and write the norm in the same kernel): each CTA takes tiles of KT
// keys and runs the three D x D products of a tile as register-tiled fp32 products
// fed from shared memory -- Y = K Pi^T, R = K - C(idx) Pi, Z = R S_mat^T -- with the
// per-key steps in between (cell search, residual, sign, norm).  A group of LPO
// lanes (16 for D <= 128, else 32) shares 4 keys of the tile, and lane l of a group
// owns the output columns l, l + LPO, ...: each loaded matrix value feeds 4 keys and
// each key value (one broadcast read of 4 keys from the transposed tile) feeds D / LPO
// columns.  A matrix row sits in shared memory with stride D + 1, so a group's rows
// (GEMMs 1 and 3) or columns (GEMM 2) fall in different banks.  For D <= 128, Pi and
// S_mat stay resident for the CTA's life; for larger D they stream through shared
// memory 128 rows at a time.  Each CTA takes one contiguous range of the keys, so the
// last partial tile occupies only the warps it needs.  The tile's codes are staged as
// bytes and packed into the little-endian bit stream by whole words; each 32-bit word
// of a sign row is one warp vote.
#include <cmath>
#include <vector>

#include "tq_internal.cuh"

namespace tq {
namespace {

template <int D>
struct CmpCfg {
  static constexpr bool kResident = D <= 128;
  static constexpr int NW = 8;                            // warps
  static constexpr int kThreads = 32 * NW;
  // a group of LPO lanes shares 4 keys and owns D / LPO output columns a lane:
  // lane l takes columns l % LPO + LPO o and keys 4 (l / LPO) .. +3 of the warp's
  static constexpr int LPO = D <= 128 ? 16 : 32;
  static constexpr int KG = 4;                            // keys per lane group
  static constexpr int KW = KG * (32 / LPO);              // keys per warp
  static constexpr int KT = NW * KW;                      // keys per tile
  static constexpr int NO = D / LPO;                      // output columns per lane
  static constexpr int LD = D + 1;                        // row stride of a staged matrix
  static constexpr int LT = KT + 4;                       // row stride of a transposed tile
  static constexpr int MR = D < 128 ? D : 128;            // matrix rows staged at once
  static constexpr int NCH = (D + MR - 1) / MR;           // row chunks of a matrix
  // floats: matrices, key tile, value/residual tile (both transposed, [D][LT]), edges;
  // then the codes (bytes)
  static constexpr size_t kMatFloats = kResident ? 2 * static_cast<size_t>(D) * LD : static_cast<size_t>(MR) * LD;
  static constexpr size_t kSmem =
      (kMatFloats + 2 * static_cast<size_t>(D) * LT + 256) * sizeof(float) + static_cast<size_t>(KT) * D;
};

// rows r0 .. r0+n-1 of a [D][D] matrix into shared memory with stride D + 1.  Each
// thread issues 16 vector loads before it stores any, so the rows cost a few round
// trips to L2 rather than one per vector.
template <int D>
__device__ __forceinline__ void stage_rows(float* dst, const float* __restrict__ src, int r0, int n) {
  constexpr int LD = CmpCfg<D>::LD, NT = CmpCfg<D>::kThreads, BATCH = 16;
  const int total = n * (D / 4);
  for (int e0 = 0; e0 < total; e0 += NT * BATCH) {
    float4 v[BATCH];
#pragma unroll
    for (int b = 0; b < BATCH; ++b) {
      const int e = e0 + b * NT + static_cast<int>(threadIdx.x);
      if (e < total) v[b] = __ldg(reinterpret_cast<const float4*>(src + static_cast<size_t>(r0 + e / (D / 4)) * D) + e % (D / 4));
    }
#pragma unroll
    for (int b = 0; b < BATCH; ++b) {
      const int e = e0 + b * NT + static_cast<int>(threadIdx.x);
      if (e < total) {
        float* d = dst + (e / (D / 4)) * LD + 4 * (e % (D / 4));
        d[0] = v[b].x; d[1] = v[b].y; d[2] = v[b].z; d[3] = v[b].w;
      }
    }
  }
}

// acc[k][o] += v.k * m for the lane group's 4 keys
template <int NO>
__device__ __forceinline__ void fma4(float (&acc)[4][NO], int o, const float4& v, float m) {
  acc[0][o] = fmaf(v.x, m, acc[0][o]);
  acc[1][o] = fmaf(v.y, m, acc[1][o]);
  acc[2][o] = fmaf(v.z, m, acc[2][o]);
  acc[3][o] = fmaf(v.w, m, acc[3][o]);
}

// PACKED: write the code plane, the sign plane and fp16 gamma; otherwise one byte per
// code and per sign and gamma as fp32 or fp16.
template <int D, bool PACKED>
__global__ void __launch_bounds__(CmpCfg<D>::kThreads, 1)
compress_tile_kernel(const float* __restrict__ keys, const float* __restrict__ Pi,
                     const float* __restrict__ Sm, const float* __restrict__ codebook, int C, int bits,
                     uint8_t* __restrict__ out_idx, uint8_t* __restrict__ out_sign,
                     float* __restrict__ gamma_f32, uint16_t* __restrict__ gamma_f16, int P, int H, int S) {
  using Cf = CmpCfg<D>;
  constexpr int KG = Cf::KG, KT = Cf::KT, NO = Cf::NO, LD = Cf::LD, MR = Cf::MR, LT = Cf::LT, LPO = Cf::LPO;
  extern __shared__ __align__(16) float smem[];
  float* sMat = smem;                                     // Pi (and S_mat) rows, stride LD
  float* sK = sMat + Cf::kMatFloats;                      // [D][LT] keys, transposed
  float* sV = sK + D * LT;                                // [D][LT] c(idx), then r, transposed
  float* sEdge = sV + D * LT;                             // [C-1] midpoints (256 floats)
  uint8_t* sCode = reinterpret_cast<uint8_t*>(sEdge + 256);   // [KT][D]
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int cl = lane % LPO;                              // first output column of the lane
  const int kb = warp * Cf::KW + KG * (lane / LPO);       // the lane group's first key in a tile
  // this CTA's keys: one contiguous range of the P*S keys laid end to end, cut into
  // tiles that do not cross a problem
  const int64_t total = static_cast<int64_t>(P) * S;
  const int64_t per = (total + gridDim.x - 1) / gridDim.x;
  const int64_t g_end = min(total, (static_cast<int64_t>(blockIdx.x) + 1) * per);
  for (int e = tid; e + 1 < C; e += Cf::kThreads) sEdge[e] = 0.5f * (__ldg(codebook + e) + __ldg(codebook + e + 1));
  int h_loaded = -1;
  for (int64_t g = static_cast<int64_t>(blockIdx.x) * per; g < g_end;) {
    const int p = static_cast<int>(g / S);
    const int s0 = static_cast<int>(g - static_cast<int64_t>(p) * S);
    const int n = static_cast<int>(min(static_cast<int64_t>(KT), min(g_end - g, static_cast<int64_t>(S - s0))));
    g += n;
    const int h = p % H;
    const float* Pih = Pi + static_cast<size_t>(h) * D * D;
    const float* Sh = Sm + static_cast<size_t>(h) * D * D;
    const bool active = warp * Cf::KW < n;                // the warp has a key of this tile
    __syncthreads();                      // the previous tile is done with every buffer
    if (Cf::kResident && h != h_loaded) {
      stage_rows<D>(sMat, Pih, 0, D);
      stage_rows<D>(sMat + D * LD, Sh, 0, D);
      h_loaded = h;
    }
    // the key tile, transposed (sK[j][s]); lane-consecutive keys; keys past n are zero;
    // every load of the thread is in flight before its first store
    {
      constexpr int NV = KT * (D / 4) / Cf::kThreads;     // vectors a thread
      static_assert(KT * (D / 4) % Cf::kThreads == 0, "key tile split");
      float4 v[NV];
#pragma unroll
      for (int b = 0; b < NV; ++b) {
        const int e = tid + b * Cf::kThreads, s = e % KT, c4 = e / KT;
        v[b] = s < n ? __ldg(reinterpret_cast<const float4*>(keys + (static_cast<size_t>(p) * S + s0 + s) * D) + c4)
                     : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int b = 0; b < NV; ++b) {
        const int e = tid + b * Cf::kThreads, s = e % KT, c4 = e / KT;
        sK[(4 * c4) * LT + s] = v[b].x;
        sK[(4 * c4 + 1) * LT + s] = v[b].y;
        sK[(4 * c4 + 2) * LT + s] = v[b].z;
        sK[(4 * c4 + 3) * LT + s] = v[b].w;
      }
    }
    float acc[KG][NO];

    // ---- GEMM 1: y[s][d] = sum_j K[s][j] Pi[d][j], the lane's d = cl + LPO o ----
#pragma unroll
    for (int k = 0; k < KG; ++k)
#pragma unroll
      for (int o = 0; o < NO; ++o) acc[k][o] = 0.f;
#pragma unroll
    for (int c = 0; c < Cf::NCH; ++c) {
      const int nrows = D - c * MR < MR ? D - c * MR : MR;   // rows of this chunk
      if (!Cf::kResident) {
        __syncthreads();
        stage_rows<D>(sMat, Pih, c * MR, nrows);
      }
      __syncthreads();
      if (active) {
        const float* m = sMat + cl * LD;
#pragma unroll 4
        for (int j = 0; j < D; ++j) {
          const float4 kv = *reinterpret_cast<const float4*>(sK + j * LT + kb);
#pragma unroll
          for (int oc = 0; oc < nrows / LPO; ++oc) fma4(acc, c * (MR / LPO) + oc, kv, m[oc * LPO * LD + j]);
        }
      }
    }
    // ---- cells: idx = number of midpoints strictly below y; V = c(idx) ----
    if (active) {
#pragma unroll
      for (int k = 0; k < KG; ++k) {
#pragma unroll
        for (int o = 0; o < NO; ++o) {
          const float y = acc[k][o];
          int lo = 0, hi = C - 1;                 // lower bound of y among the C-1 edges
          while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (sEdge[mid] < y) lo = mid + 1; else hi = mid;
          }
          const int d = cl + LPO * o;
          sCode[(kb + k) * D + d] = static_cast<uint8_t>(lo);
          sV[d * LT + kb + k] = __ldg(codebook + lo);
        }
      }
    }
    __syncwarp();

    // ---- GEMM 2: rec[s][j] = sum_d V[s][d] Pi[d][j], the lane's j = cl + LPO o ----
#pragma unroll
    for (int k = 0; k < KG; ++k)
#pragma unroll
      for (int o = 0; o < NO; ++o) acc[k][o] = 0.f;
#pragma unroll
    for (int c = 0; c < Cf::NCH; ++c) {
      const int nrows = D - c * MR < MR ? D - c * MR : MR;
      if (!Cf::kResident) {
        __syncthreads();
        stage_rows<D>(sMat, Pih, c * MR, nrows);
        __syncthreads();
      }
      if (active) {
#pragma unroll 4
        for (int dl = 0; dl < nrows; ++dl) {
          const int d = c * MR + dl;
          const float4 vv = *reinterpret_cast<const float4*>(sV + d * LT + kb);
          const float* m = sMat + dl * LD + cl;                 // columns cl + LPO o
#pragma unroll
          for (int o = 0; o < NO; ++o) fma4(acc, o, vv, m[LPO * o]);
        }
      }
    }
    // r = k - rec (kept in acc), gamma^2 per key (a sum over the lane group)
    float g2[KG];
#pragma unroll
    for (int k = 0; k < KG; ++k) {
      float sq = 0.f;
#pragma unroll
      for (int o = 0; o < NO; ++o) {
        const float r = sK[(cl + LPO * o) * LT + kb + k] - acc[k][o];
        acc[k][o] = r;
        sq = fmaf(r, r, sq);
      }
#pragma unroll
      for (int off = LPO / 2; off > 0; off >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, off);
      g2[k] = sq;
    }
    __syncwarp();                           // every lane is done reading V
#pragma unroll
    for (int k = 0; k < KG; ++k)
#pragma unroll
      for (int o = 0; o < NO; ++o) sV[(cl + LPO * o) * LT + kb + k] = acc[k][o];
    __syncwarp();

    // ---- GEMM 3: z[s][d] = sum_j R[s][j] S_mat[d][j], the lane's d = cl + LPO o ----
#pragma unroll
    for (int k = 0; k < KG; ++k)
#pragma unroll
      for (int o = 0; o < NO; ++o) acc[k][o] = 0.f;
#pragma unroll
    for (int c = 0; c < Cf::NCH; ++c) {
      const int nrows = D - c * MR < MR ? D - c * MR : MR;
      if (!Cf::kResident) {
        __syncthreads();
        stage_rows<D>(sMat, Sh, c * MR, nrows);
        __syncthreads();
      }
      if (active) {
        const float* m = sMat + (Cf::kResident ? D * LD : 0) + cl * LD;
#pragma unroll 4
        for (int j = 0; j < D; ++j) {
          const float4 rv = *reinterpret_cast<const float4*>(sV + j * LT + kb);
#pragma unroll
          for (int oc = 0; oc < nrows / LPO; ++oc) fma4(acc, c * (MR / LPO) + oc, rv, m[oc * LPO * LD + j]);
        }
      }
    }
    // ---- signs and gamma ----
    // the sign word of columns 32 w .. 32 w + 31: the lane group's votes on o = (32 w) / LPO
    // (and, with 16-lane groups, o + 1 for columns 32 w + 16 ..)
#pragma unroll
    for (int k = 0; k < KG; ++k) {
      const int s = s0 + kb + k;
      const bool live = kb + k < n;
      const size_t key = static_cast<size_t>(p) * S + s;
      if constexpr (PACKED) {
        uint32_t vote[NO];
#pragma unroll
        for (int o = 0; o < NO; ++o) vote[o] = __ballot_sync(0xffffffffu, acc[k][o] >= 0.f);
        const int gshift = LPO == 16 ? 16 * (lane / 16) : 0;
#pragma unroll
        for (int w = 0; w < D / 32; ++w) {
          uint32_t word;
          if (LPO == 32) {
            word = vote[w];
          } else {
            word = ((vote[2 * w] >> gshift) & 0xffffu) | (((vote[2 * w + 1] >> gshift) & 0xffffu) << 16);
          }
          if (cl == w && live) reinterpret_cast<uint32_t*>(out_sign + key * (D / 8))[w] = word;
        }
      } else {
#pragma unroll
        for (int o = 0; o < NO; ++o)
          if (live) reinterpret_cast<int8_t*>(out_sign)[key * D + cl + LPO * o] = acc[k][o] >= 0.f ? int8_t(1) : int8_t(-1);
      }
      if (cl == 0 && live) {
        const float gm = sqrtf(g2[k]);
        if (gamma_f32) gamma_f32[key] = gm;
        if (gamma_f16) gamma_f16[key] = __half_as_ushort(__float2half_rn(gm));
      }
    }
    __syncthreads();                        // the tile's codes are staged
    // ---- codes: bytes, or the little-endian bit stream by whole 32-bit words ----
    const int live_keys = n;
    if constexpr (PACKED) {
      const int wpk = D * bits / 32;                      // words per key row
      for (int e = tid; e < live_keys * wpk; e += Cf::kThreads) {
        const int s = e / wpk, wi = e % wpk;
        const uint8_t* cs = sCode + s * D;
        const int b0 = 32 * wi;                           // first stream bit of the word
        uint32_t w = 0u;
        for (int d = b0 / bits; d * bits < b0 + 32; ++d) {
          const int sh = d * bits - b0;                   // may be negative for a straddling code
          const uint32_t v = cs[d];
          w |= sh >= 0 ? (v << sh) : (v >> -sh);
        }
        reinterpret_cast<uint32_t*>(out_idx + (static_cast<size_t>(p) * S + s0 + s) * (D * bits / 8))[wi] = w;
      }
    } else {
      for (int e = tid; e < live_keys * (D / 4); e += Cf::kThreads) {
        const int s = e / (D / 4), c4 = e % (D / 4);
        reinterpret_cast<uint32_t*>(out_idx + (static_cast<size_t>(p) * S + s0 + s) * D)[c4] =
            reinterpret_cast<const uint32_t*>(sCode + s * D)[c4];
      }
    }
  }
}

template <int D, bool PACKED>
cudaError_t launch_compress_d(const float* keys, const float* Pi, const float* S_mat, const float* codebook,
                              int C, int bits, uint8_t* out_idx, uint8_t* out_sign, float* g32,
                              uint16_t* g16, int P, int H, int S, cudaStream_t st) {
  auto kernel = compress_tile_kernel<D, PACKED>;
  constexpr size_t smem = CmpCfg<D>::kSmem;
  static std::atomic<uint64_t> configured{0};
  static std::atomic<int> sms_cache[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (!(configured.load(std::memory_order_acquire) & bit)) {
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    sms_cache[dev & 63].store(sms, std::memory_order_relaxed);
    configured.fetch_or(bit, std::memory_order_acq_rel);
  }
  const int64_t tiles = (static_cast<int64_t>(P) * S + CmpCfg<D>::KT - 1) / CmpCfg<D>::KT;
  const int sms = sms_cache[dev & 63].load(std::memory_order_relaxed);
  const int grid = static_cast<int>(tiles < sms ? tiles : sms);
  kernel<<<grid, CmpCfg<D>::kThreads, smem, st>>>(keys, Pi, S_mat, codebook, C, bits, out_idx, out_sign, g32, g16, P, H, S);
  return cudaGetLastError();
}

template <bool PACKED>
cudaError_t launch_compress(const float* keys, const float* Pi, const float* S_mat, const float* codebook,
                            int C, int bits, uint8_t* out_idx, uint8_t* out_sign, float* g32, uint16_t* g16,
                            int P, int H, int S, int D, cudaStream_t st) {
  switch (D) {
    case 32: return launch_compress_d<32, PACKED>(keys, Pi, S_mat, codebook, C, bits, out_idx, out_sign, g32, g16, P, H, S, st);
    case 64: return launch_compress_d<64, PACKED>(keys, Pi, S_mat, codebook, C, bits, out_idx, out_sign, g32, g16, P, H, S, st);
    case 96: return launch_compress_d<96, PACKED>(keys, Pi, S_mat, codebook, C, bits, out_idx, out_sign, g32, g16, P, H, S, st);
    case 128: return launch_compress_d<128, PACKED>(keys, Pi, S_mat, codebook, C, bits, out_idx, out_sign, g32, g16, P, H, S, st);
    case 160: return launch_compress_d<160, PACKED>(keys, Pi, S_mat, codebook, C, bits, out_idx, out_sign, g32, g16, P, H, S, st);
    case 192: return launch_compress_d<192, PACKED>(keys, Pi, S_mat, codebook, C, bits, out_idx, out_sign, g32, g16, P, H, S, st);
    case 224: return launch_compress_d<224, PACKED>(keys, Pi, S_mat, codebook, C, bits, out_idx, out_sign, g32, g16, P, H, S, st);
    default: return launch_compress_d<256, PACKED>(keys, Pi, S_mat, codebook, C, bits, out_idx, out_sign, g32, g16, P, H, S, st);
  }
}

}  // namespace
}  // namespace tq

extern "C" {

tq_status tq_compress_keys(const float* keys, const float* Pi, const float* S_mat,
                           const float* codebook, int C, uint8_t* K_idx, int8_t* signs,
                           float* gamma_f32, uint16_t* gamma_f16, int P, int H, int S, int D,
                           cudaStream_t stream) {
  const void* req[] = {keys, Pi, S_mat, codebook, K_idx, signs};
  for (const void* q : req)
    if (q == nullptr) return TQ_ERR_INVALID_VALUE;
  if ((gamma_f32 == nullptr) == (gamma_f16 == nullptr)) return TQ_ERR_INVALID_VALUE;
  const void* all[] = {keys, Pi, S_mat, codebook, K_idx, signs,
                       gamma_f32 ? static_cast<const void*>(gamma_f32) : gamma_f16};
  for (const void* q : all)
    if (reinterpret_cast<uintptr_t>(q) & 15u) return TQ_ERR_MISALIGNED;
  if (P < 1 || P > 65535 || H < 1 || H > P || S < 1 || C < 1 || C > 256) return TQ_ERR_INVALID_VALUE;
  if (D < 1 || D > 256) return TQ_ERR_INVALID_VALUE;
  if (D % 32 != 0) return TQ_ERR_UNSUPPORTED;
  cudaError_t e = tq::launch_compress<false>(keys, Pi, S_mat, codebook, C, 8, K_idx,
                                             reinterpret_cast<uint8_t*>(signs), gamma_f32, gamma_f16, P, H, S, D,
                                             stream);
  return e == cudaSuccess ? TQ_OK : TQ_ERR_LAUNCH;
}

tq_status tq_compress_keys_packed(const float* keys, const float* Pi, const float* S_mat,
                                  const float* codebook, int idx_bits, uint8_t* idx_plane,
                                  uint8_t* sign_plane, uint16_t* gamma_f16, int P, int H, int S, int D,
                                  cudaStream_t stream) {
  const void* all[] = {keys, Pi, S_mat, codebook, idx_plane, sign_plane, gamma_f16};
  for (const void* q : all)
    if (q == nullptr) return TQ_ERR_INVALID_VALUE;
  for (const void* q : all)
    if (reinterpret_cast<uintptr_t>(q) & 15u) return TQ_ERR_MISALIGNED;
  if (P < 1 || P > 65535 || H < 1 || H > P || S < 1 || idx_bits < 1 || idx_bits > 3) return TQ_ERR_INVALID_VALUE;
  if (D < 1 || D > 256) return TQ_ERR_INVALID_VALUE;
  if (D % 32 != 0) return TQ_ERR_UNSUPPORTED;
  cudaError_t e = tq::launch_compress<true>(keys, Pi, S_mat, codebook, 1 << idx_bits, idx_bits, idx_plane,
                                            sign_plane, nullptr, gamma_f16, P, H, S, D, stream);
  return e == cudaSuccess ? TQ_OK : TQ_ERR_LAUNCH;
}

tq_status tq_lloyd_max_codebook(int D, int mse_bits, int grid_points, int iterations,
                                float* centroids) {
  if (centroids == nullptr || D < 3 || mse_bits < 1 || mse_bits > 8 || grid_points < 3 ||
      iterations < 0)
    return TQ_ERR_INVALID_VALUE;
  const int C = 1 << mse_bits;
  const int n = grid_points;
  // Prefix sums of the (unnormalised) density and of x * density over the grid
  // x_i = -1 + 2 i / (n-1): a cell's mass and first moment are then two lookups,
  // so each Lloyd round costs O(C log n) instead of a pass over the grid.
  std::vector<double> W(n + 1, 0.0), M(n + 1, 0.0);
  const double ex = (D - 3) / 2.0;
  for (int i = 0; i < n; ++i) {
    const double x = -1.0 + 2.0 * i / (n - 1);
    const double base = 1.0 - x * x;
    const double w = base > 0.0 ? std::pow(base, ex) : (ex == 0.0 ? 1.0 : 0.0);
    W[i + 1] = W[i] + w;
    M[i + 1] = M[i] + w * x;
  }
  // number of grid points x_i <= e (points on an edge belong to the lower cell)
  auto count_le = [n](double e) {
    long lo = 0, hi = n;   // invariant: x_i <= e for i < lo, x_i > e for i >= hi
    while (lo < hi) {
      const long mid = (lo + hi) / 2;
      if (-1.0 + 2.0 * mid / (n - 1) <= e) lo = mid + 1; else hi = mid;
    }
    return lo;
  };
  std::vector<double> c(C), bound(C + 1);
  for (int k = 0; k < C; ++k) c[k] = (-2.0 + 4.0 * k / (C - 1)) / std::sqrt(static_cast<double>(D));
  for (int it = 0; it < iterations; ++it) {
    bound[0] = 0;
    bound[C] = n;
    for (int k = 0; k + 1 < C; ++k) bound[k + 1] = static_cast<double>(count_le(0.5 * (c[k] + c[k + 1])));
    for (int k = 0; k < C; ++k) {
      const long a = static_cast<long>(bound[k]), b = static_cast<long>(bound[k + 1]);
      const double mass = W[b] - W[a];
      if (mass > 0.0) c[k] = (M[b] - M[a]) / mass;
    }
  }
  for (int k = 0; k < C; ++k) centroids[k] = static_cast<float>(c[k]);
  return TQ_OK;
}

tq_status tq_haar_rotation(const double* G, int D, float* Pi) {
  if (G == nullptr || Pi == nullptr || D < 1 || D > 4096) return TQ_ERR_INVALID_VALUE;
  // Householder QR of G (column-major working copy), Q accumulated explicitly,
  // then column j of Q multiplied by the sign of R[j][j] (zero counts as +).
  const int n = D;
  std::vector<double> R(static_cast<size_t>(n) * n), Q(static_cast<size_t>(n) * n, 0.0);
  auto r = [&](int i, int j) -> double& { return R[static_cast<size_t>(j) * n + i]; };
  auto q = [&](int i, int j) -> double& { return Q[static_cast<size_t>(j) * n + i]; };
  for (int i = 0; i < n; ++i)
    for (int j = 0; j < n; ++j) r(i, j) = G[static_cast<size_t>(i) * n + j];
  for (int i = 0; i < n; ++i) q(i, i) = 1.0;
  std::vector<double> v(n);
  for (int k = 0; k < n; ++k) {
    double norm2 = 0.0;
    for (int i = k; i < n; ++i) norm2 += r(i, k) * r(i, k);
    const double norm = std::sqrt(norm2);
    if (norm == 0.0) continue;
    const double alpha = r(k, k) > 0.0 ? -norm : norm;       // reflect away from x to avoid cancellation
    for (int i = 0; i < n; ++i) v[i] = 0.0;
    for (int i = k; i < n; ++i) v[i] = r(i, k);
    v[k] -= alpha;
    double vv = 0.0;
    for (int i = k; i < n; ++i) vv += v[i] * v[i];
    if (vv == 0.0) continue;
    for (int j = k; j < n; ++j) {                               // R <- (I - 2vv^T/v^Tv) R
      double dot = 0.0;
      for (int i = k; i < n; ++i) dot += v[i] * r(i, j);
      const double f = 2.0 * dot / vv;
      for (int i = k; i < n; ++i) r(i, j) -= f * v[i];
    }
    for (int i = 0; i < n; ++i) {                               // Q <- Q (I - 2vv^T/v^Tv)
      double dot = 0.0;
      for (int l = k; l < n; ++l) dot += q(i, l) * v[l];
      const double f = 2.0 * dot / vv;
      for (int l = k; l < n; ++l) q(i, l) -= f * v[l];
    }
  }
  for (int j = 0; j < n; ++j) {
    const double sgn = r(j, j) < 0.0 ? -1.0 : 1.0;
    for (int i = 0; i < n; ++i) Pi[static_cast<size_t>(i) * n + j] = static_cast<float>(q(i, j) * sgn);
  }
  return TQ_OK;
}

}  // extern "C"

namespace tq {
cudaError_t take_faults_compress(unsigned int* bits) { return take_unit_faults(bits); }
}  // namespace tq
