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
#include <cmath>
#include <vector>

#include "tq_internal.cuh"

namespace tq {
namespace {

constexpr int kMaxD = 128;          // compressor kernel head dimension limit
constexpr int kKeysPerCta = 64;

// One CTA of D threads (thread d owns coordinate d) walks kKeysPerCta keys.
// Pi and S_mat of the head sit in shared memory with rows padded to D+1 floats,
// so "thread d reads row d" and "thread j reads column j" are both free of bank
// conflicts.
__global__ void __launch_bounds__(kMaxD)
compress_kernel(const float* __restrict__ keys, const float* __restrict__ Pi,
                const float* __restrict__ Sm, const float* __restrict__ codebook, int C,
                uint8_t* __restrict__ K_idx, int8_t* __restrict__ signs,
                float* __restrict__ gamma_f32, uint16_t* __restrict__ gamma_f16, int H, int S,
                int D) {
  extern __shared__ float sm[];
  const int ld = D + 1;
  float* sPi = sm;                 // [D][D+1]
  float* sS = sPi + D * ld;        // [D][D+1]
  float* sK = sS + D * ld;         // [D]   current key
  float* sV = sK + D;              // [D]   c[idx] of the current key, then r
  float* sCb = sV + D;             // [256] codebook
  float* sRed = sCb + 256;         // [32]  warp partial sums

  const int p = blockIdx.y;
  const int h = p % H;
  const int d = threadIdx.x;
  const float* Pih = Pi + static_cast<size_t>(h) * D * D;
  const float* Sh = Sm + static_cast<size_t>(h) * D * D;
  for (int e = threadIdx.x; e < D * D; e += blockDim.x) {
    const int r = e / D, c = e % D;
    sPi[r * ld + c] = Pih[e];
    sS[r * ld + c] = Sh[e];
  }
  for (int e = threadIdx.x; e < C; e += blockDim.x) sCb[e] = codebook[e];
  __syncthreads();

  const int s_begin = blockIdx.x * kKeysPerCta;
  const int s_end = min(S, s_begin + kKeysPerCta);
  for (int s = s_begin; s < s_end; ++s) {
    const size_t key = static_cast<size_t>(p) * S + s;
    sK[d] = keys[key * D + d];
    __syncthreads();
    // y_d = <Pi row d, k>; idx_d = number of midpoints strictly below y_d
    float y = 0.f;
    for (int j = 0; j < D; ++j) y = fmaf(sPi[d * ld + j], sK[j], y);
    int idx = 0;
    for (int k = 0; k + 1 < C; ++k) idx += (y > 0.5f * (sCb[k] + sCb[k + 1])) ? 1 : 0;
    sV[d] = sCb[idx];
    __syncthreads();
    // r_j = k_j - sum_d Pi[d][j] c[idx_d]   (thread d plays j here)
    float rec = 0.f;
    for (int i = 0; i < D; ++i) rec = fmaf(sPi[i * ld + d], sV[i], rec);
    const float r = sK[d] - rec;
    __syncthreads();
    sV[d] = r;
    __syncthreads();
    // z_d = <S_mat row d, r>; sigma_d = +1 when z_d >= 0
    float z = 0.f;
    for (int j = 0; j < D; ++j) z = fmaf(sS[d * ld + j], sV[j], z);
    // gamma = ||r||: warp sums then one warp folds them
    float sq = r * r;
    for (int o = 16; o > 0; o >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, o);
    if ((d & 31) == 0) sRed[d >> 5] = sq;
    K_idx[key * D + d] = static_cast<uint8_t>(idx);
    signs[key * D + d] = z >= 0.f ? int8_t(1) : int8_t(-1);
    __syncthreads();
    if (d == 0) {
      float tot = 0.f;
      for (int w = 0; w < (D + 31) / 32; ++w) tot += sRed[w];
      const float g = sqrtf(tot);
      if (gamma_f32) gamma_f32[key] = g;
      if (gamma_f16) gamma_f16[key] = __half_as_ushort(__float2half_rn(g));
    }
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
  if (D < 1 || D > tq::kMaxD || D % 32 != 0) return D > 0 && D <= 256 ? TQ_ERR_UNSUPPORTED : TQ_ERR_INVALID_VALUE;
  const size_t smem = (2 * static_cast<size_t>(D) * (D + 1) + 2 * D + 256 + 32) * sizeof(float);
  cudaError_t e = cudaFuncSetAttribute(tq::compress_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return TQ_ERR_LAUNCH;
  dim3 grid(tq::ceil_div(S, tq::kKeysPerCta), P);
  tq::compress_kernel<<<grid, D, smem, stream>>>(keys, Pi, S_mat, codebook, C, K_idx, signs,
                                                 gamma_f32, gamma_f16, H, S, D);
  return cudaGetLastError() == cudaSuccess ? TQ_OK : TQ_ERR_LAUNCH;
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
