// Query transform A = Pi q, T = S_mat q for every query of every problem
// ("TurboQuant Attention in CUDA", riteshyadav.xyz, "Two kernels, two jobs":
// the first kernel; zededa.com v3 "Combined Transform": both products from one
// pass over the query).
//
// One CTA per (problem, tile of up to kQ queries), 2*D threads: thread t owns
// output coordinate d = t % D of A (t < D) or of T (t >= D) for every query of
// the tile.  It streams its own row of Pi or S_mat with independent 16-byte
// loads (the D x D matrix stays in L1/L2 across CTAs) and reads the queries as
// shared-memory broadcasts, so the whole transform is a handful of memory
// round trips regardless of B.  D % 4 == 0 uses the vector path; other D (the
// worked example has D = 2) take the scalar loop.
#include "tq_internal.cuh"

namespace tq {
namespace {

constexpr int kQ = 8;       // queries per CTA

__device__ __forceinline__ float load_q(const float* q, size_t i) { return q[i]; }
__device__ __forceinline__ float load_q(const __nv_bfloat16* q, size_t i) {
  return __bfloat162float(q[i]);
}

template <typename QT, bool VEC4>
__global__ void __launch_bounds__(512)
prepare_kernel(const QT* __restrict__ Q, const float* __restrict__ Pi,
               const float* __restrict__ Sm, float* __restrict__ A, float* __restrict__ T,
               int H, int B, int D) {
  extern __shared__ __align__(16) float sQ[];   // [kQ][D]
  const int p = blockIdx.y;
  const int h = p % H;
  const int b0 = blockIdx.x * kQ;
  const int nq = min(kQ, B - b0);
  const size_t qbase = (static_cast<size_t>(p) * B + b0) * D;
  for (int e = threadIdx.x; e < kQ * D; e += blockDim.x) {
    const int q = e / D;
    sQ[e] = q < nq ? load_q(Q, qbase + e) : 0.f;
  }
  __syncthreads();
  const int t = threadIdx.x;
  if (t >= 2 * D) return;
  const int d = t % D;
  const float* row = (t < D ? Pi : Sm) + (static_cast<size_t>(h) * D + d) * D;
  float acc[kQ];
#pragma unroll
  for (int q = 0; q < kQ; ++q) acc[q] = 0.f;
  if constexpr (VEC4) {
    const float4* r4 = reinterpret_cast<const float4*>(row);
#pragma unroll 4
    for (int j4 = 0; j4 < D / 4; ++j4) {
      const float4 m = __ldg(r4 + j4);
#pragma unroll
      for (int q = 0; q < kQ; ++q) {
        const float4 x = *reinterpret_cast<const float4*>(sQ + q * D + 4 * j4);
        acc[q] = fmaf(m.x, x.x, acc[q]);
        acc[q] = fmaf(m.y, x.y, acc[q]);
        acc[q] = fmaf(m.z, x.z, acc[q]);
        acc[q] = fmaf(m.w, x.w, acc[q]);
      }
    }
  } else {
    for (int j = 0; j < D; ++j) {
      const float m = __ldg(row + j);
#pragma unroll
      for (int q = 0; q < kQ; ++q) acc[q] = fmaf(m, sQ[q * D + j], acc[q]);
    }
  }
  float* out = (t < D ? A : T) + qbase + d;
#pragma unroll
  for (int q = 0; q < kQ; ++q)
    if (q < nq) out[static_cast<size_t>(q) * D] = acc[q];
}

template <typename QT>
void launch_typed(const QT* Q, const float* Pi, const float* S_mat, float* A, float* T, int P,
                  int H, int B, int D, cudaStream_t st) {
  dim3 grid(ceil_div(B, kQ), P);
  const int threads = (2 * D + 31) / 32 * 32;
  const size_t smem = static_cast<size_t>(kQ) * D * sizeof(float);
  if (D % 4 == 0) {
    prepare_kernel<QT, true><<<grid, threads, smem, st>>>(Q, Pi, S_mat, A, T, H, B, D);
  } else {
    prepare_kernel<QT, false><<<grid, threads, smem, st>>>(Q, Pi, S_mat, A, T, H, B, D);
  }
}

}  // namespace

cudaError_t launch_prepare(const void* Q, tq_qtype qtype, const float* Pi, const float* S_mat,
                           float* A, float* T, int P, int H, int B, int D, cudaStream_t st) {
  if (qtype == TQ_Q_BF16) {
    launch_typed(static_cast<const __nv_bfloat16*>(Q), Pi, S_mat, A, T, P, H, B, D, st);
  } else {
    launch_typed(static_cast<const float*>(Q), Pi, S_mat, A, T, P, H, B, D, st);
  }
  return cudaGetLastError();
}

}  // namespace tq
