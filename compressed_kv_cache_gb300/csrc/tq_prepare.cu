// Query transform A = Pi q, T = S_mat q for every query of every problem
// ("TurboQuant Attention in CUDA", riteshyadav.xyz, "Two kernels, two jobs":
// the first kernel; zededa.com v3 "Combined Transform": both products from one
// pass over the query).
//
// One CTA computes 32 output coordinates (rows d of Pi and S_mat) for 8 queries
// of one problem.  The 32 rows of Pi and of S_mat are streamed through shared
// memory 64 columns at a time (coalesced row reads, padded rows so that the 32
// lanes of a warp read 32 different banks); each warp owns one query and each
// lane one output coordinate, so every thread keeps two fp32 sums.
#include "tq_internal.cuh"

namespace tq {
namespace {

constexpr int kRows = 32;   // output coordinates per CTA
constexpr int kQ = 8;       // queries per CTA (one per warp)
constexpr int kCols = 64;   // columns of Pi / S_mat staged per step

__device__ __forceinline__ float load_q(const float* q, size_t i) { return q[i]; }
__device__ __forceinline__ float load_q(const __nv_bfloat16* q, size_t i) {
  return __bfloat162float(q[i]);
}

template <typename QT>
__global__ void __launch_bounds__(kRows * kQ)
prepare_kernel(const QT* __restrict__ Q, const float* __restrict__ Pi,
               const float* __restrict__ Sm, float* __restrict__ A, float* __restrict__ T,
               int H, int B, int D) {
  __shared__ float sPi[kRows][kCols + 1];
  __shared__ float sS[kRows][kCols + 1];
  __shared__ float sQ[kQ][kCols];

  const int p = blockIdx.z;
  const int h = p % H;
  const int d0 = blockIdx.x * kRows;
  const int b0 = blockIdx.y * kQ;
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const float* Pih = Pi + static_cast<size_t>(h) * D * D;
  const float* Sh = Sm + static_cast<size_t>(h) * D * D;
  const size_t qbase = (static_cast<size_t>(p) * B + b0) * D;

  float a = 0.f, t = 0.f;
  for (int j0 = 0; j0 < D; j0 += kCols) {
    const int jn = min(kCols, D - j0);
    for (int e = threadIdx.x; e < kRows * kCols; e += blockDim.x) {
      const int r = e / kCols, c = e % kCols;
      float v = 0.f, u = 0.f;
      if (d0 + r < D && c < jn) {
        const size_t off = static_cast<size_t>(d0 + r) * D + j0 + c;
        v = Pih[off];
        u = Sh[off];
      }
      sPi[r][c] = v;
      sS[r][c] = u;
    }
    for (int e = threadIdx.x; e < kQ * kCols; e += blockDim.x) {
      const int r = e / kCols, c = e % kCols;
      float v = 0.f;
      if (b0 + r < B && c < jn) v = load_q(Q, qbase + static_cast<size_t>(r) * D + j0 + c);
      sQ[r][c] = v;
    }
    __syncthreads();
#pragma unroll 8
    for (int c = 0; c < jn; ++c) {
      const float q = sQ[warp][c];
      a = fmaf(sPi[lane][c], q, a);
      t = fmaf(sS[lane][c], q, t);
    }
    __syncthreads();
  }
  if (d0 + lane < D && b0 + warp < B) {
    const size_t o = (static_cast<size_t>(p) * B + b0 + warp) * D + d0 + lane;
    A[o] = a;
    T[o] = t;
  }
}

}  // namespace

cudaError_t launch_prepare(const void* Q, tq_qtype qtype, const float* Pi, const float* S_mat,
                           float* A, float* T, int P, int H, int B, int D, cudaStream_t st) {
  dim3 grid(ceil_div(D, kRows), ceil_div(B, kQ), P);
  dim3 block(kRows * kQ);
  if (qtype == TQ_Q_BF16) {
    prepare_kernel<__nv_bfloat16><<<grid, block, 0, st>>>(
        static_cast<const __nv_bfloat16*>(Q), Pi, S_mat, A, T, H, B, D);
  } else {
    prepare_kernel<float><<<grid, block, 0, st>>>(static_cast<const float*>(Q), Pi, S_mat, A, T,
                                                  H, B, D);
  }
  return cudaGetLastError();
}

}  // namespace tq
