// Query transform A = Pi q, T = S_mat q for every query of every problem
// ("TurboQuant Attention in CUDA", riteshyadav.xyz, "Two kernels, two jobs":
// the first kernel; zededa.com v3 "Combined Transform": the rows of [Pi ; S_mat]
// against the query in one pass).
//
// One warp per output row: row r < D is row r of Pi (an entry of A), row r >= D
// is row r - D of S_mat (an entry of T).  The warp reads its row once, coalesced
// (lane l holds columns l, l+32, ...), multiplies it against up to kQ queries
// held in shared memory and reduces each product across the warp with
// shuffles.  Grid: (query tiles, problems, row chunks of 8), so even a single
// query spreads over 2D/8 CTAs and the transform costs about one memory round
// trip.  Summation order per output: lane-strided partial sums, then a
// butterfly; fp32 throughout.
//
// Randomized-Hadamard rotation (hsigns != null; "TurboQuant: Rotate-then-Quantize KV
// Caches at 3 Bits", kanthi.in §2-§3 RandomizedHadamard): A = H diag(s) q with H the
// orthonormal Walsh-Hadamard matrix, O(D log D) instead of a dense row per output.
// Slice z = 0 of the grid multiplies its query tile by s in shared memory and runs
// the log2(D) butterfly stages there (Sylvester order: within each block of 2h
// entries, (a, b) -> (a + b, a - b)), then scales by 1/sqrt(D); slices z >= 1 compute
// the rows of T = S_mat q as above.
#include "tq_internal.cuh"

namespace tq {
namespace {

constexpr int kQ = 8;        // queries per CTA
constexpr int kWarps = 8;    // output rows per CTA

__device__ __forceinline__ float load_q(const float* q, size_t i) { return q[i]; }
__device__ __forceinline__ float load_q(const __nv_bfloat16* q, size_t i) {
  return __bfloat162float(q[i]);
}

template <typename QT>
__global__ void __launch_bounds__(kWarps * 32)
prepare_kernel(const QT* __restrict__ Q, const float* __restrict__ Pi,
               const float* __restrict__ Sm, float* __restrict__ A, float* __restrict__ T,
               int H, int B, int D, uint16_t* __restrict__ Ybf, int NT, int qtiles,
               const float* __restrict__ hsigns) {
  extern __shared__ __align__(16) float sQ[];   // [kQ][D]
  // a scorer launched behind this grid may start its own prologue now (it reads A and T
  // only after this grid has completed)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int b0 = blockIdx.x * kQ;
  const int p = blockIdx.y;
  const int h = p % H;
  const int nq = min(kQ, B - b0);
  const size_t qbase = (static_cast<size_t>(p) * B + b0) * D;
  for (int e = threadIdx.x; e < kQ * D; e += blockDim.x) {
    sQ[e] = (e / D) < nq ? load_q(Q, qbase + e) : 0.f;
  }
  // one output: A or T of query b0 + q, coordinate d (and its tensor-core operand copy)
  auto put = [&](bool is_t, int q, int d, float v) {
    (is_t ? T : A)[qbase + static_cast<size_t>(q) * D + d] = v;
    if (Ybf != nullptr) {
      // tensor-core query operand: query b, K index k = d (A) or 128 + d (T), bf16 RNE,
      // 8-row x 16-byte core matrices (K-major, no swizzle) per (problem, query tile)
      const int b = b0 + q;
      const int qt = b / NT, n = b % NT, k = (is_t ? 128 : 0) + d;
      const size_t off = (static_cast<size_t>(p) * qtiles + qt) * NT * 256 +
                         ((k >> 3) * (NT >> 3) + (n >> 3)) * 64 + (n & 7) * 8 + (k & 7);
      Ybf[off] = __bfloat16_as_ushort(__float2bfloat16_rn(v));
    }
  };
  if (hsigns != nullptr && blockIdx.z == 0) {
    const float* sg = hsigns + static_cast<size_t>(h) * D;
    for (int e = threadIdx.x; e < kQ * D; e += blockDim.x) sQ[e] *= __ldg(sg + e % D);
    const int half = D >> 1;
    for (int hs = 1; hs < D; hs <<= 1) {
      __syncthreads();
      for (int e = threadIdx.x; e < kQ * half; e += blockDim.x) {
        const int q = e / half, i = e % half;
        const int j0 = (i / hs) * 2 * hs + i % hs;
        const float a = sQ[q * D + j0], b = sQ[q * D + j0 + hs];
        sQ[q * D + j0] = a + b;
        sQ[q * D + j0 + hs] = a - b;
      }
    }
    __syncthreads();
    const float scale = 1.0f / sqrtf(static_cast<float>(D));
    for (int e = threadIdx.x; e < nq * D; e += blockDim.x) put(false, e / D, e % D, sQ[e] * scale);
    return;
  }
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const int row = (hsigns != nullptr ? D + (blockIdx.z - 1) * kWarps : blockIdx.z * kWarps) + (threadIdx.x >> 5);
  if (row >= 2 * D) return;
  const bool is_t = row >= D;
  const int d = is_t ? row - D : row;
  const float* mrow = (is_t ? Sm : Pi) + (static_cast<size_t>(h) * D + d) * D;

  float acc[kQ];
#pragma unroll
  for (int q = 0; q < kQ; ++q) acc[q] = 0.f;
#pragma unroll 4
  for (int j = lane; j < D; j += 32) {
    const float m = __ldg(mrow + j);
#pragma unroll
    for (int q = 0; q < kQ; ++q) acc[q] = fmaf(m, sQ[q * D + j], acc[q]);
  }
#pragma unroll
  for (int q = 0; q < kQ; ++q) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc[q] += __shfl_xor_sync(0xffffffffu, acc[q], o);
  }
  if (lane < nq) {
    float v = acc[0];
#pragma unroll
    for (int q = 1; q < kQ; ++q)
      if (lane == q) v = acc[q];
    put(is_t, lane, d, v);
  }
}

}  // namespace

cudaError_t launch_prepare(const void* Q, tq_qtype qtype, const float* Pi, const float* S_mat,
                           float* A, float* T, int P, int H, int B, int D, cudaStream_t st,
                           uint16_t* Ybf, const float* hsigns) {
  // dense: 2D output rows in slices of kWarps; Hadamard: slice 0 for A, then the D rows of T
  dim3 grid(ceil_div(B, kQ), P, hsigns != nullptr ? 1 + ceil_div(D, kWarps) : ceil_div(2 * D, kWarps));
  const size_t smem = static_cast<size_t>(kQ) * D * sizeof(float);
  const int NT = mma_query_tile(B), qtiles = mma_query_tiles(B);
  if (D != 128) Ybf = nullptr;
  if (qtype == TQ_Q_BF16) {
    prepare_kernel<__nv_bfloat16><<<grid, kWarps * 32, smem, st>>>(
        static_cast<const __nv_bfloat16*>(Q), Pi, S_mat, A, T, H, B, D, Ybf, NT, qtiles, hsigns);
  } else {
    prepare_kernel<float><<<grid, kWarps * 32, smem, st>>>(static_cast<const float*>(Q), Pi,
                                                           S_mat, A, T, H, B, D, Ybf, NT, qtiles,
                                                           hsigns);
  }
  return cudaGetLastError();
}

}  // namespace tq
