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

// kShareSm only makes a second copy of the kernel, the one that runs ahead of a scorer
// that shares its SMs (it carries the largest shared-memory carveout; see launch_prepare).
// kR: output rows per warp (4 for grids of many problems, so that they fit in one wave).
template <typename QT, bool kShareSm, int kR>
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
  const int lane = threadIdx.x & 31;
  const bool hadamard_slice = hsigns != nullptr && blockIdx.z == 0;
  const int row0 = (hsigns != nullptr ? D + (static_cast<int>(blockIdx.z) - 1) * kWarps * kR
                                      : static_cast<int>(blockIdx.z) * kWarps * kR) +
                   (threadIdx.x >> 5) * kR;
  auto row_ptr = [&](int row) {
    const bool is_t = row >= D;
    return (is_t ? Sm : Pi) + (static_cast<size_t>(h) * D + (is_t ? row - D : row)) * D;
  };
  // The warp's rows of [Pi ; S_mat] (their first 128 columns) and the query tile are
  // requested together, four query loads a thread in flight: one memory round trip.
  constexpr int kPre = 4;
  float mpre[kR][kPre];
#pragma unroll
  for (int r = 0; r < kR; ++r) {
    const int row = row0 + r;
    const bool has = !hadamard_slice && row < 2 * D;
    const float* mrow = row_ptr(has ? row : 0);
#pragma unroll
    for (int i = 0; i < kPre; ++i) {
      const int j = lane + 32 * i;
      mpre[r][i] = has && j < D ? __ldg(mrow + j) : 0.f;
    }
  }
  constexpr int kU = 4;
  for (int e0 = threadIdx.x; e0 < kQ * D; e0 += blockDim.x * kU) {
    float v[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int e = e0 + u * static_cast<int>(blockDim.x);
      v[u] = e < kQ * D && (e / D) < nq ? load_q(Q, qbase + e) : 0.f;
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int e = e0 + u * static_cast<int>(blockDim.x);
      if (e < kQ * D) sQ[e] = v[u];
    }
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
  if (hadamard_slice) {
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

#pragma unroll
  for (int r = 0; r < kR; ++r) {
    const int row = row0 + r;
    if (row >= 2 * D) break;                  // the same for the whole warp
    const bool is_t = row >= D;
    const int d = is_t ? row - D : row;
    const float* mrow = row_ptr(row);
    float acc[kQ];
#pragma unroll
    for (int q = 0; q < kQ; ++q) acc[q] = 0.f;
#pragma unroll
    for (int i = 0; i < kPre; ++i) {
      const int j = lane + 32 * i;
      if (j < D) {
#pragma unroll
        for (int q = 0; q < kQ; ++q) acc[q] = fmaf(mpre[r][i], sQ[q * D + j], acc[q]);
      }
    }
#pragma unroll 4
    for (int j = lane + 32 * kPre; j < D; j += 32) {
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
}

template <typename QT, bool kShareSm, int kR>
cudaError_t launch_prepare_t(const QT* Q, const float* Pi, const float* S_mat, float* A, float* T,
                             int P, int H, int B, int D, cudaStream_t st, uint16_t* Ybf,
                             const float* hsigns) {
  // A scorer launched behind this grid as a programmatic dependent shares its SMs only
  // when both kernels run under the same L1 / shared-memory split.  The copy of the
  // transform that runs ahead of such a scorer takes the largest carveout, as the scorer
  // does; the other copy keeps the default, which suits kernels that cannot share an SM
  // with it anyway.
  if constexpr (kShareSm) {
    static std::atomic<uint64_t> carve{0};
    cudaError_t e = prefer_max_shared(prepare_kernel<QT, true, kR>, carve);
    if (e != cudaSuccess) return e;
  }
  // dense: 2D output rows in slices of kWarps * kR; Hadamard: slice 0 for A, then the D
  // rows of T
  dim3 grid(ceil_div(B, kQ), P,
            hsigns != nullptr ? 1 + ceil_div(D, kWarps * kR) : ceil_div(2 * D, kWarps * kR));
  const size_t smem = static_cast<size_t>(kQ) * D * sizeof(float);
  const int NT = mma_query_tile(B), qtiles = mma_query_tiles(B);
  prepare_kernel<QT, kShareSm, kR><<<grid, kWarps * 32, smem, st>>>(Q, Pi, S_mat, A, T, H, B, D, Ybf, NT,
                                                                    qtiles, hsigns);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prepare(const void* Q, tq_qtype qtype, const float* Pi, const float* S_mat,
                           float* A, float* T, int P, int H, int B, int D, cudaStream_t st,
                           uint16_t* Ybf, const float* hsigns, bool share_sm) {
  if (D != 128) Ybf = nullptr;
  // Four rows a warp once one row a warp would take more than two waves of CTAs (about
  // eight 256-thread CTAs an SM): many problems, as in a GQA decode batch.
  static std::atomic<int> sms_cache[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  int sms = sms_cache[dev & 63].load(std::memory_order_relaxed);
  if (sms == 0) {
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    sms_cache[dev & 63].store(sms, std::memory_order_relaxed);
  }
  const int64_t ctas = static_cast<int64_t>(ceil_div(B, kQ)) * P * ceil_div(2 * D, kWarps);
  const bool four = !share_sm && ctas > 2LL * 8 * sms;
  if (qtype == TQ_Q_BF16) {
    const auto* q = static_cast<const __nv_bfloat16*>(Q);
    if (share_sm) return launch_prepare_t<__nv_bfloat16, true, 1>(q, Pi, S_mat, A, T, P, H, B, D, st, Ybf, hsigns);
    if (four) return launch_prepare_t<__nv_bfloat16, false, 4>(q, Pi, S_mat, A, T, P, H, B, D, st, Ybf, hsigns);
    return launch_prepare_t<__nv_bfloat16, false, 1>(q, Pi, S_mat, A, T, P, H, B, D, st, Ybf, hsigns);
  }
  const auto* q = static_cast<const float*>(Q);
  if (share_sm) return launch_prepare_t<float, true, 1>(q, Pi, S_mat, A, T, P, H, B, D, st, Ybf, hsigns);
  if (four) return launch_prepare_t<float, false, 4>(q, Pi, S_mat, A, T, P, H, B, D, st, Ybf, hsigns);
  return launch_prepare_t<float, false, 1>(q, Pi, S_mat, A, T, P, H, B, D, st, Ybf, hsigns);
}

}  // namespace tq
