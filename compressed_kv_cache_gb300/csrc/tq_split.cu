// Outlier-split cache: two TurboQuant-MSE instances per head over disjoint channel
// sets ("TurboQuant: Rotate-then-Quantize KV Caches at 3 Bits", kanthi.in, §7
// "Fractional bits and the outlier split"; §8 "Kernel view": rotate the query once per
// instance).  The n_out outlier channels of a key (chosen ahead of time) and its other
// n_reg channels are two vectors, each with its own rotation, codebook and fp16 norm:
//
//   A_out = Pi_out q[outlier channels],  A_reg = Pi_reg q[other channels]
//   score = n_out * <A_out, c_out(idx_out)> + n_reg * <A_reg, c_reg(idx_reg)>
//
// split_prepare_kernel: one CTA per (16 output rows of [Pi_out; Pi_reg], tile of 8
// queries, problem); the query tile is staged in shared memory through the channel map
// (outlier channels in increasing order, the others after them in increasing order),
// and each warp forms two of the CTA's rows: lanes split the row (coalesced), the 8
// queries' partial sums are reduced across the warp.
// split_scores_kernel: thread per key for a tile of QB queries; both query parts as
// [n][QB] and both codebooks in shared memory; each 32-coordinate chunk of a code plane
// is BITS words whose field positions are compile-time constants.  One owner thread and
// one summation order per score.
#include <atomic>

#include "tq_internal.cuh"

namespace tq {
namespace {

constexpr int kSplitQ = 8;               // queries per transform CTA
constexpr int kSplitRows = 16;           // output rows of [Pi_out; Pi_reg] per transform CTA
constexpr int kSplitPrepThreads = 256;
constexpr int kSplitScoreThreads = 128;

template <typename QT>
__device__ __forceinline__ float widen(QT v);
template <>
__device__ __forceinline__ float widen<float>(float v) { return v; }
template <>
__device__ __forceinline__ float widen<__nv_bfloat16>(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename QT>
__global__ void __launch_bounds__(kSplitPrepThreads)
split_prepare_kernel(const QT* __restrict__ Q, const int* __restrict__ channels,
                     const float* __restrict__ Pi_out, const float* __restrict__ Pi_reg,
                     float* __restrict__ A_out, float* __restrict__ A_reg, int H, int B, int D, int n_out) {
  extern __shared__ __align__(16) float sq[];             // [kSplitQ][D] in the permuted channel order
  int* sperm = reinterpret_cast<int*>(sq + kSplitQ * D);  // [D]: original channel of permuted slot
  int* sch = sperm + D;                                   // [n_out]: the outlier channels, clamped
  const int p = blockIdx.z, h = p % H, b0 = blockIdx.y * kSplitQ;
  const int n_reg = D - n_out;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // a channel list that breaks the contract (out of range, not increasing) gives wrong
  // results but never an access outside the arrays
  for (int i = tid; i < n_out; i += kSplitPrepThreads) {
    const int c = __ldg(channels + i);
    sch[i] = c < 0 ? 0 : (c >= D ? D - 1 : c);
    sperm[i] = sch[i];
  }
  __syncthreads();
  // slot of a regular channel c: n_out + c - (outlier channels below c)
  for (int c = tid; c < D; c += kSplitPrepThreads) {
    int below = 0;
    bool outl = false;
    for (int i = 0; i < n_out; ++i) {
      below += sch[i] < c;
      outl |= sch[i] == c;
    }
    const int slot = n_out + c - below;
    if (!outl && slot < D) sperm[slot] = c;
  }
  __syncthreads();
  for (int e = tid; e < kSplitQ * D; e += kSplitPrepThreads) {
    const int q = e / D, i = e % D;
    sq[e] = b0 + q < B ? widen<QT>(Q[(static_cast<size_t>(p) * B + b0 + q) * D + sperm[i]]) : 0.f;
  }
  __syncthreads();
  const int row_end = min(D, static_cast<int>(blockIdx.x + 1) * kSplitRows);
  for (int row = blockIdx.x * kSplitRows + warp; row < row_end; row += kSplitPrepThreads / 32) {
    const bool outl = row < n_out;
    const int n = outl ? n_out : n_reg;
    const int r = outl ? row : row - n_out;
    const float* m = (outl ? Pi_out + static_cast<size_t>(h) * n_out * n_out
                           : Pi_reg + static_cast<size_t>(h) * n_reg * n_reg) + static_cast<size_t>(r) * n;
    const float* qv = sq + (outl ? 0 : n_out);
    float part[kSplitQ];
#pragma unroll
    for (int q = 0; q < kSplitQ; ++q) part[q] = 0.f;
    for (int j = lane; j < n; j += 32) {
      const float mv = __ldg(m + j);
#pragma unroll
      for (int q = 0; q < kSplitQ; ++q) part[q] = fmaf(mv, qv[q * D + j], part[q]);
    }
#pragma unroll
    for (int q = 0; q < kSplitQ; ++q) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) part[q] += __shfl_xor_sync(0xffffffffu, part[q], o);
    }
    if (lane < kSplitQ && b0 + lane < B) {
      float v = part[0];
#pragma unroll
      for (int q = 1; q < kSplitQ; ++q)
        if (lane == q) v = part[q];
      float* dst = outl ? A_out + (static_cast<size_t>(p) * B + b0 + lane) * n_out
                        : A_reg + (static_cast<size_t>(p) * B + b0 + lane) * n_reg;
      dst[r] = v;
    }
  }
}

// Sum over the codes of one key's part: sum_d A[d][q] c[code_d] for QB queries.
template <int BITS, int QB>
__device__ __forceinline__ void mse_part(const uint32_t* __restrict__ words, int chunks, const float* sA,
                                         const float* sC, float (&m)[QB]) {
  constexpr uint32_t kMask = (1u << BITS) - 1u;
  for (int ch = 0; ch < chunks; ++ch) {
    uint32_t w[BITS + 1];
#pragma unroll
    for (int i = 0; i < BITS; ++i) w[i] = __ldg(words + ch * BITS + i);
    w[BITS] = 0u;
#pragma unroll
    for (int u = 0; u < 32; ++u) {
      const int pos = BITS * u;
      const int wd = pos >> 5, sh = pos & 31;
      const uint32_t code = (sh + BITS <= 32) ? (w[wd] >> sh) & kMask : __funnelshift_r(w[wd], w[wd + 1], sh) & kMask;
      const float c = sC[code];
      const float* a = sA + (ch * 32 + u) * QB;
#pragma unroll
      for (int q = 0; q < QB; ++q) m[q] = fmaf(a[q], c, m[q]);
    }
  }
}

// The same sum from code words already in registers, for parts of at most 4 chunks.
template <int BITS, int QB>
__device__ __forceinline__ void mse_part_regs(const uint32_t (&wd)[4 * BITS], int chunks, const float* sA,
                                              const float* sC, float (&m)[QB]) {
  constexpr uint32_t kMask = (1u << BITS) - 1u;
#pragma unroll
  for (int ch = 0; ch < 4; ++ch) {
    if (ch >= chunks) break;
#pragma unroll
    for (int u = 0; u < 32; ++u) {
      const int pos = BITS * u;
      const int wi = ch * BITS + (pos >> 5), sh = pos & 31;
      const uint32_t nxt = (pos >> 5) + 1 < BITS ? wd[wi + 1] : 0u;
      const uint32_t code = (sh + BITS <= 32) ? (wd[wi] >> sh) & kMask : __funnelshift_r(wd[wi], nxt, sh) & kMask;
      const float c = sC[code];
      const float* a = sA + (ch * 32 + u) * QB;
#pragma unroll
      for (int q = 0; q < QB; ++q) m[q] = fmaf(a[q], c, m[q]);
    }
  }
}

template <int BO, int BR, int QB>
__global__ void __launch_bounds__(kSplitScoreThreads)
split_scores_kernel(const float* __restrict__ A_out, const float* __restrict__ A_reg,
                    const uint8_t* __restrict__ out_plane, const uint16_t* __restrict__ out_norm,
                    const float* __restrict__ cb_out, const uint8_t* __restrict__ reg_plane,
                    const uint16_t* __restrict__ reg_norm, const float* __restrict__ cb_reg,
                    float* __restrict__ scores, int B, int S, int n_out, int n_reg) {
  extern __shared__ __align__(16) float smem[];
  float* sAo = smem;                                      // [n_out][QB]
  float* sAr = sAo + n_out * QB;                          // [n_reg][QB]
  float* sCo = sAr + n_reg * QB;                          // [16]
  float* sCr = sCo + 16;                                  // [16]
  const int p = blockIdx.z, b0 = blockIdx.y * QB;
  const int s = blockIdx.x * blockDim.x + threadIdx.x;
  const size_t key = static_cast<size_t>(p) * S + (s < S ? s : 0);
  // parts of at most 4 chunks (the printed split: 1 and 3): this thread's code words and
  // norms are requested before the query staging below, so the two round trips overlap
  const int co = n_out / 32, cr = n_reg / 32;
  const bool early = co <= 4 && cr <= 4;
  uint32_t wo[4 * BO], wr[4 * BR];
  float no = 0.f, nr = 0.f;
  if (early && s < S) {
    const uint32_t* po = reinterpret_cast<const uint32_t*>(out_plane) + key * co * BO;
    const uint32_t* pr = reinterpret_cast<const uint32_t*>(reg_plane) + key * cr * BR;
#pragma unroll
    for (int i = 0; i < 4 * BO; ++i) wo[i] = i < co * BO ? __ldg(po + i) : 0u;
#pragma unroll
    for (int i = 0; i < 4 * BR; ++i) wr[i] = i < cr * BR ? __ldg(pr + i) : 0u;
    no = __half2float(__ushort_as_half(__ldg(out_norm + key)));
    nr = __half2float(__ushort_as_half(__ldg(reg_norm + key)));
  }
  for (int e = threadIdx.x; e < QB * n_out; e += blockDim.x) {
    const int q = e / n_out, d = e % n_out;
    sAo[d * QB + q] = b0 + q < B ? A_out[(static_cast<size_t>(p) * B + b0 + q) * n_out + d] : 0.f;
  }
  for (int e = threadIdx.x; e < QB * n_reg; e += blockDim.x) {
    const int q = e / n_reg, d = e % n_reg;
    sAr[d * QB + q] = b0 + q < B ? A_reg[(static_cast<size_t>(p) * B + b0 + q) * n_reg + d] : 0.f;
  }
  if (threadIdx.x < (1 << BO)) sCo[threadIdx.x] = cb_out[threadIdx.x];
  if (threadIdx.x < (1 << BR)) sCr[threadIdx.x] = cb_reg[threadIdx.x];
  __syncthreads();
  if (s >= S) return;
  float mo[QB], mr[QB];
#pragma unroll
  for (int q = 0; q < QB; ++q) mo[q] = mr[q] = 0.f;
  if (early) {
    mse_part_regs<BO, QB>(wo, co, sAo, sCo, mo);
    mse_part_regs<BR, QB>(wr, cr, sAr, sCr, mr);
  } else {
    mse_part<BO, QB>(reinterpret_cast<const uint32_t*>(out_plane) + key * co * BO, co, sAo, sCo, mo);
    mse_part<BR, QB>(reinterpret_cast<const uint32_t*>(reg_plane) + key * cr * BR, cr, sAr, sCr, mr);
    no = __half2float(__ushort_as_half(__ldg(out_norm + key)));
    nr = __half2float(__ushort_as_half(__ldg(reg_norm + key)));
  }
#pragma unroll
  for (int q = 0; q < QB; ++q)
    if (b0 + q < B) scores[(static_cast<size_t>(p) * B + b0 + q) * S + s] = fmaf(no, mo[q], nr * mr[q]);
}

template <int BO, int BR, int QB>
cudaError_t launch_split_qb(const float* A_out, const float* A_reg, const uint8_t* out_plane,
                            const uint16_t* out_norm, const float* cb_out, const uint8_t* reg_plane,
                            const uint16_t* reg_norm, const float* cb_reg, float* scores, int P, int B, int S,
                            int n_out, int n_reg, cudaStream_t st) {
  dim3 grid(ceil_div(S, kSplitScoreThreads), ceil_div(B, QB), P);
  const size_t smem = (static_cast<size_t>(QB) * (n_out + n_reg) + 32) * sizeof(float);
  auto kernel = split_scores_kernel<BO, BR, QB>;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  kernel<<<grid, kSplitScoreThreads, smem, st>>>(A_out, A_reg, out_plane, out_norm, cb_out, reg_plane, reg_norm,
                                                 cb_reg, scores, B, S, n_out, n_reg);
  return cudaGetLastError();
}

template <int BO, int BR>
cudaError_t launch_split_b(const float* A_out, const float* A_reg, const uint8_t* out_plane,
                           const uint16_t* out_norm, const float* cb_out, const uint8_t* reg_plane,
                           const uint16_t* reg_norm, const float* cb_reg, float* scores, int P, int B, int S,
                           int n_out, int n_reg, cudaStream_t st) {
  if (B <= 1) return launch_split_qb<BO, BR, 1>(A_out, A_reg, out_plane, out_norm, cb_out, reg_plane, reg_norm, cb_reg, scores, P, B, S, n_out, n_reg, st);
  if (B <= 2) return launch_split_qb<BO, BR, 2>(A_out, A_reg, out_plane, out_norm, cb_out, reg_plane, reg_norm, cb_reg, scores, P, B, S, n_out, n_reg, st);
  if (B <= 4) return launch_split_qb<BO, BR, 4>(A_out, A_reg, out_plane, out_norm, cb_out, reg_plane, reg_norm, cb_reg, scores, P, B, S, n_out, n_reg, st);
  return launch_split_qb<BO, BR, 8>(A_out, A_reg, out_plane, out_norm, cb_out, reg_plane, reg_norm, cb_reg, scores, P, B, S, n_out, n_reg, st);
}

template <int BO>
cudaError_t launch_split_bo(int reg_bits, const float* A_out, const float* A_reg, const uint8_t* out_plane,
                            const uint16_t* out_norm, const float* cb_out, const uint8_t* reg_plane,
                            const uint16_t* reg_norm, const float* cb_reg, float* scores, int P, int B, int S,
                            int n_out, int n_reg, cudaStream_t st) {
  switch (reg_bits) {
    case 1: return launch_split_b<BO, 1>(A_out, A_reg, out_plane, out_norm, cb_out, reg_plane, reg_norm, cb_reg, scores, P, B, S, n_out, n_reg, st);
    case 2: return launch_split_b<BO, 2>(A_out, A_reg, out_plane, out_norm, cb_out, reg_plane, reg_norm, cb_reg, scores, P, B, S, n_out, n_reg, st);
    case 3: return launch_split_b<BO, 3>(A_out, A_reg, out_plane, out_norm, cb_out, reg_plane, reg_norm, cb_reg, scores, P, B, S, n_out, n_reg, st);
    default: return launch_split_b<BO, 4>(A_out, A_reg, out_plane, out_norm, cb_out, reg_plane, reg_norm, cb_reg, scores, P, B, S, n_out, n_reg, st);
  }
}

}  // namespace
}  // namespace tq

extern "C" {

tq_status tq_prepare_queries_split(const void* Q, tq_qtype qtype, const int* channels, const float* Pi_out,
                                   const float* Pi_reg, float* A_out, float* A_reg, int P, int H, int B,
                                   int D, int n_out, cudaStream_t stream) {
  const void* all[] = {Q, channels, Pi_out, Pi_reg, A_out, A_reg};
  for (const void* q : all)
    if (q == nullptr) return TQ_ERR_INVALID_VALUE;
  for (const void* q : all)
    if (reinterpret_cast<uintptr_t>(q) & 15u) return TQ_ERR_MISALIGNED;
  if (P < 1 || P > 65535 || H < 1 || H > P || B < 1 || D < 2 || D > 256 || n_out < 1 || n_out >= D)
    return TQ_ERR_INVALID_VALUE;
  if (qtype != TQ_Q_F32 && qtype != TQ_Q_BF16) return TQ_ERR_INVALID_VALUE;
  if ((B + tq::kSplitQ - 1) / tq::kSplitQ > 65535) return TQ_ERR_INVALID_VALUE;
  dim3 grid((D + tq::kSplitRows - 1) / tq::kSplitRows, (B + tq::kSplitQ - 1) / tq::kSplitQ, P);
  const size_t smem = static_cast<size_t>(tq::kSplitQ) * D * sizeof(float) + 2 * D * sizeof(int);
  if (qtype == TQ_Q_BF16)
    tq::split_prepare_kernel<__nv_bfloat16><<<grid, tq::kSplitPrepThreads, smem, stream>>>(
        static_cast<const __nv_bfloat16*>(Q), channels, Pi_out, Pi_reg, A_out, A_reg, H, B, D, n_out);
  else
    tq::split_prepare_kernel<float><<<grid, tq::kSplitPrepThreads, smem, stream>>>(
        static_cast<const float*>(Q), channels, Pi_out, Pi_reg, A_out, A_reg, H, B, D, n_out);
  return cudaGetLastError() == cudaSuccess ? TQ_OK : TQ_ERR_LAUNCH;
}

tq_status tq_scores_split(const float* A_out, const float* A_reg, const uint8_t* out_plane,
                          const uint16_t* out_norm, const float* out_codebook, int out_bits,
                          const uint8_t* reg_plane, const uint16_t* reg_norm, const float* reg_codebook,
                          int reg_bits, float* scores, int P, int B, int S, int n_out, int n_reg,
                          cudaStream_t stream) {
  const void* all[] = {A_out, A_reg, out_plane, out_norm, out_codebook, reg_plane, reg_norm, reg_codebook, scores};
  for (const void* q : all)
    if (q == nullptr) return TQ_ERR_INVALID_VALUE;
  for (const void* q : all)
    if (reinterpret_cast<uintptr_t>(q) & 15u) return TQ_ERR_MISALIGNED;
  if (P < 1 || P > 65535 || B < 1 || B > 65535 || S < 1 || out_bits < 1 || out_bits > 4 || reg_bits < 1 ||
      reg_bits > 4 || n_out < 1 || n_reg < 1 || n_out + n_reg > 4096)
    return TQ_ERR_INVALID_VALUE;
  if (n_out % 32 != 0 || n_reg % 32 != 0) return TQ_ERR_UNSUPPORTED;
  cudaError_t e;
  switch (out_bits) {
    case 1: e = tq::launch_split_bo<1>(reg_bits, A_out, A_reg, out_plane, out_norm, out_codebook, reg_plane, reg_norm, reg_codebook, scores, P, B, S, n_out, n_reg, stream); break;
    case 2: e = tq::launch_split_bo<2>(reg_bits, A_out, A_reg, out_plane, out_norm, out_codebook, reg_plane, reg_norm, reg_codebook, scores, P, B, S, n_out, n_reg, stream); break;
    case 3: e = tq::launch_split_bo<3>(reg_bits, A_out, A_reg, out_plane, out_norm, out_codebook, reg_plane, reg_norm, reg_codebook, scores, P, B, S, n_out, n_reg, stream); break;
    default: e = tq::launch_split_bo<4>(reg_bits, A_out, A_reg, out_plane, out_norm, out_codebook, reg_plane, reg_norm, reg_codebook, scores, P, B, S, n_out, n_reg, stream); break;
  }
  return e == cudaSuccess ? TQ_OK : TQ_ERR_LAUNCH;
}

}  // extern "C"
