// Fused decode in the rotated domain ("TurboQuant: Rotate-then-Quantize KV Caches at
// 3 Bits", kanthi.in, §8 "Kernel view: never un-rotate a key", the kernel form of
// tq_rotated_domain), over an MSE-quantized or a TurboQuant_prod key cache and an
// MSE-quantized value cache:
//
//   s[b,i]  = scale * nk_i * <A_b, ck[kidx_i]>                      MSE keys
//   s[b,i]  = scale * (<A_b, ck[kidx_i]> + kappa g_i <T_b, sigma_i>)  product keys
//             (A_b = Pi_k q_b, T_b = S_mat q_b; "Implementing TurboQuant on NVIDIA's
//             AGX Thor", zededa.com, v2 kernel 3 and v6 fused hybrid kernel: TQ score,
//             value dequant, accumulate)
//   p[b,:]  = softmax(s[b,:])
//   acc[b]  = sum_i p[b,i] nv_i cv[vidx_i]              accumulated in the rotated basis
//   out[b]  = Pi_v^T acc[b]                             one inverse rotation per query
//
// Split-KV (flash decoding): decode_split_kernel takes one chunk of keys and one tile
// of QB queries of a problem.  Each of its 16 warps owns a contiguous run of the
// chunk's keys and starts the asynchronous copies of their key rows (and sign rows)
// and value rows into shared memory, 32 keys to a copy group.  The CTA builds the key
// lookup tables (code tables from A, sign tables from T) meanwhile.  Then every warp
// runs an online softmax over its groups as they land: logits (lane per key), the
// group maximum, the rescale of the running sum and accumulator by exp(old max - new
// max), and the weighted value centroids.  The warps merge in shared memory and write
// (max, sum, acc[128]) per (query, chunk) to the workspace.  decode_combine_kernel
// merges the chunks of a query with the same rescaling and applies Pi_v^T.  D = 128,
// 1-3 bit codes.
#include <atomic>

#include "tq_internal.cuh"
#include "tq_lut.cuh"

namespace tq {
namespace {

constexpr int kD = 128;
constexpr int kDecThreads = 512;
constexpr int kMaxChunk = 1024;          // keys per split CTA (rows staged in shared memory)
constexpr int kAcc = 4;                  // acc offset in a partial row (16-byte aligned)
constexpr int kPart = kAcc + kD;         // floats per (query, chunk): max, sum, 2 pad, acc

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

// One bulk copy global -> shared through the copy engine, completing on a local mbarrier.
__device__ __forceinline__ void bulk_copy(void* dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}
__device__ __forceinline__ void expect_bytes(uint32_t bar, uint32_t bytes) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(bar),
               "r"(bytes)
               : "memory");
}
// Bounded wait for phase 0 of a local mbarrier (kWaitBudgetNs); false if it gave up.
__device__ __forceinline__ bool wait_phase0(uint32_t bar) { return wait_parity_bounded(bar, 0, kFaultDecode); }

// Shared memory: key rows [chunk][16 KBITS B] | value rows [chunk][16 VBITS B] |
// copy barriers [warps][steps] | lut [QB][NPI*NV] | rotated queries [QB][128] |
// warp acc [warps][QB][128] | warp max and sum [warps][QB] each | value centroids [8]
constexpr int kDecWarps = kDecThreads / 32;
constexpr int kStep = 32;                                  // keys per warp step (lane per key)
constexpr int kMaxSteps = kMaxChunk / kDecWarps / kStep;   // warp steps, at most

// Arguments of one split launch (PROD: product keys with sign rows and gamma).
struct SplitArgs {
  const float* A;                 // [P,B,128] rotated queries
  const float* T;                 // [P,B,128] projected queries (product keys only)
  const uint8_t* k_plane;         // [P,S,16 KBITS] key codes
  const uint8_t* k_sign;          // [P,S,16] key sign rows (product keys only)
  const uint16_t* k_scale;        // [P,S] fp16: key norms (MSE keys) or residual norms gamma
  const float* k_cb;
  const uint8_t* v_plane;
  const uint16_t* v_norm;
  const float* v_cb;
  float* part;
  int B, S, chunk, nchunks;
  float scale, kappa;
};

template <int KBITS, bool PROD>
__host__ __device__ constexpr int key_tab_floats() {
  return LutShape<KBITS>::NPI * LutShape<KBITS>::NV + (PROD ? LutShape<KBITS>::NPS * 16 : 0);
}

template <int KBITS, int VBITS, int QB, bool PROD>
constexpr size_t split_smem_bytes(int chunk) {
  return static_cast<size_t>(chunk) * 16 * (KBITS + VBITS + (PROD ? 1 : 0)) + 8 * kDecWarps * kMaxSteps +
         sizeof(float) * (static_cast<size_t>(QB) * key_tab_floats<KBITS, PROD>() +
                          static_cast<size_t>(QB) * kD * (PROD ? 2 : 1) +
                          static_cast<size_t>(kDecWarps) * QB * (kD + 2) + 8);
}

template <int KBITS, int VBITS, int QB, bool PROD>
__global__ void __launch_bounds__(kDecThreads)
decode_split_kernel(const SplitArgs args) {
  using L = LutShape<KBITS>;
  constexpr int kW = kDecWarps;
  constexpr int kKRow = 16 * KBITS, kVRow = 16 * VBITS;   // bytes of one key / value row
  constexpr int kSRow = PROD ? 16 : 0;                    // bytes of one sign row
  constexpr int kTab = key_tab_floats<KBITS, PROD>();     // table floats per query
  constexpr int kQ = PROD ? 2 * kD : kD;                  // query-side floats per query (A, T)
  constexpr int kBlk = kStep;
  constexpr int kMaxBlk = kMaxSteps;
  const int B = args.B, S = args.S, chunk = args.chunk, nchunks = args.nchunks;
  const float scale = args.scale;
  extern __shared__ __align__(16) uint8_t smem_raw[];
  uint8_t* kst = smem_raw;
  uint8_t* sst = kst + static_cast<size_t>(chunk) * kKRow;
  uint8_t* vst = sst + static_cast<size_t>(chunk) * kSRow;
  uint64_t* bars = reinterpret_cast<uint64_t*>(vst + static_cast<size_t>(chunk) * kVRow);
  float* lut = reinterpret_cast<float*>(bars + kW * kMaxBlk);
  float* sA = lut + QB * kTab;                            // [QB][A | T]
  float* racc = sA + QB * kQ;
  float* rmax = racc + kW * QB * kD;
  float* rsum = rmax + kW * QB;
  float* vtab = rsum + kW * QB;
  const int c = blockIdx.x, p = blockIdx.z, b0 = blockIdx.y * QB;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int k0 = c * chunk;
  const int n = min(chunk, S - k0);                        // >= 1
  const size_t kbase = static_cast<size_t>(p) * S + k0;
  // the merge kernel behind this grid may launch now; it reads the partials only after
  // this grid has completed
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  // rotated queries into registers first (stored once the copies are under way)
  constexpr int kAPer = (QB * kQ + kDecThreads - 1) / kDecThreads;
  float av[kAPer];
#pragma unroll
  for (int j = 0; j < kAPer; ++j) {
    const int e = tid + j * kDecThreads, q = e / kQ, x = e % kQ;
    const size_t row = (static_cast<size_t>(p) * B + b0 + q) * kD;
    av[j] = e < QB * kQ && b0 + q < B ? (x < kD ? __ldg(args.A + row + x) : __ldg(args.T + row + x - kD)) : 0.f;
  }
  const float vt = tid < (1 << VBITS) ? __ldg(args.v_cb + tid) : 0.f;
  __shared__ float sKcb[1 << KBITS];
  stage_codebook<KBITS>(args.k_cb, sKcb, 0);   // read after the barrier before the table build

  // this warp's keys [w0, w1) of the chunk, in steps of 32: per step one bulk copy of
  // the key rows and one of the value rows, both completing on the step's barrier
  const int per = (n + kW - 1) / kW;
  const int w0 = min(n, warp * per), w1 = min(n, w0 + per);
  const int nsteps = (w1 - w0 + kBlk - 1) / kBlk;
  const uint32_t bar0 = static_cast<uint32_t>(__cvta_generic_to_shared(bars + warp * kMaxBlk));
  if (lane == 0) {
    for (int t = 0; t < nsteps; ++t)
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bar0 + 8 * t) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    for (int t = 0; t < nsteps; ++t) {
      const int r0 = w0 + t * kBlk, rows = min(kBlk, w1 - r0);
      const uint32_t bar = bar0 + 8 * t;
      expect_bytes(bar, static_cast<uint32_t>(rows * (kKRow + kSRow + kVRow)));
      bulk_copy(kst + static_cast<size_t>(r0) * kKRow, args.k_plane + (kbase + r0) * kKRow,
                static_cast<uint32_t>(rows * kKRow), bar);
      if constexpr (PROD)
        bulk_copy(sst + static_cast<size_t>(r0) * kSRow, args.k_sign + (kbase + r0) * kSRow,
                  static_cast<uint32_t>(rows * kSRow), bar);
      bulk_copy(vst + static_cast<size_t>(r0) * kVRow, args.v_plane + (kbase + r0) * kVRow,
                static_cast<uint32_t>(rows * kVRow), bar);
    }
  }
  __syncwarp();
  // key norms (MSE keys) or residual norms (product keys) and value norms of this
  // lane's keys w0 + 32 t + lane
  float nk[kMaxBlk], nv[kMaxBlk];
#pragma unroll
  for (int t = 0; t < kMaxBlk; ++t) {
    const int i = w0 + t * kBlk + lane;
    nk[t] = i < w1 ? __half2float(__ushort_as_half(__ldg(args.k_scale + kbase + i))) : 0.f;
    nv[t] = i < w1 ? __half2float(__ushort_as_half(__ldg(args.v_norm + kbase + i))) : 0.f;
  }

#pragma unroll
  for (int j = 0; j < kAPer; ++j) {
    const int e = tid + j * kDecThreads;
    if (e < QB * kQ) sA[e] = av[j];
  }
  if (tid < (1 << VBITS)) vtab[tid] = vt;
  // key tables of the query tile (rows past B give zero tables): code tables from A,
  // then (product keys) 32 sign tables of 4 signs each from T
  __syncthreads();
  {
    float cv[L::G];
    table_centroids<KBITS>(sKcb, cv);
    const int v = tid % L::NV;
    for (int q = 0; q < QB; ++q) {
      const float* a = sA + q * kQ;
      float* tq = lut + q * kTab;
      for (int g = tid / L::NV; g < L::NPI; g += kDecThreads / L::NV) {
        float acc = 0.f;
#pragma unroll
        for (int k = 0; k < L::G; ++k) acc = fmaf(a[g * L::G + k], cv[k], acc);
        tq[g * L::NV + v] = acc;
      }
      if constexpr (PROD) {
        const int vs = tid & 15;
        for (int g = tid >> 4; g < L::NPS; g += kDecThreads / 16) {
          float acc = 0.f;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float t = a[kD + 4 * g + i];
            acc += ((vs >> i) & 1) ? t : -t;
          }
          tq[L::NPI * L::NV + g * 16 + vs] = acc;
        }
      }
    }
  }
  __syncthreads();

  // online softmax over the warp's steps: logits (lane per key), the step maximum, the
  // rescale of what came before, then the weighted value centroids.  Values: KPI keys
  // at a time, LPK = 32 / KPI lanes per key, lane sub = lane % LPK owning CPL = 128 / LPK
  // coordinates CPL*sub .. CPL*sub + CPL-1, whose codes are the bits from VBITS*CPL*sub
  // on of the value row; a code becomes its centroid by one read of the shared table.
  // Four keys at a time (8 lanes per key) for up to two queries, else one.
  constexpr int KPI = QB <= 2 ? 4 : 1;
  constexpr int LPK = 32 / KPI, CPL = kD / LPK, NB = VBITS * CPL;
  constexpr uint32_t kMask = (1u << VBITS) - 1u;
  const int slot = lane / LPK, sub = lane % LPK;
  const int bit0 = NB * sub;
  const int wlo = bit0 >> 5, bsh = bit0 & 31;
  const bool two = bsh + NB > 32;          // the lane's codes straddle two words
  bool landed = true;
  float M[QB], Lp[QB], acc[QB][CPL];
#pragma unroll
  for (int q = 0; q < QB; ++q) {
    M[q] = -INFINITY;
    Lp[q] = 0.f;
#pragma unroll
    for (int j = 0; j < CPL; ++j) acc[q][j] = 0.f;
  }
#pragma unroll
  for (int t = 0; t < kMaxBlk; ++t) {
    if (t < nsteps) {
      landed &= wait_phase0(bar0 + 8 * t);
      const int r0 = w0 + t * kBlk;
      const int i = r0 + lane;
      float sc[QB];
#pragma unroll
      for (int q = 0; q < QB; ++q) sc[q] = -INFINITY;
      if (i < w1) {
        const uint4* kp = reinterpret_cast<const uint4*>(kst + static_cast<size_t>(i) * kKRow);
        uint32_t wd[4 * KBITS + 1];
#pragma unroll
        for (int r = 0; r < KBITS; ++r) {
          const uint4 x = kp[r];
          wd[4 * r] = x.x; wd[4 * r + 1] = x.y; wd[4 * r + 2] = x.z; wd[4 * r + 3] = x.w;
        }
        wd[4 * KBITS] = 0u;
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
          for (int q = 0; q < QB; ++q) m[gi & 1][q] += lut[q * kTab + gi * L::NV + val];
        }
        if constexpr (PROD) {
          // the sign row: 32 lookups of 4 signs each, then score = mse + kappa g res
          const uint4 sr = *reinterpret_cast<const uint4*>(sst + static_cast<size_t>(i) * kSRow);
          unsigned long long r2[QB][2];
#pragma unroll
          for (int q = 0; q < QB; ++q) r2[q][0] = r2[q][1] = 0ull;
          lut_nibbles<QB, kTab>(lut + L::NPI * L::NV, sr.x, 0, r2);
          lut_nibbles<QB, kTab>(lut + L::NPI * L::NV, sr.y, 8, r2);
          lut_nibbles<QB, kTab>(lut + L::NPI * L::NV, sr.z, 16, r2);
          lut_nibbles<QB, kTab>(lut + L::NPI * L::NV, sr.w, 24, r2);
          const float kg = args.kappa * nk[t];
#pragma unroll
          for (int q = 0; q < QB; ++q)
            sc[q] = scale * fmaf(kg, sum2(r2[q][0]) + sum2(r2[q][1]), m[0][q] + m[1][q]);
        } else {
#pragma unroll
          for (int q = 0; q < QB; ++q) sc[q] = scale * nk[t] * (m[0][q] + m[1][q]);
        }
      }
      float w[QB];
#pragma unroll
      for (int q = 0; q < QB; ++q) {
        const float mn = fmaxf(M[q], warp_max(sc[q]));     // finite: the step has a key
        const float r = expf(M[q] - mn);                    // 0 on the first step
        const float e = i < w1 ? expf(sc[q] - mn) : 0.f;
        Lp[q] = fmaf(Lp[q], r, e);
        w[q] = e * nv[t];
#pragma unroll
        for (int j = 0; j < CPL; ++j) acc[q][j] *= r;
        M[q] = mn;
      }
      const int cnt = min(kBlk, w1 - r0);
#pragma unroll 2
      for (int k = 0; k < cnt; k += KPI) {
        const int kk = k + slot;                            // this lane's key of the step
        const uint32_t* vr =
            reinterpret_cast<const uint32_t*>(vst + static_cast<size_t>(r0 + min(kk, cnt - 1)) * kVRow);
        const uint32_t lo = vr[wlo];
        const uint32_t hi = two ? vr[wlo + 1] : 0u;
        const uint32_t c0 = __funnelshift_r(lo, hi, bsh);  // code bits 0..31 of the lane
        const uint32_t c1 = hi >> bsh;                      // code bits 32..63
        float cw[CPL];
#pragma unroll
        for (int j = 0; j < CPL; ++j) {
          const int pj = VBITS * j;
          const uint32_t code = pj + VBITS <= 32 ? (c0 >> pj) & kMask
                                : pj >= 32       ? (c1 >> (pj - 32)) & kMask
                                                 : __funnelshift_r(c0, c1, pj) & kMask;
          cw[j] = vtab[code];
        }
#pragma unroll
        for (int q = 0; q < QB; ++q) {
          const float wsh = __shfl_sync(0xffffffffu, w[q], kk & 31);
          const float wq = kk < cnt ? wsh : 0.f;
#pragma unroll
          for (int j = 0; j < CPL; ++j) acc[q][j] = fmaf(wq, cw[j], acc[q][j]);
        }
      }
    }
  }
  // the key slots of a lane group hold partial sums of the same coordinates
#pragma unroll
  for (int o = LPK; o < 32; o <<= 1) {
#pragma unroll
    for (int q = 0; q < QB; ++q) {
#pragma unroll
      for (int j = 0; j < CPL; ++j) acc[q][j] += __shfl_xor_sync(0xffffffffu, acc[q][j], o);
    }
  }

  // merge the warps: max, rescaled sums and accumulators, to the workspace
  landed = __all_sync(0xffffffffu, landed);
#pragma unroll
  for (int q = 0; q < QB; ++q) {
    const float ls = warp_sum(Lp[q]);
    if (lane == 0) {
      rmax[warp * QB + q] = M[q];                            // -inf for a warp without keys
      rsum[warp * QB + q] = landed ? ls : __int_as_float(0x7fc00000);   // NaN: rows never landed
    }
    if (slot == 0) {
#pragma unroll
      for (int j = 0; j < CPL; ++j) racc[(warp * QB + q) * kD + CPL * sub + j] = acc[q][j];
    }
  }
  __syncthreads();
  for (int e = tid; e < QB * kD; e += kDecThreads) {
    const int q = e / kD, d = e % kD;
    if (b0 + q >= B) continue;
    float mx = rmax[q];
    for (int w = 1; w < kW; ++w) mx = fmaxf(mx, rmax[w * QB + q]);
    float s = 0.f, ls = 0.f;
    for (int w = 0; w < kW; ++w) {
      const float f = expf(rmax[w * QB + q] - mx);
      s = fmaf(racc[(w * QB + q) * kD + d], f, s);
      ls = fmaf(rsum[w * QB + q], f, ls);
    }
    float* pp = args.part + ((static_cast<size_t>(p) * B + b0 + q) * nchunks + c) * kPart;
    pp[kAcc + d] = s;
    if (d == 0) {
      pp[0] = mx;
      pp[1] = ls;
    }
  }
}

// One query: merge the chunks (rescale by exp(max_c - max)), normalise, out = acc Pi_v.
// 512 threads.  Thread t first holds rows 32g .. 32g+31 of column d of Pi_v (g = t / 128,
// d = t % 128), loaded before the wait on the split grid so that they overlap it.  Warp
// w then takes the chunks w, w + 16, ..., ten at a time with all their loads in flight
// at once (lane l: the chunk's max and sum, and acc coordinates 4l .. 4l+3), and keeps
// a running (max, sum, acc) with the usual rescaling.  The 16 warps merge in shared
// memory, the result is normalised, and thread (g, d) sums its 32 terms of out[d].
constexpr int kCombThreads = 512;
constexpr int kCombWarps = kCombThreads / 32;
constexpr int kCombSlots = 10;            // chunks per warp and round

__global__ void __launch_bounds__(kCombThreads)
decode_combine_kernel(const float* __restrict__ part, const float* __restrict__ Pi_v,
                      float* __restrict__ out, int H, int B, int nchunks) {
  constexpr int kGroups = kCombThreads / kD;
  constexpr int kRows = kD / kGroups;
  __shared__ float wmax[kCombWarps];
  __shared__ float wsum[kCombWarps];
  __shared__ __align__(16) float wacc[kCombWarps][kD];
  __shared__ float snorm[kD];
  const int b = blockIdx.x, p = blockIdx.y, h = p % H, tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  const int d = tid & (kD - 1), g = tid / kD;
  const float* Pv = Pi_v + static_cast<size_t>(h) * kD * kD + static_cast<size_t>(g) * kRows * kD + d;
  float pv[kRows];
#pragma unroll
  for (int k = 0; k < kRows; ++k) pv[k] = __ldg(Pv + k * kD);
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const float* pp = part + (static_cast<size_t>(p) * B + b) * nchunks * kPart;
  float Mw = -INFINITY, Lw = 0.f;
  float a[4] = {0.f, 0.f, 0.f, 0.f};
  for (int c0 = warp; c0 < nchunks; c0 += kCombWarps * kCombSlots) {
    float2 ml[kCombSlots];
    float4 x[kCombSlots];
#pragma unroll
    for (int j = 0; j < kCombSlots; ++j) {
      const int c = c0 + j * kCombWarps;
      if (c < nchunks) {
        const float* pc = pp + static_cast<size_t>(c) * kPart;
        ml[j] = *reinterpret_cast<const float2*>(pc);
        x[j] = *reinterpret_cast<const float4*>(pc + kAcc + 4 * lane);
      } else {
        ml[j] = make_float2(-INFINITY, 0.f);
        x[j] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
    float mb = Mw;
#pragma unroll
    for (int j = 0; j < kCombSlots; ++j) mb = fmaxf(mb, ml[j].x);   // finite: chunk c0 exists
    const float r = expf(Mw - mb);                                     // 0 on the first round
    Lw *= r;
#pragma unroll
    for (int k = 0; k < 4; ++k) a[k] *= r;
#pragma unroll
    for (int j = 0; j < kCombSlots; ++j) {
      const float e = expf(ml[j].x - mb);
      Lw = fmaf(ml[j].y, e, Lw);
      a[0] = fmaf(x[j].x, e, a[0]);
      a[1] = fmaf(x[j].y, e, a[1]);
      a[2] = fmaf(x[j].z, e, a[2]);
      a[3] = fmaf(x[j].w, e, a[3]);
    }
    Mw = mb;
  }
  if (lane == 0) {
    wmax[warp] = Mw;                      // -inf for a warp without chunks
    wsum[warp] = Lw;
  }
  *reinterpret_cast<float4*>(&wacc[warp][4 * lane]) = make_float4(a[0], a[1], a[2], a[3]);
  __syncthreads();
  if (tid < kD) {
    float M = wmax[0];
    for (int w = 1; w < kCombWarps; ++w) M = fmaxf(M, wmax[w]);
    float t = 0.f, l = 0.f;
    for (int w = 0; w < kCombWarps; ++w) {
      const float f = expf(wmax[w] - M);
      t = fmaf(wacc[w][tid], f, t);
      l = fmaf(wsum[w], f, l);
    }
    snorm[tid] = t / l;
  }
  __syncthreads();
  float o = 0.f;
#pragma unroll
  for (int k = 0; k < kRows; ++k) o = fmaf(snorm[g * kRows + k], pv[k], o);
  wacc[g][d] = o;
  __syncthreads();
  if (g == 0) {
    float t = 0.f;
#pragma unroll
    for (int j = 0; j < kGroups; ++j) t += wacc[j][d];
    out[(static_cast<size_t>(p) * B + b) * kD + d] = t;
  }
}

template <int KBITS, int VBITS, int QB, bool PROD>
cudaError_t launch_decode_qb(SplitArgs a, const float* Pi_v, float* out, int P, int H, cudaStream_t st) {
  auto kernel = decode_split_kernel<KBITS, VBITS, QB, PROD>;
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
                             static_cast<int>(split_smem_bytes<KBITS, VBITS, QB, PROD>(kMaxChunk)));
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (e != cudaSuccess) return e;
    configured.fetch_or(bit, std::memory_order_acq_rel);
  }
  static std::atomic<uint64_t> carve_combine{0};
  e = prefer_max_shared(decode_combine_kernel, carve_combine);
  if (e != cudaSuccess) return e;
  // chunks of 256..1024 keys, as many as give every SM one CTA (equal chunks, so that
  // no SM gets more keys than another)
  const int B = a.B, S = a.S;
  const int qtiles = ceil_div(B, QB);
  const int64_t units = static_cast<int64_t>(P) * qtiles;
  const int64_t per_unit = (static_cast<int64_t>(sms) + units - 1) / units;
  int chunk = ceil_div(S, per_unit < 1 ? 1 : per_unit);
  chunk = chunk < 256 ? 256 : (chunk > kMaxChunk ? kMaxChunk : chunk);
  a.chunk = chunk;
  a.nchunks = ceil_div(S, chunk);
  const size_t smem = split_smem_bytes<KBITS, VBITS, QB, PROD>(chunk);
  dim3 grid(a.nchunks, qtiles, P);
  kernel<<<grid, kDecThreads, smem, st>>>(a);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(B, P);
  cfg.blockDim = dim3(kCombThreads);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, decode_combine_kernel, static_cast<const float*>(a.part), Pi_v, out, H, B,
                         a.nchunks);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <int KBITS, int VBITS, bool PROD>
cudaError_t launch_decode_kv(const SplitArgs& a, const float* Pi_v, float* out, int P, int H, cudaStream_t st) {
  if (a.B <= 1) return launch_decode_qb<KBITS, VBITS, 1, PROD>(a, Pi_v, out, P, H, st);
  if (a.B <= 2) return launch_decode_qb<KBITS, VBITS, 2, PROD>(a, Pi_v, out, P, H, st);
  if (a.B <= 4 || KBITS == 3) return launch_decode_qb<KBITS, VBITS, 4, PROD>(a, Pi_v, out, P, H, st);
  return launch_decode_qb<KBITS, VBITS, 8, PROD>(a, Pi_v, out, P, H, st);
}

template <int KBITS, bool PROD>
cudaError_t launch_decode_k(const SplitArgs& a, int v_bits, const float* Pi_v, float* out, int P, int H,
                            cudaStream_t st) {
  switch (v_bits) {
    case 1: return launch_decode_kv<KBITS, 1, PROD>(a, Pi_v, out, P, H, st);
    case 2: return launch_decode_kv<KBITS, 2, PROD>(a, Pi_v, out, P, H, st);
    default: return launch_decode_kv<KBITS, 3, PROD>(a, Pi_v, out, P, H, st);
  }
}

template <bool PROD>
cudaError_t launch_decode(const SplitArgs& a, int k_bits, int v_bits, const float* Pi_v, float* out, int P,
                          int H, cudaStream_t st) {
  switch (k_bits) {
    case 1: return launch_decode_k<1, PROD>(a, v_bits, Pi_v, out, P, H, st);
    case 2: return launch_decode_k<2, PROD>(a, v_bits, Pi_v, out, P, H, st);
    default: return launch_decode_k<3, PROD>(a, v_bits, Pi_v, out, P, H, st);
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
  SplitArgs a = {A, nullptr, k_plane, nullptr, k_norm, k_cb, v_plane, v_norm, v_cb, part, B, S, 0, 0, scale, 0.f};
  return launch_decode<false>(a, k_bits, v_bits, Pi_v, out, P, H, st);
}

cudaError_t launch_decode_prod(const float* A, const float* T, const uint8_t* k_plane,
                               const uint8_t* k_sign, const uint16_t* k_gamma, const float* k_cb,
                               int k_bits, const uint8_t* v_plane, const uint16_t* v_norm,
                               const float* v_cb, int v_bits, const float* Pi_v, float* out,
                               float* part, int P, int H, int B, int S, float scale, cudaStream_t st) {
  SplitArgs a = {A, T, k_plane, k_sign, k_gamma, k_cb, v_plane, v_norm, v_cb, part, B, S, 0, 0, scale,
                 qjl_scale(128)};
  return launch_decode<true>(a, k_bits, v_bits, Pi_v, out, P, H, st);
}

}  // namespace tq

namespace tq {
cudaError_t take_faults_decode(unsigned int* bits) { return take_unit_faults(bits); }
}  // namespace tq
