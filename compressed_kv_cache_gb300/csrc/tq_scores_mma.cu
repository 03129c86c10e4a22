// bf16 tensor-core scorer (TQ_PATH_BF16_MMA), D = 128, tcgen05 + TMEM.
//
// The extended-2D form of the TurboQuant_prod score ("Implementing TurboQuant
// on NVIDIA's AGX Thor", zededa.com, v5 "Extended 2D": <[Pi q | S q], [c | sigma]>
// over R^{2D}) makes a block of scores one dense contraction with K = 2D = 256:
//
//   X[s, 0:128]   = c[idx[s, :]]      (bf16, dequantised in shared memory)
//   X[s, 128:256] = sigma[s, :]       (+1 / -1, exact in bf16)
//   Y[b, 0:128]   = A[b, :],  Y[b, 128:256] = T[b, :]   (bf16, round to nearest even)
//   mse[s, b] = sum_{k<128} X Y,  res[s, b] = sum_{k>=128} X Y   (fp32, in TMEM)
//   score[b, s] = mse[s, b] + (sqrt(pi/2)/D) gamma[s] res[s, b]   (fp32 epilogue)
//
// Tile: M = 128 keys (TMEM lanes) x N = up to 128 queries x K = 256, as 16
// tcgen05.mma.kind::f16 instructions of K = 16 (8 into the mse accumulator,
// 8 into the residual accumulator).  Both operands are K-major in the
// no-swizzle canonical layout: 8-row x 16-byte core matrices, row groups 128 B
// apart (SBO), K-adjacent core matrices one row-group column apart (LBO).
//
// One persistent CTA per SM, warp-specialised, 17 warps:
//   warps 0-7   producers: thread = (key row, half); load the next tile's rows into
//               registers, wait for a free shared-memory stage, dequantise into it,
//               arrive on x_full;
//   warps 8-15  epilogue: two warps per TMEM lane quarter (each drains half of the N
//               columns); wait for a full accumulator stage, tcgen05.ld, apply
//               gamma, coalesced global stores, arrive on acc_empty;
//   warp 16     MMA: allocates TMEM; one lane waits for x_full and acc_empty, issues
//               the 16 MMAs of a tile and commits them to x_empty and acc_full.
// Two shared-memory stages and two TMEM accumulator stages, so dequantisation of tile
// i+1, the MMAs of tile i and the stores of tile i-1 run at the same time.  Every wait
// on an mbarrier is bounded; a wait that runs out raises a CTA-wide abort flag, every
// role leaves its loop (the epilogue writes NaN for a tile it could not drain), and
// TMEM is still released.
#include <atomic>

#include "tq_internal.cuh"

namespace tq {
namespace {

constexpr int kM = 128;                 // keys per tile
constexpr int kK = 256;                 // 2D
constexpr int kProducerThreads = 256;   // warps 0-7
constexpr int kEpilogueThreads = 256;   // warps 8-15
constexpr int kMmaWarp = 16;
constexpr int kThreads = kProducerThreads + kEpilogueThreads + 32;
constexpr int kMaxN = 128;              // queries per tile
constexpr int kXBytes = kM * kK * 2;    // 64 KB per key-tile buffer
constexpr uint32_t kWaitPolls = 1u << 22;

enum Layout { kUnpackedSmallC = 0, kUnpackedLargeC = 1, kPacked1 = 2, kPacked2 = 3, kPacked3 = 4 };

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---- mbarrier --------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// ---- tcgen05 ---------------------------------------------------------------
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void tmem_alloc(uint32_t slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
// Shared-memory matrix descriptor, no swizzle, K-major canonical layout.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return static_cast<uint64_t>((saddr >> 4) & 0x3FFFu) |
         (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
         (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46);
}
// Instruction descriptor of kind::f16: fp32 accumulator, bf16 A and B, both K-major.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t (&v)[8]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]),
                 "=r"(v[6]), "=r"(v[7])
               : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}

__device__ __forceinline__ uint32_t bf16_bits(float x) {
  return static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(x)));
}

// +1/-1 bf16 pair for sign bits b0 (low element) and b1 (high element), bit = 1 means +1.
__device__ __forceinline__ uint32_t sign_pair(uint32_t neg_bits, int j) {
  return 0x3F803F80u | (((neg_bits >> (2 * j)) & 1u) << 15) | (((neg_bits >> (2 * j + 1)) & 1u) << 31);
}

struct Params {
  const float* A;
  const float* T;
  const uint8_t* idx;      // [P,S,D] codes (unpacked) or [P,S,D*bits/8] plane (packed)
  const uint8_t* signs;    // [P,S,D] int8 (unpacked) or [P,S,D/8] plane (packed)
  const void* gamma;       // fp32 (unpacked) or fp16 (packed) [P,S]
  const float* codebook;
  float* scores;
  int B, S, C, NT, key_tiles, tmem_cols;
  float kappa;
};

// Raw bytes of one key row held in registers between the load and the dequantisation,
// so that the next tile's loads are in flight while the producer waits for a stage.
// Producer thread t: row r = t % 128, half t / 128 (0: the code row, 1: the sign row).
template <int LAYOUT>
struct RawRow {
  static constexpr int kBits = LAYOUT >= kPacked1 ? LAYOUT - kPacked1 + 1 : 8;
  static constexpr int kVec = LAYOUT >= kPacked1 ? kBits : 8;   // uint4 per code row
  uint4 v[kVec];
  bool valid;
};

template <int LAYOUT>
__device__ __forceinline__ void load_row(const Params& prm, int p, int kt, RawRow<LAYOUT>& raw) {
  const int r = threadIdx.x & (kM - 1);
  const int half = threadIdx.x >> 7;
  const int s = kt * kM + r;
  raw.valid = s < prm.S;
  if (!raw.valid) return;
  const size_t key = static_cast<size_t>(p) * prm.S + s;
  if constexpr (LAYOUT >= kPacked1) {
    constexpr int kBits = RawRow<LAYOUT>::kBits;
    if (half == 0) {
      const uint4* src = reinterpret_cast<const uint4*>(prm.idx + key * (16 * kBits));
#pragma unroll
      for (int i = 0; i < kBits; ++i) raw.v[i] = __ldg(src + i);
    } else {
      raw.v[0] = __ldg(reinterpret_cast<const uint4*>(prm.signs + key * 16));
    }
  } else {
    const uint4* src = reinterpret_cast<const uint4*>((half == 0 ? prm.idx : prm.signs) + key * 128);
#pragma unroll
    for (int i = 0; i < 8; ++i) raw.v[i] = __ldg(src + i);
  }
}

// Dequantise the row into the X buffer at `xbuf` (shared address): half 0 writes the
// 128 centroids (core-matrix columns 0..15), half 1 the 128 signs (columns 16..31).
template <int LAYOUT>
__device__ __forceinline__ void store_row(const Params& prm, const RawRow<LAYOUT>& raw,
                                          uint32_t xbuf, const uint32_t* lut,
                                          const uint16_t* cbf) {
  constexpr int kBits = RawRow<LAYOUT>::kBits;
  const int r = threadIdx.x & (kM - 1);
  const int half = threadIdx.x >> 7;
  const uint32_t rowbase = xbuf + r * 16 + (half ? 16 * 2048 : 0);
  if (!raw.valid) {
#pragma unroll
    for (int kc = 0; kc < 16; ++kc) st_shared_v4(rowbase + kc * 2048, 0, 0, 0, 0);
    return;
  }
  if (half == 0) {
    if constexpr (LAYOUT >= kPacked1) {
      constexpr int kWords = 4 * kBits;
      uint32_t w[kWords + 1];
#pragma unroll
      for (int i = 0; i < kBits; ++i) {
        w[4 * i] = raw.v[i].x; w[4 * i + 1] = raw.v[i].y; w[4 * i + 2] = raw.v[i].z; w[4 * i + 3] = raw.v[i].w;
      }
      w[kWords] = 0u;
#pragma unroll
      for (int kc = 0; kc < 16; ++kc) {
        const int off = 8 * kBits * kc;                 // 8 codes = 8*bits bits
        const int wi = off >> 5, sh = off & 31;
        const uint64_t pair = (static_cast<uint64_t>(w[wi + 1]) << 32) | w[wi];
        const uint32_t v = static_cast<uint32_t>(pair >> sh);
        constexpr uint32_t kPm = (1u << (2 * kBits)) - 1u;
        st_shared_v4(rowbase + kc * 2048, lut[v & kPm], lut[(v >> (2 * kBits)) & kPm],
                     lut[(v >> (4 * kBits)) & kPm], lut[(v >> (6 * kBits)) & kPm]);
      }
    } else {
#pragma unroll
      for (int c2 = 0; c2 < 8; ++c2) {                  // 16 codes per 16-byte vector
        const uint32_t ws[4] = {raw.v[c2].x, raw.v[c2].y, raw.v[c2].z, raw.v[c2].w};
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t o[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const uint32_t word = ws[2 * h + (q >> 1)];
            const uint32_t b0 = (word >> (16 * (q & 1))) & 0xFFu;
            const uint32_t b1 = (word >> (16 * (q & 1) + 8)) & 0xFFu;
            if constexpr (LAYOUT == kUnpackedSmallC) {
              o[q] = lut[b0 + prm.C * b1];
            } else {
              o[q] = static_cast<uint32_t>(cbf[b0]) | (static_cast<uint32_t>(cbf[b1]) << 16);
            }
          }
          st_shared_v4(rowbase + (2 * c2 + h) * 2048, o[0], o[1], o[2], o[3]);
        }
      }
    }
  } else {
    if constexpr (LAYOUT >= kPacked1) {
      const uint32_t ws[4] = {~raw.v[0].x, ~raw.v[0].y, ~raw.v[0].z, ~raw.v[0].w};  // 1 = sigma -1
#pragma unroll
      for (int kc = 0; kc < 16; ++kc) {
        const uint32_t nb = (ws[kc >> 2] >> (8 * (kc & 3))) & 0xFFu;
        st_shared_v4(rowbase + kc * 2048, sign_pair(nb, 0), sign_pair(nb, 1), sign_pair(nb, 2),
                     sign_pair(nb, 3));
      }
    } else {
#pragma unroll
      for (int c2 = 0; c2 < 8; ++c2) {
        const uint32_t ws[4] = {raw.v[c2].x, raw.v[c2].y, raw.v[c2].z, raw.v[c2].w};
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t o[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const uint32_t u = ws[2 * h + (q >> 1)] >> (16 * (q & 1));   // bytes b0 (low), b1
            o[q] = 0x3F803F80u | ((u & 0x80u) << 8) | ((u & 0x8000u) << 16);
          }
          st_shared_v4(rowbase + (2 * c2 + h) * 2048, o[0], o[1], o[2], o[3]);
        }
      }
    }
  }
}

// Bounded wait that also gives up once another role has raised the abort flag.
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
  for (uint32_t i = 0; i < kWaitPolls; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 255u) == 255u && *abort_flag) return false;
  }
  *abort_flag = 1;
  return false;
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(bar) : "memory");
}

template <int LAYOUT>
__global__ void __launch_bounds__(kThreads, 1) scores_mma_kernel(Params prm) {
  extern __shared__ __align__(1024) uint8_t smem[];
  // [X0 64K][X1 64K][Y NT*512][lut 256 words][cbf 256 halves][8 mbarriers][tmem slot]
  uint8_t* X = smem;
  uint8_t* Yp = X + 2 * kXBytes;
  uint32_t* lut = reinterpret_cast<uint32_t*>(Yp + prm.NT * kK * 2);
  uint16_t* cbf = reinterpret_cast<uint16_t*>(lut + 256);
  uint64_t* bars = reinterpret_cast<uint64_t*>(cbf + 256);   // x_full[2], x_empty[2], acc_full[2], acc_empty[2]
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 8);
  __shared__ int abort_flag;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int p = blockIdx.z;
  const int q0 = blockIdx.y * prm.NT;
  const int NT = prm.NT;
  const uint32_t x_full = smem_u32(bars), x_empty = smem_u32(bars + 2);
  const uint32_t acc_full = smem_u32(bars + 4), acc_empty = smem_u32(bars + 6);

  // --- set-up: TMEM, barriers, tables, the query operand ---
  if (warp == kMmaWarp) tmem_alloc(smem_u32(tslot), prm.tmem_cols);
  if (tid == 0) {
    for (int b = 0; b < 2; ++b) {
      mbar_init(x_full + 8 * b, kProducerThreads);
      mbar_init(x_empty + 8 * b, 1);
      mbar_init(acc_full + 8 * b, 1);
      mbar_init(acc_empty + 8 * b, kEpilogueThreads);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    abort_flag = 0;
  }
  const int C = prm.C;
  for (int e = tid; e < 256; e += kThreads) {
    cbf[e] = e < C ? static_cast<uint16_t>(bf16_bits(prm.codebook[e])) : 0;
  }
  __syncthreads();
  if constexpr (LAYOUT == kUnpackedSmallC) {
    for (int e = tid; e < C * C; e += kThreads) lut[e] = cbf[e % C] | (static_cast<uint32_t>(cbf[e / C]) << 16);
  } else if constexpr (LAYOUT >= kPacked1) {
    constexpr int kBits = LAYOUT - kPacked1 + 1;
    constexpr int kPc = 1 << kBits;
    for (int e = tid; e < kPc * kPc; e += kThreads)
      lut[e] = cbf[e & (kPc - 1)] | (static_cast<uint32_t>(cbf[e >> kBits]) << 16);
  }
  {  // Y: query n (row) x 256 K, bf16, core-matrix layout; queries past B are zero
    const uint32_t ybase = smem_u32(Yp);
    const int ngroups = NT / 8;
    for (int e = tid; e < NT * 32; e += kThreads) {
      const int n = e >> 5, kc = e & 31;
      uint32_t o[4] = {0u, 0u, 0u, 0u};
      const int b = q0 + n;
      if (b < prm.B) {
        const float* src = (kc < 16 ? prm.A : prm.T) + (static_cast<size_t>(p) * prm.B + b) * 128 + (kc & 15) * 8;
        const float4 lo = __ldg(reinterpret_cast<const float4*>(src));
        const float4 hi = __ldg(reinterpret_cast<const float4*>(src + 4));
        o[0] = bf16_bits(lo.x) | (bf16_bits(lo.y) << 16);
        o[1] = bf16_bits(lo.z) | (bf16_bits(lo.w) << 16);
        o[2] = bf16_bits(hi.x) | (bf16_bits(hi.y) << 16);
        o[3] = bf16_bits(hi.z) | (bf16_bits(hi.w) << 16);
      }
      st_shared_v4(ybase + (kc * ngroups + (n >> 3)) * 128 + (n & 7) * 16, o[0], o[1], o[2], o[3]);
    }
  }
  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  const uint32_t xaddr0 = smem_u32(X);
  volatile int* abort_v = &abort_flag;

  if (warp < kProducerThreads / 32) {
    // ------------------------------ producers ------------------------------
    RawRow<LAYOUT> raw;
    int i = 0;
    if (static_cast<int>(blockIdx.x) < prm.key_tiles) load_row<LAYOUT>(prm, p, blockIdx.x, raw);
    for (int kt = blockIdx.x; kt < prm.key_tiles; kt += gridDim.x, ++i) {
      const int st = i & 1;
      if (!wait_or_abort(x_empty + 8 * st, ((i >> 1) & 1) ^ 1, abort_v)) break;
      store_row<LAYOUT>(prm, raw, xaddr0 + st * kXBytes, lut, cbf);
      fence_async_smem();
      mbar_arrive(x_full + 8 * st);
      if (kt + static_cast<int>(gridDim.x) < prm.key_tiles) load_row<LAYOUT>(prm, p, kt + gridDim.x, raw);
    }
  } else if (warp < (kProducerThreads + kEpilogueThreads) / 32) {
    // ------------------------------ epilogue -------------------------------
    const int e = warp - kProducerThreads / 32;      // 0..7
    const int lg = warp & 3;                         // TMEM lane quarter this warp may read
    const int colhalf = e >> 2;
    const int r = lg * 32 + lane;
    const int half_n = NT / 2;
    int i = 0;
    for (int kt = blockIdx.x; kt < prm.key_tiles; kt += gridDim.x, ++i) {
      const int as = i & 1;
      const int s = kt * kM + r;
      float g = 0.f;
      if (s < prm.S) {
        const size_t key = static_cast<size_t>(p) * prm.S + s;
        g = LAYOUT >= kPacked1
                ? __half2float(__ushort_as_half(__ldg(static_cast<const uint16_t*>(prm.gamma) + key)))
                : __ldg(static_cast<const float*>(prm.gamma) + key);
      }
      const float kg = prm.kappa * g;
      // tcgen05.ld is warp-collective: the whole warp takes the same branch
      const bool ok = __all_sync(0xffffffffu, wait_or_abort(acc_full + 8 * as, (i >> 1) & 1, abort_v));
      tc_fence_after();
      const uint32_t trow = tmem + (static_cast<uint32_t>(lg * 32) << 16) + as * 2 * NT;
      float* out = prm.scores + (static_cast<size_t>(p) * prm.B + q0) * prm.S + s;
      for (int c = colhalf * half_n; c < (colhalf + 1) * half_n; c += 8) {
        uint32_t m[8], q[8];
        if (ok) {
          tmem_ld8(trow + c, m);
          tmem_ld8(trow + NT + c, q);
          tmem_ld_wait();
        }
        if (s < prm.S) {
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            if (q0 + c + j < prm.B) {
              out[static_cast<size_t>(c + j) * prm.S] =
                  ok ? fmaf(kg, __uint_as_float(q[j]), __uint_as_float(m[j])) : __int_as_float(0x7fc00000);
            }
          }
        }
      }
      if (!ok) break;
      tc_fence_before();
      mbar_arrive(acc_empty + 8 * as);
    }
  } else {
    // -------------------------------- MMA ----------------------------------
    if (lane == 0) {
      const uint32_t yaddr = smem_u32(Yp);
      const uint32_t idesc = idesc_bf16(kM, NT);
      const uint32_t ylbo = (NT / 8) * 128;
      int i = 0;
      for (int kt = blockIdx.x; kt < prm.key_tiles; kt += gridDim.x, ++i) {
        const int st = i & 1;
        if (!wait_or_abort(x_full + 8 * st, (i >> 1) & 1, abort_v)) break;
        if (!wait_or_abort(acc_empty + 8 * st, ((i >> 1) & 1) ^ 1, abort_v)) break;
        tc_fence_after();
        const uint32_t xbuf = xaddr0 + st * kXBytes;
        const uint32_t dm = tmem + st * 2 * NT;
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const uint64_t ad = smem_desc(xbuf + k * 2 * 2048, 2048, 128);
          const uint64_t bd = smem_desc(yaddr + k * 2 * ylbo, ylbo, 128);
          mma_bf16(k < 8 ? dm : dm + NT, ad, bd, idesc, (k & 7) != 0);
        }
        mma_commit(x_empty + 8 * st);
        mma_commit(acc_full + 8 * st);
      }
    }
    __syncwarp();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tmem, prm.tmem_cols);
}

template <int LAYOUT>
cudaError_t launch_layout(const Params& prm, int P, int qtiles, cudaStream_t st) {
  // The opt-in shared-memory size is a per-device function attribute: on the first
  // launch on each device the kernel is given everything the device allows next to
  // its static shared memory (one CTA per SM either way), so every descriptor the
  // kernel builds addresses memory it owns.
  static std::atomic<int> dyn_bytes[64];
  constexpr size_t need = 2 * kXBytes + static_cast<size_t>(kMaxN) * kK * 2 + 256 * 4 + 256 * 2 +
                          8 * 8 + 16;
  int dev = 0, sms = 148;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  int smem = dyn_bytes[dev & 63].load(std::memory_order_acquire);
  if (smem == 0) {
    int optin = 0;
    e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess) return e;
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, scores_mma_kernel<LAYOUT>);
    if (e != cudaSuccess) return e;
    smem = optin - static_cast<int>(fa.sharedSizeBytes);
    if (smem < static_cast<int>(need)) return cudaErrorInvalidConfiguration;
    e = cudaFuncSetAttribute(scores_mma_kernel<LAYOUT>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    dyn_bytes[dev & 63].store(smem, std::memory_order_release);
  }
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int per = P * qtiles;
  int gx = (sms + per - 1) / per;
  gx = gx < 1 ? 1 : (gx > prm.key_tiles ? prm.key_tiles : gx);
  dim3 grid(gx, qtiles, P);
  scores_mma_kernel<LAYOUT><<<grid, kThreads, static_cast<size_t>(smem), st>>>(prm);
  return cudaGetLastError();
}

}  // namespace

bool mma_path_available() { return true; }

cudaError_t launch_scores_mma(const float* A, const float* T, const uint8_t* idx,
                              const void* signs, const void* gamma, const float* codebook,
                              float* scores, int P, int B, int S, int C, int idx_bits,
                              bool packed, cudaStream_t st) {
  Params prm;
  prm.A = A;
  prm.T = T;
  prm.idx = idx;
  prm.signs = static_cast<const uint8_t*>(signs);
  prm.gamma = gamma;
  prm.codebook = codebook;
  prm.scores = scores;
  prm.B = B;
  prm.S = S;
  prm.C = C;
  const int nt = B < kMaxN ? B : kMaxN;
  prm.NT = (nt + 15) / 16 * 16;
  const int qtiles = (B + prm.NT - 1) / prm.NT;
  prm.key_tiles = (S + kM - 1) / kM;
  int cols = 32;
  while (cols < 4 * prm.NT) cols <<= 1;
  prm.tmem_cols = cols;
  prm.kappa = qjl_scale(128);
  if (!packed) {
    return C <= 16 ? launch_layout<kUnpackedSmallC>(prm, P, qtiles, st)
                   : launch_layout<kUnpackedLargeC>(prm, P, qtiles, st);
  }
  switch (idx_bits) {
    case 1: return launch_layout<kPacked1>(prm, P, qtiles, st);
    case 2: return launch_layout<kPacked2>(prm, P, qtiles, st);
    default: return launch_layout<kPacked3>(prm, P, qtiles, st);
  }
}

}  // namespace tq
