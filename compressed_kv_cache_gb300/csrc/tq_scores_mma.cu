// bf16 tensor-core scorer (TQ_PATH_BF16_MMA), D = 128, tcgen05 + TMEM.
//
// The extended-2D form of the TurboQuant_prod score ("Implementing TurboQuant
// on NVIDIA's AGX Thor", zededa.com, v5 "Extended 2D": <[Pi q | S q], [c | sigma]>
// over R^{2D}) makes a block of scores one dense contraction with K = 2D = 256:
//
//   X[s, 0:128]   = c[idx[s, :]]                      (bf16, dequantised in shared memory)
//   X[s, 128:256] = sigma[s, :] * bf16(kappa gamma[s])  (the sign flips a bf16 magnitude)
//   Y[b, 0:128]   = A[b, :],  Y[b, 128:256] = T[b, :]   (bf16, round to nearest even)
//   score[b, s]   = sum_k X[s, k] Y[b, k]               (fp32, accumulated in TMEM)
// with kappa = sqrt(pi/2)/D.  Folding kappa*gamma into the sign operand rounds it to
// bf16 (relative 2^-9 on the residual term), well inside the path's bound, and leaves
// one accumulator per tile, so the epilogue only copies TMEM to memory (the HBM write of
// the scores is what bounds this kernel).
//
// Tile: M = 128 keys (TMEM lanes) x N = up to 128 queries x K = 256, as 16
// tcgen05.mma.kind::f16 instructions of K = 16 into one fp32 accumulator.  Both operands are K-major in the
// no-swizzle canonical layout: 8-row x 16-byte core matrices, row groups 128 B
// apart (SBO), K-adjacent core matrices one row-group column apart (LBO).
//
// Persistent CTAs, warp-specialised.  Full configuration (one CTA per SM, 26 warps):
//   warps 0-7   producers: thread = (key row, half of K); take the tile's rows from a
//               shared-memory stage (packed rows, filled by the loader) or from registers
//               (unpacked rows, loaded after the set-up), wait for their half of X to be
//               free, dequantise into it, arrive on that half's x_full;
//   warps 8-23  epilogue: four warps per TMEM lane quarter, a column group of 32 queries
//               each; wait for a full accumulator stage, tcgen05.ld, stage the 32 x 128
//               scores in shared memory and write them with one tensor store, arrive on
//               acc_empty;
//   warp 24     MMA: allocates TMEM; one lane waits for each half of X and for a free
//               accumulator stage, issues the tile's 16 MMAs (8 a half) and commits them
//               to the halves' x_empty and to acc_full;
//   warp 25     loader: bulk-copies packed code and sign rows into three stages, three
//               tiles ahead, and asks L2 for their gamma.
// One X stage split by K into halves with their own barriers, and four TMEM accumulator
// stages, so one half is dequantised while the MMAs read the other and the draining of
// earlier tiles overlaps both.  The lite configuration (two CTAs per SM, at most two
// tiles an SM) has four epilogue warps and no loader; at up to 32 queries its score tile
// sits in the unused half of the query operand region.  Every wait on an mbarrier is
// bounded; a wait that runs out raises a CTA-wide abort flag, every role leaves its loop
// (the epilogue writes NaN for a tile it could not drain), and TMEM is still released.
#include <atomic>

#include <cuda.h>            // CUtensorMap (types only; the encoder comes from the runtime)
#include <cudaTypedefs.h>

#include "tq_internal.cuh"

namespace tq {
namespace {

constexpr int kM = 128;                 // keys per tile
constexpr int kK = 256;                 // 2D
constexpr int kProducerThreads = 256;   // warps 0-7
// Two configurations: "full" (16 epilogue warps, 2 shared-memory stages, one CTA per SM)
// and "lite" (4 epilogue warps, 1 stage, two CTAs per SM) for problems with few tiles.
template <int EPIW> struct Cfg {
  static constexpr int kEpilogueThreads = EPIW * 32;
  static constexpr int kMmaWarp = 8 + EPIW;
  // the full configuration has one more warp: the loader of packed key rows
  static constexpr int kThreads = kProducerThreads + kEpilogueThreads + 32 + (EPIW == 16 ? 32 : 0);
};
constexpr int kRawStages = 3;           // packed key-row stages in flight (full configuration)
constexpr int kMaxN = 128;              // queries per tile
constexpr int kXBytes = kM * kK * 2;    // 64 KB per key-tile buffer

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
__device__ __forceinline__ void tmem_ld4(uint32_t taddr, uint32_t* v) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3])
               : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void st_shared_f32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared.b32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
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

// bf16 pair (+-mag, +-mag) for sign bits 2j (low element) and 2j+1 (high element) of
// neg_bits, where a set bit means sigma = -1; mag2 holds the magnitude in both halves.
__device__ __forceinline__ uint32_t sign_pair(uint32_t mag2, uint32_t neg_bits, int j) {
  return mag2 | (((neg_bits >> (2 * j)) & 1u) << 15) | (((neg_bits >> (2 * j + 1)) & 1u) << 31);
}

struct Params {
  const float* A;
  const float* T;
  const uint8_t* idx;      // [P,S,D] codes (unpacked) or [P,S,D*bits/8] plane (packed)
  const uint8_t* signs;    // [P,S,D] int8 (unpacked) or [P,S,D/8] plane (packed)
  const void* gamma;       // fp32 (unpacked) or fp16 (packed) [P,S]
  const float* codebook;
  const uint16_t* Ybf;     // query operand prepared by the transform (bulk-copied), or null
  float* scores;
  int B, S, C, NT, key_tiles, tmem_cols, acc_stages;
  float kappa;
  int tma_scores;          // smap describes scores as [P][B][S] fp32 (boxes of 128 keys x 32 queries)
  CUtensorMap smap;        // 64-byte aligned by its type
};

// Raw key bytes held in registers between the load and the dequantisation, so that the
// next tile's loads are in flight while the producer waits for a stage.
//
// Packed layouts: producer thread t owns row r = t % 128 and half t / 128 (0: the code
// row, 1: the sign row).
//
// Unpacked layouts (128-byte code and sign rows): producer warp w, lane l = 8g + j holds
// for rg, ch in {0, 1} the 16-byte chunk c = 4*ch + g of row r = 64*rg + 8*w + j, of the
// code rows (v[2*rg + ch]) and of the sign rows (v[4 + 2*rg + ch]).  One load instruction
// of a warp then reads 64 contiguous bytes of each of 8 consecutive rows (every sector it
// touches is used whole), and the eight lanes of a quarter-warp store 8 consecutive rows
// of one core-matrix column (no bank conflict).
template <int LAYOUT>
struct RawRow {
  static constexpr int kBits = LAYOUT >= kPacked1 ? LAYOUT - kPacked1 + 1 : 8;
  static constexpr int kVec = LAYOUT >= kPacked1 ? kBits : 8;
  uint4 v[kVec];
  float g[2];    // gamma: of the row (packed, sign half) or of rows r(rg = 0, 1) (unpacked)
  bool ok[2];    // the row (packed: ok[0]) or rows r(rg) exist (s < S)
};

template <int LAYOUT>
__device__ __forceinline__ void load_row(const Params& prm, int p, int kt, RawRow<LAYOUT>& raw) {
  if constexpr (LAYOUT >= kPacked1) {
    const int r = threadIdx.x & (kM - 1);
    const int half = threadIdx.x >> 7;
    const int s = kt * kM + r;
    raw.ok[0] = s < prm.S;
    if (!raw.ok[0]) return;
    const size_t key = static_cast<size_t>(p) * prm.S + s;
    constexpr int kBits = RawRow<LAYOUT>::kBits;
    if (half == 0) {
      const uint4* src = reinterpret_cast<const uint4*>(prm.idx + key * (16 * kBits));
#pragma unroll
      for (int i = 0; i < kBits; ++i) raw.v[i] = __ldg(src + i);
    } else {
      raw.v[0] = __ldg(reinterpret_cast<const uint4*>(prm.signs + key * 16));
      raw.g[0] = __half2float(__ushort_as_half(__ldg(static_cast<const uint16_t*>(prm.gamma) + key)));
    }
  } else {
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
#pragma unroll
    for (int rg = 0; rg < 2; ++rg) {
      const int s = kt * kM + 64 * rg + 8 * w + (l & 7);
      raw.ok[rg] = s < prm.S;
      if (!raw.ok[rg]) continue;
      const size_t key = static_cast<size_t>(p) * prm.S + s;
      const uint4* ci = reinterpret_cast<const uint4*>(prm.idx + key * 128);
      const uint4* cs = reinterpret_cast<const uint4*>(prm.signs + key * 128);
#pragma unroll
      for (int ch = 0; ch < 2; ++ch) {
        raw.v[2 * rg + ch] = __ldg(ci + 4 * ch + (l >> 3));
        raw.v[4 + 2 * rg + ch] = __ldg(cs + 4 * ch + (l >> 3));
      }
      raw.g[rg] = __ldg(static_cast<const float*>(prm.gamma) + key);
    }
  }
}

// Sixteen unpacked codes (one 16-byte chunk, coordinates 16c .. 16c+15) as two 16-byte
// core-matrix rows of centroids at `dst` (column 2c) and dst + 2048 (column 2c+1).
template <int LAYOUT>
__device__ __forceinline__ void store_code_chunk(const Params& prm, uint4 raw, uint32_t dst,
                                                 const uint32_t* lut, const uint16_t* cbf) {
  const uint32_t ws[4] = {raw.x, raw.y, raw.z, raw.w};
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
    st_shared_v4(dst + h * 2048, o[0], o[1], o[2], o[3]);
  }
}

// Sixteen unpacked int8 signs as +-mag bf16 (bit 7 of each byte is the sign of sigma).
__device__ __forceinline__ void store_sign_chunk(uint4 raw, uint32_t mag2, uint32_t dst) {
  const uint32_t ws[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    uint32_t o[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint32_t u = ws[2 * h + (q >> 1)] >> (16 * (q & 1));   // bytes b0 (low), b1
      o[q] = mag2 | ((u & 0x80u) << 8) | ((u & 0x8000u) << 16);
    }
    st_shared_v4(dst + h * 2048, o[0], o[1], o[2], o[3]);
  }
}

// Dequantise into the X buffer at `xbuf` (shared address): centroids in core-matrix
// columns 0..15, signs times bf16(kappa gamma) in columns 16..31; rows past S are zero.
// Words of the centroid lookup table in shared memory.  Packed codes: one copy of the
// table of code pairs per lane (entry e of lane l at word 32 e + l), so that the 32
// lookups of a warp, whatever their codes, fall in 32 distinct banks.  Unpacked codes
// with a small codebook: one table of C x C code pairs.
template <int LAYOUT>
constexpr int lut_words() {
  return LAYOUT >= kPacked1 ? 32 << (2 * RawRow<LAYOUT>::kBits) : 256;
}

template <int LAYOUT>
__device__ __forceinline__ void store_row(const Params& prm, const RawRow<LAYOUT>& raw,
                                          uint32_t xbuf, const uint32_t* lut,
                                          const uint16_t* cbf) {
  constexpr int kBits = RawRow<LAYOUT>::kBits;
  if constexpr (LAYOUT < kPacked1) {
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
#pragma unroll
    for (int rg = 0; rg < 2; ++rg) {
      const uint32_t rowbase = xbuf + (64 * rg + 8 * w + (l & 7)) * 16;
      const uint32_t mag = bf16_bits(prm.kappa * raw.g[rg]);      // kappa*gamma >= 0
#pragma unroll
      for (int ch = 0; ch < 2; ++ch) {
        const int c = 4 * ch + (l >> 3);
        const uint32_t dcode = rowbase + (2 * c) * 2048;
        const uint32_t dsign = rowbase + (16 + 2 * c) * 2048;
        if (raw.ok[rg]) {
          store_code_chunk<LAYOUT>(prm, raw.v[2 * rg + ch], dcode, lut, cbf);
          store_sign_chunk(raw.v[4 + 2 * rg + ch], mag | (mag << 16), dsign);
        } else {
          st_shared_v4(dcode, 0, 0, 0, 0);
          st_shared_v4(dcode + 2048, 0, 0, 0, 0);
          st_shared_v4(dsign, 0, 0, 0, 0);
          st_shared_v4(dsign + 2048, 0, 0, 0, 0);
        }
      }
    }
  } else {
    const int r = threadIdx.x & (kM - 1);
    const int half = threadIdx.x >> 7;
    const uint32_t rowbase = xbuf + r * 16 + (half ? 16 * 2048 : 0);
    if (!raw.ok[0]) {
#pragma unroll
      for (int kc = 0; kc < 16; ++kc) st_shared_v4(rowbase + kc * 2048, 0, 0, 0, 0);
      return;
    }
    if (half == 0) {
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
        const uint32_t ln = threadIdx.x & 31u;
        st_shared_v4(rowbase + kc * 2048, lut[((v & kPm) << 5) | ln], lut[(((v >> (2 * kBits)) & kPm) << 5) | ln],
                     lut[(((v >> (4 * kBits)) & kPm) << 5) | ln], lut[(((v >> (6 * kBits)) & kPm) << 5) | ln]);
      }
    } else {
      const uint32_t mag = bf16_bits(prm.kappa * raw.g[0]);      // kappa*gamma >= 0
      const uint32_t mag2 = mag | (mag << 16);
      const uint32_t ws[4] = {~raw.v[0].x, ~raw.v[0].y, ~raw.v[0].z, ~raw.v[0].w};  // 1 = sigma -1
#pragma unroll
      for (int kc = 0; kc < 16; ++kc) {
        const uint32_t nb = (ws[kc >> 2] >> (8 * (kc & 3))) & 0xFFu;
        st_shared_v4(rowbase + kc * 2048, sign_pair(mag2, nb, 0), sign_pair(mag2, nb, 1),
                     sign_pair(mag2, nb, 2), sign_pair(mag2, nb, 3));
      }
    }
  }
}

// Bounded wait (kWaitBudgetNs of the global timer) that also gives up once another
// role has raised the abort flag; the first role to run out records the fault.
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity, volatile int* abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 255u) == 0u) {
      if (*abort_flag) return false;
      if (global_ns() - t0 > kWaitBudgetNs) break;
    }
  }
  *abort_flag = 1;
  atomicOr(&g_wait_fault, kFaultMma);
  return false;
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(bar) : "memory");
}

// ---- named barriers and bulk stores (epilogue of the full configuration) ----
__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}
// Barrier over `nthreads` threads that also returns the AND of every thread's `pred`.
__device__ __forceinline__ bool named_bar_and(int id, int nthreads, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
      "barrier.red.and.pred q, %2, %3, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(pred)), "r"(id), "r"(nthreads)
      : "memory");
  return r != 0;
}
// Store one shared-memory box [1][32][128] fp32 to scores[z][y .. y+31][x .. x+127]
// (the tensor map clips the parts past S and past B).
__device__ __forceinline__ void tma_store_box(const CUtensorMap* map, int x, int y, int z, uint32_t ssrc) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y), "r"(z), "r"(ssrc)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

template <int LAYOUT, int EPIW, int XS>
// The lite configuration keeps to 64 registers a thread: two of its CTAs then fit on an
// SM next to a CTA of the query transform, so that none of them waits for the transform's
// CTAs to leave before it can start (programmatic dependent launch).
__global__ void __launch_bounds__(Cfg<EPIW>::kThreads) __maxnreg__(EPIW == 4 ? 64 : 72)
scores_mma_kernel(const __grid_constant__ Params prm) {
  constexpr int kEpilogueThreads = Cfg<EPIW>::kEpilogueThreads;
  constexpr int kMmaWarp = Cfg<EPIW>::kMmaWarp;
  constexpr int kThreads = Cfg<EPIW>::kThreads;
  extern __shared__ __align__(1024) uint8_t smem[];
  // [X: XS x 64K][Y NT*512][scores NT*512][key rows: kRawStages x 128 x (code row + sign
  // row), full and packed][lut lut_words()][cbf 256 halves][24 mbarriers][tmem slot]
  constexpr bool kRawTma = EPIW == 16 && LAYOUT >= kPacked1;     // key rows by the copy engine
  // The score tile of the tensor-store epilogue: a region of its own in the full
  // configuration; in the lite one, whose query operand region is sized for 64 queries,
  // the half that a tile of at most 32 queries leaves unused.
  const bool sbuf_on = EPIW == 16 || prm.NT <= 32;
  constexpr int kCodeRow = 16 * RawRow<LAYOUT>::kBits;             // bytes of codes per packed key
  constexpr int kRawIdx = kM * kCodeRow, kRawSgn = kM * 16;        // bytes per stage
  uint8_t* X = smem;
  uint8_t* Yp = X + XS * kXBytes;
  float* sbuf = reinterpret_cast<float*>(Yp + prm.NT * kK * 2);   // [NT columns][128 keys]
  uint8_t* rawp = reinterpret_cast<uint8_t*>(sbuf) + (sbuf_on ? prm.NT * 512 : 0);
  uint32_t* lut = reinterpret_cast<uint32_t*>(rawp + (kRawTma ? kRawStages * (kRawIdx + kRawSgn) : 0));
  uint16_t* cbf = reinterpret_cast<uint16_t*>(lut + lut_words<LAYOUT>());
  // x_full[2] x_empty[2] acc_full[4] acc_empty[4] y raw_full[3] raw_empty[3]
  uint64_t* bars = reinterpret_cast<uint64_t*>(cbf + 256);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 24);
  __shared__ int abort_flag;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int p = blockIdx.z;
  const int q0 = blockIdx.y * prm.NT;
  const int NT = prm.NT;
  const uint32_t x_full = smem_u32(bars), x_empty = smem_u32(bars + 2);
  const uint32_t acc_full = smem_u32(bars + 4), acc_empty = smem_u32(bars + 8);
  const uint32_t y_bar = smem_u32(bars + 12);
  const uint32_t raw_full = smem_u32(bars + 13), raw_empty = smem_u32(bars + 16);
  const int AS = prm.acc_stages;
  const int gx = gridDim.x;
  // Stage j of this CTA's packed key rows (tile blockIdx.x + j*gx) into raw stage j % 3:
  // code rows and sign rows, two bulk copies completing bytes on raw_full.
  auto issue_rows = [&](int j) {
    const int kt = static_cast<int>(blockIdx.x) + j * gx;
    const int n = min(kM, prm.S - kt * kM);
    const int rs = j % kRawStages;
    const size_t key0 = static_cast<size_t>(p) * prm.S + static_cast<size_t>(kt) * kM;
    const uint32_t fb = raw_full + 8 * rs;
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(fb),
                 "r"(static_cast<uint32_t>(n * (kCodeRow + 16)))
                 : "memory");
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(rawp + rs * kRawIdx)),
                 "l"(prm.idx + key0 * kCodeRow), "r"(static_cast<uint32_t>(n * kCodeRow)), "r"(fb)
                 : "memory");
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(rawp + kRawStages * kRawIdx + rs * kRawSgn)),
                 "l"(prm.signs + key0 * 16), "r"(static_cast<uint32_t>(n * 16)), "r"(fb)
                 : "memory");
    // gamma stays a register load of the sign-half producers, one tile ahead; asked of L2
    // here, three tiles ahead, it no longer stalls them on HBM latency (measured on c4:
    // 1.85 to 1.57 us a tile)
    prefetch_l2(static_cast<const uint16_t*>(prm.gamma) + key0, static_cast<size_t>(n) * 2);
  };

  // With packed rows staged by the loader, the single X stage is split by K: barrier 0
  // guards the centroid columns (producer warps 0-3), barrier 1 the sign columns (warps
  // 4-7), and the MMA frees each half as soon as its 8 MMAs have read it.
  constexpr bool kSplitX = kRawTma && XS == 1;
  if (tid == 0) {
    if constexpr (kSplitX) {
      for (int b = 0; b < 2; ++b) {
        mbar_init(x_full + 8 * b, kProducerThreads / 64);   // one arrival per warp of the half
        mbar_init(x_empty + 8 * b, 1);
      }
    } else {
      for (int b = 0; b < XS; ++b) {
        mbar_init(x_full + 8 * b, kProducerThreads / 32);   // one arrival per producer warp
        mbar_init(x_empty + 8 * b, 1);
      }
    }
    for (int b = 0; b < 4; ++b) {
      mbar_init(acc_full + 8 * b, 1);
      mbar_init(acc_empty + 8 * b, kEpilogueThreads / 32);  // one arrival per epilogue warp
    }
    mbar_init(y_bar, 1);
    for (int b = 0; b < kRawStages; ++b) {
      mbar_init(raw_full + 8 * b, 1);
      mbar_init(raw_empty + 8 * b, kProducerThreads / 32);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    abort_flag = 0;
    // the first stages of key rows are requested at once (the stages start empty); the
    // copy engine reads them while the rest of the set-up runs
    if constexpr (kRawTma) {
      for (int j = 0; j < kRawStages && static_cast<int>(blockIdx.x) + j * gx < prm.key_tiles; ++j) issue_rows(j);
    }
  }
  // The codebook (independent of the transform) is requested first, ahead of the key rows.
  const int C = prm.C;
  const float cval = tid < C ? __ldg(prm.codebook + tid) : 0.f;
  // Without the loader warp, one thread asks L2 for the first tile's key rows at entry
  // (a hint, carried out by the copy engine), and the producers load them into registers
  // only after the set-up.  Loaded into registers at entry, the rows of every CTA queue
  // in the SMs' load path ahead of the set-up's own reads and of the transform running
  // beside this grid, and hold up the query operand (measured on c1: the query operand
  // arrived 2.2 us later that way).
  constexpr bool kTwoDeep = false;   // one tile ahead: the register budget of 800 threads
  RawRow<LAYOUT> raw0, raw1;
  if (!kRawTma && tid == 0 && static_cast<int>(blockIdx.x) < prm.key_tiles) {
    const size_t k0 = static_cast<size_t>(p) * prm.S + static_cast<size_t>(blockIdx.x) * kM;
    const size_t n = static_cast<size_t>(min(kM, prm.S - static_cast<int>(blockIdx.x) * kM));
    if constexpr (LAYOUT >= kPacked1) {
      prefetch_l2(prm.idx + k0 * kCodeRow, n * kCodeRow);
      prefetch_l2(prm.signs + k0 * 16, n * 16);
      prefetch_l2(static_cast<const uint16_t*>(prm.gamma) + k0, n * 2);
    } else {
      prefetch_l2(prm.idx + k0 * 128, n * 128);
      prefetch_l2(prm.signs + k0 * 128, n * 128);
      prefetch_l2(static_cast<const float*>(prm.gamma) + k0, n * 4);
    }
  }

  // --- set-up: TMEM, barriers, tables, the query operand ---
  if (warp == kMmaWarp) tmem_alloc(smem_u32(tslot), prm.tmem_cols);
  const uint32_t ybytes = static_cast<uint32_t>(NT) * 512u;
  // With the query operand prepared by the transform, only the MMA issuer reads what the
  // transform wrote: it alone waits for that grid (below), and the set-up and the
  // producers' first tiles proceed while the transform is still running.
  if (prm.Ybf == nullptr) {
    // A and T are read after this wait, which returns once a transform launched right
    // before this grid (programmatic dependent launch) is complete.  One round trip for
    // the set-up's global inputs: each thread requests its chunks of A/T, then converts
    // and stores them.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // Y: query n (row) x 256 K, bf16, core-matrix layout; queries past B are zero
    const uint32_t ybase = smem_u32(Yp);
    const int ngroups = NT / 8;
    // pairs of float4 in flight per thread (fewer next to the larger unpacked key registers)
    constexpr int kBatch = LAYOUT >= kPacked1 ? 4 : 2;
    for (int e0 = tid; e0 < NT * 32; e0 += kThreads * kBatch) {
      float4 lo[kBatch], hi[kBatch];
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int e = e0 + u * kThreads;
        const int n = e >> 5, kc = e & 31;
        lo[u] = hi[u] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (e < NT * 32 && q0 + n < prm.B) {
          const float* src = (kc < 16 ? prm.A : prm.T) + (static_cast<size_t>(p) * prm.B + q0 + n) * 128 + (kc & 15) * 8;
          lo[u] = __ldcg(reinterpret_cast<const float4*>(src));
          hi[u] = __ldcg(reinterpret_cast<const float4*>(src + 4));
        }
      }
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int e = e0 + u * kThreads;
        if (e < NT * 32) {
          const int n = e >> 5, kc = e & 31;
          st_shared_v4(ybase + (kc * ngroups + (n >> 3)) * 128 + (n & 7) * 16,
                       bf16_bits(lo[u].x) | (bf16_bits(lo[u].y) << 16), bf16_bits(lo[u].z) | (bf16_bits(lo[u].w) << 16),
                       bf16_bits(hi[u].x) | (bf16_bits(hi[u].y) << 16), bf16_bits(hi[u].z) | (bf16_bits(hi[u].w) << 16));
        }
      }
    }
  }
  if (tid < 256) cbf[tid] = tid < C ? static_cast<uint16_t>(bf16_bits(cval)) : 0;
  __syncthreads();
  if constexpr (LAYOUT == kUnpackedSmallC) {
    for (int e = tid; e < C * C; e += kThreads) lut[e] = cbf[e % C] | (static_cast<uint32_t>(cbf[e / C]) << 16);
  } else if constexpr (LAYOUT >= kPacked1) {
    constexpr int kBits = LAYOUT - kPacked1 + 1;
    constexpr int kPc = 1 << kBits;
    for (int i = tid; i < kPc * kPc * 32; i += kThreads) {
      const int e = i >> 5;
      lut[i] = cbf[e & (kPc - 1)] | (static_cast<uint32_t>(cbf[e >> kBits]) << 16);
    }
  }
  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (!kRawTma && warp < kProducerThreads / 32) {
    if (static_cast<int>(blockIdx.x) < prm.key_tiles) load_row<LAYOUT>(prm, p, blockIdx.x, raw0);
    if (kTwoDeep && static_cast<int>(blockIdx.x) + gx < prm.key_tiles)
      load_row<LAYOUT>(prm, p, blockIdx.x + gx, raw1);
  }
  const uint32_t tmem = *tslot;
  const uint32_t xaddr0 = smem_u32(X);
  volatile int* abort_v = &abort_flag;

  if (warp < kProducerThreads / 32) {
    // ------------------------------ producers ------------------------------
    auto consume = [&](const RawRow<LAYOUT>& raw, int i) -> bool {
      const int st = i % XS;
      const int b = kSplitX ? (tid >> 7) : st;          // split: this thread's half of X
      const uint32_t parity = kSplitX ? ((i & 1) ^ 1) : (((i / XS) & 1) ^ 1);
      if (!wait_or_abort(x_empty + 8 * b, parity, abort_v)) return false;
      store_row<LAYOUT>(prm, raw, xaddr0 + st * kXBytes, lut, cbf);
      fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(x_full + 8 * b);
      return true;
    };
    if constexpr (kRawTma) {
      // key rows from the shared-memory stages the loader fills; gamma (2 bytes a key,
      // sign half only) is read from global memory one tile ahead
      const int r = tid & (kM - 1), half = tid >> 7;
      auto load_g = [&](int kt) -> float {
        const int s = kt * kM + r;
        return half == 1 && s < prm.S
                   ? __half2float(__ushort_as_half(__ldg(static_cast<const uint16_t*>(prm.gamma) +
                                                         static_cast<size_t>(p) * prm.S + s)))
                   : 0.f;
      };
      float g_cur = static_cast<int>(blockIdx.x) < prm.key_tiles ? load_g(blockIdx.x) : 0.f;
      int i = 0;
      for (int kt = blockIdx.x; kt < prm.key_tiles; kt += gx, ++i) {
        const float g_next = kt + gx < prm.key_tiles ? load_g(kt + gx) : 0.f;
        const int rs = i % kRawStages;
        if (!wait_or_abort(raw_full + 8 * rs, (i / kRawStages) & 1, abort_v)) break;
        RawRow<LAYOUT> raw;
        raw.ok[0] = kt * kM + r < prm.S;
        if (half == 0) {
#pragma unroll
          for (int v = 0; v < RawRow<LAYOUT>::kBits; ++v)
            raw.v[v] = *reinterpret_cast<const uint4*>(rawp + rs * kRawIdx + r * kCodeRow + 16 * v);
        } else {
          raw.v[0] = *reinterpret_cast<const uint4*>(rawp + kRawStages * kRawIdx + rs * kRawSgn + r * 16);
          raw.g[0] = g_cur;
        }
        // the rows are in registers: the stage may be refilled
        __syncwarp();
        if (lane == 0) mbar_arrive(raw_empty + 8 * rs);
        g_cur = g_next;
        if (!consume(raw, i)) break;
      }
    } else if constexpr (kTwoDeep) {
      // two register sets: tile i+2 is requested as soon as tile i has been stored
      int i = 0;
      for (int kt = blockIdx.x; kt < prm.key_tiles; kt += 2 * gx, i += 2) {
        if (!consume(raw0, i)) break;
        if (kt + 2 * gx < prm.key_tiles) load_row<LAYOUT>(prm, p, kt + 2 * gx, raw0);
        if (kt + gx >= prm.key_tiles) break;
        if (!consume(raw1, i + 1)) break;
        if (kt + 3 * gx < prm.key_tiles) load_row<LAYOUT>(prm, p, kt + 3 * gx, raw1);
      }
    } else {
      int i = 0;
      for (int kt = blockIdx.x; kt < prm.key_tiles; kt += gx, ++i) {
        if (!consume(raw0, i)) break;
        if (kt + gx < prm.key_tiles) load_row<LAYOUT>(prm, p, kt + gx, raw0);
      }
    }
  } else if (warp < (kProducerThreads + kEpilogueThreads) / 32) {
    // ------------------------------ epilogue -------------------------------
    const int e = warp - kProducerThreads / 32;      // 0..EPIW-1
    const int lg = warp & 3;                         // TMEM lane quarter this warp may read
    const int width = NT / (EPIW / 4);               // columns per warp, a multiple of 4
    const int cbeg = (e >> 2) * width;
    const int r = lg * 32 + lane;
    int i = 0;
    if (sbuf_on && prm.tma_scores && width == 32) {
      // 32 columns a warp (128 queries in the full configuration, 32 in the lite one) and
      // a tensor map of the scores.  The four warps of a column
      // group (one per lane quarter) drain their 32 columns into the shared score tile and
      // free the TMEM stage at once; one thread of the group then writes the 32 x 128
      // block with one tensor store, so the scores leave through the copy engine while
      // the warps go on to the next tile.
      const int grp = e >> 2;
      const bool issuer = lg == 0 && lane == 0;
      const uint32_t sb = smem_u32(sbuf) + cbeg * 512;
      for (int kt = blockIdx.x; kt < prm.key_tiles; kt += gridDim.x, ++i) {
        const int as = i % AS;
        const bool okw = __all_sync(0xffffffffu, wait_or_abort(acc_full + 8 * as, (i / AS) & 1, abort_v));
        if (issuer) bulk_wait_read();                 // the previous tile has left the buffer
        // the whole group takes the same branch (and may overwrite the buffer)
        const bool ok = named_bar_and(1 + grp, 128, okw);
        tc_fence_after();
        uint32_t v[32];
        if (ok) {
#pragma unroll
          for (int t = 0; t < 8; ++t) tmem_ld4(tmem + (static_cast<uint32_t>(lg * 32) << 16) + as * NT + cbeg + 4 * t, v + 4 * t);
          tmem_ld_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(acc_empty + 8 * as);
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = 0x7fc00000u;
        }
#pragma unroll
        for (int j = 0; j < 32; ++j) st_shared_f32(sb + j * 512 + r * 4, v[j]);
        fence_async_smem();
        named_bar_sync(1 + grp, 128);
        if (issuer && q0 + cbeg < prm.B) {
          tma_store_box(&prm.smap, kt * kM, q0 + cbeg, p, sb);
          bulk_commit();
        }
        if (!ok) break;
      }
      if (issuer) bulk_wait_all();
    } else {
    for (int kt = blockIdx.x; kt < prm.key_tiles; kt += gridDim.x, ++i) {
      const int as = i % AS;
      const int s = kt * kM + r;
      // tcgen05.ld is warp-collective: the whole warp takes the same branch
      const bool ok = __all_sync(0xffffffffu, wait_or_abort(acc_full + 8 * as, (i / AS) & 1, abort_v));
      tc_fence_after();
      const uint32_t trow = tmem + (static_cast<uint32_t>(lg * 32) << 16) + as * NT + cbeg;
      float* out = prm.scores + (static_cast<size_t>(p) * prm.B + q0 + cbeg) * prm.S + s;
      const int ncol = min(width, prm.B - (q0 + cbeg));
      for (int c0 = 0; c0 < width; c0 += 32) {        // batches of up to 32 columns, one wait each
        uint32_t v[32];
        if (ok) {
#pragma unroll
          for (int t = 0; t < 8; ++t)
            if (c0 + 4 * t < width) tmem_ld4(trow + c0 + 4 * t, v + 4 * t);
          tmem_ld_wait();
        }
        if (s < prm.S) {
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            if (c0 + j < ncol)
              out[static_cast<size_t>(c0 + j) * prm.S] = ok ? __uint_as_float(v[j]) : __int_as_float(0x7fc00000);
          }
        }
      }
      if (!ok) break;
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acc_empty + 8 * as);
    }
    }
  } else if (warp == kMmaWarp) {
    // -------------------------------- MMA ----------------------------------
    if (lane == 0) {
      const uint32_t yaddr = smem_u32(Yp);
      if (prm.Ybf != nullptr) {
        // the transform wrote this tile of the query operand: wait for that grid, then
        // one bulk copy
        asm volatile("griddepcontrol.wait;" ::: "memory");
        asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(y_bar),
                     "r"(ybytes)
                     : "memory");
        const uint16_t* src = prm.Ybf + (static_cast<size_t>(p) * gridDim.y + blockIdx.y) * NT * 256;
        asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(smem_u32(Yp)),
                     "l"(src), "r"(ybytes), "r"(y_bar)
                     : "memory");
      }
      bool y_ready = prm.Ybf == nullptr || wait_or_abort(y_bar, 0, abort_v);
      const uint32_t idesc = idesc_bf16(kM, NT);
      const uint32_t ylbo = (NT / 8) * 128;
      int i = 0;
      for (int kt = blockIdx.x; kt < prm.key_tiles && y_ready; kt += gridDim.x, ++i) {
        const int st = i % XS;
        const int as = i % AS;
        const uint32_t xbuf = xaddr0 + st * kXBytes;
        const uint32_t dm = tmem + as * NT;
        if constexpr (kSplitX) {
          // centroid half (K 0..127), then sign half (K 128..255), each freed on its own
          if (!wait_or_abort(x_full, i & 1, abort_v)) break;
          if (!wait_or_abort(acc_empty + 8 * as, ((i / AS) & 1) ^ 1, abort_v)) break;
          tc_fence_after();
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const uint64_t ad = smem_desc(xbuf + k * 2 * 2048, 2048, 128);
            const uint64_t bd = smem_desc(yaddr + k * 2 * ylbo, ylbo, 128);
            mma_bf16(dm, ad, bd, idesc, k != 0);
          }
          mma_commit(x_empty);
          if (!wait_or_abort(x_full + 8, i & 1, abort_v)) break;
          tc_fence_after();
#pragma unroll
          for (int k = 8; k < 16; ++k) {
            const uint64_t ad = smem_desc(xbuf + k * 2 * 2048, 2048, 128);
            const uint64_t bd = smem_desc(yaddr + k * 2 * ylbo, ylbo, 128);
            mma_bf16(dm, ad, bd, idesc, true);
          }
          mma_commit(x_empty + 8);
        } else {
          if (!wait_or_abort(x_full + 8 * st, (i / XS) & 1, abort_v)) break;
          if (!wait_or_abort(acc_empty + 8 * as, ((i / AS) & 1) ^ 1, abort_v)) break;
          tc_fence_after();
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            const uint64_t ad = smem_desc(xbuf + k * 2 * 2048, 2048, 128);
            const uint64_t bd = smem_desc(yaddr + k * 2 * ylbo, ylbo, 128);
            mma_bf16(dm, ad, bd, idesc, k != 0);
          }
          mma_commit(x_empty + 8 * st);
        }
        mma_commit(acc_full + 8 * as);
      }
    }
    __syncwarp();
  } else {
    // ------------------ loader (full configuration, packed rows) ------------------
    if (kRawTma && lane == 0) {
      int j = kRawStages;
      for (int kt = blockIdx.x + kRawStages * gx; kt < prm.key_tiles; kt += gx, ++j) {
        const int rs = j % kRawStages;
        if (!wait_or_abort(raw_empty + 8 * rs, ((j / kRawStages) & 1) ^ 1, abort_v)) break;
        issue_rows(j);
      }
    }
    __syncwarp();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tmem, prm.tmem_cols);
}

template <int LAYOUT, int EPIW, int XS>
cudaError_t launch_cfg(const Params& prm, int P, int qtiles, bool after_prepare, int sms,
                       cudaStream_t st) {
  using K = Cfg<EPIW>;
  constexpr bool kLite = EPIW == 4;
  // Dynamic shared memory: the lite configuration takes exactly its layout so that two
  // CTAs share an SM; the full one takes what the device allows next to its static
  // shared memory (one CTA per SM).  The opt-in size is a per-device attribute, set on
  // the first launch on each device.
  static std::atomic<int> dyn_bytes[64];
  constexpr int kNMax = kLite ? 64 : kMaxN;           // the lite configuration serves NT <= 64
  constexpr int kCodeRow = 16 * RawRow<LAYOUT>::kBits;
  constexpr size_t kRaw = (!kLite && LAYOUT >= kPacked1) ? kRawStages * kM * (kCodeRow + 16) : 0;
  constexpr size_t need = XS * static_cast<size_t>(kXBytes) + static_cast<size_t>(kNMax) * kK * 2 +
                          (kLite ? 0 : static_cast<size_t>(kNMax) * 512) + kRaw + lut_words<LAYOUT>() * 4 + 256 * 2 + 24 * 8 + 16;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  int smem = dyn_bytes[dev & 63].load(std::memory_order_acquire);
  if (smem == 0) {
    int optin = 0;
    e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess) return e;
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, scores_mma_kernel<LAYOUT, EPIW, XS>);
    if (e != cudaSuccess) return e;
    smem = kLite ? static_cast<int>(need) : optin - static_cast<int>(fa.sharedSizeBytes);
    if (smem < static_cast<int>(need) || smem > optin) return cudaErrorInvalidConfiguration;
    e = cudaFuncSetAttribute(scores_mma_kernel<LAYOUT, EPIW, XS>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(scores_mma_kernel<LAYOUT, EPIW, XS>,
                             cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (e != cudaSuccess) return e;
    dyn_bytes[dev & 63].store(smem, std::memory_order_release);
  }
  const int per = P * qtiles;
  const int slots = kLite ? 2 * sms : sms;
  int gx = (slots + per - 1) / per;
  gx = gx < 1 ? 1 : (gx > prm.key_tiles ? prm.key_tiles : gx);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(gx, qtiles, P);
  cfg.blockDim = dim3(K::kThreads);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = after_prepare ? 1 : 0;
  e = cudaLaunchKernelEx(&cfg, scores_mma_kernel<LAYOUT, EPIW, XS>, prm);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// At most two tiles per SM: two lighter CTAs per SM run every tile at once.
bool lite_layout(int NT, int64_t tiles, int sms) { return NT <= 64 && tiles <= 2LL * sms; }

template <int LAYOUT>
cudaError_t launch_layout(const Params& prm, int P, int qtiles, bool after_prepare, cudaStream_t st) {
  int dev = 0, sms = 148;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t tiles = static_cast<int64_t>(prm.key_tiles) * qtiles * P;
  if (lite_layout(prm.NT, tiles, sms)) return launch_cfg<LAYOUT, 4, 1>(prm, P, qtiles, after_prepare, sms, st);
  return launch_cfg<LAYOUT, 16, 1>(prm, P, qtiles, after_prepare, sms, st);
}

// Tensor map of the scores [P][B][S] fp32 for the bulk epilogue: boxes of 128 keys x 32
// queries x 1 problem.  Needs 16-byte row pitch (S % 4 == 0); false when it cannot be
// built, and the epilogue then stores from registers.
bool encode_scores_map(CUtensorMap* map, float* scores, int P, int B, int S) {
  static std::atomic<void*> encode{nullptr};
  static std::atomic<int> looked{0};
  if (S % 4 != 0) return false;
  if (!looked.load(std::memory_order_acquire)) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      fn = nullptr;
    encode.store(fn, std::memory_order_release);
    looked.store(1, std::memory_order_release);
  }
  auto fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(encode.load(std::memory_order_acquire));
  if (fn == nullptr) {
    (void)cudaGetLastError();
    return false;
  }
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(S), static_cast<cuuint64_t>(B), static_cast<cuuint64_t>(P)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(S) * 4, static_cast<cuuint64_t>(B) * S * 4};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(kM), 32, 1};
  const cuuint32_t estride[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, scores, dims, strides, box, estride,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool mma_path_available() { return true; }

bool mma_shares_sm(int P, int B, int S) {
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t tiles = static_cast<int64_t>((S + kM - 1) / kM) * mma_query_tiles(B) * P;
  return lite_layout(mma_query_tile(B), tiles, sms);
}

cudaError_t launch_scores_mma(const float* A, const float* T, const uint8_t* idx,
                              const void* signs, const void* gamma, const float* codebook,
                              float* scores, int P, int B, int S, int C, int idx_bits,
                              bool packed, bool after_prepare, cudaStream_t st,
                              const uint16_t* Ybf) {
  Params prm;
  prm.Ybf = Ybf;
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
  prm.NT = mma_query_tile(B);
  const int qtiles = mma_query_tiles(B);
  prm.key_tiles = (S + kM - 1) / kM;
  prm.acc_stages = 4;                      // 4 x NT <= 512 TMEM columns for NT <= 128
  int cols = 32;
  while (cols < prm.acc_stages * prm.NT) cols <<= 1;
  prm.tmem_cols = cols;
  prm.kappa = qjl_scale(128);
  prm.tma_scores = encode_scores_map(&prm.smap, scores, P, B, S) ? 1 : 0;
  if (!packed) {
    return C <= 16 ? launch_layout<kUnpackedSmallC>(prm, P, qtiles, after_prepare, st)
                   : launch_layout<kUnpackedLargeC>(prm, P, qtiles, after_prepare, st);
  }
  switch (idx_bits) {
    case 1: return launch_layout<kPacked1>(prm, P, qtiles, after_prepare, st);
    case 2: return launch_layout<kPacked2>(prm, P, qtiles, after_prepare, st);
    default: return launch_layout<kPacked3>(prm, P, qtiles, after_prepare, st);
  }
}

}  // namespace tq

namespace tq {
cudaError_t take_faults_mma(unsigned int* bits) { return take_unit_faults(bits); }
}  // namespace tq
