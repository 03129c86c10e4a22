/*
 * tq.h -- C ABI of libtq: raw TurboQuant_prod attention scores read straight
 * from a compressed key cache, on one NVIDIA Blackwell GPU (sm_103a).
 *
 * For query b and cached key s of a problem, the library computes
 *
 *   score[b,s] = <A_b, codebook[K_idx[s,:]]> + (sqrt(pi/2)/D) * gamma[s] * <T_b, sign[s,:]>
 *   with A_b = Pi q_b and T_b = S_mat q_b,
 *
 * with no softmax, no value read and no 1/sqrt(D) scale.  The query-side
 * transform is the identity of "TurboQuant Attention in CUDA: Transform the
 * Query, Reuse the Work" (riteshyadav.xyz), section "Move the transforms to
 * the query"; the estimator is TurboQuant_prod ("Implementing TurboQuant on
 * NVIDIA's AGX Thor", zededa.com, "Theorem 2: Unbiased Inner Products";
 * "TurboQuant: Rotate-then-Quantize KV Caches at 3 Bits", kanthi.in, §3,
 * TurboQuantProd).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Memory: unless stated otherwise every pointer is a DEVICE pointer owned by
 *   the caller.  The library allocates no memory.  Its only mutable device state
 *   is the fault bits of the bounded waits (tq_device_faults) and the fixed
 *   scratch array of tq_solve_packed_noalloc; every other call is safe to run
 *   concurrently on different streams as long as their output and workspace
 *   buffers do not overlap.
 * - Streams: every call is asynchronous on `stream` (0 = legacy default
 *   stream).  Outputs are valid once the stream reaches the call.
 * - Errors: argument errors are reported synchronously, before anything is
 *   launched (nothing is written).  A launch error reported by CUDA maps to
 *   TQ_ERR_LAUNCH.  Faults during execution surface at the caller's next
 *   synchronisation, as for any CUDA library.  Nothing is printed and no C++
 *   exception crosses the ABI.
 * - Layouts are dense and row-major.  P independent problems are laid out
 *   back to back: queries [P,B,D], keys [P,S,...], scores [P,B,S].  Problem p
 *   uses rotation and projection head p % H (grouped-query attention: all
 *   problems of one KV head share its Pi and S_mat).  The codebook is shared.
 * - Alignment: every array pointer must be 16-byte aligned
 *   (TQ_ERR_MISALIGNED otherwise).  Row pitches need no alignment.
 * - Indices: every code must be < C (unpacked) or < 2^idx_bits (packed); this
 *   is the caller's contract and is not checked on the device.
 */
#ifndef TQ_H
#define TQ_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  TQ_OK = 0,
  TQ_ERR_INVALID_VALUE = 1, /* null pointer, size <= 0 or out of range               */
  TQ_ERR_UNSUPPORTED = 2,   /* valid arguments no kernel of this library implements     */
  TQ_ERR_MISALIGNED = 3,    /* an array pointer is not 16-byte aligned                  */
  TQ_ERR_WORKSPACE = 4,     /* workspace null or smaller than tq_workspace_bytes()      */
  TQ_ERR_LAUNCH = 5         /* CUDA reported an error when the kernels were launched    */
} tq_status;

/* Element type of the queries Q. */
typedef enum { TQ_Q_F32 = 0, TQ_Q_BF16 = 1 } tq_qtype;

/* Arithmetic path of a scoring call.
 * TQ_PATH_FP32: CUDA-core fp32 throughout; max |err| <= 1e-5 (1 + |score|) against
 *   the float64 definition.
 * TQ_PATH_BF16_MMA: A and T rounded to bf16, centroids rounded to bf16, signs exact,
 *   products summed by the tensor cores in fp32; max |err| <= 2e-3 ||q_b||_2.
 *   Requires D == 128.
 * TQ_PATH_AUTO: the path tq_auto_path(B, D) names. */
typedef enum { TQ_PATH_AUTO = 0, TQ_PATH_FP32 = 1, TQ_PATH_BF16_MMA = 2 } tq_path;

/* Human-readable name of a status code (static string, never NULL). */
const char* tq_status_string(tq_status status);

/* The path TQ_PATH_AUTO resolves to for B queries of length D per problem. */
tq_path tq_auto_path(int B, int D);

/* Faults of the bounded waits.  Every wait of a kernel on an mbarrier (a bulk copy
 * landing, a peer CTA's rows arriving, a tensor-core stage) gives up after one second
 * of the GPU's global timer; the kernel then finishes with NaN in the outputs it could
 * not compute and sets a fault bit on the device instead of hanging it.
 * tq_device_faults ORs into *bits the fault bits set on the CURRENT device since the
 * last call and clears them: 1 = fp32 lookup-table scorers, 2 = tensor-core scorer,
 * 4 = fused decode, 8 = compressor, 16 = tq_check_wait_expiry.  It synchronises with the device (it reads device
 * memory) and is not for use inside stream capture.  bits: host pointer, not NULL.
 * Errors: TQ_ERR_INVALID_VALUE (bits NULL), TQ_ERR_LAUNCH (the device read failed). */
tq_status tq_device_faults(unsigned int* bits);

/* Failure path of the bounded waits, run on purpose (no counterpart in the pages).
 * Launches one warp on `stream` whose only mbarrier wait can never complete: nothing
 * arrives on it.  After the one-second budget the wait gives up, sets fault bit 16 and
 * the kernel returns; the context stays usable and nothing else is written.  Read the
 * bit with tq_device_faults once the stream has passed the call (about one second).
 * For tests of a caller's fault handling; it computes nothing.
 * Errors: TQ_ERR_LAUNCH. */
tq_status tq_check_wait_expiry(cudaStream_t stream);

/* ------------------------------------------------------------------------
 * Query transform (riteshyadav.xyz, "Two kernels, two jobs", first kernel;
 * zededa.com v3 "Combined Transform": one [Pi | S_mat] product per query).
 *
 *   A[p,b,d] = sum_j Pi[h,d,j]    * Q[p,b,j]
 *   T[p,b,d] = sum_j S_mat[h,d,j] * Q[p,b,j]      h = p % H
 *
 * Q: [P,B,D] of `qtype` (bf16 values are widened exactly).  Pi, S_mat: [H,D,D]
 * fp32.  A, T: [P,B,D] fp32 outputs.  1 <= D <= 256, 1 <= H <= P.
 * ---------------------------------------------------------------------- */
tq_status tq_prepare_queries(const void* Q, tq_qtype qtype, const float* Pi, const float* S_mat,
                             float* A, float* T, int P, int H, int B, int D, cudaStream_t stream);

/* ------------------------------------------------------------------------
 * The same transform with a randomized-Hadamard rotation Pi = H diag(s)
 * (kanthi.in §2 "A dense Haar rotation costs O(d^2) ... randomized Hadamard
 * transform y = H D x", §3 RandomizedHadamard): A = H (s * q) by a fast
 * Walsh-Hadamard transform in O(D log D), H orthonormal in Sylvester order
 * (H[i][j] = (-1)^popcount(i & j) / sqrt(D)); T = S_mat q as above.
 *
 * hsigns: [H,D] fp32, each +1 or -1 (device).  D a power of two, 2 <= D <= 256.
 * Other arguments and errors as for tq_prepare_queries.
 *
 * tq_hadamard_rotation (HOST pointers): writes the dense fp32 row-major
 * Pi = H diag(s) for the D signs at `signs`, D a power of two <= 4096, so that
 * the compressor and every other entry taking Pi use the same rotation.
 * ---------------------------------------------------------------------- */
tq_status tq_prepare_queries_hadamard(const void* Q, tq_qtype qtype, const float* hsigns,
                                      const float* S_mat, float* A, float* T, int P, int H, int B,
                                      int D, cudaStream_t stream);
tq_status tq_hadamard_rotation(const float* signs, int D, float* Pi);

/* ------------------------------------------------------------------------
 * Scores from an UNPACKED cache (riteshyadav.xyz, "Two kernels, two jobs",
 * second kernel, and "Full CUDA solution"): one byte per index and per sign.
 *
 * A, T: [P,B,D] fp32 (from tq_prepare_queries).  K_idx: [P,S,D] uint8 codes < C.
 * signs: [P,S,D] int8, each +1 or -1.  gamma: [P,S] fp32 residual norms.
 * codebook: [C] fp32.  scores: [P,B,S] fp32 output.
 * 1 <= D <= 256, 1 <= C <= 256.  TQ_PATH_BF16_MMA needs D == 128.
 * ---------------------------------------------------------------------- */
tq_status tq_scores(const float* A, const float* T, const uint8_t* K_idx, const int8_t* signs,
                    const float* gamma, const float* codebook, float* scores,
                    int P, int B, int S, int D, int C, tq_path path, cudaStream_t stream);

/* ------------------------------------------------------------------------
 * Scores from a BIT-PACKED cache: two bit planes per key plus an fp16 norm
 * (kanthi.in §8 "Kernel view", packed slot sizes; zededa.com v6 tile scorer,
 * (packed >> sub*BITS) & MASK).
 *
 * idx_plane: [P,S,D*idx_bits/8] bytes.  Within a key, bit t of coordinate d is
 *   stream bit idx_bits*d + t, and stream bit i is bit (i mod 8) of byte i/8
 *   (little-endian; 3-bit fields straddle bytes).
 * sign_plane: [P,S,D/8] bytes; bit d (same numbering) is 1 exactly when sigma_d = +1.
 * gamma_f16: [P,S] IEEE binary16 residual norms (raw 16-bit patterns).
 * codebook: [2^idx_bits] fp32.  A, T, scores as for tq_scores.
 * D % 32 == 0, 32 <= D <= 256, idx_bits in {1,2,3}.
 * ---------------------------------------------------------------------- */
tq_status tq_scores_packed(const float* A, const float* T, const uint8_t* idx_plane,
                           const uint8_t* sign_plane, const uint16_t* gamma_f16,
                           const float* codebook, float* scores, int P, int B, int S, int D,
                           int idx_bits, tq_path path, cudaStream_t stream);

/* ------------------------------------------------------------------------
 * MSE-only variant (TurboQuant-MSE: no residual sketch, one stored norm per key;
 * kanthi.in "TurboQuant: Rotate-then-Quantize KV Caches at 3 Bits", §3
 * TurboQuantMSE, §6 on why attention prefers it, §8 "Kernel view: never
 * un-rotate a key"):
 *
 *   score[b,s] = n_s * sum_d A[b,d] c[idx[s,d]]
 *   score[b,s] = n_s * sum_d A[b,d] c[idx[s,d]] / sqrt(sum_d c[idx[s,d]]^2)
 *                                           (norm_correction = 1: the codeword
 *                                            is put back on the unit sphere)
 *
 * A         [P,B,D] fp32 = Pi q (the A output of tq_prepare_queries).
 * idx_plane [P,S,D*idx_bits/8] bytes, the packed code format above, codes
 *           of the rotated unit key k/||k||.
 * norm_f16  [P,S] IEEE fp16 key lengths ||k||.
 * codebook  2^idx_bits fp32 centroids.  scores [P,B,S] fp32.
 * D % 32 == 0 (32 <= D <= 4096), idx_bits in {1,2,3,4}; fp32 arithmetic
 * (D = 128 with 1-3 bit codes uses the lookup-table kernel).  Every pointer is
 * a caller-owned device pointer, 16-byte aligned; nothing is allocated.
 * Errors: TQ_ERR_INVALID_VALUE (null pointer, size or flag out of range),
 * TQ_ERR_MISALIGNED, TQ_ERR_UNSUPPORTED (D % 32 != 0), TQ_ERR_LAUNCH.
 * ---------------------------------------------------------------------- */
tq_status tq_scores_mse(const float* A, const uint8_t* idx_plane, const uint16_t* norm_f16,
                        const float* codebook, float* scores, int P, int B, int S, int D,
                        int idx_bits, int norm_correction, cudaStream_t stream);

/* ------------------------------------------------------------------------
 * Outlier-split cache: fractional bits from two TurboQuant-MSE instances per head
 * over disjoint channel sets (kanthi.in §7 "Fractional bits and the outlier split":
 * the channels hot across the sequence are known ahead of time and get their own,
 * wider instance; each instance has its own rotation, codebook and norm):
 *
 *   A_out = Pi_out q[channels],  A_reg = Pi_reg q[other channels, increasing]
 *   score = n_out * <A_out, c_out(idx_out)> + n_reg * <A_reg, c_reg(idx_reg)>
 *
 * tq_prepare_queries_split: Q [P,B,D] (f32 or bf16); channels: n_out int32 device
 * values, strictly increasing, each in [0, D) (the caller's contract: a list that
 * breaks it gives wrong results, never an out-of-bounds access); Pi_out [H,n_out,n_out],
 * Pi_reg [H,D-n_out,D-n_out] fp32; A_out [P,B,n_out], A_reg [P,B,D-n_out] fp32
 * outputs.  2 <= D <= 256, 1 <= n_out < D.
 *
 * tq_scores_split: each instance's cache in the tq_scores_mse format of its own
 * width: out_plane [P,S,n_out*out_bits/8] + out_norm [P,S] fp16 + out_codebook
 * [2^out_bits], reg_plane [P,S,n_reg*reg_bits/8] + reg_norm + reg_codebook;
 * scores [P,B,S] fp32.  n_out and n_reg multiples of 32, bits in {1,...,4}.  The
 * printed split is n_out = 32 at 3 bits and n_reg = 96 at 2: 36 bytes of codes and
 * two fp16 norms, 40 bytes (2.5 bits a coordinate) a key.  fp32 arithmetic.
 * Errors: TQ_ERR_INVALID_VALUE, TQ_ERR_MISALIGNED, TQ_ERR_UNSUPPORTED, TQ_ERR_LAUNCH.
 * ---------------------------------------------------------------------- */
tq_status tq_prepare_queries_split(const void* Q, tq_qtype qtype, const int* channels, const float* Pi_out,
                                   const float* Pi_reg, float* A_out, float* A_reg, int P, int H, int B,
                                   int D, int n_out, cudaStream_t stream);
tq_status tq_scores_split(const float* A_out, const float* A_reg, const uint8_t* out_plane,
                          const uint16_t* out_norm, const float* out_codebook, int out_bits,
                          const uint8_t* reg_plane, const uint16_t* reg_norm, const float* reg_codebook,
                          int reg_bits, float* scores, int P, int B, int S, int n_out, int n_reg,
                          cudaStream_t stream);

/* ------------------------------------------------------------------------
 * Fused decode over an MSE-quantized key AND value cache, in the rotated
 * domain (kanthi.in §8 "Kernel view: never un-rotate a key", the kernel form
 * of tq_rotated_domain; §7 on values):
 *
 *   s[b,i] = scale * nk_i * <A_b, ck[kidx_i]>     A = Pi_k q (tq_prepare_queries)
 *   p[b,:] = softmax(s[b,:])
 *   out[b] = Pi_v^T sum_i p[b,i] nv_i cv[vidx_i]  (one inverse rotation per query)
 *
 * Keys and values use the tq_scores_mse format: packed code planes
 * k_plane [P,S,D*k_bits/8] and v_plane [P,S,D*v_bits/8] of the rotated unit
 * vectors, fp16 lengths k_norm, v_norm [P,S], fp32 codebooks of 2^bits
 * centroids.  Pi_v: [H,D,D] fp32 (problem p uses head p % H).  out: [P,B,D]
 * fp32.  scale: the logit scale (1/sqrt(D) on the page).  D == 128,
 * k_bits, v_bits in {1,2,3}.  Split-KV: the caller passes `workspace` of at
 * least tq_decode_workspace_bytes(P, B, S, D) bytes (scratch, contents
 * unspecified on return, not shared by concurrent calls).  fp32 arithmetic.
 * Errors: TQ_ERR_INVALID_VALUE, TQ_ERR_MISALIGNED, TQ_ERR_UNSUPPORTED (D != 128),
 * TQ_ERR_WORKSPACE, TQ_ERR_LAUNCH.
 * ---------------------------------------------------------------------- */
size_t tq_decode_workspace_bytes(int P, int B, int S, int D);
tq_status tq_decode_mse(const float* A, const uint8_t* k_plane, const uint16_t* k_norm,
                        const float* k_codebook, int k_bits, const uint8_t* v_plane,
                        const uint16_t* v_norm, const float* v_codebook, int v_bits,
                        const float* Pi_v, float* out, int P, int H, int B, int S, int D,
                        float scale, void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* ------------------------------------------------------------------------
 * Fused decode over a TurboQuant_prod KEY cache and an MSE-quantized VALUE cache
 * ("Implementing TurboQuant on NVIDIA's AGX Thor", zededa.com, "The Optimization
 * Journey", v2 kernel 3 and v6 "Fused hybrid Triton kernel": per compressed block
 * the TQ score, the value dequantization and the accumulation, with online softmax):
 *
 *   s[b,i] = scale * (<A_b, kcb[kidx_i]> + (sqrt(pi/2)/D) gamma_i <T_b, sigma_i>)
 *            (the raw score of tq_scores_packed, times scale)
 *   p[b,:] = softmax(s[b,:])
 *   out[b] = Pi_v^T sum_i p[b,i] nv_i vcb[vidx_i]
 *
 * A, T: [P,B,D] fp32 from tq_prepare_queries.  Keys in the tq_scores_packed format:
 * k_plane [P,S,D*k_bits/8], k_sign_plane [P,S,D/8], k_gamma [P,S] fp16, codebook
 * k_codebook of 2^k_bits fp32 centroids.  Values, Pi_v, out, scale, workspace and
 * errors as for tq_decode_mse (the same workspace size).  D == 128, k_bits and v_bits
 * in {1,2,3}.  fp32 arithmetic.
 * ---------------------------------------------------------------------- */
tq_status tq_decode_prod(const float* A, const float* T, const uint8_t* k_plane,
                         const uint8_t* k_sign_plane, const uint16_t* k_gamma,
                         const float* k_codebook, int k_bits, const uint8_t* v_plane,
                         const uint16_t* v_norm, const float* v_codebook, int v_bits,
                         const float* Pi_v, float* out, int P, int H, int B, int S, int D,
                         float scale, void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* ------------------------------------------------------------------------
 * Fused query transform + scoring: the challenge's `solve` without its
 * per-call cudaMalloc/cudaFree (riteshyadav.xyz, "What the rearrangement
 * saves": its solve "allocates temporary arrays on every call").  The caller
 * passes `workspace`, a device buffer of at least tq_workspace_bytes(P, B, D)
 * bytes that holds A and T between the two steps (and, for D = 128 and B >= 16,
 * their bf16 copy laid out for the tensor cores); it is scratch, its contents
 * on return are unspecified, and calls that may run concurrently must not
 * share it.  (tq_solve_packed on the fp32 path with B <= 8 and D = 128 runs the
 * transform inside its single scoring kernel and leaves the workspace untouched.)
 * ---------------------------------------------------------------------- */
size_t tq_workspace_bytes(int P, int B, int D);

tq_status tq_solve(const void* Q, tq_qtype qtype, const uint8_t* K_idx, const int8_t* signs,
                   const float* gamma, const float* Pi, const float* S_mat, const float* codebook,
                   float* scores, int P, int H, int B, int S, int D, int C,
                   void* workspace, size_t workspace_bytes, tq_path path, cudaStream_t stream);

tq_status tq_solve_packed(const void* Q, tq_qtype qtype, const uint8_t* idx_plane,
                          const uint8_t* sign_plane, const uint16_t* gamma_f16, const float* Pi,
                          const float* S_mat, const float* codebook, float* scores,
                          int P, int H, int B, int S, int D, int idx_bits,
                          void* workspace, size_t workspace_bytes, tq_path path,
                          cudaStream_t stream);

/* ------------------------------------------------------------------------
 * Bit packing of the cache format above, bit-exact in both directions
 * (kanthi.in §11 "Verification plan", item 4: pack then unpack is the
 * identity for every slot size and head dimension).
 *
 * n_keys rows of D coordinates.  Packing ignores code bits at and above
 * `bits`; packing signs stores 1 for every strictly positive int8.
 * Unpacked signs are +1 / -1.  D % 8 == 0, 8 <= D <= 4096, bits in {1,...,8}.
 * ---------------------------------------------------------------------- */
tq_status tq_pack_indices(const uint8_t* K_idx, uint8_t* idx_plane, int64_t n_keys, int D,
                          int bits, cudaStream_t stream);
tq_status tq_unpack_indices(const uint8_t* idx_plane, uint8_t* K_idx, int64_t n_keys, int D,
                            int bits, cudaStream_t stream);
tq_status tq_pack_signs(const int8_t* signs, uint8_t* sign_plane, int64_t n_keys, int D,
                        cudaStream_t stream);
tq_status tq_unpack_signs(const uint8_t* sign_plane, int8_t* signs, int64_t n_keys, int D,
                          cudaStream_t stream);

/* ------------------------------------------------------------------------
 * Compressor: the write side of the cache (TurboQuant_prod, kanthi.in §3
 * TurboQuantProd and "Kernel checklist" of §8: rotate, search the midpoints,
 * residual sketch; zededa.com "Theorem 2").
 *
 * tq_compress_keys (device): for each unit-norm key k of problem p (head
 * h = p % H): y = Pi_h k; idx_d = number of codebook midpoints strictly below
 * y_d (ties go to the lower index); r = k - Pi_h^T c[idx]; sign_d = +1 when
 * (S_mat_h r)_d >= 0, else -1; gamma = ||r||_2.  keys: [P,S,D] fp32; Pi,
 * S_mat: [H,D,D]; codebook: [C] fp32 sorted ascending; outputs K_idx [P,S,D]
 * uint8, signs [P,S,D] int8 and exactly one of gamma_f32 / gamma_f16 [P,S]
 * (the other NULL).  Computed in fp32: a coordinate within ~1e-6 of a cell
 * edge may fall on either side.  D % 32 == 0, 32 <= D <= 256, C <= 256.  Keys
 * are taken as unit length (the score has no key-norm term).
 *
 * tq_compress_keys_packed (device): the same compression in one pass that
 * writes the packed cache of tq_scores_packed directly (kanthi.in §8 "Kernel
 * checklist": rotate, search the midpoints, pack the bits and write the norm in
 * the store kernel): idx_plane [P,S,D*idx_bits/8], sign_plane [P,S,D/8],
 * gamma_f16 [P,S], codebook of 2^idx_bits centroids sorted ascending.
 * D % 32 == 0, 32 <= D <= 256, idx_bits in {1,2,3}.  Errors: TQ_ERR_INVALID_VALUE,
 * TQ_ERR_MISALIGNED, TQ_ERR_UNSUPPORTED (D % 32 != 0), TQ_ERR_LAUNCH.
 *
 * tq_lloyd_max_codebook (HOST pointer out): the 2^mse_bits Lloyd-Max centroids
 * of one coordinate of a uniform unit vector in R^D, density proportional to
 * (1-x^2)^((D-3)/2) on [-1,1] sampled at grid_points even points (kanthi.in
 * §2-§4: 400001 points, 300 rounds, start evenly spaced on +-2/sqrt(D)).
 * D >= 3, 1 <= mse_bits <= 8.
 *
 * tq_haar_rotation (HOST pointers): Pi = Q diag(sign(diag R)) for the QR
 * factorisation G = QR of a D x D float64 matrix G (row-major), written as
 * fp32 row-major (kanthi.in §3, HaarRotation).  D <= 4096.
 * ---------------------------------------------------------------------- */
tq_status tq_compress_keys(const float* keys, const float* Pi, const float* S_mat,
                           const float* codebook, int C, uint8_t* K_idx, int8_t* signs,
                           float* gamma_f32, uint16_t* gamma_f16, int P, int H, int S, int D,
                           cudaStream_t stream);
tq_status tq_compress_keys_packed(const float* keys, const float* Pi, const float* S_mat,
                                  const float* codebook, int idx_bits, uint8_t* idx_plane,
                                  uint8_t* sign_plane, uint16_t* gamma_f16, int P, int H, int S, int D,
                                  cudaStream_t stream);
tq_status tq_lloyd_max_codebook(int D, int mse_bits, int grid_points, int iterations,
                                float* centroids);
tq_status tq_haar_rotation(const double* G, int D, float* Pi);

/* ------------------------------------------------------------------------
 * tq_solve_packed_noalloc: tq_solve_packed for callers that cannot allocate
 * device memory.  The pages have no counterpart: this is a deployment entry
 * point of this library.
 *
 * Some callers have no way to hand over a workspace: an inference-engine
 * plugin that receives only its input and output buffers while the engine owns
 * all device memory, or a service that reserves its device memory once at
 * start-up and must not allocate later (an allocation can fail or synchronise
 * the device).  This entry point takes the same arguments as tq_solve_packed
 * minus the workspace and keeps A and T in a fixed 1 MiB array inside libtq
 * (a file-scope device array that every GPU loading the library holds until the
 * process exits).  It calls no allocator.
 *
 * Limit: tq_workspace_bytes(P, B, D) must be <= 1048576 (for D = 128 that is
 * about 1 KB per query, 1.5 KB per query when B >= 16); larger calls return
 * TQ_ERR_WORKSPACE and launch nothing.
 * The first call on each device looks up the array's device address (once per
 * device, with that device current); make that first call before any stream
 * capture.  The looked-up address is kept for the life of the process, so do not
 * call this entry point on a device after cudaDeviceReset on it (the reset unloads
 * the array and the kept address would be stale).  Nothing in the array needs to start at zero (the transform writes
 * all of A and T before scoring reads them).  All calls on one device share the
 * array: calls that may overlap on the GPU (other streams, other host threads)
 * race on it and must be serialised by the caller.
 * ---------------------------------------------------------------------- */
tq_status tq_solve_packed_noalloc(const void* Q, tq_qtype qtype, const uint8_t* idx_plane,
                                  const uint8_t* sign_plane, const uint16_t* gamma_f16,
                                  const float* Pi, const float* S_mat, const float* codebook,
                                  float* scores, int P, int H, int B, int S, int D, int idx_bits,
                                  tq_path path, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* TQ_H */
