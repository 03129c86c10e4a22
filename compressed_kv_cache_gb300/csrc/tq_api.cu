// C ABI of libtq (declared in include/tq.h): argument validation and dispatch.
// Every check runs on the host before any CUDA call, so an invalid call
// returns its status without touching the device.
#include <climits>
#include <cmath>

#include "tq_internal.cuh"

namespace {

constexpr int kMaxGridYZ = 65535;

bool misaligned(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; }

template <typename... Ptrs>
tq_status check_ptrs(Ptrs... ptrs) {
  const void* all[] = {static_cast<const void*>(ptrs)...};
  for (const void* p : all)
    if (p == nullptr) return TQ_ERR_INVALID_VALUE;
  for (const void* p : all)
    if (misaligned(p)) return TQ_ERR_MISALIGNED;
  return TQ_OK;
}

tq_status from_cuda(cudaError_t e) { return e == cudaSuccess ? TQ_OK : TQ_ERR_LAUNCH; }

size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

size_t at_bytes(int P, int B, int D) {
  return round_up(static_cast<size_t>(P) * B * D * sizeof(float), 256);
}

// Workspace: [A][T][bf16 query operand of the tensor-core path (D = 128, B >= 16 only)].
size_t y_bytes(int P, int B, int D) {
  return (D == 128 && B >= 16) ? round_up(tq::mma_y_bytes(P, B), 256) : 0;
}

tq_status check_prepare_sizes(int P, int H, int B, int D, tq_qtype qtype) {
  if (P < 1 || H < 1 || H > P || B < 1 || D < 1 || D > 256) return TQ_ERR_INVALID_VALUE;
  if (P > kMaxGridYZ || (B + 7) / 8 > kMaxGridYZ) return TQ_ERR_INVALID_VALUE;
  if (qtype != TQ_Q_F32 && qtype != TQ_Q_BF16) return TQ_ERR_INVALID_VALUE;
  return TQ_OK;
}

tq_status check_score_sizes(int P, int B, int S, int D) {
  if (P < 1 || B < 1 || S < 1 || D < 1 || D > 256) return TQ_ERR_INVALID_VALUE;
  if (P > kMaxGridYZ || B > kMaxGridYZ || S > INT_MAX - 1024) return TQ_ERR_INVALID_VALUE;
  return TQ_OK;
}

// Resolves AUTO and checks that the requested path exists for this shape.
tq_status resolve_path(tq_path path, int B, int D, tq_path* out) {
  if (path != TQ_PATH_AUTO && path != TQ_PATH_FP32 && path != TQ_PATH_BF16_MMA)
    return TQ_ERR_INVALID_VALUE;
  if (path == TQ_PATH_AUTO) path = tq_auto_path(B, D);
  if (path == TQ_PATH_BF16_MMA && (D != 128 || !tq::mma_path_available()))
    return TQ_ERR_UNSUPPORTED;
  *out = path;
  return TQ_OK;
}

tq_status check_unpacked(const float* A, const float* T, const uint8_t* K_idx, const int8_t* signs,
                         const float* gamma, const float* codebook, float* scores, int P, int B,
                         int S, int D, int C, tq_path path, tq_path* resolved) {
  tq_status st = check_ptrs(A, T, K_idx, signs, gamma, codebook, scores);
  if (st != TQ_OK) return st;
  if ((st = check_score_sizes(P, B, S, D)) != TQ_OK) return st;
  if (C < 1 || C > 256) return TQ_ERR_INVALID_VALUE;
  return resolve_path(path, B, D, resolved);
}

tq_status check_packed(const float* A, const float* T, const uint8_t* idx_plane,
                       const uint8_t* sign_plane, const uint16_t* gamma_f16,
                       const float* codebook, float* scores, int P, int B, int S, int D,
                       int idx_bits, tq_path path, tq_path* resolved) {
  tq_status st = check_ptrs(A, T, idx_plane, sign_plane, gamma_f16, codebook, scores);
  if (st != TQ_OK) return st;
  if ((st = check_score_sizes(P, B, S, D)) != TQ_OK) return st;
  if (idx_bits < 1 || idx_bits > 3) return TQ_ERR_INVALID_VALUE;
  if (D % 32 != 0) return TQ_ERR_UNSUPPORTED;
  return resolve_path(path, B, D, resolved);
}

tq_status run_unpacked(const float* A, const float* T, const uint8_t* K_idx, const int8_t* signs,
                       const float* gamma, const float* codebook, float* scores, int P, int B,
                       int S, int D, int C, tq_path path, cudaStream_t stream,
                       bool after_prepare = false, const uint16_t* Ybf = nullptr) {
  if (path == TQ_PATH_BF16_MMA)
    return from_cuda(tq::launch_scores_mma(A, T, K_idx, signs, gamma, codebook, scores, P, B, S,
                                           C, 0, false, after_prepare, stream, Ybf));
  return from_cuda(tq::launch_scores_unpacked_fp32(A, T, K_idx, signs, gamma, codebook, scores,
                                                   P, B, S, D, C, stream));
}

tq_status run_packed(const float* A, const float* T, const uint8_t* idx_plane,
                     const uint8_t* sign_plane, const uint16_t* gamma_f16, const float* codebook,
                     float* scores, int P, int B, int S, int D, int idx_bits, tq_path path,
                     cudaStream_t stream, bool after_prepare = false, const uint16_t* Ybf = nullptr) {
  if (path == TQ_PATH_BF16_MMA)
    return from_cuda(tq::launch_scores_mma(A, T, idx_plane, sign_plane, gamma_f16, codebook,
                                           scores, P, B, S, 1 << idx_bits, idx_bits, true,
                                           after_prepare, stream, Ybf));
  return from_cuda(tq::launch_scores_packed_fp32(A, T, idx_plane, sign_plane, gamma_f16, codebook,
                                                 scores, P, B, S, D, idx_bits, after_prepare, stream));
}

tq_status check_pack_sizes(int64_t n_keys, int D, int bits) {
  if (n_keys < 1 || D < 8 || D > 4096 || D % 8 != 0 || bits < 1 || bits > 8)
    return TQ_ERR_INVALID_VALUE;
  if (n_keys > (static_cast<int64_t>(1) << 40) / D) return TQ_ERR_INVALID_VALUE;
  return TQ_OK;
}

}  // namespace

namespace tq {
// tq_faults.cu: one warp whose only bounded wait runs out, and that unit's fault word
cudaError_t launch_wait_expiry(cudaStream_t st);
cudaError_t take_faults_check(unsigned int* bits);
}  // namespace tq

extern "C" {

const char* tq_status_string(tq_status status) {
  switch (status) {
    case TQ_OK: return "TQ_OK";
    case TQ_ERR_INVALID_VALUE: return "TQ_ERR_INVALID_VALUE: null pointer or size out of range";
    case TQ_ERR_UNSUPPORTED: return "TQ_ERR_UNSUPPORTED: no kernel implements this combination";
    case TQ_ERR_MISALIGNED: return "TQ_ERR_MISALIGNED: an array pointer is not 16-byte aligned";
    case TQ_ERR_WORKSPACE: return "TQ_ERR_WORKSPACE: workspace null or too small";
    case TQ_ERR_LAUNCH: return "TQ_ERR_LAUNCH: CUDA reported a launch error";
  }
  return "unknown tq_status";
}

tq_status tq_device_faults(unsigned int* bits) {
  if (bits == nullptr) return TQ_ERR_INVALID_VALUE;
  unsigned int v = 0;
  cudaError_t e = tq::take_faults_simt(&v);
  if (e == cudaSuccess) e = tq::take_faults_mma(&v);
  if (e == cudaSuccess) e = tq::take_faults_decode(&v);
  if (e == cudaSuccess) e = tq::take_faults_compress(&v);
  if (e == cudaSuccess) e = tq::take_faults_check(&v);
  if (e != cudaSuccess) return TQ_ERR_LAUNCH;
  *bits |= v;
  return TQ_OK;
}

tq_status tq_check_wait_expiry(cudaStream_t stream) {
  return tq::launch_wait_expiry(stream) == cudaSuccess ? TQ_OK : TQ_ERR_LAUNCH;
}

tq_path tq_auto_path(int B, int D) {
  return (B >= 16 && D == 128 && tq::mma_path_available()) ? TQ_PATH_BF16_MMA : TQ_PATH_FP32;
}

tq_status tq_prepare_queries(const void* Q, tq_qtype qtype, const float* Pi, const float* S_mat,
                             float* A, float* T, int P, int H, int B, int D,
                             cudaStream_t stream) {
  tq_status st = check_ptrs(Q, Pi, S_mat, A, T);
  if (st != TQ_OK) return st;
  if ((st = check_prepare_sizes(P, H, B, D, qtype)) != TQ_OK) return st;
  return from_cuda(tq::launch_prepare(Q, qtype, Pi, S_mat, A, T, P, H, B, D, stream));
}

tq_status tq_prepare_queries_hadamard(const void* Q, tq_qtype qtype, const float* hsigns,
                                      const float* S_mat, float* A, float* T, int P, int H, int B,
                                      int D, cudaStream_t stream) {
  tq_status st = check_ptrs(Q, hsigns, S_mat, A, T);
  if (st != TQ_OK) return st;
  if ((st = check_prepare_sizes(P, H, B, D, qtype)) != TQ_OK) return st;
  if (D < 2 || (D & (D - 1)) != 0) return TQ_ERR_INVALID_VALUE;
  // the dense rows are unused in this mode; S_mat stands in for Pi
  return from_cuda(tq::launch_prepare(Q, qtype, S_mat, S_mat, A, T, P, H, B, D, stream, nullptr, hsigns));
}

tq_status tq_hadamard_rotation(const float* signs, int D, float* Pi) {
  if (signs == nullptr || Pi == nullptr || D < 1 || D > 4096 || (D & (D - 1)) != 0)
    return TQ_ERR_INVALID_VALUE;
  // Pi[i][j] = H[i][j] s_j / sqrt(D), H[i][j] = (-1)^popcount(i & j) (Sylvester order)
  const double scale = 1.0 / std::sqrt(static_cast<double>(D));
  for (int i = 0; i < D; ++i)
    for (int j = 0; j < D; ++j) {
      const double h = (__builtin_popcount(static_cast<unsigned>(i & j)) & 1) ? -scale : scale;
      Pi[static_cast<size_t>(i) * D + j] = static_cast<float>(h * signs[j]);
    }
  return TQ_OK;
}

tq_status tq_scores(const float* A, const float* T, const uint8_t* K_idx, const int8_t* signs,
                    const float* gamma, const float* codebook, float* scores, int P, int B, int S,
                    int D, int C, tq_path path, cudaStream_t stream) {
  tq_path p;
  tq_status st = check_unpacked(A, T, K_idx, signs, gamma, codebook, scores, P, B, S, D, C, path, &p);
  if (st != TQ_OK) return st;
  return run_unpacked(A, T, K_idx, signs, gamma, codebook, scores, P, B, S, D, C, p, stream);
}

tq_status tq_scores_packed(const float* A, const float* T, const uint8_t* idx_plane,
                           const uint8_t* sign_plane, const uint16_t* gamma_f16,
                           const float* codebook, float* scores, int P, int B, int S, int D,
                           int idx_bits, tq_path path, cudaStream_t stream) {
  tq_path p;
  tq_status st = check_packed(A, T, idx_plane, sign_plane, gamma_f16, codebook, scores, P, B, S, D,
                              idx_bits, path, &p);
  if (st != TQ_OK) return st;
  return run_packed(A, T, idx_plane, sign_plane, gamma_f16, codebook, scores, P, B, S, D, idx_bits,
                    p, stream);
}

size_t tq_workspace_bytes(int P, int B, int D) {
  if (P < 1 || B < 1 || D < 1) return 0;
  return 2 * at_bytes(P, B, D) + y_bytes(P, B, D);
}

tq_status tq_solve(const void* Q, tq_qtype qtype, const uint8_t* K_idx, const int8_t* signs,
                   const float* gamma, const float* Pi, const float* S_mat, const float* codebook,
                   float* scores, int P, int H, int B, int S, int D, int C, void* workspace,
                   size_t workspace_bytes, tq_path path, cudaStream_t stream) {
  tq_status st = check_ptrs(Q, Pi, S_mat);
  if (st != TQ_OK) return st;
  if ((st = check_prepare_sizes(P, H, B, D, qtype)) != TQ_OK) return st;
  if (workspace == nullptr) return TQ_ERR_WORKSPACE;
  if (misaligned(workspace)) return TQ_ERR_MISALIGNED;
  if (workspace_bytes < tq_workspace_bytes(P, B, D)) return TQ_ERR_WORKSPACE;
  float* A = static_cast<float*>(workspace);
  float* T = reinterpret_cast<float*>(static_cast<char*>(workspace) + at_bytes(P, B, D));
  tq_path p;
  if ((st = check_unpacked(A, T, K_idx, signs, gamma, codebook, scores, P, B, S, D, C, path, &p)) != TQ_OK)
    return st;
  uint16_t* Y = (p == TQ_PATH_BF16_MMA && y_bytes(P, B, D) > 0)
                    ? reinterpret_cast<uint16_t*>(static_cast<char*>(workspace) + 2 * at_bytes(P, B, D))
                    : nullptr;
  if ((st = from_cuda(tq::launch_prepare(Q, qtype, Pi, S_mat, A, T, P, H, B, D, stream, Y, nullptr,
                                         Y != nullptr && tq::mma_shares_sm(P, B, S)))) != TQ_OK)
    return st;
  return run_unpacked(A, T, K_idx, signs, gamma, codebook, scores, P, B, S, D, C, p, stream, true, Y);
}

tq_status tq_solve_packed(const void* Q, tq_qtype qtype, const uint8_t* idx_plane,
                          const uint8_t* sign_plane, const uint16_t* gamma_f16, const float* Pi,
                          const float* S_mat, const float* codebook, float* scores, int P, int H,
                          int B, int S, int D, int idx_bits, void* workspace,
                          size_t workspace_bytes, tq_path path, cudaStream_t stream) {
  tq_status st = check_ptrs(Q, Pi, S_mat);
  if (st != TQ_OK) return st;
  if ((st = check_prepare_sizes(P, H, B, D, qtype)) != TQ_OK) return st;
  if (workspace == nullptr) return TQ_ERR_WORKSPACE;
  if (misaligned(workspace)) return TQ_ERR_MISALIGNED;
  if (workspace_bytes < tq_workspace_bytes(P, B, D)) return TQ_ERR_WORKSPACE;
  float* A = static_cast<float*>(workspace);
  float* T = reinterpret_cast<float*>(static_cast<char*>(workspace) + at_bytes(P, B, D));
  tq_path p;
  if ((st = check_packed(A, T, idx_plane, sign_plane, gamma_f16, codebook, scores, P, B, S, D,
                         idx_bits, path, &p)) != TQ_OK)
    return st;
  if (p == TQ_PATH_FP32 && tq::fused_packed_supported(P, B, D))   // one kernel, workspace untouched
    return from_cuda(tq::launch_solve_packed_fused(Q, qtype, Pi, S_mat, H, idx_plane, sign_plane,
                                                   gamma_f16, codebook, scores, P, B, S,
                                                   idx_bits, stream));
  uint16_t* Y = (p == TQ_PATH_BF16_MMA && y_bytes(P, B, D) > 0)
                    ? reinterpret_cast<uint16_t*>(static_cast<char*>(workspace) + 2 * at_bytes(P, B, D))
                    : nullptr;
  if ((st = from_cuda(tq::launch_prepare(Q, qtype, Pi, S_mat, A, T, P, H, B, D, stream, Y, nullptr,
                                         Y != nullptr && tq::mma_shares_sm(P, B, S)))) != TQ_OK)
    return st;
  return run_packed(A, T, idx_plane, sign_plane, gamma_f16, codebook, scores, P, B, S, D, idx_bits,
                    p, stream, true, Y);
}

tq_status tq_scores_mse(const float* A, const uint8_t* idx_plane, const uint16_t* norm_f16,
                        const float* codebook, float* scores, int P, int B, int S, int D,
                        int idx_bits, int norm_correction, cudaStream_t stream) {
  tq_status st = check_ptrs(A, idx_plane, norm_f16, codebook, scores);
  if (st != TQ_OK) return st;
  if (P < 1 || B < 1 || S < 1 || D < 32 || D > 4096) return TQ_ERR_INVALID_VALUE;
  if (P > kMaxGridYZ || B > kMaxGridYZ || S > INT_MAX - 1024) return TQ_ERR_INVALID_VALUE;
  if (idx_bits < 1 || idx_bits > 4 || (norm_correction != 0 && norm_correction != 1))
    return TQ_ERR_INVALID_VALUE;
  if (D % 32 != 0) return TQ_ERR_UNSUPPORTED;
  return from_cuda(tq::launch_scores_mse(A, idx_plane, norm_f16, codebook, scores, P, B, S, D,
                                         idx_bits, norm_correction != 0, stream));
}

size_t tq_decode_workspace_bytes(int P, int B, int S, int D) {
  if (P < 1 || B < 1 || S < 1 || D != 128) return 0;
  return round_up(tq::decode_part_floats(P, B, S) * sizeof(float), 256);
}

tq_status tq_decode_mse(const float* A, const uint8_t* k_plane, const uint16_t* k_norm,
                        const float* k_codebook, int k_bits, const uint8_t* v_plane,
                        const uint16_t* v_norm, const float* v_codebook, int v_bits,
                        const float* Pi_v, float* out, int P, int H, int B, int S, int D,
                        float scale, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  tq_status st = check_ptrs(A, k_plane, k_norm, k_codebook, v_plane, v_norm, v_codebook, Pi_v, out);
  if (st != TQ_OK) return st;
  if (P < 1 || H < 1 || H > P || B < 1 || S < 1 || D < 1) return TQ_ERR_INVALID_VALUE;
  if (P > kMaxGridYZ || B > kMaxGridYZ || S > INT_MAX - 4096) return TQ_ERR_INVALID_VALUE;
  if (k_bits < 1 || k_bits > 3 || v_bits < 1 || v_bits > 3 || !std::isfinite(scale))
    return TQ_ERR_INVALID_VALUE;
  if (D != 128) return TQ_ERR_UNSUPPORTED;
  if (workspace == nullptr) return TQ_ERR_WORKSPACE;
  if (misaligned(workspace)) return TQ_ERR_MISALIGNED;
  if (workspace_bytes < tq_decode_workspace_bytes(P, B, S, D)) return TQ_ERR_WORKSPACE;
  return from_cuda(tq::launch_decode_mse(A, k_plane, k_norm, k_codebook, k_bits, v_plane, v_norm,
                                         v_codebook, v_bits, Pi_v, out, static_cast<float*>(workspace),
                                         P, H, B, S, scale, stream));
}

tq_status tq_decode_prod(const float* A, const float* T, const uint8_t* k_plane,
                         const uint8_t* k_sign_plane, const uint16_t* k_gamma,
                         const float* k_codebook, int k_bits, const uint8_t* v_plane,
                         const uint16_t* v_norm, const float* v_codebook, int v_bits,
                         const float* Pi_v, float* out, int P, int H, int B, int S, int D,
                         float scale, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  tq_status st = check_ptrs(A, T, k_plane, k_sign_plane, k_gamma, k_codebook, v_plane, v_norm, v_codebook,
                            Pi_v, out);
  if (st != TQ_OK) return st;
  if (P < 1 || H < 1 || H > P || B < 1 || S < 1 || D < 1) return TQ_ERR_INVALID_VALUE;
  if (P > kMaxGridYZ || B > kMaxGridYZ || S > INT_MAX - 4096) return TQ_ERR_INVALID_VALUE;
  if (k_bits < 1 || k_bits > 3 || v_bits < 1 || v_bits > 3 || !std::isfinite(scale))
    return TQ_ERR_INVALID_VALUE;
  if (D != 128) return TQ_ERR_UNSUPPORTED;
  if (workspace == nullptr) return TQ_ERR_WORKSPACE;
  if (misaligned(workspace)) return TQ_ERR_MISALIGNED;
  if (workspace_bytes < tq_decode_workspace_bytes(P, B, S, D)) return TQ_ERR_WORKSPACE;
  return from_cuda(tq::launch_decode_prod(A, T, k_plane, k_sign_plane, k_gamma, k_codebook, k_bits, v_plane,
                                          v_norm, v_codebook, v_bits, Pi_v, out,
                                          static_cast<float*>(workspace), P, H, B, S, scale, stream));
}

tq_status tq_pack_indices(const uint8_t* K_idx, uint8_t* idx_plane, int64_t n_keys, int D,
                          int bits, cudaStream_t stream) {
  tq_status st = check_ptrs(K_idx, idx_plane);
  if (st != TQ_OK) return st;
  if ((st = check_pack_sizes(n_keys, D, bits)) != TQ_OK) return st;
  return from_cuda(tq::launch_pack_indices(K_idx, idx_plane, n_keys, D, bits, stream));
}

tq_status tq_unpack_indices(const uint8_t* idx_plane, uint8_t* K_idx, int64_t n_keys, int D,
                            int bits, cudaStream_t stream) {
  tq_status st = check_ptrs(idx_plane, K_idx);
  if (st != TQ_OK) return st;
  if ((st = check_pack_sizes(n_keys, D, bits)) != TQ_OK) return st;
  return from_cuda(tq::launch_unpack_indices(idx_plane, K_idx, n_keys, D, bits, stream));
}

tq_status tq_pack_signs(const int8_t* signs, uint8_t* sign_plane, int64_t n_keys, int D,
                        cudaStream_t stream) {
  tq_status st = check_ptrs(signs, sign_plane);
  if (st != TQ_OK) return st;
  if ((st = check_pack_sizes(n_keys, D, 1)) != TQ_OK) return st;
  return from_cuda(tq::launch_pack_signs(signs, sign_plane, n_keys, D, stream));
}

tq_status tq_unpack_signs(const uint8_t* sign_plane, int8_t* signs, int64_t n_keys, int D,
                          cudaStream_t stream) {
  tq_status st = check_ptrs(sign_plane, signs);
  if (st != TQ_OK) return st;
  if ((st = check_pack_sizes(n_keys, D, 1)) != TQ_OK) return st;
  return from_cuda(tq::launch_unpack_signs(sign_plane, signs, n_keys, D, stream));
}

}  // extern "C"
