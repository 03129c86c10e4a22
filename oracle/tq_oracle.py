"""Float64 reference implementation of TurboQuant_prod compression and scoring.

TEST INFRASTRUCTURE ONLY: used by tests, the smoke check and the CPU baseline
of the benchmark; never by the product path.

Sources (page title, then section):

* [RY] "TurboQuant Attention in CUDA: Transform the Query, Reuse the Work"
  (riteshyadav.xyz): "Move the transforms to the query", "A tiny example
  before CUDA", "Two kernels, two jobs", "Full CUDA solution".
* [KB] "TurboQuant: Rotate-then-Quantize KV Caches at 3 Bits" (kanthi.in):
  §2 mental model, §3 "The quantizer in NumPy", §4 "Check the codebook
  against the paper", §6 "The trap: unbiased is not the same as better",
  §8 "Kernel view: never un-rotate a key".
* [ZT] "Implementing TurboQuant on NVIDIA's AGX Thor" (zededa.com):
  "Theorem 2: Unbiased Inner Products", v6 tile scorer.

Where the pages are silent or garbled, the reading taken is stated in the
docstring of the function concerned: tie-breaks, sign(0), the float32
storage of Π, S_mat and the codebook, and the bit-packing format.
"""
from __future__ import annotations

import math

import numpy as np

__all__ = [
    "SQRT_HALF_PI",
    "kappa",
    "haar_rotation",
    "fwht",
    "hadamard_rotation",
    "lloyd_max_sphere",
    "nearest_cell",
    "compress_prod",
    "compress_mse",
    "prepare_queries",
    "scores",
    "scores_from_queries",
    "scores_sampled",
    "scores_mse",
    "decode_mse",
    "decode_prod",
    "outlier_channels",
    "compress_split",
    "prepare_queries_split",
    "scores_split",
    "pack_indices",
    "unpack_indices",
    "pack_signs",
    "unpack_signs",
]

SQRT_HALF_PI = math.sqrt(math.pi / 2.0)


def kappa(D: int) -> float:
    """QJL scale sqrt(pi/2)/D ([KB] §3 TurboQuantProd; [ZT] Theorem 2 item 1)."""
    return SQRT_HALF_PI / D


# ---------------------------------------------------------------------------
# Rotation and codebook (inputs of the scorer, produced on the CPU)
# ---------------------------------------------------------------------------

def haar_rotation(G: np.ndarray) -> np.ndarray:
    """Uniformly random orthogonal Π from a Gaussian matrix G ([KB] §3, HaarRotation).

    G = Q R (Householder QR, LAPACK).  Each column j of Q is multiplied by the
    sign of R[j, j] so that G = Π R' with R' upper triangular and a positive
    diagonal; a zero diagonal entry keeps its column (sign taken as +1).  The
    rotation acts on column vectors: y = Π k.
    """
    Q, R = np.linalg.qr(np.asarray(G, dtype=np.float64))
    col_sign = np.where(np.diag(R) < 0.0, -1.0, 1.0)
    return Q * col_sign[np.newaxis, :]


def fwht(x: np.ndarray) -> np.ndarray:
    """Orthonormal Walsh-Hadamard transform along the last axis ([KB] §2 "randomized
    Hadamard transform"; the length n must be a power of two).

    The n x n Walsh-Hadamard matrix in Sylvester order is the k-fold Kronecker
    power of H_2 = [[1, 1], [1, -1]] / sqrt(2) (n = 2^k), so its entry (i, j) is
    (-1)^popcount(i & j) / sqrt(n).  Viewing the last axis as k axes of length 2
    (index bits, most significant first), the transform applies H_2 along each of
    those axes in turn.  The result is orthonormal and its own inverse.
    """
    y = np.array(x, dtype=np.float64, copy=True)
    n = y.shape[-1]
    if n < 1 or n & (n - 1):
        raise ValueError("length must be a power of two")
    k = n.bit_length() - 1
    lead = y.shape[:-1]
    h2 = np.array([[1.0, 1.0], [1.0, -1.0]]) / math.sqrt(2.0)
    t = y.reshape(lead + (2,) * k)
    for axis in range(len(lead), len(lead) + k):
        # contract H_2 with this bit axis, then put the new axis back in its place
        t = np.moveaxis(np.tensordot(t, h2, axes=([axis], [1])), -1, axis)
    return t.reshape(lead + (n,))


def hadamard_rotation(signs: np.ndarray) -> np.ndarray:
    """Dense matrix of the randomized Hadamard rotation y = H diag(s) x ([KB] §2-§3
    RandomizedHadamard): Π[i, j] = H[i, j] s_j with H the orthonormal Walsh-Hadamard
    matrix, so that Π x = fwht(x * s).  ``signs`` holds +1 / -1."""
    s = np.asarray(signs, dtype=np.float64)
    return fwht(np.eye(s.size)).T * s[np.newaxis, :]


def nearest_cell(values: np.ndarray, edges: np.ndarray) -> np.ndarray:
    """Index of the codebook cell of each value: the number of edges strictly below it.

    With sorted centroids the nearest-centroid rule is a search over the
    midpoints ([KB] §3 "Indices are searched against midpoints").  A value
    exactly on a midpoint goes to the lower cell (left-sided search).
    """
    v = np.asarray(values, dtype=np.float64)
    out = np.zeros(v.shape, dtype=np.int64)
    for e in np.asarray(edges, dtype=np.float64):
        out += v > e
    return out


def _sphere_coordinate_moments(d: int):
    """Exact cell moments of one coordinate x of a uniform unit vector in R^d.

    Its density is f(x) = (1 - x^2)^m / Z on [-1, 1] with m = (d - 3) / 2 ([KB] §2,
    fact 1).  Substituting t = (1 + x) / 2 turns the mass below x into the
    regularised incomplete beta function I_t(m + 1, m + 1).  The first moment has
    the antiderivative -(1 - x^2)^(m+1) / (2 (m + 1)), and x^2 = 1 - (1 - x^2) writes
    the second moment through the density of exponent m + 1, whose normaliser is
    Z_{m+1} = Z_m (d - 1) / d (so that E[x^2] = 1 / d).  Returns three functions of
    the cell edges (a, b): mass, first moment and second moment.
    """
    from scipy import special

    m = (d - 3) / 2.0
    log_z = (2.0 * m + 1.0) * math.log(2.0) + special.betaln(m + 1.0, m + 1.0)

    def cdf(x, e):
        t = np.clip((1.0 + np.asarray(x, dtype=np.float64)) / 2.0, 0.0, 1.0)
        return special.betainc(e + 1.0, e + 1.0, t)

    def mass(a, b):
        return cdf(b, m) - cdf(a, m)

    def first(a, b):
        g = lambda x: np.clip(1.0 - np.asarray(x, dtype=np.float64) ** 2, 0.0, None) ** (m + 1.0)
        return (g(a) - g(b)) / (2.0 * (m + 1.0)) / math.exp(log_z)

    def second(a, b):
        return mass(a, b) - (d - 1.0) / d * (cdf(b, m + 1.0) - cdf(a, m + 1.0))

    return mass, first, second


def lloyd_max_sphere(d: int, mse_bits: int, tol: float = 1e-13, max_rounds: int = 200_000):
    """Lloyd-Max codebook for one coordinate of a uniform unit vector in R^d ([KB] §2-§4).

    The codebook is the fixed point of Lloyd's two conditions for the density
    (1 - x^2)^((d-3)/2) on [-1, 1]: every cell edge is the midpoint of its two
    centroids, and every centroid is the mean of its cell.  Cell masses and
    moments are evaluated exactly (:func:`_sphere_coordinate_moments`), not on a
    grid.  The 2^b centroids start at the medians of 2^b equal-probability cells;
    rounds of "edges from centroids, then centroids from edges" repeat until no
    centroid moves by more than ``tol`` times the largest one (the float64 cell
    moments carry about 1e-15 of rounding noise, so ``tol`` stays above it).  The
    density is log-concave, so the fixed point is unique and the start does not
    matter.

    Returns ``(centroids, edges, d_mse)`` in float64, where ``d_mse`` is
    d * E[(x - Q(x))^2], the expected squared error of a unit vector.
    """
    if d < 3:
        raise ValueError("the sphere-coordinate density needs d >= 3")
    from scipy import special

    mass, first, second = _sphere_coordinate_moments(d)
    C = 1 << mse_bits
    m = (d - 3) / 2.0
    probs = (np.arange(C) + 0.5) / C
    centroids = 2.0 * special.betaincinv(m + 1.0, m + 1.0, probs) - 1.0
    for _ in range(max_rounds):
        edges = 0.5 * (centroids[1:] + centroids[:-1])
        lo = np.concatenate(([-1.0], edges))
        hi = np.concatenate((edges, [1.0]))
        new = first(lo, hi) / mass(lo, hi)
        moved = float(np.max(np.abs(new - centroids)))
        centroids = new
        if moved <= tol * float(np.max(np.abs(centroids))):
            break
    else:
        raise RuntimeError("Lloyd-Max rounds did not converge")
    edges = 0.5 * (centroids[1:] + centroids[:-1])
    lo = np.concatenate(([-1.0], edges))
    hi = np.concatenate((edges, [1.0]))
    err = second(lo, hi) - 2.0 * centroids * first(lo, hi) + centroids ** 2 * mass(lo, hi)
    return centroids, edges, d * float(np.sum(err))


# ---------------------------------------------------------------------------
# Compressor: TurboQuant_prod on unit-norm keys
# ---------------------------------------------------------------------------

def compress_prod(keys: np.ndarray, Pi: np.ndarray, S_mat: np.ndarray, codebook: np.ndarray,
                  gamma_dtype: str = "f32"):
    """TurboQuant_prod compression of unit-norm keys ([KB] §3 TurboQuantProd; [ZT] Theorem 2).

    Steps, in the pages' order, for each key k (a row of ``keys``):

    1. y = Π k (rotate; keys are unit length, so the stored norm is 1 and is
       not kept -- the score has no norm term, [RY] "Move the transforms").
    2. idx_d = nearest centroid of y_d (search over midpoints, ties to the
       lower index).
    3. r = k - Πᵀ c[idx] (residual of the MSE stage).
    4. σ = sign(S_mat r) with sign(0) = +1 (the scorer needs ±1, [RY]).
    5. γ = ‖r‖₂, stored as float32 or float16.

    Π, S_mat and the codebook are used exactly as stored (float32 values
    widened to float64), so the residual is taken against the keys the scorer
    can reconstruct.  Returns ``(idx uint8 [S,D], signs int8 [S,D], gamma)``
    with gamma float32 or float16.
    """
    k = np.asarray(keys, dtype=np.float64)
    P = np.asarray(Pi, dtype=np.float64)
    Sm = np.asarray(S_mat, dtype=np.float64)
    c = np.asarray(codebook, dtype=np.float64)
    y = k @ P.T
    edges = 0.5 * (c[1:] + c[:-1])
    idx = nearest_cell(y, edges)
    r = k - c[idx] @ P
    z = r @ Sm.T
    signs = np.where(z >= 0.0, 1, -1).astype(np.int8)
    g = np.sqrt(np.sum(r * r, axis=1))
    if gamma_dtype == "f32":
        gamma = g.astype(np.float32)
    elif gamma_dtype == "f16":
        gamma = g.astype(np.float16)
    else:
        raise ValueError(gamma_dtype)
    return idx.astype(np.uint8), signs, gamma


# ---------------------------------------------------------------------------
# Scorer
# ---------------------------------------------------------------------------

def prepare_queries(Q: np.ndarray, Pi: np.ndarray, S_mat: np.ndarray):
    """A_b = Π q_b and T_b = S_mat q_b for every query row ([RY] "Two kernels, two jobs").

    A[b, d] = sum_j Π[d, j] q[b, j]; T[b, d] = sum_j S_mat[d, j] q[b, j].
    """
    q = np.asarray(Q, dtype=np.float64)
    return q @ np.asarray(Pi, dtype=np.float64).T, q @ np.asarray(S_mat, dtype=np.float64).T


def scores(A: np.ndarray, T: np.ndarray, idx: np.ndarray, signs: np.ndarray, gamma: np.ndarray,
           codebook: np.ndarray) -> np.ndarray:
    """Raw TurboQuant_prod scores from the transformed queries ([RY]; [ZT] Theorem 2).

    score[b, s] = sum_d A[b,d] c[idx[s,d]] + sqrt(pi/2)/D * gamma[s] * sum_d T[b,d] sigma[s,d]

    with no softmax, no value read and no 1/sqrt(D).  float64 throughout,
    from the stored inputs widened exactly.
    """
    A = np.asarray(A, dtype=np.float64)
    T = np.asarray(T, dtype=np.float64)
    D = A.shape[1]
    cvals = np.asarray(codebook, dtype=np.float64)[np.asarray(idx, dtype=np.int64)]
    mse = A @ cvals.T
    res = T @ np.asarray(signs, dtype=np.float64).T
    return mse + kappa(D) * np.asarray(gamma, dtype=np.float64)[np.newaxis, :] * res


def scores_from_queries(Q, Pi, S_mat, idx, signs, gamma, codebook) -> np.ndarray:
    """Query transform followed by the scorer (the whole path, [RY] solve)."""
    A, T = prepare_queries(Q, Pi, S_mat)
    return scores(A, T, idx, signs, gamma, codebook)


def scores_sampled(A, T, idx_rows, sign_rows, gamma_vals, codebook, b_index) -> np.ndarray:
    """Scores of selected (query, key) pairs, one at a time.

    ``idx_rows``/``sign_rows``/``gamma_vals`` hold the keys of the pairs and
    ``b_index`` their query rows; used to check outputs of workloads too large
    to score in full.
    """
    A = np.asarray(A, dtype=np.float64)
    T = np.asarray(T, dtype=np.float64)
    D = A.shape[1]
    c = np.asarray(codebook, dtype=np.float64)
    out = np.empty(len(b_index))
    for n, b in enumerate(b_index):
        mse = float(np.dot(A[b], c[np.asarray(idx_rows[n], dtype=np.int64)]))
        res = float(np.dot(T[b], np.asarray(sign_rows[n], dtype=np.float64)))
        out[n] = mse + kappa(D) * float(gamma_vals[n]) * res
    return out


# ---------------------------------------------------------------------------
# MSE-only variant (no residual sketch; one stored norm per key)
# ---------------------------------------------------------------------------

def compress_mse(keys: np.ndarray, Pi: np.ndarray, codebook: np.ndarray):
    """TurboQuant-MSE compression of keys of any length ([KB] §3 TurboQuantMSE.quantize).

    For each key k: n = ‖k‖₂, stored as IEEE float16; y = Π (k / n); idx_d = the
    cell of y_d among the codebook's midpoints (ties to the lower index, as in
    :func:`compress_prod`).  Π and the codebook are used as stored (float32
    widened).  Returns ``(idx uint8 [S,D], norm float16 [S])``.
    """
    k = np.asarray(keys, dtype=np.float64)
    P = np.asarray(Pi, dtype=np.float64)
    c = np.asarray(codebook, dtype=np.float64)
    n = np.sqrt(np.sum(k * k, axis=1))
    y = (k / n[:, np.newaxis]) @ P.T
    idx = nearest_cell(y, 0.5 * (c[1:] + c[:-1]))
    return idx.astype(np.uint8), n.astype(np.float16)


def scores_mse(A: np.ndarray, idx: np.ndarray, norm: np.ndarray, codebook: np.ndarray,
               norm_correction: bool = False) -> np.ndarray:
    """Raw MSE-only scores from the rotated queries A = Π q ([KB] §8 "Kernel view":
    ⟨q, k̂⟩ = ‖k‖ ⟨Π q, c_idx⟩; §3 TurboQuantMSE.dequantize).

    score[b, s] = norm[s] * sum_d A[b,d] c[idx[s,d]], and with norm correction the
    codeword is first put back on the unit sphere:
    score[b, s] = norm[s] * sum_d A[b,d] c[idx[s,d]] / sqrt(sum_d c[idx[s,d]]^2).
    float64 throughout, from the stored inputs widened exactly.
    """
    A = np.asarray(A, dtype=np.float64)
    cvals = np.asarray(codebook, dtype=np.float64)[np.asarray(idx, dtype=np.int64)]
    dots = A @ cvals.T
    if norm_correction:
        dots = dots / np.sqrt(np.sum(cvals * cvals, axis=1))[np.newaxis, :]
    return dots * np.asarray(norm, dtype=np.float64)[np.newaxis, :]


def decode_mse(A: np.ndarray, k_idx: np.ndarray, k_norm: np.ndarray, k_codebook: np.ndarray,
               v_idx: np.ndarray, v_norm: np.ndarray, v_codebook: np.ndarray, Pi_v: np.ndarray,
               scale: float) -> np.ndarray:
    """Attention output over an MSE-quantized key and value cache, computed in the
    rotated domain ([KB] §8 "Kernel view", the kernel form of tq_rotated_domain):

        s[b, i]  = scale * k_norm[i] * <A[b], c_k[k_idx[i]]>        (A = Pi_k q)
        p[b, :]  = softmax(s[b, :])                                 (max subtracted)
        acc[b]   = sum_i p[b, i] v_norm[i] c_v[v_idx[i]]            (stays rotated)
        out[b]   = Pi_v^T acc[b]                                    (one inverse rotation)

    The page's scale is 1/sqrt(D).  float64 throughout.
    """
    A = np.asarray(A, dtype=np.float64)
    kc = np.asarray(k_codebook, dtype=np.float64)[np.asarray(k_idx, dtype=np.int64)]
    vc = np.asarray(v_codebook, dtype=np.float64)[np.asarray(v_idx, dtype=np.int64)]
    s = scale * (A @ kc.T) * np.asarray(k_norm, dtype=np.float64)[np.newaxis, :]
    p = np.exp(s - s.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    acc = (p * np.asarray(v_norm, dtype=np.float64)[np.newaxis, :]) @ vc
    return acc @ np.asarray(Pi_v, dtype=np.float64)


def decode_prod(A: np.ndarray, T: np.ndarray, k_idx: np.ndarray, k_signs: np.ndarray,
                k_gamma: np.ndarray, k_codebook: np.ndarray, v_idx: np.ndarray, v_norm: np.ndarray,
                v_codebook: np.ndarray, Pi_v: np.ndarray, scale: float) -> np.ndarray:
    """Attention output over a TurboQuant_prod key cache and an MSE-quantized value cache
    ([ZT] "The Optimization Journey", v2 kernel 3 and v6 "Fused hybrid Triton kernel":
    per compressed block the TQ score, the value dequantization and the accumulation;
    the score is TurboQuant_prod's <y, x_mse> + ||r|| sqrt(pi/2)/d <S y, qjl>, [ZT]
    "Relevance to v6"):

        s[b, i]  = scale * score[b, i]        (score: :func:`scores`, from A = Pi q, T = S_mat q)
        p[b, :]  = softmax(s[b, :])           (max subtracted)
        acc[b]   = sum_i p[b, i] v_norm[i] c_v[v_idx[i]]          (rotated value basis)
        out[b]   = Pi_v^T acc[b]

    Values as in :func:`decode_mse`.  float64 throughout.
    """
    s = scale * scores(A, T, k_idx, k_signs, k_gamma, k_codebook)
    p = np.exp(s - s.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    vc = np.asarray(v_codebook, dtype=np.float64)[np.asarray(v_idx, dtype=np.int64)]
    acc = (p * np.asarray(v_norm, dtype=np.float64)[np.newaxis, :]) @ vc
    return acc @ np.asarray(Pi_v, dtype=np.float64)


# ---------------------------------------------------------------------------
# Outlier split: two TurboQuant-MSE instances per head over disjoint channel sets
# ---------------------------------------------------------------------------

def outlier_channels(keys: np.ndarray, n_out: int) -> np.ndarray:
    """The n_out channels with the largest mean |k| over ``keys`` ([KB] §7 "Fractional
    bits and the outlier split": channels hot across the whole sequence are known ahead
    of time; §11 picks the 32 channels with the largest mean |k|).  Returned in
    increasing order; among equal means the lower channel index is taken first."""
    k = np.asarray(keys, dtype=np.float64)
    D = k.shape[1]
    if not 0 < n_out < D:
        raise ValueError("both channel sets must be non-empty")
    mean_abs = np.mean(np.abs(k), axis=0)
    ranked = sorted(range(D), key=lambda c: (-mean_abs[c], c))
    return np.array(sorted(ranked[:n_out]), dtype=np.int64)


def _regular_channels(channels: np.ndarray, D: int) -> np.ndarray:
    mask = np.ones(D, dtype=bool)
    mask[np.asarray(channels, dtype=np.int64)] = False
    return np.nonzero(mask)[0]


def compress_split(keys: np.ndarray, channels: np.ndarray, Pi_out: np.ndarray, Pi_reg: np.ndarray,
                   cb_out: np.ndarray, cb_reg: np.ndarray):
    """Fractional-bit compression ([KB] §7): the outlier channels of each key and the
    remaining channels are two vectors, each compressed by its own TurboQuant-MSE
    instance (:func:`compress_mse`) with its own rotation, codebook and norm; for 2.5
    bits, 32 outlier channels at 3 bits and 96 at 2.  Returns
    ``(idx_out, norm_out, idx_reg, norm_reg)``."""
    k = np.asarray(keys, dtype=np.float64)
    ch = np.asarray(channels, dtype=np.int64)
    reg = _regular_channels(ch, k.shape[1])
    io, no = compress_mse(k[:, ch], Pi_out, cb_out)
    ir, nr = compress_mse(k[:, reg], Pi_reg, cb_reg)
    return io, no, ir, nr


def prepare_queries_split(Q: np.ndarray, channels: np.ndarray, Pi_out: np.ndarray, Pi_reg: np.ndarray):
    """Each instance's rotated query: A_out = Pi_out q[outlier channels] and
    A_reg = Pi_reg q[other channels] ([KB] §8: rotate the query once per instance)."""
    q = np.asarray(Q, dtype=np.float64)
    ch = np.asarray(channels, dtype=np.int64)
    reg = _regular_channels(ch, q.shape[1])
    return (q[:, ch] @ np.asarray(Pi_out, dtype=np.float64).T,
            q[:, reg] @ np.asarray(Pi_reg, dtype=np.float64).T)


def scores_split(A_out: np.ndarray, A_reg: np.ndarray, idx_out: np.ndarray, norm_out: np.ndarray,
                 cb_out: np.ndarray, idx_reg: np.ndarray, norm_reg: np.ndarray,
                 cb_reg: np.ndarray) -> np.ndarray:
    """<q, k_hat> for the split cache: the sum of the two instances' MSE scores
    (:func:`scores_mse` without norm correction), since the channel sets partition q
    and k.  float64."""
    return scores_mse(A_out, idx_out, norm_out, cb_out) + scores_mse(A_reg, idx_reg, norm_reg, cb_reg)


# ---------------------------------------------------------------------------
# Bit packing (the library's storage format)
# ---------------------------------------------------------------------------

def pack_indices(idx: np.ndarray, bits: int) -> np.ndarray:
    """Pack b-bit indices of each key into a little-endian bit stream.

    Bit t of coordinate d is stream bit bits*d + t; stream bit i is bit
    (i mod 8) of byte i // 8.  A key of D coordinates takes D*bits/8 bytes
    (a 128-dim 2-bit key is 32 bytes, a 3-bit key 48 bytes: [KB] §8).
    """
    idx = np.asarray(idx, dtype=np.int64)
    S, D = idx.shape
    if (D * bits) % 8:
        raise ValueError("D*bits must be a whole number of bytes")
    stream = np.zeros((S, D * bits), dtype=np.uint8)
    for t in range(bits):
        stream[:, t::bits] = (idx >> t) & 1
    return np.packbits(stream.reshape(S, -1, 8), axis=2, bitorder="little").reshape(S, -1)


def unpack_indices(plane: np.ndarray, bits: int, D: int) -> np.ndarray:
    """Inverse of :func:`pack_indices`."""
    plane = np.asarray(plane, dtype=np.uint8)
    S = plane.shape[0]
    stream = np.unpackbits(plane, axis=1, bitorder="little")[:, :D * bits].astype(np.int64)
    idx = np.zeros((S, D), dtype=np.int64)
    for t in range(bits):
        idx |= stream[:, t::bits] << t
    return idx.astype(np.uint8)


def pack_signs(signs: np.ndarray) -> np.ndarray:
    """One bit per coordinate, little-endian: bit d is 1 exactly when sigma_d = +1."""
    s = np.asarray(signs)
    return np.packbits((s > 0).astype(np.uint8), axis=1, bitorder="little")


def unpack_signs(plane: np.ndarray, D: int) -> np.ndarray:
    """Inverse of :func:`pack_signs`: int8 +1 / -1."""
    bits = np.unpackbits(np.asarray(plane, dtype=np.uint8), axis=1, bitorder="little")[:, :D]
    return np.where(bits == 1, 1, -1).astype(np.int8)
