"""Test inputs: raw draws from ``synth``, compressed and scored by the CPU oracle.

Nothing here comes from the GPU path.  ``build_case`` returns NumPy arrays for a
whole workload (all problems), ready to be copied to the device.
"""
from __future__ import annotations

import functools

import numpy as np

import oracle
import synth
from conftest import codebook as _lloyd


@functools.lru_cache(maxsize=None)
def rotation(seed: int, head: int, D: int) -> np.ndarray:
    return oracle.haar_rotation(synth.rotation_seed_matrix(seed, head, D)).astype(np.float32)


def codebook_for(D: int, mse_bits: int, seed: int | None = None) -> np.ndarray:
    """Lloyd-Max codebook for D >= 3; for tiny D (or when a seed is given, to save time
    on shape sweeps) a sorted random codebook -- the scorer's contract is any fp32 table."""
    if seed is None and D >= 3:
        return _lloyd(D, mse_bits)[0].astype(np.float32)
    rng = np.random.default_rng(seed if seed is not None else 0)
    return np.sort(rng.standard_normal(1 << mse_bits) / np.sqrt(max(D, 1))).astype(np.float32)


class Case:
    """A compressed workload: P problems x (B queries, S keys of length D)."""

    def __init__(self, P, H, B, S, D, mse_bits, seed, gamma_dtype="f32", q_dtype="f32",
                 random_codebook=False):
        self.P, self.H, self.B, self.S, self.D = P, H, B, S, D
        self.mse_bits, self.bits, self.seed = mse_bits, mse_bits, seed
        self.cb = codebook_for(D, mse_bits, seed if random_codebook else None)
        self.Pi = np.stack([rotation(seed, h, D) for h in range(H)])
        self.S_mat = np.stack([synth.s_matrix(seed, h, D) for h in range(H)])
        self.idx = np.empty((P, S, D), np.uint8)
        self.signs = np.empty((P, S, D), np.int8)
        self.gamma = np.empty((P, S), np.float32 if gamma_dtype == "f32" else np.float16)
        self.Q = np.empty((P, B, D), np.float32)
        self.Q_raw = np.empty((P, B, D), np.float32 if q_dtype == "f32" else np.uint16)
        self.q_dtype = q_dtype
        for p in range(P):
            h = p % H
            keys = synth.unit_keys(seed, p, 0, S, D)
            self.idx[p], self.signs[p], self.gamma[p] = oracle.compress_prod(
                keys, self.Pi[h], self.S_mat[h], self.cb, gamma_dtype)
            self.Q[p], self.Q_raw[p] = synth.queries(seed, p, B, D, q_dtype)
        self._A = self._T = None

    # ---- oracle side ----
    def AT(self):
        if self._A is None:
            A = np.empty((self.P, self.B, self.D))
            T = np.empty((self.P, self.B, self.D))
            for p in range(self.P):
                A[p], T[p] = oracle.prepare_queries(self.Q[p], self.Pi[p % self.H], self.S_mat[p % self.H])
            self._A, self._T = A, T
        return self._A, self._T

    def expected(self):
        A, T = self.AT()
        return np.stack([oracle.scores(A[p], T[p], self.idx[p], self.signs[p], self.gamma[p], self.cb)
                         for p in range(self.P)])

    def expected_sampled(self, p_idx, b_idx, s_idx):
        A, T = self.AT()
        out = np.empty(len(p_idx))
        for p in np.unique(p_idx):
            sel = np.nonzero(p_idx == p)[0]
            out[sel] = oracle.scores_sampled(A[p], T[p], self.idx[p][s_idx[sel]], self.signs[p][s_idx[sel]],
                                             self.gamma[p][s_idx[sel]], self.cb, b_idx[sel])
        return out

    def qnorm(self):
        return np.linalg.norm(self.Q.astype(np.float64), axis=2)      # [P,B]

    def packed(self):
        ip = np.stack([oracle.pack_indices(self.idx[p], self.bits) for p in range(self.P)])
        sp = np.stack([oracle.pack_signs(self.signs[p]) for p in range(self.P)])
        return ip, sp


@functools.lru_cache(maxsize=None)
def workload_case(key: str) -> Case:
    w = synth.WORKLOADS[key]
    return Case(w.P, w.H, w.B, w.S, w.D, w.mse_bits, w.seed, w.gamma_dtype, w.q_dtype)


def fp32_tol(expected):
    """Parity bound of the fp32 path: 1e-5 (1 + |score|)."""
    return 1e-5 * (1.0 + np.abs(expected))


def bf16_tol(qnorm_b):
    """Parity bound of the bf16 tensor-core path: 2e-3 ||q_b||_2."""
    return 2e-3 * qnorm_b
