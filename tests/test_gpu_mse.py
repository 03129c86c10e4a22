"""GPU parity of the MSE-only scorer (tq_scores_mse) against the oracle, through the C ABI.

fp32 arithmetic, so the bound is the fp32 path's: max |err| <= 1e-5 (1 + |score|).
"""
import numpy as np
import pytest

import oracle
from cases import fp32_tol
from conftest import codebook

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tq():
    from compressed_kv_cache_gb300 import build as tqbuild
    tqbuild.build()
    from compressed_kv_cache_gb300 import tq as mod
    assert torch.cuda.is_available()
    return mod


def dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


class MseCase:
    """P problems of S keys and B queries; one rotation per problem.  Keys are unit
    directions scaled to lengths 0.5-3, queries N(0,1): the fp32 bound, written for the
    unit keys of the workloads, keeps its meaning when the lengths stay of order one."""

    def __init__(self, P, B, S, D, bits, seed):
        rng = np.random.default_rng(seed)
        self.bits = bits
        self.cb = codebook(D, bits)[0].astype(np.float32)
        self.Pi = np.stack([oracle.haar_rotation(rng.standard_normal((D, D))) for _ in range(P)]).astype(np.float32)
        self.Q = rng.standard_normal((P, B, D)).astype(np.float32)
        self.idx = np.empty((P, S, D), np.uint8)
        self.norm = np.empty((P, S), np.float16)
        for p in range(P):
            keys = rng.standard_normal((S, D))
            keys *= rng.uniform(0.5, 3.0, (S, 1)) / np.linalg.norm(keys, axis=1, keepdims=True)
            self.idx[p], self.norm[p] = oracle.compress_mse(keys, self.Pi[p], self.cb)
        self.plane = np.stack([oracle.pack_indices(self.idx[p], bits) for p in range(P)])

    def expected(self, corr):
        out = []
        for p in range(self.Q.shape[0]):
            A, _ = oracle.prepare_queries(self.Q[p], self.Pi[p], self.Pi[p])
            out.append(oracle.scores_mse(A, self.idx[p], self.norm[p], self.cb, corr))
        return np.stack(out)

    def run(self, tq, corr):
        A, _ = tq.prepare_queries(dev(self.Q), dev(self.Pi), dev(self.Pi))
        return tq.scores_mse(A, dev(self.plane), dev(self.norm), dev(self.cb), self.bits,
                             norm_correction=corr).cpu().numpy()


def assert_fp32(got, want):
    err = np.abs(got.astype(np.float64) - want)
    bad = err > fp32_tol(want)
    assert not bad.any(), f"{bad.sum()} of {bad.size} outside 1e-5(1+|s|); max err {err.max():.3e}"


@pytest.mark.parametrize("bits", [1, 2, 3, 4])
@pytest.mark.parametrize("D", [32, 128, 256])
@pytest.mark.parametrize("B", [1, 3, 8, 11])
def test_scores_mse(tq, bits, D, B):
    c = MseCase(2, B, 300, D, bits, seed=500 + 7 * D + 3 * bits + B)
    for corr in (False, True):
        assert_fp32(c.run(tq, corr), c.expected(corr))


def test_scores_mse_stream_k_many_problems(tq):
    """D = 128 lookup-table kernel with CTA ranges that start and end inside problems."""
    c = MseCase(100, 3, 1001, 128, 2, seed=601)
    for corr in (False, True):
        assert_fp32(c.run(tq, corr), c.expected(corr))


def test_scores_mse_decode_batch(tq):
    """A GQA-shaped decode batch (8 problems x 4 queries x 32768 keys, 3-bit codes)."""
    c = MseCase(8, 4, 32768, 128, 3, seed=602)
    assert_fp32(c.run(tq, True), c.expected(True))


def test_scores_mse_deterministic(tq):
    c = MseCase(1, 5, 4000, 128, 2, seed=603)
    a = c.run(tq, True)
    assert np.array_equal(a, c.run(tq, True))
