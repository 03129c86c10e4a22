"""GPU parity of the fused decode over MSE keys and values (tq_decode_mse) against the
oracle's rotated-domain decode, through the C ABI.  fp32 bound on the outputs:
max |err| <= 1e-5 (1 + |out|)."""
import math

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


def run_case(tq, P, H, B, S, kbits, vbits, seed, scale=None):
    D = 128
    rng = np.random.default_rng(seed)
    Pk = np.stack([oracle.haar_rotation(rng.standard_normal((D, D))) for _ in range(H)]).astype(np.float32)
    Pv = np.stack([oracle.haar_rotation(rng.standard_normal((D, D))) for _ in range(H)]).astype(np.float32)
    kcb = codebook(D, kbits)[0].astype(np.float32)
    vcb = codebook(D, vbits)[0].astype(np.float32)
    Q = rng.standard_normal((P, B, D)).astype(np.float32)
    ki = np.empty((P, S, D), np.uint8); kn = np.empty((P, S), np.float16)
    vi = np.empty((P, S, D), np.uint8); vn = np.empty((P, S), np.float16)
    for p in range(P):
        K = rng.standard_normal((S, D))
        K *= rng.uniform(0.5, 3.0, (S, 1)) / np.linalg.norm(K, axis=1, keepdims=True)
        V = rng.standard_normal((S, D))
        ki[p], kn[p] = oracle.compress_mse(K, Pk[p % H], kcb)
        vi[p], vn[p] = oracle.compress_mse(V, Pv[p % H], vcb)
    kp = np.stack([oracle.pack_indices(ki[p], kbits) for p in range(P)])
    vp = np.stack([oracle.pack_indices(vi[p], vbits) for p in range(P)])
    sc = 1.0 / math.sqrt(D) if scale is None else scale
    A, _ = tq.prepare_queries(dev(Q), dev(Pk), dev(Pk))
    got = tq.decode_mse(A, dev(kp), dev(kn), dev(kcb), kbits, dev(vp), dev(vn), dev(vcb), vbits, dev(Pv),
                        scale=sc).cpu().numpy()
    want = np.stack([oracle.decode_mse(Q[p].astype(np.float64) @ Pk[p % H].astype(np.float64).T, ki[p], kn[p],
                                       kcb, vi[p], vn[p], vcb, Pv[p % H], sc) for p in range(P)])
    err = np.abs(got.astype(np.float64) - want)
    bad = err > fp32_tol(want)
    assert not bad.any(), f"{bad.sum()} of {bad.size} outside 1e-5(1+|o|); max err {err.max():.3e}"
    return got


@pytest.mark.parametrize("kbits,vbits", [(1, 1), (2, 3), (3, 2), (3, 3)])
@pytest.mark.parametrize("B", [1, 3, 8])
def test_decode_mse(tq, kbits, vbits, B):
    run_case(tq, 2, 2, B, 3001, kbits, vbits, seed=800 + 10 * kbits + vbits + B)


def test_decode_mse_long_context_and_shapes(tq):
    """Many chunks and a ragged last chunk (S = 70001), a single key, query tiles past B,
    problems sharing heads, and a logit scale other than 1/sqrt(D)."""
    run_case(tq, 1, 1, 1, 70001, 3, 3, seed=811)
    run_case(tq, 3, 1, 2, 1, 2, 2, seed=812)
    run_case(tq, 4, 2, 13, 777, 2, 3, seed=813, scale=0.3)


def test_decode_mse_deterministic(tq):
    a = run_case(tq, 1, 1, 4, 9000, 3, 3, seed=814)
    b = run_case(tq, 1, 1, 4, 9000, 3, 3, seed=814)
    assert np.array_equal(a, b)
