"""GPU parity of the fused decode over a TurboQuant_prod key cache (tq_decode_prod)
against the oracle's decode_prod, through the C ABI.  fp32 bound on the outputs:
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
    """P problems (head p % H) of S unit keys compressed by TurboQuant_prod with kbits-bit
    codes plus signs and fp16 gamma, and S values of length 0.5-3 compressed by
    TurboQuant-MSE with vbits-bit codes; B queries per problem."""
    D = 128
    rng = np.random.default_rng(seed)
    Pk = np.stack([oracle.haar_rotation(rng.standard_normal((D, D))) for _ in range(H)]).astype(np.float32)
    Sm = rng.standard_normal((H, D, D)).astype(np.float32)
    Pv = np.stack([oracle.haar_rotation(rng.standard_normal((D, D))) for _ in range(H)]).astype(np.float32)
    kcb = codebook(D, kbits)[0].astype(np.float32)
    vcb = codebook(D, vbits)[0].astype(np.float32)
    Q = rng.standard_normal((P, B, D)).astype(np.float32)
    ki = np.empty((P, S, D), np.uint8); ks = np.empty((P, S, D), np.int8); kg = np.empty((P, S), np.float16)
    vi = np.empty((P, S, D), np.uint8); vn = np.empty((P, S), np.float16)
    for p in range(P):
        K = rng.standard_normal((S, D))
        K /= np.linalg.norm(K, axis=1, keepdims=True)
        V = rng.standard_normal((S, D))
        V *= rng.uniform(0.5, 3.0, (S, 1)) / np.linalg.norm(V, axis=1, keepdims=True)
        ki[p], ks[p], kg[p] = oracle.compress_prod(K, Pk[p % H], Sm[p % H], kcb, "f16")
        vi[p], vn[p] = oracle.compress_mse(V, Pv[p % H], vcb)
    kp = np.stack([oracle.pack_indices(ki[p], kbits) for p in range(P)])
    sp = np.stack([oracle.pack_signs(ks[p]) for p in range(P)])
    vp = np.stack([oracle.pack_indices(vi[p], vbits) for p in range(P)])
    sc = 1.0 / math.sqrt(D) if scale is None else scale
    A, T = tq.prepare_queries(dev(Q), dev(Pk), dev(Sm))
    got = tq.decode_prod(A, T, dev(kp), dev(sp), dev(kg), dev(kcb), kbits, dev(vp), dev(vn), dev(vcb), vbits,
                         dev(Pv), scale=sc).cpu().numpy()
    want = np.empty((P, B, D))
    for p in range(P):
        Ao, To = oracle.prepare_queries(Q[p], Pk[p % H], Sm[p % H])
        want[p] = oracle.decode_prod(Ao, To, ki[p], ks[p], kg[p], kcb, vi[p], vn[p], vcb, Pv[p % H], sc)
    err = np.abs(got.astype(np.float64) - want)
    bad = err > fp32_tol(want)
    assert not bad.any(), f"{bad.sum()} of {bad.size} outside 1e-5(1+|o|); max err {err.max():.3e}"
    return got


@pytest.mark.parametrize("kbits,vbits", [(1, 1), (2, 3), (3, 2), (2, 2)])
@pytest.mark.parametrize("B", [1, 3, 8])
def test_decode_prod(tq, kbits, vbits, B):
    run_case(tq, 2, 2, B, 3001, kbits, vbits, seed=900 + 10 * kbits + vbits + B)


def test_decode_prod_long_context_and_shapes(tq):
    """Many chunks and a ragged last chunk (S = 70001), a single key, S between one and
    two chunks, query tiles past B, problems sharing heads, a scale other than 1/sqrt(D)."""
    run_case(tq, 1, 1, 1, 70001, 2, 3, seed=911)
    run_case(tq, 3, 1, 2, 1, 2, 2, seed=912)
    run_case(tq, 1, 1, 5, 300, 3, 3, seed=913)
    run_case(tq, 4, 2, 13, 777, 2, 3, seed=914, scale=0.3)


def test_decode_prod_deterministic(tq):
    a = run_case(tq, 1, 1, 4, 9000, 2, 3, seed=915)
    b = run_case(tq, 1, 1, 4, 9000, 2, 3, seed=915)
    assert np.array_equal(a, b)


def test_decode_prod_argument_errors(tq):
    L = tq.lib()
    f = 0x100000
    # D != 128, a null sign plane, bits out of range, a short workspace
    assert L.tq_decode_prod(f, f, f, f, f, f, 2, f, f, f, 3, f, f, 1, 1, 1, 64, 64, 0.1, f, 1 << 20, None) == 2
    assert L.tq_decode_prod(f, f, f, None, f, f, 2, f, f, f, 3, f, f, 1, 1, 1, 64, 128, 0.1, f, 1 << 20, None) == 1
    assert L.tq_decode_prod(f, f, f, f, f, f, 4, f, f, f, 3, f, f, 1, 1, 1, 64, 128, 0.1, f, 1 << 20, None) == 1
    assert L.tq_decode_prod(f, f, f, f, f, f, 2, f, f, f, 3, f, f, 1, 1, 1, 64, 128, 0.1, f, 16, None) == 4
