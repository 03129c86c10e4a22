"""GPU parity of the randomized-Hadamard query transform (tq_prepare_queries_hadamard)
against the oracle, and a whole path with a Hadamard rotation: compressor, transform,
packed scorer.  fp32 bound: max |err| <= 1e-5 (1 + |value|)."""
import numpy as np
import pytest

import oracle
import synth
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


def assert_fp32(got, want):
    err = np.abs(np.asarray(got, dtype=np.float64) - want)
    bad = err > fp32_tol(want)
    assert not bad.any(), f"{bad.sum()} of {bad.size} outside 1e-5(1+|x|); max err {err.max():.3e}"


@pytest.mark.parametrize("D", [2, 8, 32, 64, 128, 256])
@pytest.mark.parametrize("B", [1, 5, 8, 13, 40])
@pytest.mark.parametrize("qdt", ["f32", "bf16"])
def test_prepare_hadamard(tq, D, B, qdt):
    P, H = 3, 2
    rng = np.random.default_rng(700 + D + B)
    signs = rng.choice([-1.0, 1.0], size=(H, D)).astype(np.float32)
    S_mat = rng.standard_normal((H, D, D)).astype(np.float32)
    Qv = np.empty((P, B, D), np.float32)
    Qraw = np.empty((P, B, D), np.float32 if qdt == "f32" else np.uint16)
    for p in range(P):
        Qv[p], Qraw[p] = synth.queries(700 + D, p, B, D, qdt)
    Qt = dev(Qraw) if qdt == "f32" else dev(Qraw.view(np.int16)).view(torch.bfloat16)
    A, T = tq.prepare_queries_hadamard(Qt, dev(signs), dev(S_mat))
    for p in range(P):
        h = p % H
        q = Qv[p].astype(np.float64)
        assert_fp32(A[p].cpu().numpy(), oracle.fwht(q * signs[h]))
        assert_fp32(T[p].cpu().numpy(), q @ S_mat[h].astype(np.float64).T)


@pytest.mark.parametrize("P,D", [(200, 64), (130, 128)])
def test_prepare_hadamard_many_problems(tq, P, D):
    """Enough problems that every warp of the transform takes four rows of S_mat."""
    H, B = 4, 3
    rng = np.random.default_rng(800 + P + D)
    signs = rng.choice([-1.0, 1.0], size=(H, D)).astype(np.float32)
    S_mat = rng.standard_normal((H, D, D)).astype(np.float32)
    Q = rng.standard_normal((P, B, D)).astype(np.float32)
    A, T = tq.prepare_queries_hadamard(dev(Q), dev(signs), dev(S_mat))
    A, T = A.cpu().numpy(), T.cpu().numpy()
    for p in range(P):
        h = p % H
        q = Q[p].astype(np.float64)
        assert_fp32(A[p], oracle.fwht(q * signs[h]))
        assert_fp32(T[p], q @ S_mat[h].astype(np.float64).T)


def test_hadamard_rotation_through_the_whole_path(tq):
    """Keys compressed on the GPU with the dense H diag(s), queries transformed by the fast
    transform, packed fp32 scorer: the oracle's scores for the same rotation."""
    D, S, B, bits = 128, 5000, 3, 2
    rng = np.random.default_rng(710)
    s = rng.choice([-1.0, 1.0], size=D).astype(np.float32)
    Pi = tq.hadamard_rotation(s)
    S_mat = rng.standard_normal((D, D)).astype(np.float32)
    cb = codebook(D, bits)[0].astype(np.float32)
    keys = synth.unit_keys(710, 0, 0, S, D).astype(np.float32)
    Q = synth.queries(710, 0, B, D, "f32")[0]
    k_idx, k_sg, k_g = tq.compress_keys(dev(keys), dev(Pi), dev(S_mat), dev(cb), torch.float16)
    A, T = tq.prepare_queries_hadamard(dev(Q), dev(s), dev(S_mat))
    out = tq.scores_packed(A, T, tq.pack_indices(k_idx, bits), tq.pack_signs(k_sg), k_g, dev(cb), bits,
                           path="fp32").cpu().numpy()
    # the oracle scores the GPU's own codes (a code on a cell edge may differ between the
    # fp32 compressor and an exact one) with its float64 transform of the same rotation
    Ao, To = oracle.prepare_queries(Q, oracle.hadamard_rotation(s), S_mat)
    want = oracle.scores(Ao, To, k_idx.cpu().numpy(), k_sg.cpu().numpy(),
                         k_g.cpu().numpy().astype(np.float64), cb)
    assert_fp32(out, want)
    # the rotation really is the one the codes were made with: the GPU codes agree with
    # the oracle's compression of the same keys except at cell edges
    idx_o, _, _ = oracle.compress_prod(keys, Pi, S_mat, cb, "f16")
    assert np.mean(idx_o == k_idx.cpu().numpy()) > 0.999
