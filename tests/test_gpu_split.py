"""GPU parity of the outlier-split cache (tq_prepare_queries_split, tq_scores_split)
against the oracle's split compressor, transform and scorer, through the C ABI.  fp32
bound: max |err| <= 1e-5 (1 + |x|) on the rotated queries and on the scores."""
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


def run_case(tq, P, H, B, S, D, n_out, bo, br, seed, qdt="f32"):
    rng = np.random.default_rng(seed)
    n_reg = D - n_out
    keys = [synth.unit_keys(seed, p, 0, S, D) * rng.uniform(0.5, 3.0, (S, 1)) for p in range(P)]
    ch = oracle.outlier_channels(keys[0], n_out)             # known ahead of time, shared
    Po = np.stack([oracle.haar_rotation(rng.standard_normal((n_out, n_out))) for _ in range(H)]).astype(np.float32)
    Pr = np.stack([oracle.haar_rotation(rng.standard_normal((n_reg, n_reg))) for _ in range(H)]).astype(np.float32)
    co = codebook(n_out, bo)[0].astype(np.float32)
    cr = codebook(n_reg, br)[0].astype(np.float32)
    Q32, Qraw = synth.queries(seed, 0, P * B, D, qdt)
    Q32 = Q32.reshape(P, B, D)
    io = np.empty((P, S, n_out), np.uint8); no = np.empty((P, S), np.float16)
    ir = np.empty((P, S, n_reg), np.uint8); nr = np.empty((P, S), np.float16)
    for p in range(P):
        io[p], no[p], ir[p], nr[p] = oracle.compress_split(keys[p], ch, Po[p % H], Pr[p % H], co, cr)
    op = np.stack([oracle.pack_indices(io[p], bo) for p in range(P)])
    rp = np.stack([oracle.pack_indices(ir[p], br) for p in range(P)])
    if qdt == "bf16":
        Qt = dev(Qraw.reshape(P, B, D).view(np.int16)).view(torch.bfloat16)
    else:
        Qt = dev(Q32)
    Ao, Ar = tq.prepare_queries_split(Qt, dev(ch.astype(np.int32)), dev(Po), dev(Pr))
    got = tq.scores_split(Ao, Ar, dev(op), dev(no), dev(co), bo, dev(rp), dev(nr), dev(cr), br).cpu().numpy()
    for p in range(P):
        wo, wr = oracle.prepare_queries_split(Q32[p], ch, Po[p % H], Pr[p % H])
        for name, g, w in (("A_out", Ao[p].cpu().numpy(), wo), ("A_reg", Ar[p].cpu().numpy(), wr)):
            err = np.abs(g.astype(np.float64) - w)
            assert (err <= fp32_tol(w)).all(), f"{name}: max err {err.max():.3e}"
        want = oracle.scores_split(wo, wr, io[p], no[p], co, ir[p], nr[p], cr)
        err = np.abs(got[p].astype(np.float64) - want)
        bad = err > fp32_tol(want)
        assert not bad.any(), f"{bad.sum()} of {bad.size} scores outside 1e-5(1+|s|); max err {err.max():.3e}"


@pytest.mark.parametrize("bo,br", [(3, 2), (2, 1), (4, 3)])
@pytest.mark.parametrize("B", [1, 3, 9])
def test_split_scores(tq, bo, br, B):
    """The printed split (32 outlier channels of 128, 3 + 2 bits) and other widths."""
    run_case(tq, 2, 2, B, 1500, 128, 32, bo, br, seed=600 + 10 * bo + br + B)


def test_split_shapes(tq):
    """Other splits and head sizes, ragged S, one key, problems sharing heads, bf16 queries."""
    run_case(tq, 3, 1, 2, 777, 64, 32, 3, 2, seed=611)
    run_case(tq, 1, 1, 4, 1, 128, 64, 3, 2, seed=612)
    run_case(tq, 4, 2, 5, 300, 256, 96, 3, 2, seed=613)
    run_case(tq, 1, 1, 16, 2000, 128, 32, 3, 2, seed=614, qdt="bf16")


def test_split_argument_errors(tq):
    L = tq.lib()
    f = 0x100000
    # n_out not a multiple of 32, 5-bit codes, a null plane (nothing is launched)
    assert L.tq_scores_split(f, f, f, f, f, 3, f, f, f, 2, f, 1, 1, 10, 16, 112, None) == 2
    assert L.tq_scores_split(f, f, f, f, f, 5, f, f, f, 2, f, 1, 1, 10, 32, 96, None) == 1
    assert L.tq_scores_split(f, f, None, f, f, 3, f, f, f, 2, f, 1, 1, 10, 32, 96, None) == 1
    # n_out >= D, misaligned channels
    assert L.tq_prepare_queries_split(f, 0, f, f, f, f, f, 1, 1, 1, 128, 128, None) == 1
    assert L.tq_prepare_queries_split(f, 0, f + 4, f, f, f, f, 1, 1, 1, 128, 32, None) == 3
