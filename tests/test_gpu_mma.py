"""GPU parity of the bf16 tensor-core path (tcgen05) against the CPU oracle.

Parity bound: max |err| <= 2e-3 ||q_b||_2 against the float64 oracle on the
original queries.  The path rounds A, T and the centroids to bf16 (signs are exact)
and sums in fp32.
"""
import numpy as np
import pytest

from cases import Case, workload_case

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tq():
    from compressed_kv_cache_gb300 import build as tqbuild
    tqbuild.build()
    from compressed_kv_cache_gb300 import tq as mod
    return mod


def dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def f16(x):
    return dev(np.ascontiguousarray(x).astype(np.float16))


def q_tensor(c):
    if c.q_dtype == "bf16":
        return dev(c.Q_raw.view(np.int16)).view(torch.bfloat16)
    return dev(c.Q)


def assert_bf16(got, want, qn_b):
    err = np.abs(got.astype(np.float64) - want)
    bound = 2e-3 * qn_b
    bad = err > bound
    assert np.isfinite(got).all(), "non-finite scores"
    assert not bad.any(), f"{bad.sum()} of {bad.size} outside 2e-3||q||; max err/bound {(err / bound).max():.3f}"


def test_auto_selects_tensor_cores(tq):
    assert tq.auto_path(16, 128) == "bf16_mma"
    assert tq.auto_path(128, 128) == "bf16_mma"
    assert tq.auto_path(8, 128) == "fp32"


UNPACKED = [  # P, B, S, mse_bits (C = 2^bits)
    (1, 16, 129, 2),
    (1, 32, 1000, 2),
    (2, 17, 300, 6),        # C = 64: per-code codebook lookup
    (1, 133, 257, 3),       # two query tiles, ragged last tile
    (1, 32, 40963, 2),      # more tiles than two per SM: full configuration, unpacked rows
]


@pytest.mark.parametrize("P,B,S,bits", UNPACKED)
def test_mma_unpacked(tq, P, B, S, bits):
    c = Case(P, 1, B, S, 128, bits, seed=300 + B + S, random_codebook=True)
    A, T = tq.prepare_queries(q_tensor(c), dev(c.Pi), dev(c.S_mat))
    out = tq.scores(A, T, dev(c.idx), dev(c.signs), dev(c.gamma), dev(c.cb), path="bf16_mma").cpu().numpy()
    want = c.expected()
    assert_bf16(out, want, c.qnorm()[:, :, None])


PACKED = [  # P, H, B, S, bits
    (1, 1, 16, 128, 2),
    (1, 1, 40, 513, 2),
    (2, 2, 128, 300, 3),
    (3, 3, 130, 200, 1),
    (1, 1, 256, 1024, 3),
    (1, 1, 128, 1027, 2),     # rows not 16-byte aligned: epilogue stores from registers
    (1, 1, 64, 41037, 2),     # more tiles than two per SM: full configuration with 64 queries
    (1, 1, 96, 5125, 3),      # full configuration, 96 queries (24 columns an epilogue warp)
]


@pytest.mark.parametrize("P,H,B,S,bits", PACKED)
def test_mma_packed(tq, P, H, B, S, bits):
    c = Case(P, H, B, S, 128, bits, seed=400 + B + S + bits, gamma_dtype="f16", q_dtype="bf16")
    ip, sp = c.packed()
    out = tq.solve_packed(q_tensor(c), dev(ip), dev(sp), f16(c.gamma), dev(c.Pi), dev(c.S_mat), dev(c.cb),
                          bits, path="bf16_mma").cpu().numpy()
    assert_bf16(out, c.expected(), c.qnorm()[:, :, None])


def test_mma_deterministic(tq):
    c = Case(1, 1, 64, 2000, 128, 2, seed=5, gamma_dtype="f16", random_codebook=True)
    ip, sp = c.packed()
    A, T = tq.prepare_queries(dev(c.Q), dev(c.Pi), dev(c.S_mat))
    args = (A, T, dev(ip), dev(sp), f16(c.gamma), dev(c.cb), 2)
    r1 = tq.scores_packed(*args, path="bf16_mma")
    r2 = tq.scores_packed(*args, path="bf16_mma")
    assert torch.equal(r1, r2)


def test_c1_challenge_shape_auto_path(tq):
    c = workload_case("c1")
    out = tq.solve(dev(c.Q[0]), dev(c.idx[0]), dev(c.signs[0]), dev(c.gamma[0]), dev(c.Pi[0]),
                   dev(c.S_mat[0]), dev(c.cb)).cpu().numpy()
    assert_bf16(out, c.expected()[0], c.qnorm()[0][:, None])


def test_c4_prefill_auto_path_sampled(tq):
    c = workload_case("c4")
    ip, sp = c.packed()
    out = tq.solve_packed(q_tensor(c), dev(ip), dev(sp), f16(c.gamma), dev(c.Pi), dev(c.S_mat), dev(c.cb),
                          c.bits).cpu().numpy()
    assert np.isfinite(out).all()
    rng = np.random.default_rng(44)
    n = 40000
    p = np.zeros(n, np.int64)
    b = rng.integers(0, c.B, n)
    s = rng.integers(0, c.S, n)
    b[:2], s[:2] = [0, c.B - 1], [0, c.S - 1]
    assert_bf16(out[p, b, s], c.expected_sampled(p, b, s), c.qnorm()[p, b])
