"""GPU parity: every kernel of libtq against the CPU oracle, through the C ABI.

Tolerances are the parity bounds: fp32 path max |err| <= 1e-5 (1 + |score|);
bf16 tensor-core path max |err| <= 2e-3 ||q_b||_2; packing bit-exact.
"""
import time

import numpy as np
import pytest

import oracle
from cases import Case, bf16_tol, fp32_tol, workload_case
from conftest import golden

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


def f16(x):
    return dev(np.ascontiguousarray(x).astype(np.float16))


def q_tensor(case):
    if case.q_dtype == "bf16":
        return dev(case.Q_raw.view(np.int16)).view(torch.bfloat16)
    return dev(case.Q)


def assert_fp32(got, want):
    err = np.abs(got.astype(np.float64) - want)
    bad = err > fp32_tol(want)
    assert not bad.any(), f"{bad.sum()} of {bad.size} outside 1e-5(1+|s|); max err {err.max():.3e}"


def assert_bf16(got, want, qn):
    err = np.abs(got.astype(np.float64) - want)
    bad = err > bf16_tol(qn)
    assert not bad.any(), f"{bad.sum()} of {bad.size} outside 2e-3||q||; max err {err.max():.3e}"


# ---------------------------------------------------------------------------
# the page's worked example (D = 2) through the generic kernels
# ---------------------------------------------------------------------------

def test_worked_example(tq):
    g = golden("worked_example.json")
    Q = dev(np.array(g["Q"], np.float32))
    Pi, Sm = dev(np.array(g["Pi"], np.float32)), dev(np.array(g["S_mat"], np.float32))
    idx = dev(np.array(g["K_idx"], np.uint8))
    sg = dev(np.array(g["signs"], np.int8))
    gamma = dev(np.array(g["gamma"], np.float32))
    cb = dev(np.array(g["codebook"], np.float32))
    A, T = tq.prepare_queries(Q, Pi, Sm)
    assert A.cpu().tolist() == g["A"] and T.cpu().tolist() == g["T"]
    out = tq.scores(A, T, idx, sg, gamma, cb, path="fp32").cpu().numpy()
    assert np.round(out.astype(np.float64), g["decimals"]).tolist() == g["scores"]
    fused = tq.solve(Q, idx, sg, gamma, Pi, Sm, cb, path="fp32").cpu().numpy()
    np.testing.assert_array_equal(fused, out)


# ---------------------------------------------------------------------------
# query transform
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("P,H,B,D", [(1, 1, 1, 2), (3, 2, 5, 37), (2, 2, 9, 128), (4, 4, 3, 256), (8, 8, 4, 128),
                                     # 32 queries per CTA from B = 32 on (D <= 256), ragged last tile
                                     (2, 1, 37, 128), (1, 1, 64, 256), (2, 2, 33, 37), (1, 1, 96, 200),
                                     # many problems: four rows a warp, ragged last slice at D = 37
                                     (100, 4, 3, 128), (300, 3, 2, 37)])
@pytest.mark.parametrize("qdt", ["f32", "bf16"])
def test_prepare_queries(tq, P, H, B, D, qdt):
    c = Case(P, H, B, 1, D, 2, seed=50 + P + D, q_dtype=qdt, random_codebook=True)
    Qt = q_tensor(c)
    A, T = tq.prepare_queries(Qt, dev(c.Pi), dev(c.S_mat))
    Aw, Tw = c.AT()
    # fp32 dot products of length D: bound the error by D * 2^-24 * sum |Pi_dj q_j|
    for got, want, M in ((A, Aw, c.Pi), (T, Tw, c.S_mat)):
        mag = np.stack([np.abs(c.Q[p].astype(np.float64)) @ np.abs(M[p % H].astype(np.float64)).T for p in range(P)])
        err = np.abs(got.cpu().numpy().astype(np.float64) - want)
        assert (err <= D * 2.0 ** -24 * mag + 1e-30).all(), err.max()


# ---------------------------------------------------------------------------
# unpacked scorer (generic D, any C)
# ---------------------------------------------------------------------------

UNPACKED_SHAPES = [
    # P, B, S, D, mse_bits (C = 2^bits)
    (1, 1, 1, 3, 0),
    (1, 3, 130, 2, 2),
    (2, 5, 257, 37, 4),
    (1, 17, 300, 128, 2),
    (3, 8, 1000, 64, 8),
    (1, 40, 129, 128, 3),
    (2, 2, 513, 256, 1),
]


@pytest.mark.parametrize("P,B,S,D,bits", UNPACKED_SHAPES)
def test_scores_unpacked_fp32(tq, P, B, S, D, bits):
    c = Case(P, 1, B, S, D, bits, seed=100 + S, random_codebook=True)
    A, T = c.AT()
    out = tq.scores(dev(A.astype(np.float32)), dev(T.astype(np.float32)), dev(c.idx), dev(c.signs),
                    dev(c.gamma), dev(c.cb), path="fp32").cpu().numpy()
    # the oracle from the fp32-rounded A, T (what the kernel is given)
    want = np.stack([oracle.scores(A[p].astype(np.float32), T[p].astype(np.float32), c.idx[p], c.signs[p],
                                   c.gamma[p], c.cb) for p in range(P)])
    assert_fp32(out.reshape(want.shape), want)


# ---------------------------------------------------------------------------
# packed scorer
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("bits", [1, 2, 3])
@pytest.mark.parametrize("D", [32, 64, 96, 128, 256])
@pytest.mark.parametrize("B", [1, 3, 8, 11])
def test_scores_packed_fp32(tq, bits, D, B):
    P, S = 2, 300
    c = Case(P, 2, B, S, D, bits, seed=7 * D + bits, gamma_dtype="f16", random_codebook=True)
    ip, sp = c.packed()
    Qt = q_tensor(c)
    A, T = tq.prepare_queries(Qt, dev(c.Pi), dev(c.S_mat))
    out = tq.scores_packed(A, T, dev(ip), dev(sp), f16(c.gamma), dev(c.cb), bits, path="fp32").cpu().numpy()
    assert_fp32(out, c.expected())
    # the fused entry (for B <= 8 at D = 128 a single kernel that also does the transform)
    fused = tq.solve_packed(Qt, dev(ip), dev(sp), f16(c.gamma), dev(c.Pi), dev(c.S_mat), dev(c.cb), bits,
                            path="fp32").cpu().numpy()
    assert_fp32(fused, c.expected())


# ---------------------------------------------------------------------------
# bit packing (bit-exact both ways)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("bits", [1, 2, 3, 4, 5, 8])
@pytest.mark.parametrize("D", [8, 32, 96, 128, 256])
def test_pack_unpack_bit_exact(tq, bits, D):
    rng = np.random.default_rng(bits * 31 + D)
    idx = rng.integers(0, 1 << bits, (129, D)).astype(np.uint8)
    sg = np.where(rng.random((129, D)) < 0.5, 1, -1).astype(np.int8)
    want_plane = oracle.pack_indices(idx, bits)
    got_plane = tq.pack_indices(dev(idx), bits).cpu().numpy()
    np.testing.assert_array_equal(got_plane, want_plane)
    np.testing.assert_array_equal(tq.unpack_indices(dev(want_plane), D, bits).cpu().numpy(), idx)
    want_sp = oracle.pack_signs(sg)
    np.testing.assert_array_equal(tq.pack_signs(dev(sg)).cpu().numpy(), want_sp)
    np.testing.assert_array_equal(tq.unpack_signs(dev(want_sp), D).cpu().numpy(), sg)


def test_pack_hand_worked_bytes(tq):
    for case in golden("pack_bytes.json")["cases"]:
        if case["kind"] == "indices":
            got = tq.pack_indices(dev(np.array([case["idx"]], np.uint8)), case["bits"]).cpu().numpy()
        else:
            sg = -np.ones((1, case["D"]), np.int8)
            sg[0, case["plus_at"]] = 1
            got = tq.pack_signs(dev(sg)).cpu().numpy()
        assert got[0].tolist() == case["bytes"]


# ---------------------------------------------------------------------------
# the five workloads at full size
# ---------------------------------------------------------------------------

def test_c0_oracle_scale_fused(tq):
    c = workload_case("c0")
    ws = torch.empty(tq.workspace_bytes(1, c.B, c.D), dtype=torch.uint8, device="cuda")
    out = tq.solve(dev(c.Q[0]), dev(c.idx[0]), dev(c.signs[0]), dev(c.gamma[0]), dev(c.Pi[0]),
                   dev(c.S_mat[0]), dev(c.cb), path="fp32", workspace=ws).cpu().numpy()
    assert_fp32(out, c.expected()[0])


def test_c1_challenge_shape_fp32(tq):
    c = workload_case("c1")
    out = tq.solve(dev(c.Q[0]), dev(c.idx[0]), dev(c.signs[0]), dev(c.gamma[0]), dev(c.Pi[0]),
                   dev(c.S_mat[0]), dev(c.cb), path="fp32").cpu().numpy()
    assert_fp32(out, c.expected()[0])


def test_c2_single_query_decode(tq):
    c = workload_case("c2")
    ip, sp = c.packed()
    out = tq.solve_packed(dev(c.Q[0]), dev(ip[0]), dev(sp[0]), f16(c.gamma[0]), dev(c.Pi[0]),
                          dev(c.S_mat[0]), dev(c.cb), c.bits).cpu().numpy()
    assert_fp32(out, c.expected()[0])


def _sample(c, n, seed):
    rng = np.random.default_rng(seed)
    p = rng.integers(0, c.P, n)
    b = rng.integers(0, c.B, n)
    s = rng.integers(0, c.S, n)
    # always include both ends of the key range of the first and last problem
    p[:4], b[:4], s[:4] = [0, 0, c.P - 1, c.P - 1], [0, c.B - 1, 0, c.B - 1], [0, c.S - 1, 0, c.S - 1]
    return p, b, s


def test_c3_gqa_batch_sampled(tq):
    c = workload_case("c3")
    ip, sp = c.packed()
    out = tq.solve_packed(dev(c.Q), dev(ip), dev(sp), f16(c.gamma), dev(c.Pi), dev(c.S_mat), dev(c.cb),
                          c.bits).cpu().numpy()
    p, b, s = _sample(c, 20000, 3)
    assert_fp32(out[p, b, s], c.expected_sampled(p, b, s))
    # problem p = sequence * 8 + kv_head uses head p % 8: a whole problem of the last head
    full = oracle.scores_from_queries(c.Q[15], c.Pi[7], c.S_mat[7], c.idx[15], c.signs[15], c.gamma[15], c.cb)
    assert_fp32(out[15], full)


def test_c4_prefill_fp32_path_sampled(tq):
    c = workload_case("c4")
    ip, sp = c.packed()
    out = tq.solve_packed(q_tensor(c), dev(ip), dev(sp), f16(c.gamma), dev(c.Pi), dev(c.S_mat), dev(c.cb),
                          c.bits, path="fp32").cpu().numpy()
    p, b, s = _sample(c, 20000, 4)
    assert_fp32(out[p, b, s], c.expected_sampled(p, b, s))


def test_fused_solve_many_keys_per_thread(tq):
    """One problem with far more keys than the fused kernel's threads: each CTA's range
    spans several key tiles, so its two-stage ring of tiles is refilled; S is ragged and
    the queries are bf16."""
    c = Case(1, 1, 2, 400_001, 128, 3, seed=91, gamma_dtype="f16", q_dtype="bf16")
    ip, sp = c.packed()
    out = tq.solve_packed(q_tensor(c), dev(ip), dev(sp), f16(c.gamma), dev(c.Pi), dev(c.S_mat), dev(c.cb),
                          c.bits, path="fp32").cpu().numpy()
    p, b, s = _sample(c, 20000, 5)
    assert_fp32(out[p, b, s], c.expected_sampled(p, b, s))


@pytest.mark.parametrize("bits,S", [(2, 172_801), (3, 161_281)])
def test_fused_solve_staged_range_two_keys_per_thread(tq, bits, S):
    """Key ranges of one to three tiles of the fused kernel's ring (a tile holds one key
    per thread), so some threads score keys of two tiles; the last range is ragged."""
    c = Case(1, 1, 2, S, 128, bits, seed=93 + bits, gamma_dtype="f16")
    ip, sp = c.packed()
    out = tq.solve_packed(q_tensor(c), dev(ip), dev(sp), f16(c.gamma), dev(c.Pi), dev(c.S_mat), dev(c.cb),
                          c.bits, path="fp32").cpu().numpy()
    assert_fp32(out, c.expected())


def test_stream_k_ranges_cross_problems(tq):
    """Enough problems for the transform + stream-K scorer: CTA key ranges start and end
    inside problems, S is not a multiple of the block, and heads repeat every 4 problems."""
    c = Case(100, 4, 3, 1001, 128, 2, seed=92, gamma_dtype="f16")
    ip, sp = c.packed()
    Qt = q_tensor(c)
    out = tq.solve_packed(Qt, dev(ip), dev(sp), f16(c.gamma), dev(c.Pi), dev(c.S_mat), dev(c.cb), c.bits,
                          path="fp32").cpu().numpy()
    assert_fp32(out, c.expected())
    A, T = tq.prepare_queries(Qt, dev(c.Pi), dev(c.S_mat))
    direct = tq.scores_packed(A, T, dev(ip), dev(sp), f16(c.gamma), dev(c.cb), c.bits, path="fp32").cpu().numpy()
    assert_fp32(direct, c.expected())


# ---------------------------------------------------------------------------
# degenerate inputs, on every scoring path
# ---------------------------------------------------------------------------

DEGENERATE_PATHS = ["unpacked_fp32", "unpacked_bf16_mma", "packed_fused", "packed_stream_k"]


@pytest.mark.parametrize("path", DEGENERATE_PATHS)
@pytest.mark.parametrize("case", ["zero_queries", "zero_gamma", "constant_codes"])
def test_degenerate_inputs(tq, path, case):
    """Zero queries score exactly 0; zero gamma leaves only the codebook term; one code and
    one sign everywhere make every key the same vector.  S is ragged (300 keys)."""
    D, S, bits = 128, 300, 2
    B = {"unpacked_fp32": 3, "unpacked_bf16_mma": 16, "packed_fused": 1, "packed_stream_k": 4}[path]
    rng = np.random.default_rng(1234 + DEGENERATE_PATHS.index(path))
    from conftest import codebook
    cb = codebook(D, bits)[0].astype(np.float32)
    Pi = oracle.haar_rotation(rng.standard_normal((D, D))).astype(np.float32)
    Sm = rng.standard_normal((D, D)).astype(np.float32)
    Q = rng.standard_normal((B, D)).astype(np.float32)
    idx = rng.integers(0, 1 << bits, (S, D)).astype(np.uint8)
    sg = rng.choice(np.array([-1, 1], np.int8), (S, D))
    gm = (0.1 + rng.random(S)).astype(np.float32)
    if case == "zero_queries":
        Q[:] = 0.0
    elif case == "zero_gamma":
        gm[:] = 0.0
    else:
        idx[:] = (1 << bits) - 1
        sg[:] = 1
    packed = path.startswith("packed")
    if packed:
        gm = gm.astype(np.float16)
    want = oracle.scores_from_queries(Q, Pi, Sm, idx, sg, gm, cb)
    if path == "unpacked_fp32" or path == "unpacked_bf16_mma":
        got = tq.solve(dev(Q), dev(idx), dev(sg), dev(gm), dev(Pi), dev(Sm), dev(cb),
                       path="fp32" if path == "unpacked_fp32" else "bf16_mma")
    else:
        ip, sp = dev(oracle.pack_indices(idx, bits)), dev(oracle.pack_signs(sg))
        if path == "packed_fused":
            got = tq.solve_packed(dev(Q), ip, sp, dev(gm), dev(Pi), dev(Sm), dev(cb), bits, path="fp32")
        else:
            A, T = tq.prepare_queries(dev(Q), dev(Pi), dev(Sm))
            got = tq.scores_packed(A, T, ip, sp, dev(gm), dev(cb), bits, path="fp32")
    got = got.cpu().numpy()
    if case == "zero_queries":
        assert (got == 0).all()
    elif path == "unpacked_bf16_mma":
        assert_bf16(got, want, np.linalg.norm(Q.astype(np.float64), axis=1)[:, np.newaxis])
    else:
        assert_fp32(got, want)


# ---------------------------------------------------------------------------
# properties
# ---------------------------------------------------------------------------

def test_deterministic_and_fused_equals_two_step(tq):
    c = workload_case("c0")
    args = (dev(c.idx[0]), dev(c.signs[0]), dev(c.gamma[0]), dev(c.cb))
    A, T = tq.prepare_queries(dev(c.Q[0]), dev(c.Pi[0]), dev(c.S_mat[0]))
    r1 = tq.scores(A, T, *args, path="fp32")
    r2 = tq.scores(A, T, *args, path="fp32")
    fused = tq.solve(dev(c.Q[0]), dev(c.idx[0]), dev(c.signs[0]), dev(c.gamma[0]), dev(c.Pi[0]),
                     dev(c.S_mat[0]), dev(c.cb), path="fp32")
    assert torch.equal(r1, r2) and torch.equal(r1, fused)


def test_device_errors_raise(tq):
    c = Case(1, 1, 2, 64, 128, 2, seed=9, random_codebook=True)
    A, T = tq.prepare_queries(dev(c.Q[0]), dev(c.Pi[0]), dev(c.S_mat[0]))
    big = dev(np.concatenate([c.idx[0].ravel(), np.zeros(16, np.uint8)]))
    with pytest.raises(tq.TQError, match="MISALIGNED"):
        tq.lib()  # loaded
        st = tq.lib().tq_scores(A.data_ptr(), T.data_ptr(), big.data_ptr() + 1, dev(c.signs[0]).data_ptr(),
                                dev(c.gamma[0]).data_ptr(), dev(c.cb).data_ptr(),
                                torch.empty(2, 64, device="cuda").data_ptr(), 1, 2, 64, 128, 4, 1,
                                torch.cuda.current_stream().cuda_stream)
        tq._check("tq_scores", st)
    ws = torch.empty(8, dtype=torch.uint8, device="cuda")
    with pytest.raises(tq.TQError, match="WORKSPACE"):
        tq.solve(dev(c.Q[0]), dev(c.idx[0]), dev(c.signs[0]), dev(c.gamma[0]), dev(c.Pi[0]),
                 dev(c.S_mat[0]), dev(c.cb), workspace=ws)


@pytest.mark.gpu
def test_no_bounded_wait_ran_out(tq):
    """Every bounded wait of the kernels above completed: no fault bit is set (reading clears them)."""
    tq.device_faults()
    test_c2_single_query_decode(tq)
    torch.cuda.synchronize()
    assert tq.device_faults() == 0


def test_bounded_wait_runs_out_and_reports(tq):
    """A wait that nothing completes gives up after its budget: the kernel returns, the
    fault bit reaches the host, reading clears it, and the context still computes."""
    tq.device_faults()
    t0 = time.perf_counter()
    tq.check_wait_expiry()
    torch.cuda.synchronize()
    waited = time.perf_counter() - t0
    assert tq.device_faults() == 16
    assert tq.device_faults() == 0
    assert 0.9 <= waited < 30.0
    test_c2_single_query_decode(tq)
    torch.cuda.synchronize()
    assert tq.device_faults() == 0
