"""Pins for the CPU oracle: each check ties it to something other than itself.

* the worked example printed on the riteshyadav.xyz page (intermediates and output);
* brute-force key reconstruction followed by a plain dot product (pure Python loops);
* closed forms and tables of the Lloyd-Max codebook from the kanthi.in chapter, the
  exact 1-bit centroid from the Gamma function, and the centroid fixed point checked by
  adaptive quadrature of the exact density;
* the defining property of the sign-fixed QR rotation;
* nearest-centroid / sign / norm properties of the compressor on brute force;
* the unbiasedness of the estimator (zededa.com Theorem 2) and the slope table of the
  kanthi.in chapter, section 6;
* hand-worked bytes of the packed format.
"""
import math

import numpy as np
import pytest

import oracle
import synth
from conftest import codebook, golden


# ---------------------------------------------------------------------------
# Scorer
# ---------------------------------------------------------------------------

def test_worked_example_matches_page():
    g = golden("worked_example.json")
    A, T = oracle.prepare_queries(np.array(g["Q"]), np.array(g["Pi"]), np.array(g["S_mat"]))
    np.testing.assert_array_equal(A, np.array(g["A"]))
    np.testing.assert_array_equal(T, np.array(g["T"]))
    gamma = np.array(g["gamma"], dtype=np.float32)
    out = oracle.scores(A, T, np.array(g["K_idx"], dtype=np.uint8), np.array(g["signs"], dtype=np.int8),
                        gamma, np.array(g["codebook"], dtype=np.float32))
    assert np.round(out, g["decimals"]).tolist() == g["scores"]
    # the two parts the page spells out for token 0 and token 1
    no_corr = oracle.scores(A, T, np.array(g["K_idx"], dtype=np.uint8), np.array(g["signs"], dtype=np.int8),
                            np.zeros(2, dtype=np.float32), np.array(g["codebook"], dtype=np.float32))
    np.testing.assert_allclose(no_corr, g["centroid_score"], rtol=0, atol=1e-15)
    corr0 = out[0, 0] - no_corr[0, 0]
    assert round(corr0, 6) == g["correction_token0"]
    assert corr0 / (oracle.kappa(2) * float(gamma[0])) == pytest.approx(g["residual_dot"][0][0], rel=1e-12)


def _bruteforce_scores(Q, Pi, Smat, idx, signs, gamma, cb):
    """Reconstruct every key as Pi^T c[idx] + sqrt(pi/2)/D * gamma * S_mat^T sigma and dot it
    with the query, all in plain Python floats (kanthi.in §3, TurboQuantProd.dequantize)."""
    B, D = len(Q), len(Q[0])
    S = len(idx)
    k = math.sqrt(math.pi / 2.0) / D
    out = [[0.0] * S for _ in range(B)]
    for s in range(S):
        key = [0.0] * D
        for j in range(D):
            acc = 0.0
            for d in range(D):
                acc += float(Pi[d][j]) * float(cb[int(idx[s][d])])
                acc += k * float(gamma[s]) * float(Smat[d][j]) * float(signs[s][d])
            key[j] = acc
        for b in range(B):
            out[b][s] = sum(float(Q[b][j]) * key[j] for j in range(D))
    return np.array(out)


@pytest.mark.parametrize("D,C,B,S", [(2, 4, 1, 3), (4, 2, 2, 5), (8, 8, 3, 16), (5, 16, 2, 7)])
def test_scores_equal_bruteforce_reconstruction(D, C, B, S):
    rng = np.random.default_rng(100 + D * 7 + C)
    Pi = rng.standard_normal((D, D)).astype(np.float32)      # deliberately not orthogonal or symmetric
    Smat = rng.standard_normal((D, D)).astype(np.float32)
    cb = np.sort(rng.standard_normal(C)).astype(np.float32)
    Q = rng.standard_normal((B, D)).astype(np.float32)
    idx = rng.integers(0, C, (S, D)).astype(np.uint8)
    signs = np.where(rng.random((S, D)) < 0.5, 1, -1).astype(np.int8)
    gamma = rng.random(S).astype(np.float32)
    got = oracle.scores_from_queries(Q, Pi, Smat, idx, signs, gamma, cb)
    want = _bruteforce_scores(Q, Pi, Smat, idx, signs, gamma, cb)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)
    # gamma = 0: the rotated-domain identity <Pi q, c[idx]> = <q, Pi^T c[idx]> (kanthi.in §8)
    got0 = oracle.scores_from_queries(Q, Pi, Smat, idx, signs, np.zeros(S, np.float32), cb)
    want0 = _bruteforce_scores(Q, Pi, Smat, idx, signs, np.zeros(S), cb)
    np.testing.assert_allclose(got0, want0, rtol=1e-12, atol=1e-12)
    # sampled one-by-one scorer agrees with the full scorer
    A, T = oracle.prepare_queries(Q, Pi, Smat)
    bs = np.arange(B).repeat(S)
    ss = np.tile(np.arange(S), B)
    one = oracle.scores_sampled(A, T, idx[ss], signs[ss], gamma[ss], cb, bs)
    np.testing.assert_allclose(one, got[bs, ss], rtol=1e-13, atol=1e-13)


def test_exact_binary_case():
    """Pi = S_mat = I, integer codebook, kappa*gamma = 1/8: every term is exact in binary."""
    D = 4
    gamma = np.float32(0.125 / oracle.kappa(D))       # kappa*gamma rounds back to 1/8 within 1e-8
    cb = np.array([-3.0, -1.0, 1.0, 3.0], dtype=np.float32)
    Q = np.array([[1.0, 2.0, -4.0, 8.0]], dtype=np.float32)
    idx = np.array([[0, 1, 2, 3]], dtype=np.uint8)
    sg = np.array([[1, -1, -1, 1]], dtype=np.int8)
    out = oracle.scores_from_queries(Q, np.eye(D), np.eye(D), idx, sg, np.array([gamma]), cb)
    # centroid part: 1*-3 + 2*-1 + -4*1 + 8*3 = 15 ; sign part: 1 - 2 + 4 + 8 = 11 ; 15 + 11/8
    assert out[0, 0] == pytest.approx(15.0 + 11.0 / 8.0, abs=1e-6)


# ---------------------------------------------------------------------------
# Codebook
# ---------------------------------------------------------------------------

def test_codebook_matches_printed_table():
    g = golden("codebook_d128.json")
    d = g["d"]
    for b, vals in g["centroids_times_sqrt_d"].items():
        c, _, _ = codebook(d, int(b))
        np.testing.assert_allclose(c * math.sqrt(d), vals, atol=0.5 * 10 ** -g["centroid_decimals"] + 1e-4)
    for b, dm in g["d_mse"].items():
        _, _, got = codebook(d, int(b))
        assert abs(got - dm) <= 0.5 * 10 ** -g["d_mse_decimals"] + 1e-6, (b, got, dm)
        lo, hi = 4.0 ** -int(b), math.sqrt(3) * math.pi / 2 * 4.0 ** -int(b)
        assert lo < got < hi


def test_codebook_gaussian_closed_forms():
    g = golden("codebook_d128.json")["gaussian_closed_forms"]
    d = 128
    c1, _, _ = codebook(d, 1)
    c2, _, _ = codebook(d, 2)
    tol = g["abs_tolerance_times_sqrt_d"]
    assert abs(c1[1] * math.sqrt(d) - g["1"][0]) < tol
    np.testing.assert_allclose(np.abs(c2[2:]) * math.sqrt(d), g["2"], atol=tol)


def test_one_bit_codebook_exact_closed_form():
    """1 bit: the cell edge is 0 and each centroid is E|x| = Gamma(d/2) / (sqrt(pi) Gamma((d+1)/2));
    the distortion is 1 - d c^2 because E[x^2] = 1/d on the sphere."""
    for d in (4, 16, 64, 128):
        c, edges, dm = codebook(d, 1) if d == 128 else oracle.lloyd_max_sphere(d, 1)
        exact = math.exp(math.lgamma(d / 2) - math.lgamma((d + 1) / 2)) / math.sqrt(math.pi)
        np.testing.assert_allclose([-c[0], c[1]], [exact, exact], rtol=1e-12)
        assert abs(edges[0]) < 1e-15
        assert dm == pytest.approx(1.0 - d * exact * exact, rel=1e-10)


def test_uniform_density_at_d3():
    """d = 3 makes the coordinate uniform on [-1, 1] (Archimedes): the Lloyd-Max codebook is the
    uniform quantizer, centroids -1 + (2k + 1)/C, and the distortion is 3 * (2/C)^2 / 12."""
    for b in (1, 2, 3):
        C = 1 << b
        c, edges, dm = oracle.lloyd_max_sphere(3, b)
        np.testing.assert_allclose(c, -1.0 + (2.0 * np.arange(C) + 1.0) / C, atol=1e-13)
        np.testing.assert_allclose(edges, -1.0 + 2.0 * np.arange(1, C) / C, atol=1e-13)
        assert dm == pytest.approx(3.0 * (2.0 / C) ** 2 / 12.0, rel=1e-12)


def test_codebook_is_a_lloyd_fixed_point_under_quadrature():
    """Each centroid is the conditional mean of its cell under the exact density and the
    distortion is the integral of the squared error, both checked with adaptive quadrature
    (scipy.integrate.quad) instead of the oracle's incomplete-beta moments."""
    integrate = pytest.importorskip("scipy.integrate")
    for d in (16, 128):
        for b in (2, 3, 4):
            c, edges, dm = codebook(d, b) if d == 128 else oracle.lloyd_max_sphere(d, b)
            f = lambda x: (1.0 - x * x) ** ((d - 3) / 2.0)
            z = integrate.quad(f, -1.0, 1.0, epsabs=0, epsrel=1e-13, limit=200)[0]
            lims = [-1.0] + list(edges) + [1.0]
            sq = 0.0
            for k in range(len(c)):
                a, e = lims[k], lims[k + 1]
                mass = integrate.quad(f, a, e, epsabs=0, epsrel=1e-13, limit=200)[0]
                mom = integrate.quad(lambda x: x * f(x), a, e, epsabs=0, epsrel=1e-13, limit=200)[0]
                sq += integrate.quad(lambda x: (x - c[k]) ** 2 * f(x), a, e, epsabs=0, epsrel=1e-13,
                                     limit=200)[0]
                # converged to the fixed point; a wrong density exponent moves centroids ~1e-2
                assert c[k] == pytest.approx(mom / mass, rel=1e-9)
            assert dm == pytest.approx(d * sq / z, rel=1e-8)
            # symmetry of a symmetric density: c_k = -c_{C-1-k}
            np.testing.assert_allclose(c, -c[::-1], atol=1e-13)


# ---------------------------------------------------------------------------
# Rotation
# ---------------------------------------------------------------------------

def test_haar_rotation_is_sign_fixed_qr_factor():
    for D in (2, 7, 128):
        G = synth.rotation_seed_matrix(5, 0, D)
        Pi = oracle.haar_rotation(G)
        assert np.abs(Pi @ Pi.T - np.eye(D)).max() < 1e-12
        R = Pi.T @ G                       # G = Pi R with R upper triangular, positive diagonal
        assert np.abs(np.tril(R, -1)).max() < 1e-11 * max(1.0, np.abs(R).max())
        assert (np.diag(R) > 0).all()


def test_haar_rotation_second_moment():
    """Entries of a Haar matrix have E[Pi_ij^2] = 1/D."""
    D = 16
    acc = np.zeros((D, D))
    n = 400
    for seed in range(n):
        acc += oracle.haar_rotation(np.random.default_rng(seed).standard_normal((D, D))) ** 2
    assert np.abs(acc / n - 1.0 / D).max() < 6 * math.sqrt(2.0 / n) / D


# ---------------------------------------------------------------------------
# Compressor
# ---------------------------------------------------------------------------

def test_compressor_bruteforce_properties():
    D, S = 16, 64
    rng = np.random.default_rng(3)
    keys = rng.standard_normal((S, D))
    keys /= np.linalg.norm(keys, axis=1, keepdims=True)
    Pi = oracle.haar_rotation(rng.standard_normal((D, D))).astype(np.float32)
    Smat = rng.standard_normal((D, D)).astype(np.float32)
    cb = (oracle.lloyd_max_sphere(D, 2)[0]).astype(np.float32)
    idx, sg, gamma = oracle.compress_prod(keys, Pi, Smat, cb, "f32")
    P64, S64, c64 = Pi.astype(float), Smat.astype(float), cb.astype(float)
    for s in range(S):
        r = keys[s].copy()
        for d in range(D):
            y = sum(P64[d][j] * keys[s][j] for j in range(D))
            dist = [abs(y - c64[k]) for k in range(len(cb))]
            assert idx[s][d] == min(range(len(cb)), key=lambda k: (dist[k], k))
            for j in range(D):
                r[j] -= P64[d][j] * c64[idx[s][d]]
        for d in range(D):
            z = sum(S64[d][j] * r[j] for j in range(D))
            assert sg[s][d] == (1 if z >= 0 else -1)
        assert float(gamma[s]) == pytest.approx(math.sqrt(sum(v * v for v in r)), rel=1e-7)


def test_compressor_ties_and_zero_sign():
    """A coordinate on a cell edge takes the lower index; sign(0) is +1."""
    D = 4
    cb = np.array([-3.0, -1.0, 1.0, 3.0], dtype=np.float32) / 8   # edges -0.25, 0, 0.25
    key = np.array([[0.0, 0.25, -0.25, math.sqrt(1 - 2 * 0.0625)]])
    Smat = np.zeros((D, D), dtype=np.float32)
    Smat[1, 0] = 1.0
    idx, sg, gamma = oracle.compress_prod(key, np.eye(D, dtype=np.float32), Smat, cb, "f16")
    assert idx[0].tolist() == [1, 2, 0, 3]
    r0 = key[0, 0] - cb[1]
    assert sg[0].tolist() == [1, 1 if r0 >= 0 else -1, 1, 1]
    assert gamma.dtype == np.float16


def _prod_estimates(mse_bits, n, seed, D=128):
    """The kanthi.in §6 Part 1 protocol: unit keys, correlated unit queries, estimate <q, k>."""
    rng = np.random.default_rng(seed)
    k = rng.standard_normal((n, D))
    k /= np.linalg.norm(k, axis=1, keepdims=True)
    q = k + 0.6 * rng.standard_normal((n, D)) / math.sqrt(D)
    q /= np.linalg.norm(q, axis=1, keepdims=True)
    Pi = oracle.haar_rotation(rng.standard_normal((D, D))).astype(np.float32)
    Smat = rng.standard_normal((D, D)).astype(np.float32)
    cb = codebook(D, mse_bits)[0].astype(np.float32)
    idx, sg, gamma = oracle.compress_prod(k, Pi, Smat, cb, "f32")
    A, T = oracle.prepare_queries(q, Pi, Smat)
    rows = np.arange(n)
    est = oracle.scores_sampled(A, T, idx, sg, gamma, cb, rows)
    return np.sum(q * k, axis=1), est


def test_slope_table_of_mse_plus_qjl():
    g = golden("prod_slope.json")
    for name, row in g["rows"].items():
        true, est = _prod_estimates(row["mse_bits"], 512, seed=11 + row["mse_bits"])
        slope = float(est @ true / (true @ true))
        resid = est - slope * true
        se = float(np.std(resid) / math.sqrt(true @ true))
        assert abs(slope - 1.0) < 5 * se + 1e-3, (name, slope, se)
        assert abs(slope - row["slope"]) < 5 * se + 2e-3, (name, slope)
        assert np.std(resid) == pytest.approx(row["resid_std"], rel=0.25), name
        # zededa.com Theorem 3: no inner-product quantizer beats 1/(d 4^b) for unit queries
        b_total = row["mse_bits"] + 1
        assert np.mean((est - true) ** 2) > 1.0 / (128 * 4 ** b_total)


def test_estimator_is_unbiased_over_rotations():
    """zededa.com Theorem 2: E[<y, x~>] = <y, x> over the random rotation and projection.
    Without the QJL term the estimate is visibly biased, so the test can fail."""
    D, n_keys, reps = 128, 8, 96
    rng = np.random.default_rng(21)
    k = rng.standard_normal((n_keys, D))
    k /= np.linalg.norm(k, axis=1, keepdims=True)
    q = k + 0.6 * rng.standard_normal((n_keys, D)) / math.sqrt(D)
    true = np.sum(q * k, axis=1)
    cb = codebook(D, 2)[0].astype(np.float32)
    err, err_mse_only = [], []
    for rep in range(reps):
        r2 = np.random.default_rng(1000 + rep)
        Pi = oracle.haar_rotation(r2.standard_normal((D, D))).astype(np.float32)
        Smat = r2.standard_normal((D, D)).astype(np.float32)
        idx, sg, gamma = oracle.compress_prod(k, Pi, Smat, cb, "f32")
        A, T = oracle.prepare_queries(q, Pi, Smat)
        rows = np.arange(n_keys)
        err.append(oracle.scores_sampled(A, T, idx, sg, gamma, cb, rows) - true)
        err_mse_only.append(oracle.scores_sampled(A, T, idx, sg, np.zeros(n_keys), cb, rows) - true)
    err = np.array(err)
    mean, se = err.mean(), err.std() / math.sqrt(err.size)
    assert abs(mean) < 4 * se, (mean, se)
    e2 = np.array(err_mse_only)
    assert abs(e2.mean()) > 4 * e2.std() / math.sqrt(e2.size)


# ---------------------------------------------------------------------------
# Packer
# ---------------------------------------------------------------------------

def test_pack_hand_worked_bytes():
    for case in golden("pack_bytes.json")["cases"]:
        if case["kind"] == "indices":
            idx = np.array([case["idx"]], dtype=np.uint8)
            plane = oracle.pack_indices(idx, case["bits"])
            assert plane[0].tolist() == case["bytes"]
            np.testing.assert_array_equal(oracle.unpack_indices(plane, case["bits"], case["D"]), idx)
        else:
            sg = -np.ones((1, case["D"]), dtype=np.int8)
            sg[0, case["plus_at"]] = 1
            plane = oracle.pack_signs(sg)
            assert plane[0].tolist() == case["bytes"]
            np.testing.assert_array_equal(oracle.unpack_signs(plane, case["D"]), sg)


@pytest.mark.parametrize("bits", [1, 2, 3])
@pytest.mark.parametrize("D", [32, 64, 96, 128, 256])
def test_pack_round_trip(bits, D):
    rng = np.random.default_rng(bits * 1000 + D)
    idx = rng.integers(0, 1 << bits, (37, D)).astype(np.uint8)
    plane = oracle.pack_indices(idx, bits)
    assert plane.shape == (37, D * bits // 8)
    np.testing.assert_array_equal(oracle.unpack_indices(plane, bits, D), idx)
    sg = np.where(rng.random((37, D)) < 0.5, 1, -1).astype(np.int8)
    sp = oracle.pack_signs(sg)
    assert sp.shape == (37, D // 8)
    np.testing.assert_array_equal(oracle.unpack_signs(sp, D), sg)


def test_synth_keys_are_unit_and_reproducible():
    a = synth.unit_keys(7, 0, 4090, 20, 128)
    b = synth.unit_keys(7, 0, 4000, 200, 128)[90:110]
    np.testing.assert_array_equal(a, b)
    np.testing.assert_allclose(np.linalg.norm(a, axis=1), 1.0, atol=1e-14)
    q, raw = synth.queries(7, 0, 4, 128, "bf16")
    assert raw.dtype == np.uint16
    assert np.abs(q - synth.queries(7, 0, 4, 128, "f32")[0]).max() <= 2.0 ** -8 * np.abs(q).max()


# ---------------------------------------------------------------------------
# MSE-only variant (kanthi.in §3 TurboQuantMSE, §6 Part 1, §8 "Kernel view")
# ---------------------------------------------------------------------------

def _mse_pair_estimates(mse_bits, n, seed, D=128, norm_correction=False):
    """kanthi.in §6 Part 1 protocol for the MSE-only quantizer: est_i = <q_i, k^_i>."""
    rng = np.random.default_rng(seed)
    k = rng.standard_normal((n, D))
    k /= np.linalg.norm(k, axis=1, keepdims=True)
    q = k + 0.6 * rng.standard_normal((n, D)) / math.sqrt(D)
    q /= np.linalg.norm(q, axis=1, keepdims=True)
    Pi = oracle.haar_rotation(rng.standard_normal((D, D))).astype(np.float32)
    cb = codebook(D, mse_bits)[0].astype(np.float32)
    idx, nrm = oracle.compress_mse(k, Pi, cb)
    A = q @ Pi.astype(np.float64).T
    est = np.concatenate([np.diag(oracle.scores_mse(A[i:i + 256], idx[i:i + 256], nrm[i:i + 256], cb,
                                                    norm_correction)) for i in range(0, n, 256)])
    return np.sum(q * k, axis=1), est


def test_mse_score_equals_unrotated_reconstruction():
    """kanthi.in §8: scoring in the rotated domain equals the dot product with the
    reconstructed key n * Pi^T c_idx (the dequantize route of §3), built here coordinate
    by coordinate; keys are not unit length, so the stored norm matters."""
    D, S, B = 8, 6, 3
    rng = np.random.default_rng(31)
    keys = rng.standard_normal((S, D)) * rng.uniform(0.5, 3.0, (S, 1))
    Q = rng.standard_normal((B, D))
    Pi = oracle.haar_rotation(rng.standard_normal((D, D))).astype(np.float32)
    cb = codebook(D, 2)[0].astype(np.float32)
    idx, nrm = oracle.compress_mse(keys, Pi, cb)
    A = Q @ Pi.astype(np.float64).T
    for corr in (False, True):
        got = oracle.scores_mse(A, idx, nrm, cb, norm_correction=corr)
        for s in range(S):
            cw = [float(cb[idx[s, d]]) for d in range(D)]
            scale = math.sqrt(sum(x * x for x in cw)) if corr else 1.0
            khat = [float(nrm[s]) * sum(float(Pi[d, j]) * cw[d] for d in range(D)) / scale for j in range(D)]
            for b in range(B):
                want = sum(Q[b, j] * khat[j] for j in range(D))
                assert got[b, s] == pytest.approx(want, rel=1e-12, abs=1e-12)
    # the stored norm is the key's length rounded to float16, the codes the nearest cells
    assert np.allclose(nrm.astype(np.float64), np.linalg.norm(keys, axis=1), rtol=1e-3)
    y = (keys / np.linalg.norm(keys, axis=1, keepdims=True)) @ Pi.astype(np.float64).T
    dist = np.abs(y[:, :, None] - cb.astype(np.float64)[None, None, :])
    assert np.all(dist[np.arange(S)[:, None], np.arange(D)[None, :], idx] <= dist.min(axis=2) + 1e-15)


def test_mse_norm_correction_puts_the_codeword_on_the_sphere():
    """With norm correction the reconstructed key has exactly the stored length: scored
    against its own unit direction it returns the stored norm (kanthi.in §3 dequantize)."""
    D = 16
    rng = np.random.default_rng(32)
    keys = rng.standard_normal((5, D)) * 2.5
    Pi = oracle.haar_rotation(rng.standard_normal((D, D))).astype(np.float32)
    cb = codebook(D, 3)[0].astype(np.float32)
    idx, nrm = oracle.compress_mse(keys, Pi, cb)
    c = cb.astype(np.float64)[idx.astype(np.int64)]
    u = c / np.linalg.norm(c, axis=1, keepdims=True)          # unit codewords, rotated domain
    got = oracle.scores_mse(u, idx, nrm, cb, norm_correction=True)
    assert np.allclose(np.diag(got), nrm.astype(np.float64), rtol=1e-12)
    plain = oracle.scores_mse(u, idx, nrm, cb, norm_correction=False)
    assert np.allclose(np.diag(plain), nrm.astype(np.float64) * np.linalg.norm(c, axis=1), rtol=1e-12)


def test_mse_slope_table():
    """kanthi.in §6 Part 1 table: the MSE quantizer shrinks inner products by the printed
    slopes at 2, 3 and 4 bits."""
    g = golden("mse_slope.json")
    for name, row in g["rows"].items():
        true, est = _mse_pair_estimates(row["mse_bits"], 4096, seed=41 + row["mse_bits"])
        slope = float(est @ true / (true @ true))
        resid = est - slope * true
        se = float(np.std(resid) / math.sqrt(true @ true))
        assert abs(slope - row["slope"]) < 5 * se + 5e-4 + 2e-3, (name, slope, se)
        assert np.std(resid) == pytest.approx(row["resid_std"], rel=0.25), name


def test_mse_one_bit_shrinkage_closed_form():
    """At 1 bit the codebook is +-E|y_1| for y uniform on the sphere, so the shrinkage is
    d E|y_1|^2 = d Gamma(d/2)^2 / (pi Gamma((d+1)/2)^2), which tends to 2/pi (kanthi.in §6)."""
    D = 128
    c1 = math.exp(math.lgamma(D / 2) - math.lgamma((D + 1) / 2)) / math.sqrt(math.pi)
    shrink = D * c1 * c1
    assert shrink == pytest.approx(golden("mse_slope.json")["one_bit_shrinkage"], abs=4e-3)
    assert float(codebook(D, 1)[0][1]) == pytest.approx(c1, rel=1e-4)
    true, est = _mse_pair_estimates(1, 4096, seed=40)
    slope = float(est @ true / (true @ true))
    se = float(np.std(est - slope * true) / math.sqrt(true @ true))
    assert abs(slope - shrink) < 5 * se + 2e-3, (slope, shrink, se)


# ---------------------------------------------------------------------------
# randomized Hadamard rotation (kanthi.in §2-§3 RandomizedHadamard)
# ---------------------------------------------------------------------------

def test_fwht_matches_the_sylvester_matrix():
    """The butterfly transform equals the Sylvester-order Hadamard matrix of the library
    routine, scaled to be orthonormal, for every power-of-two length up to 256."""
    scipy_linalg = pytest.importorskip("scipy.linalg")
    rng = np.random.default_rng(51)
    for n in (1, 2, 4, 8, 32, 128, 256):
        x = rng.standard_normal((3, n))
        want = x @ (scipy_linalg.hadamard(n).astype(np.float64) / math.sqrt(n)).T
        assert np.allclose(oracle.fwht(x), want, rtol=1e-12, atol=1e-12)
    assert np.allclose(oracle.fwht(np.array([1.0, 0.0])), [1 / math.sqrt(2), 1 / math.sqrt(2)])
    with pytest.raises(ValueError):
        oracle.fwht(np.ones(6))


def test_randomized_hadamard_is_orthogonal_and_inverts_as_printed():
    """y = H D x is exactly orthogonal, and x = D H y recovers x (the page's inverse)."""
    rng = np.random.default_rng(52)
    for n in (8, 64, 128):
        s = rng.choice([-1.0, 1.0], size=n)
        Pi = oracle.hadamard_rotation(s)
        assert np.allclose(Pi @ Pi.T, np.eye(n), atol=1e-12)
        x = rng.standard_normal(n)
        y = Pi @ x
        assert np.allclose(y, oracle.fwht(x * s), atol=1e-12)
        assert np.allclose(oracle.fwht(y) * s, x, atol=1e-12)
        # entries are +-1/sqrt(n): every coordinate of y mixes all of x
        assert np.allclose(np.abs(Pi), 1.0 / math.sqrt(n))


# ---------------------------------------------------------------------------
# fused decode over MSE keys and values (kanthi.in §8 "Kernel view")
# ---------------------------------------------------------------------------

def _decode_case(n, D, seed, kbits=3, vbits=3):
    rng = np.random.default_rng(seed)
    K = rng.standard_normal((n, D))
    V = rng.standard_normal((n, D))
    q = rng.standard_normal((2, D))
    Pk = oracle.haar_rotation(rng.standard_normal((D, D))).astype(np.float32)
    Pv = oracle.haar_rotation(rng.standard_normal((D, D))).astype(np.float32)
    kcb = codebook(D, kbits)[0].astype(np.float32)
    vcb = codebook(D, vbits)[0].astype(np.float32)
    ki, kn = oracle.compress_mse(K, Pk, kcb)
    vi, vn = oracle.compress_mse(V, Pv, vcb)
    return q, K, V, Pk, Pv, kcb, vcb, ki, kn, vi, vn


def test_decode_equals_dequantize_everything():
    """The rotated-domain decode equals attention over fully dequantized keys and values
    (kanthi.in §8 prints both routes agreeing to 1e-15): every key and value is rebuilt
    as n * Pi^T c_idx, scored against q / sqrt(d), softmaxed, and the values averaged."""
    D, n = 32, 300
    q, K, V, Pk, Pv, kcb, vcb, ki, kn, vi, vn = _decode_case(n, D, 61)
    A = q @ Pk.astype(np.float64).T
    got = oracle.decode_mse(A, ki, kn, kcb, vi, vn, vcb, Pv, 1.0 / math.sqrt(D))
    Kh = kn.astype(np.float64)[:, None] * (kcb.astype(np.float64)[ki.astype(np.int64)] @ Pk.astype(np.float64))
    Vh = vn.astype(np.float64)[:, None] * (vcb.astype(np.float64)[vi.astype(np.int64)] @ Pv.astype(np.float64))
    for b in range(q.shape[0]):
        logits = [float(np.dot(Kh[i], q[b])) / math.sqrt(D) for i in range(n)]
        m = max(logits)
        w = [math.exp(x - m) for x in logits]
        tot = sum(w)
        want = sum(w[i] / tot * Vh[i] for i in range(n))
        assert np.allclose(got[b], want, rtol=1e-12, atol=1e-12)


def test_decode_special_cases():
    """One key: the output is that value's reconstruction.  A key whose logit exceeds
    every other by a wide margin takes all the weight.  Keys with equal logits weigh their
    values equally: the output is the plain mean of the reconstructed values."""
    D = 16
    q, K, V, Pk, Pv, kcb, vcb, ki, kn, vi, vn = _decode_case(40, D, 62)
    A = q @ Pk.astype(np.float64).T
    Vh = vn.astype(np.float64)[:, None] * (vcb.astype(np.float64)[vi.astype(np.int64)] @ Pv.astype(np.float64))
    one = oracle.decode_mse(A, ki[:1], kn[:1], kcb, vi[:1], vn[:1], vcb, Pv, 0.25)
    assert np.allclose(one, np.broadcast_to(Vh[0], one.shape), rtol=1e-12)
    # key 0's logit for query 0 is s0 = 0.25 * n0 * <A0, c_k0>; a norm of 1e4 with the
    # sign of <A0, c_k0> puts it far above the others (whose norms are about 4)
    dot0 = float(A[0] @ kcb.astype(np.float64)[ki[0].astype(np.int64)])
    big = kn.astype(np.float64).copy()
    big[0] = math.copysign(1e4, dot0)
    out = oracle.decode_mse(A[:1], ki, big, kcb, vi, vn, vcb, Pv, 0.25)
    assert np.allclose(out[0], Vh[0], rtol=1e-9, atol=1e-9)
    same = np.zeros_like(ki)                          # one code row for every key
    ones = np.ones(len(kn), dtype=np.float16)
    o1 = oracle.decode_mse(A, same, ones, kcb, vi, vn, vcb, Pv, 0.25)
    assert np.allclose(o1, np.broadcast_to(Vh.mean(axis=0), o1.shape), rtol=1e-12, atol=1e-12)


def test_nearest_cell_is_a_left_sided_search():
    """The cell rule equals NumPy's left-sided binary search over the sorted midpoints
    (a value on a midpoint takes the lower cell), on random values and on the edges."""
    rng = np.random.default_rng(5)
    edges = np.sort(rng.standard_normal(7))
    vals = np.concatenate([rng.standard_normal(500), edges, [-np.inf, np.inf]])
    assert np.array_equal(oracle.nearest_cell(vals, edges), np.searchsorted(edges, vals, side="left"))


def test_qjl_constant_is_the_half_normal_mean():
    """sqrt(pi/2) = 1 / E|g| for g ~ N(0, 1), and E|g| = sqrt(2) / Gamma(1/2)."""
    assert oracle.SQRT_HALF_PI == pytest.approx(math.gamma(0.5) / math.sqrt(2.0), rel=1e-15)
    assert oracle.kappa(128) == pytest.approx(oracle.SQRT_HALF_PI / 128, rel=1e-15)


def _prod_decode_case(n, D, seed, kbits=3, vbits=3):
    """Unit keys compressed by TurboQuant_prod (b = kbits: (kbits-1)-bit codes + signs),
    values by TurboQuant-MSE; two queries."""
    rng = np.random.default_rng(seed)
    K = rng.standard_normal((n, D))
    K /= np.linalg.norm(K, axis=1, keepdims=True)
    V = rng.standard_normal((n, D))
    q = rng.standard_normal((2, D))
    Pk = oracle.haar_rotation(rng.standard_normal((D, D))).astype(np.float32)
    Sm = rng.standard_normal((D, D)).astype(np.float32)
    Pv = oracle.haar_rotation(rng.standard_normal((D, D))).astype(np.float32)
    kcb = codebook(D, kbits - 1)[0].astype(np.float32)
    vcb = codebook(D, vbits)[0].astype(np.float32)
    ki, ks, kg = oracle.compress_prod(K, Pk, Sm, kcb, "f16")
    vi, vn = oracle.compress_mse(V, Pv, vcb)
    return q, Pk, Sm, Pv, kcb, vcb, ki, ks, kg, vi, vn


def _prod_reconstructions(D, Pk, Sm, Pv, kcb, vcb, ki, ks, kg, vi, vn):
    """Keys and values rebuilt in the original basis, as the page's first version does
    before any matrix product (zededa.com v1: unpack, centroids, rotate back; the QJL part
    sqrt(pi/2)/d * gamma * S^T sigma, kanthi.in §3 TurboQuantProd.dequantize)."""
    P = Pk.astype(np.float64)
    Kh = kcb.astype(np.float64)[ki.astype(np.int64)] @ P
    Kh += (math.sqrt(math.pi / 2) / D) * kg.astype(np.float64)[:, None] * (ks.astype(np.float64) @ Sm.astype(np.float64))
    Vh = vn.astype(np.float64)[:, None] * (vcb.astype(np.float64)[vi.astype(np.int64)] @ Pv.astype(np.float64))
    return Kh, Vh


def test_prod_decode_equals_dequantize_everything():
    """Attention over the product cache equals softmax(scale <q, k_hat>) weights on the
    rebuilt values, with every key rebuilt in the original basis and scored from q itself
    (no A, no T), one pair at a time."""
    for D, n, kb, vb in ((8, 13, 3, 2), (32, 200, 3, 3), (16, 64, 4, 1)):
        q, Pk, Sm, Pv, kcb, vcb, ki, ks, kg, vi, vn = _prod_decode_case(n, D, 71 + D, kb, vb)
        A, T = oracle.prepare_queries(q, Pk, Sm)
        got = oracle.decode_prod(A, T, ki, ks, kg, kcb, vi, vn, vcb, Pv, 1.0 / math.sqrt(D))
        Kh, Vh = _prod_reconstructions(D, Pk, Sm, Pv, kcb, vcb, ki, ks, kg, vi, vn)
        for b in range(q.shape[0]):
            logits = [float(np.dot(Kh[i], q[b])) / math.sqrt(D) for i in range(n)]
            m = max(logits)
            w = [math.exp(x - m) for x in logits]
            tot = sum(w)
            want = sum(w[i] / tot * Vh[i] for i in range(n))
            assert np.allclose(got[b], want, rtol=1e-11, atol=1e-12)


def test_prod_decode_special_cases():
    """One key: the output is that value's reconstruction.  A dominant key (its logit far
    above every other) takes all the weight.  Equal logits (q = 0) weigh the values
    equally: the output is the plain mean of the rebuilt values."""
    D = 16
    q, Pk, Sm, Pv, kcb, vcb, ki, ks, kg, vi, vn = _prod_decode_case(40, D, 81)
    A, T = oracle.prepare_queries(q, Pk, Sm)
    _, Vh = _prod_reconstructions(D, Pk, Sm, Pv, kcb, vcb, ki, ks, kg, vi, vn)
    one = oracle.decode_prod(A, T, ki[:1], ks[:1], kg[:1], kcb, vi[:1], vn[:1], vcb, Pv, 0.25)
    assert np.allclose(one, np.broadcast_to(Vh[0], one.shape), rtol=1e-12)
    # the query along key 7's reconstruction, scaled up: its logit exceeds the rest by
    # far more than log(n / eps)
    Kh, _ = _prod_reconstructions(D, Pk, Sm, Pv, kcb, vcb, ki, ks, kg, vi, vn)
    qd = 400.0 * Kh[7:8] / np.linalg.norm(Kh[7])
    Ad, Td = oracle.prepare_queries(qd, Pk, Sm)
    logits = (Kh @ qd[0])
    assert logits[7] - np.delete(logits, 7).max() > 50.0
    out = oracle.decode_prod(Ad, Td, ki, ks, kg, kcb, vi, vn, vcb, Pv, 1.0)
    assert np.allclose(out[0], Vh[7], rtol=1e-12, atol=1e-12)
    z = np.zeros_like(A)
    o0 = oracle.decode_prod(z, z, ki, ks, kg, kcb, vi, vn, vcb, Pv, 0.25)
    assert np.allclose(o0, np.broadcast_to(Vh.mean(axis=0), o0.shape), rtol=1e-12, atol=1e-12)


def _split_case(S, D, n_out, seed, bo=3, br=2):
    rng = np.random.default_rng(seed)
    K = synth.unit_keys(seed, 0, 0, S, D) * rng.uniform(0.5, 3.0, (S, 1))
    q = rng.standard_normal((3, D))
    ch = oracle.outlier_channels(K, n_out)
    Po = oracle.haar_rotation(rng.standard_normal((n_out, n_out))).astype(np.float32)
    Pr = oracle.haar_rotation(rng.standard_normal((D - n_out, D - n_out))).astype(np.float32)
    co = codebook(n_out, bo)[0].astype(np.float32)
    cr = codebook(D - n_out, br)[0].astype(np.float32)
    return K, q, ch, Po, Pr, co, cr


def test_split_scores_equal_reconstruction():
    """The split score equals <q, k_hat> with k_hat rebuilt in the original basis: the
    outlier channels from norm_out Pi_out^T c_out(idx_out), the others from
    norm_reg Pi_reg^T c_reg(idx_reg), one pair at a time."""
    for S, D, n_out in ((40, 128, 32), (25, 64, 16)):
        K, q, ch, Po, Pr, co, cr = _split_case(S, D, n_out, 301 + D)
        io, no, ir, nr = oracle.compress_split(K, ch, Po, Pr, co, cr)
        Ao, Ar = oracle.prepare_queries_split(q, ch, Po, Pr)
        got = oracle.scores_split(Ao, Ar, io, no, co, ir, nr, cr)
        reg = np.array([c for c in range(D) if c not in set(ch.tolist())])
        for s in range(S):
            kh = np.zeros(D)
            kh[ch] = float(no[s]) * (co.astype(np.float64)[io[s].astype(np.int64)] @ Po.astype(np.float64))
            kh[reg] = float(nr[s]) * (cr.astype(np.float64)[ir[s].astype(np.int64)] @ Pr.astype(np.float64))
            for b in range(q.shape[0]):
                assert got[b, s] == pytest.approx(float(np.dot(q[b], kh)), rel=1e-12, abs=1e-12)


def test_split_storage_of_the_printed_split():
    """The split kanthi.in §7 prints: 32 channels at 3 bits and 96 at 2.  Its codes take
    (32*3 + 96*2)/128 = 2.25 bits a coordinate (the page writes 2.5 for that expression);
    with the two fp16 norms a key of D = 128 takes 12 + 24 + 4 = 40 bytes, 2.5 bits a
    coordinate in all."""
    assert (32 * 3 + 96 * 2) / 128 == 2.25
    K, q, ch, Po, Pr, co, cr = _split_case(8, 128, 32, 311)
    io, no, ir, nr = oracle.compress_split(K, ch, Po, Pr, co, cr)
    code_bytes = oracle.pack_indices(io, 3).shape[1] + oracle.pack_indices(ir, 2).shape[1]
    assert code_bytes == 36
    assert code_bytes + no.itemsize + nr.itemsize == 40 == 2.5 * 128 / 8


def test_outlier_channels_pick_the_hot_channels():
    """Keys with channels {3, 17, 64, 101} scaled x15 before normalisation: those four are
    among the 32 picked.  With channel magnitudes strictly ordered by construction, the
    pick is exactly the top of that order; equal means take the lower index."""
    K = synth.unit_keys(1234, 0, 0, 2000, 128)
    ch = oracle.outlier_channels(K, 32)
    assert len(ch) == 32 and np.all(np.diff(ch) > 0)
    assert {3, 17, 64, 101} <= set(ch.tolist())
    scale = np.arange(1, 9, dtype=np.float64)[::-1]             # channel 0 hottest
    Ks = np.ones((5, 8)) * scale
    assert oracle.outlier_channels(Ks, 3).tolist() == [0, 1, 2]
    assert oracle.outlier_channels(np.ones((4, 6)), 2).tolist() == [0, 1]


def test_split_distortion_sits_between_the_uniform_widths():
    """On keys with outlier channels, the reconstruction error of the 2.5-bit split lies
    between uniform 2-bit and uniform 3-bit TurboQuant-MSE (kanthi.in §7: the extra bits
    of the outlier instance are not worthless)."""
    rng = np.random.default_rng(321)
    S, D = 3000, 128
    K = synth.unit_keys(321, 0, 0, S, D)
    def err_uniform(bits):
        P = oracle.haar_rotation(rng.standard_normal((D, D))).astype(np.float32)
        cb = codebook(D, bits)[0].astype(np.float32)
        idx, n = oracle.compress_mse(K, P, cb)
        kh = n.astype(np.float64)[:, None] * (cb.astype(np.float64)[idx.astype(np.int64)] @ P.astype(np.float64))
        return float(np.mean(np.sum((K - kh) ** 2, axis=1)))
    _, _, ch, Po, Pr, co, cr = _split_case(S, D, 32, 322)
    ch = oracle.outlier_channels(K, 32)
    io, no, ir, nr = oracle.compress_split(K, ch, Po, Pr, co, cr)
    reg = np.array([c for c in range(D) if c not in set(ch.tolist())])
    kh = np.zeros_like(K)
    kh[:, ch] = no.astype(np.float64)[:, None] * (co.astype(np.float64)[io.astype(np.int64)] @ Po.astype(np.float64))
    kh[:, reg] = nr.astype(np.float64)[:, None] * (cr.astype(np.float64)[ir.astype(np.int64)] @ Pr.astype(np.float64))
    e_split = float(np.mean(np.sum((K - kh) ** 2, axis=1)))
    assert err_uniform(3) < e_split < err_uniform(2)
