"""libtq's host-side setup helpers (codebook, rotation) against the CPU oracle.
Both run on the host, so these tests need no GPU."""
import numpy as np
import pytest

import oracle
import synth
from conftest import codebook
from compressed_kv_cache_gb300 import build as tqbuild
from compressed_kv_cache_gb300 import tq


@pytest.fixture(scope="module", autouse=True)
def _built():
    tqbuild.build()


# The host helper follows the page's procedure: the density sampled on an even grid of
# 400001 points, 300 rounds.  A grid point that lies exactly on a cell edge joins the
# lower cell, so each centroid is biased by about one grid step's share of its cell's
# mass: ~2e-5 relative for the two 1-bit cells at d = 128, growing as cells narrow.
# The oracle is the exact fixed point, so they agree to that resolution.
GRID_BIAS = {1: 1e-4, 2: 3e-4, 3: 1e-3, 4: 4e-3}


@pytest.mark.parametrize("bits", [1, 2, 3, 4])
def test_lloyd_max_matches_oracle(bits):
    want = codebook(128, bits)[0]
    got = tq.lloyd_max_codebook(128, bits)
    np.testing.assert_allclose(got, want, rtol=GRID_BIAS[bits])
    assert np.all(np.diff(got) > 0)


def test_lloyd_max_other_dims():
    for D in (16, 64):
        want = oracle.lloyd_max_sphere(D, 2)[0]
        np.testing.assert_allclose(tq.lloyd_max_codebook(D, 2, 400_001, 80), want, rtol=GRID_BIAS[2])


@pytest.mark.parametrize("D", [2, 5, 128])
def test_haar_rotation_matches_oracle(D):
    G = synth.rotation_seed_matrix(1234, 3, D)
    want = oracle.haar_rotation(G).astype(np.float32)
    got = tq.haar_rotation(G)
    np.testing.assert_allclose(got, want, rtol=0, atol=4e-7)
    assert np.abs(got.astype(np.float64) @ got.T.astype(np.float64) - np.eye(D)).max() < 1e-6


def test_host_helper_argument_errors():
    L = tq.lib()
    out = np.empty(4, np.float32)
    assert L.tq_lloyd_max_codebook(2, 2, 1001, 10, out.ctypes.data) == 1
    assert L.tq_lloyd_max_codebook(128, 9, 1001, 10, out.ctypes.data) == 1
    assert L.tq_haar_rotation(None, 4, out.ctypes.data) == 1
    f = 0x100000
    assert L.tq_compress_keys(f, f, f, f, 4, f, f, f, f, 1, 1, 8, 128, None) == 1   # both gammas
    assert L.tq_compress_keys(f, f, f, f, 4, f, f, f, None, 1, 1, 8, 100, None) == 2  # D % 32 != 0
    assert L.tq_compress_keys(f, f, f, f, 4, f, f, f, None, 1, 1, 8, 288, None) == 1  # D > 256
    assert L.tq_compress_keys_packed(f, f, f, f, 2, f, f, f, 1, 1, 8, 100, None) == 2
    assert L.tq_compress_keys_packed(f, f, f, f, 4, f, f, f, 1, 1, 8, 128, None) == 1  # 4-bit codes
    assert L.tq_compress_keys_packed(f, f, f, f, 2, f, f, None, 1, 1, 8, 128, None) == 1


def test_hadamard_rotation_matches_oracle():
    """tq_hadamard_rotation (host) writes H diag(s) in fp32: the oracle's matrix rounded."""
    import oracle
    rng = np.random.default_rng(71)
    for D in (1, 2, 16, 128, 256):
        s = rng.choice([-1.0, 1.0], size=D).astype(np.float32)
        got = tq.hadamard_rotation(s)
        assert np.array_equal(got, oracle.hadamard_rotation(s).astype(np.float32))
    with pytest.raises(Exception):
        tq.hadamard_rotation(np.ones(12, dtype=np.float32))
