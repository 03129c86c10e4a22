"""The byte accounting behind bench.py's roofline, checked on CPU against the storage
layout and the shapes of the workloads.

Per key (D = 128): the unpacked cache holds a uint8 code and an int8 sign per coordinate
and an fp32 gamma (260 B).  The packed cache holds the bit stream of the codes, one
sign bit per coordinate and an fp16 gamma: 32 + 16 + 2 = 50 B for 2-bit codes and
48 + 16 + 2 = 66 B for 3-bit codes ("TurboQuant: Rotate-then-Quantize KV Caches at
3 Bits", kanthi.in, §8: a 128-dimensional 3-bit key is 48 bytes).  The MSE-only cache
drops the sign plane and stores an fp16 norm; the fused decode reads the key's and the
value's code planes and norms.  A scoring launch reads the cache once and writes every
score once (4 B), plus A and T and the codebook."""
import pytest

import bench
import synth

W = synth.WORKLOADS


@pytest.mark.parametrize("key,per_key", [("c0", 260), ("c1", 260), ("c2", 50), ("c3", 50), ("c4", 66),
                                         ("m1", 50), ("d1", 100), ("d2", 100), ("s1", 40)])
def test_bytes_per_key(key, per_key):
    assert bench.key_bytes(W[key]) == per_key


def test_scoring_launch_bytes_of_the_workloads():
    # cache + scores + A and T + codebook, written out for each workload's shape
    c1 = 32768 * 260 + 4 * 32 * 32768 + 2 * 4 * 32 * 128 + 4 * 4
    c2 = 131072 * 50 + 4 * 131072 + 2 * 4 * 128 + 4 * 4
    c3 = 128 * 32768 * 50 + 4 * 128 * 4 * 32768 + 2 * 4 * 128 * 4 * 128 + 4 * 4
    c4 = 262144 * 66 + 4 * 128 * 262144 + 2 * 4 * 128 * 128 + 4 * 8
    assert bench.score_kernel_bytes(W["c1"]) == c1
    assert bench.score_kernel_bytes(W["c2"]) == c2
    assert bench.score_kernel_bytes(W["c3"]) == c3
    assert bench.score_kernel_bytes(W["c4"]) == c4
    # the totals quoted for the workloads: about 12.75, 7.08, 277 and 151.5 MB
    assert abs(c1 / 1e6 - 12.75) < 0.01 and abs(c2 / 1e6 - 7.08) < 0.01
    assert abs(c3 / 1e6 - 277) < 0.5 and abs(c4 / 1e6 - 151.5) < 0.2
    # c4's output alone is the 134 MB of fp32 scores
    assert 4 * 128 * 262144 == 134217728


def test_mse_and_decode_launch_bytes():
    m1 = 131072 * 50 + 4 * 131072 + 4 * 128 + 4 * 8          # A only, no T
    d1 = 131072 * 100 + 2 * 4 * 128 + 4 * 128 * 128 + 8 * 8  # A and the output, Pi_v, two codebooks
    assert bench.score_kernel_bytes(W["m1"]) == m1
    assert bench.score_kernel_bytes(W["d1"]) == d1
    # the product-key decode: 2-bit codes + signs + gamma (50 B) and 3-bit values + norm
    # (50 B) a key; A, T and the output; Pi_v; a 4- and an 8-entry codebook
    d2 = 131072 * 100 + 3 * 4 * 128 + 4 * 128 * 128 + 4 * 4 + 4 * 8
    assert bench.score_kernel_bytes(W["d2"]) == d2


def test_fused_kernel_also_reads_queries_and_rotations():
    # the single fused kernel of c2 reads the query and Pi, S_mat instead of A and T
    extra = bench.fused_kernel_extra_bytes(W["c2"])
    assert extra == 4 * 128 + 2 * 4 * 128 * 128 - 8 * 128
