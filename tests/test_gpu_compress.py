"""GPU compressor (tq_compress_keys) against the CPU oracle's compressor.

The kernel decides codes and signs in fp32, the oracle in float64, so a coordinate
that sits within rounding distance of a cell edge (or an S_mat r entry within rounding
distance of 0) may legitimately go either way.  The test compares what is unique --
every decision away from such ties, gamma where all of a key's decisions agree -- and
checks that every differing decision is such a tie."""
import numpy as np
import pytest

import oracle
import synth
from cases import codebook_for, rotation

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tq():
    from compressed_kv_cache_gb300 import build as tqbuild
    tqbuild.build()
    from compressed_kv_cache_gb300 import tq as mod
    return mod


CASES = [(1, 1, 4096, 128, 2, "f32"), (4, 2, 777, 128, 3, "f16"), (2, 2, 300, 64, 1, "f32"),
         (1, 1, 129, 32, 2, "f16"), (2, 1, 333, 256, 2, "f16"), (1, 1, 100, 160, 3, "f32"),
         (3, 3, 65, 96, 2, "f16")]


def _inputs(P, H, S, D, bits):
    seed = 900 + D + bits
    cb = codebook_for(D, bits)
    Pi = np.stack([rotation(seed, h, D) for h in range(H)])
    Sm = np.stack([synth.s_matrix(seed, h, D) for h in range(H)])
    keys = np.stack([synth.unit_keys(seed, p, 0, S, D) for p in range(P)]).astype(np.float32)
    return cb, Pi, Sm, keys


@pytest.mark.parametrize("P,H,S,D,bits,gdt", CASES)
def test_compress_matches_oracle(tq, P, H, S, D, bits, gdt):
    cb, Pi, Sm, keys = _inputs(P, H, S, D, bits)
    gd = torch.float32 if gdt == "f32" else torch.float16
    gi, gs, gg = tq.compress_keys(torch.from_numpy(keys).cuda(), torch.from_numpy(Pi).cuda(),
                                  torch.from_numpy(Sm).cuda(), torch.from_numpy(cb).cuda(), gd)
    gi, gs, gg = gi.cpu().numpy(), gs.cpu().numpy(), gg.cpu().numpy().astype(np.float64)
    _check_against_oracle(P, H, S, D, gdt, cb, Pi, Sm, keys, gi, gs, gg)


@pytest.mark.parametrize("P,H,S,D,bits,gdt", [c for c in CASES if c[5] == "f16"] + [(1, 1, 4096, 128, 2, "f16"),
                                                                                     (2, 1, 999, 128, 1, "f16")])
def test_compress_packed_matches_oracle(tq, P, H, S, D, bits, gdt):
    """The one-pass compressor writes the packed cache: unpacked with the oracle's
    unpackers, its codes, signs and fp16 gamma pass the same tie-aware comparison."""
    cb, Pi, Sm, keys = _inputs(P, H, S, D, bits)
    ip, sp, g = tq.compress_keys_packed(torch.from_numpy(keys).cuda(), torch.from_numpy(Pi).cuda(),
                                        torch.from_numpy(Sm).cuda(), torch.from_numpy(cb).cuda(), bits)
    ip, sp = ip.cpu().numpy(), sp.cpu().numpy()
    gi = np.stack([oracle.unpack_indices(ip[p], bits, D) for p in range(P)])
    gs = np.stack([oracle.unpack_signs(sp[p], D) for p in range(P)])
    _check_against_oracle(P, H, S, D, "f16", cb, Pi, Sm, keys, gi, gs, g.cpu().numpy().astype(np.float64))


def _check_against_oracle(P, H, S, D, gdt, cb, Pi, Sm, keys, gi, gs, gg):
    edges = 0.5 * (cb[1:].astype(np.float64) + cb[:-1])
    n_tie_idx = n_tie_sign = 0
    for p in range(P):
        h = p % H
        k = keys[p].astype(np.float64)          # the kernel is given the fp32-rounded keys
        idx, sg, gamma = oracle.compress_prod(k, Pi[h], Sm[h], cb, gdt)
        y = k @ Pi[h].astype(np.float64).T
        near_edge = np.min(np.abs(y[..., None] - edges), axis=-1) < 2e-6
        diff = gi[p] != idx
        assert not (diff & ~near_edge).any(), "code differs away from a cell edge"
        n_tie_idx += int(diff.sum())
        same_rows = ~diff.any(axis=1)
        r = k - cb[idx].astype(np.float64) @ Pi[h].astype(np.float64)
        z = r @ Sm[h].astype(np.float64).T
        near_zero = np.abs(z) < 2e-5
        sdiff = (gs[p] != sg) & same_rows[:, None]
        assert not (sdiff & ~near_zero).any(), "sign differs away from zero"
        n_tie_sign += int(sdiff.sum())
        g_or = gamma.astype(np.float64)[same_rows]
        tol = 2e-6 * g_or if gdt == "f32" else np.maximum(2.0 ** -10 * g_or, 1e-7)
        assert (np.abs(gg[p][same_rows] - g_or) <= tol).all()
    assert set(np.unique(gs)) <= {-1, 1}
    assert n_tie_idx <= 1e-3 * P * S * D and n_tie_sign <= 1e-3 * P * S * D


def test_compressed_cache_scores_like_oracle_cache(tq):
    """Scores from the GPU-compressed cache equal the oracle's scores of that same cache."""
    D, S, B, bits = 128, 2048, 4, 2
    seed = 77
    cb = codebook_for(D, bits)
    Pi, Sm = rotation(seed, 0, D), synth.s_matrix(seed, 0, D)
    keys = synth.unit_keys(seed, 0, 0, S, D).astype(np.float32)
    gi, gs, gg = tq.compress_keys(torch.from_numpy(keys).cuda(), torch.from_numpy(Pi).cuda(),
                                  torch.from_numpy(Sm).cuda(), torch.from_numpy(cb).cuda(), torch.float16)
    Q = synth.queries(seed, 0, B, D)[0]
    ip, sp = tq.pack_indices(gi, bits), tq.pack_signs(gs)
    out = tq.solve_packed(torch.from_numpy(Q).cuda(), ip, sp, gg, torch.from_numpy(Pi).cuda(),
                          torch.from_numpy(Sm).cuda(), torch.from_numpy(cb).cuda(), bits, path="fp32")
    want = oracle.scores_from_queries(Q, Pi, Sm, gi.cpu().numpy(), gs.cpu().numpy(),
                                      gg.cpu().numpy(), cb)
    err = np.abs(out.cpu().numpy().astype(np.float64) - want)
    assert (err <= 1e-5 * (1 + np.abs(want))).all()
