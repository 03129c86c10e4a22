"""Host-only checks of the C ABI: the library loads without a GPU, exports every
function include/tq.h declares, and rejects bad arguments before any CUDA call."""
import ctypes

import pytest

from compressed_kv_cache_gb300 import build as tqbuild
from compressed_kv_cache_gb300 import tq


@pytest.fixture(scope="module")
def L():
    tqbuild.build()
    return tq.lib()


def test_exports_every_declared_symbol(L):
    names = tq.declared_functions()
    assert len(names) >= 12
    missing = [n for n in names if not hasattr(L, n)]
    assert not missing, missing


def test_status_strings(L):
    for code, name in tq.STATUS_NAMES.items():
        assert tq.status_string(code).startswith(name)
    assert tq.status_string(99) == "unknown tq_status"


def test_workspace_bytes(L):
    assert tq.workspace_bytes(1, 32, 128) == 2 * 32 * 128 * 4 + 32 * 512     # A, T, bf16 query operand
    assert tq.workspace_bytes(1, 1, 2) == 2 * 256          # each half rounded up to 256 bytes
    assert tq.workspace_bytes(1, 8, 128) == 2 * 8 * 128 * 4                 # no tensor-core copy below B = 16
    assert tq.workspace_bytes(0, 1, 1) == 0


def test_auto_path_small_batch_is_fp32(L):
    for B in (1, 4, 8):
        assert tq.auto_path(B, 128) == "fp32"
    assert tq.auto_path(64, 96) == "fp32"                   # tensor-core path needs D == 128


FAKE = 0x100000       # 16-byte aligned, never dereferenced: every call below fails validation first
ODD = 0x100004


def _scores(L, A=FAKE, K=FAKE, S=10, D=128, C=4, P=1, B=1, path=1):
    return L.tq_scores(A, FAKE, K, FAKE, FAKE, FAKE, FAKE, P, B, S, D, C, path, None)


def test_scores_argument_errors(L):
    assert _scores(L, A=None) == 1
    assert _scores(L, A=ODD) == 3
    assert _scores(L, S=0) == 1
    assert _scores(L, D=257) == 1
    assert _scores(L, C=0) == 1 and _scores(L, C=257) == 1
    assert _scores(L, P=70000) == 1
    assert _scores(L, path=7) == 1
    assert _scores(L, D=64, path=2) == 2                    # tensor-core path needs D == 128


def test_packed_argument_errors(L):
    def call(D=128, bits=2, ptr=FAKE):
        return L.tq_scores_packed(FAKE, FAKE, ptr, FAKE, FAKE, FAKE, FAKE, 1, 1, 8, D, bits, 1, None)
    assert call(D=40) == 2
    assert call(bits=0) == 1 and call(bits=4) == 1
    assert call(ptr=ODD) == 3
    assert call(ptr=None) == 1


def test_prepare_and_solve_argument_errors(L):
    assert L.tq_prepare_queries(FAKE, 0, FAKE, FAKE, FAKE, FAKE, 2, 3, 4, 128, None) == 1   # H > P
    assert L.tq_prepare_queries(FAKE, 5, FAKE, FAKE, FAKE, FAKE, 1, 1, 4, 128, None) == 1   # bad qtype
    assert L.tq_prepare_queries(FAKE, 0, FAKE, FAKE, FAKE, ODD, 1, 1, 4, 128, None) == 3
    need = tq.workspace_bytes(1, 4, 128)
    args = (FAKE, 0, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 1, 4, 16, 128, 4)
    assert L.tq_solve(*args, None, need, 1, None) == 4
    assert L.tq_solve(*args, FAKE, need - 1, 1, None) == 4
    assert L.tq_solve(*args, ODD, need, 1, None) == 3


def test_pack_argument_errors(L):
    assert L.tq_pack_indices(FAKE, FAKE, 0, 128, 2, None) == 1
    assert L.tq_pack_indices(FAKE, FAKE, 4, 12, 2, None) == 1          # D % 8 != 0
    assert L.tq_pack_indices(FAKE, FAKE, 4, 128, 9, None) == 1
    assert L.tq_unpack_signs(None, FAKE, 4, 128, None) == 1
    assert L.tq_pack_signs(FAKE, ODD, 4, 128, None) == 3


def test_binding_refuses_cpu_tensors(L):
    import torch
    x = torch.zeros(4, 128)
    with pytest.raises(ValueError, match="CUDA"):
        tq.prepare_queries(x, torch.eye(128), torch.eye(128))


def test_mse_argument_errors(L):
    def call(A=FAKE, norm=FAKE, D=128, bits=2, corr=0, S=10):
        return L.tq_scores_mse(A, FAKE, norm, FAKE, FAKE, 1, 1, S, D, bits, corr, None)
    assert call(A=None) == 1
    assert call(norm=ODD) == 3
    assert call(D=48) == 2                                   # D % 32 != 0
    assert call(D=16) == 1 and call(D=8192) == 1
    assert call(bits=0) == 1 and call(bits=5) == 1
    assert call(corr=2) == 1
    assert call(S=0) == 1


def test_hadamard_prepare_argument_errors(L):
    def call(D=128, signs=FAKE, H=1, P=1):
        return L.tq_prepare_queries_hadamard(FAKE, 0, signs, FAKE, FAKE, FAKE, P, H, 4, D, None)
    assert call(D=96) == 1 and call(D=1) == 1 and call(D=512) == 1   # a power of two, 2..256
    assert call(signs=None) == 1
    assert call(signs=ODD) == 3
    assert call(H=2) == 1                                              # H > P
    assert L.tq_hadamard_rotation(None, 8, None) == 1


def test_decode_argument_errors(L):
    assert L.tq_decode_workspace_bytes(1, 1, 131072, 128) >= 4 * 130 * 512
    assert L.tq_decode_workspace_bytes(1, 1, 10, 64) == 0

    def call(A=FAKE, D=128, kb=3, vb=3, scale=0.1, ws=FAKE, wsb=1 << 20, H=1):
        return L.tq_decode_mse(A, FAKE, FAKE, FAKE, kb, FAKE, FAKE, FAKE, vb, FAKE, FAKE, 1, H, 2, 100, D,
                               scale, ws, wsb, None)
    assert call(A=None) == 1 and call(A=ODD) == 3
    assert call(D=64) == 2                                    # D must be 128
    assert call(kb=0) == 1 and call(kb=4) == 1 and call(vb=4) == 1
    assert call(scale=float("inf")) == 1
    assert call(H=2) == 1                                     # H > P
    assert call(ws=None) == 4 and call(wsb=16) == 4 and call(ws=ODD) == 3
