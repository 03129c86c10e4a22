"""Thin Python binding of libtq (argument marshalling only).

Every function takes torch tensors that already live on a CUDA device, checks
their dtype, device, contiguity and shape, and passes raw device pointers and
the current CUDA stream to the C ABI declared in ``include/tq.h``.  All work
runs in libtq's kernels; there is no CPU fallback.  A missing libtq.so, a
tensor on the CPU, or a non-OK status raises.
"""
from __future__ import annotations

import ctypes
import os
import re

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libtq.so")
HEADER = os.path.join(os.path.dirname(_HERE), "include", "tq.h")

TQ_OK = 0
STATUS_NAMES = {0: "TQ_OK", 1: "TQ_ERR_INVALID_VALUE", 2: "TQ_ERR_UNSUPPORTED",
                3: "TQ_ERR_MISALIGNED", 4: "TQ_ERR_WORKSPACE", 5: "TQ_ERR_LAUNCH"}
QTYPE = {torch.float32: 0, torch.bfloat16: 1}
PATHS = {"auto": 0, "fp32": 1, "bf16_mma": 2}
PATH_NAMES = {v: k for k, v in PATHS.items()}

_lib = None


class TQError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} returned {status_string(status)}")


_P, _I, _L, _Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
_SIGNATURES = {
    "tq_status_string": ([_I], ctypes.c_char_p),
    "tq_auto_path": ([_I, _I], _I),
    "tq_device_faults": ([ctypes.POINTER(ctypes.c_uint)], _I),
    "tq_check_wait_expiry": ([_P], _I),
    "tq_prepare_queries": ([_P, _I, _P, _P, _P, _P, _I, _I, _I, _I, _P], _I),
    "tq_scores": ([_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P], _I),
    "tq_scores_packed": ([_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P], _I),
    "tq_scores_mse": ([_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P], _I),
    "tq_prepare_queries_hadamard": ([_P, _I, _P, _P, _P, _P, _I, _I, _I, _I, _P], _I),
    "tq_hadamard_rotation": ([_P, _I, _P], _I),
    "tq_decode_workspace_bytes": ([_I, _I, _I, _I], ctypes.c_size_t),
    "tq_decode_mse": ([_P, _P, _P, _P, _I, _P, _P, _P, _I, _P, _P, _I, _I, _I, _I, _I, ctypes.c_float,
                       _P, ctypes.c_size_t, _P], _I),
    "tq_decode_prod": ([_P, _P, _P, _P, _P, _P, _I, _P, _P, _P, _I, _P, _P, _I, _I, _I, _I, _I, ctypes.c_float,
                        _P, ctypes.c_size_t, _P], _I),
    "tq_prepare_queries_split": ([_P, _I, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P], _I),
    "tq_scores_split": ([_P, _P, _P, _P, _P, _I, _P, _P, _P, _I, _P, _I, _I, _I, _I, _I, _P], _I),
    "tq_workspace_bytes": ([_I, _I, _I], _Z),
    "tq_solve": ([_P, _I, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _Z, _I, _P], _I),
    "tq_solve_packed": ([_P, _I, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _Z, _I, _P], _I),
    "tq_pack_indices": ([_P, _P, _L, _I, _I, _P], _I),
    "tq_unpack_indices": ([_P, _P, _L, _I, _I, _P], _I),
    "tq_pack_signs": ([_P, _P, _L, _I, _P], _I),
    "tq_unpack_signs": ([_P, _P, _L, _I, _P], _I),
    "tq_compress_keys": ([_P, _P, _P, _P, _I, _P, _P, _P, _P, _I, _I, _I, _I, _P], _I),
    "tq_compress_keys_packed": ([_P, _P, _P, _P, _I, _P, _P, _P, _I, _I, _I, _I, _P], _I),
    "tq_lloyd_max_codebook": ([_I, _I, _I, _I, _P], _I),
    "tq_haar_rotation": ([_P, _I, _P], _I),
    "tq_solve_packed_noalloc": ([_P, _I, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _P], _I),
}


def lib() -> ctypes.CDLL:
    """Loads libtq.so once; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it with compressed_kv_cache_gb300.build.build()")
        handle = ctypes.CDLL(LIB_PATH)
        for name, (args, res) in _SIGNATURES.items():
            fn = getattr(handle, name)
            fn.argtypes = args
            fn.restype = res
        _lib = handle
    return _lib


def declared_functions() -> list[str]:
    """Names of the functions include/tq.h declares."""
    with open(HEADER) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*(tq_[a-z0-9_]+)\s*\(",
                                 text, flags=re.M)))


def status_string(status: int) -> str:
    return lib().tq_status_string(status).decode()


def auto_path(B: int, D: int) -> str:
    return PATH_NAMES[lib().tq_auto_path(B, D)]


def device_faults() -> int:
    """Fault bits the bounded waits of libtq's kernels set on the current device since the
    last call (0 = none; 1 lookup-table scorers, 2 tensor-core scorer, 4 decode, 8
    compressor, 16 check_wait_expiry); reading clears them.  Synchronises with the device."""
    v = ctypes.c_uint(0)
    _check("tq_device_faults", lib().tq_device_faults(ctypes.byref(v)))
    return int(v.value)


def check_wait_expiry() -> None:
    """Runs one warp whose only bounded wait can never complete, on the current stream:
    after about a second it sets fault bit 16 and returns (see device_faults)."""
    _check("tq_check_wait_expiry", lib().tq_check_wait_expiry(_stream()))


def _check(fn: str, status: int) -> None:
    if status != TQ_OK:
        raise TQError(fn, status)


def _stream() -> int:
    return torch.cuda.current_stream().cuda_stream


def _dev(t: torch.Tensor, name: str, dtypes) -> int:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (libtq has no CPU path)")
    if t.dtype not in dtypes:
        raise TypeError(f"{name} has dtype {t.dtype}, expected one of {dtypes}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _as3(t: torch.Tensor) -> tuple[int, int, int]:
    if t.dim() == 2:
        return 1, t.shape[0], t.shape[1]
    if t.dim() == 3:
        return t.shape[0], t.shape[1], t.shape[2]
    raise ValueError(f"expected a [B,D] or [P,B,D] tensor, got shape {tuple(t.shape)}")


def prepare_queries(Q, Pi, S_mat, out=None):
    """A = Pi q and T = S_mat q.  Q [P,B,D] (or [B,D]) fp32/bf16; Pi, S_mat [H,D,D] (or [D,D])."""
    P, B, D = _as3(Q)
    H = 1 if Pi.dim() == 2 else Pi.shape[0]
    if tuple(Pi.shape[-2:]) != (D, D) or Pi.shape != S_mat.shape:
        raise ValueError("Pi and S_mat must be [H,D,D] or [D,D]")
    A, T = out if out is not None else (torch.empty((P, B, D), device=Q.device, dtype=torch.float32),
                                         torch.empty((P, B, D), device=Q.device, dtype=torch.float32))
    _check("tq_prepare_queries", lib().tq_prepare_queries(
        _dev(Q, "Q", QTYPE), QTYPE[Q.dtype], _dev(Pi, "Pi", (torch.float32,)),
        _dev(S_mat, "S_mat", (torch.float32,)), _dev(A, "A", (torch.float32,)),
        _dev(T, "T", (torch.float32,)), P, H, B, D, _stream()))
    if Q.dim() == 2:
        return A.view(B, D), T.view(B, D)
    return A, T


def prepare_queries_hadamard(Q, signs, S_mat, out=None):
    """A = H diag(s) q (fast Walsh-Hadamard transform) and T = S_mat q.  signs [H,D] (or [D])
    fp32 +-1; S_mat [H,D,D] (or [D,D]); D a power of two."""
    P, B, D = _as3(Q)
    H = 1 if signs.dim() == 1 else signs.shape[0]
    if signs.shape[-1] != D or tuple(S_mat.shape[-2:]) != (D, D):
        raise ValueError("signs must be [H,D] and S_mat [H,D,D]")
    A, T = out if out is not None else (torch.empty((P, B, D), device=Q.device, dtype=torch.float32),
                                         torch.empty((P, B, D), device=Q.device, dtype=torch.float32))
    _check("tq_prepare_queries_hadamard", lib().tq_prepare_queries_hadamard(
        _dev(Q, "Q", QTYPE), QTYPE[Q.dtype], _dev(signs, "signs", (torch.float32,)),
        _dev(S_mat, "S_mat", (torch.float32,)), _dev(A, "A", (torch.float32,)),
        _dev(T, "T", (torch.float32,)), P, H, B, D, _stream()))
    if Q.dim() == 2:
        return A.view(B, D), T.view(B, D)
    return A, T


def hadamard_rotation(signs):
    """Dense Pi = H diag(s) as a float32 [D,D] numpy matrix (host computation in libtq), for
    the compressor and the dense paths."""
    import numpy as np
    s = np.ascontiguousarray(signs, dtype=np.float32)
    D = s.size
    out = np.empty((D, D), dtype=np.float32)
    _check("tq_hadamard_rotation", lib().tq_hadamard_rotation(s.ctypes.data, D, out.ctypes.data))
    return out


def _keys3(t: torch.Tensor, P: int):
    if t.dim() == 2 and P == 1:
        return t.shape[0], t.shape[1]
    if t.dim() == 3 and t.shape[0] == P:
        return t.shape[1], t.shape[2]
    raise ValueError(f"key tensor shape {tuple(t.shape)} does not match P={P}")


def _scores_out(out, P, B, S, like):
    if out is None:
        out = torch.empty((P, B, S), device=like.device, dtype=torch.float32)
    if out.numel() != P * B * S:
        raise ValueError("scores output has the wrong size")
    return out


def scores(A, T, K_idx, signs, gamma, codebook, path="auto", out=None):
    """Scores from an unpacked cache: K_idx uint8 [P,S,D], signs int8 [P,S,D], gamma fp32 [P,S]."""
    P, B, D = _as3(A)
    S, Dk = _keys3(K_idx, P)
    if Dk != D or signs.shape != K_idx.shape or gamma.numel() != P * S:
        raise ValueError("inconsistent key shapes")
    o = _scores_out(out, P, B, S, A)
    _check("tq_scores", lib().tq_scores(
        _dev(A, "A", (torch.float32,)), _dev(T, "T", (torch.float32,)),
        _dev(K_idx, "K_idx", (torch.uint8,)), _dev(signs, "signs", (torch.int8,)),
        _dev(gamma, "gamma", (torch.float32,)), _dev(codebook, "codebook", (torch.float32,)),
        _dev(o, "scores", (torch.float32,)), P, B, S, D, codebook.numel(), PATHS[path], _stream()))
    return o if (out is not None or A.dim() == 3) else o.view(B, S)


def scores_packed(A, T, idx_plane, sign_plane, gamma_f16, codebook, idx_bits, path="auto", out=None):
    """Scores from a bit-packed cache: idx_plane uint8 [P,S,D*bits/8], sign_plane uint8
    [P,S,D/8], gamma_f16 float16 [P,S]."""
    P, B, D = _as3(A)
    S, row = _keys3(idx_plane, P)
    if row * 8 != D * idx_bits or sign_plane.shape[-1] * 8 != D or gamma_f16.numel() != P * S:
        raise ValueError("inconsistent packed key shapes")
    o = _scores_out(out, P, B, S, A)
    _check("tq_scores_packed", lib().tq_scores_packed(
        _dev(A, "A", (torch.float32,)), _dev(T, "T", (torch.float32,)),
        _dev(idx_plane, "idx_plane", (torch.uint8,)), _dev(sign_plane, "sign_plane", (torch.uint8,)),
        _dev(gamma_f16, "gamma_f16", (torch.float16,)), _dev(codebook, "codebook", (torch.float32,)),
        _dev(o, "scores", (torch.float32,)), P, B, S, D, idx_bits, PATHS[path], _stream()))
    return o if (out is not None or A.dim() == 3) else o.view(B, S)


def scores_mse(A, idx_plane, norm_f16, codebook, idx_bits, norm_correction=False, out=None):
    """MSE-only scores: A = Pi q [P,B,D] fp32, idx_plane uint8 [P,S,D*bits/8] (codes of
    the rotated unit keys), norm_f16 float16 [P,S] (key lengths)."""
    P, B, D = _as3(A)
    S, row = _keys3(idx_plane, P)
    if row * 8 != D * idx_bits or norm_f16.numel() != P * S:
        raise ValueError("inconsistent packed key shapes")
    o = _scores_out(out, P, B, S, A)
    _check("tq_scores_mse", lib().tq_scores_mse(
        _dev(A, "A", (torch.float32,)), _dev(idx_plane, "idx_plane", (torch.uint8,)),
        _dev(norm_f16, "norm_f16", (torch.float16,)), _dev(codebook, "codebook", (torch.float32,)),
        _dev(o, "scores", (torch.float32,)), P, B, S, D, idx_bits, 1 if norm_correction else 0,
        _stream()))
    return o if (out is not None or A.dim() == 3) else o.view(B, S)


def decode_mse(A, k_plane, k_norm, k_codebook, k_bits, v_plane, v_norm, v_codebook, v_bits, Pi_v,
               scale=None, workspace=None, out=None):
    """Attention output over MSE-quantized keys and values (rotated-domain decode).
    A = Pi_k q [P,B,128]; planes uint8 [P,S,128*bits/8]; norms float16 [P,S];
    Pi_v [H,128,128] (or [128,128]).  Returns [P,B,128] (or [B,128])."""
    P, B, D = _as3(A)
    S, krow = _keys3(k_plane, P)
    _, vrow = _keys3(v_plane, P)
    H = 1 if Pi_v.dim() == 2 else Pi_v.shape[0]
    if krow * 8 != D * k_bits or vrow * 8 != D * v_bits or k_norm.numel() != P * S or v_norm.numel() != P * S:
        raise ValueError("inconsistent key/value shapes")
    need = int(lib().tq_decode_workspace_bytes(P, B, S, D))
    if workspace is None:
        workspace = torch.empty(max(need, 16), device=A.device, dtype=torch.uint8)
    o = out if out is not None else torch.empty((P, B, D), device=A.device, dtype=torch.float32)
    if scale is None:
        scale = 1.0 / float(D) ** 0.5
    _check("tq_decode_mse", lib().tq_decode_mse(
        _dev(A, "A", (torch.float32,)), _dev(k_plane, "k_plane", (torch.uint8,)),
        _dev(k_norm, "k_norm", (torch.float16,)), _dev(k_codebook, "k_codebook", (torch.float32,)), k_bits,
        _dev(v_plane, "v_plane", (torch.uint8,)), _dev(v_norm, "v_norm", (torch.float16,)),
        _dev(v_codebook, "v_codebook", (torch.float32,)), v_bits, _dev(Pi_v, "Pi_v", (torch.float32,)),
        _dev(o, "out", (torch.float32,)), P, H, B, S, D, float(scale),
        _dev(workspace, "workspace", (torch.uint8,)), workspace.numel(), _stream()))
    return o if (out is not None or A.dim() == 3) else o.view(B, D)


def decode_prod(A, T, k_plane, k_sign_plane, k_gamma, k_codebook, k_bits, v_plane, v_norm, v_codebook,
                v_bits, Pi_v, scale=None, workspace=None, out=None):
    """Attention output over a TurboQuant_prod key cache and MSE-quantized values.
    A, T [P,B,128] from prepare_queries; k_plane uint8 [P,S,128*k_bits/8], k_sign_plane
    uint8 [P,S,16], k_gamma float16 [P,S]; values as for decode_mse.  Returns [P,B,128]
    (or [B,128])."""
    P, B, D = _as3(A)
    if _as3(T) != (P, B, D):
        raise ValueError("A and T must have the same shape")
    S, krow = _keys3(k_plane, P)
    S2, srow = _keys3(k_sign_plane, P)
    _, vrow = _keys3(v_plane, P)
    H = 1 if Pi_v.dim() == 2 else Pi_v.shape[0]
    if (krow * 8 != D * k_bits or srow * 8 != D or S2 != S or vrow * 8 != D * v_bits
            or k_gamma.numel() != P * S or v_norm.numel() != P * S):
        raise ValueError("inconsistent key/value shapes")
    need = int(lib().tq_decode_workspace_bytes(P, B, S, D))
    if workspace is None:
        workspace = torch.empty(max(need, 16), device=A.device, dtype=torch.uint8)
    o = out if out is not None else torch.empty((P, B, D), device=A.device, dtype=torch.float32)
    if scale is None:
        scale = 1.0 / float(D) ** 0.5
    _check("tq_decode_prod", lib().tq_decode_prod(
        _dev(A, "A", (torch.float32,)), _dev(T, "T", (torch.float32,)), _dev(k_plane, "k_plane", (torch.uint8,)),
        _dev(k_sign_plane, "k_sign_plane", (torch.uint8,)), _dev(k_gamma, "k_gamma", (torch.float16,)),
        _dev(k_codebook, "k_codebook", (torch.float32,)), k_bits,
        _dev(v_plane, "v_plane", (torch.uint8,)), _dev(v_norm, "v_norm", (torch.float16,)),
        _dev(v_codebook, "v_codebook", (torch.float32,)), v_bits, _dev(Pi_v, "Pi_v", (torch.float32,)),
        _dev(o, "out", (torch.float32,)), P, H, B, S, D, float(scale),
        _dev(workspace, "workspace", (torch.uint8,)), workspace.numel(), _stream()))
    return o if (out is not None or A.dim() == 3) else o.view(B, D)


def prepare_queries_split(Q, channels, Pi_out, Pi_reg, out=None):
    """A_out = Pi_out q[channels], A_reg = Pi_reg q[other channels] for Q [P,B,D] (or [B,D])
    f32/bf16; channels int32 [n_out] increasing; Pi_out [H,n_out,n_out] (or 2-D), Pi_reg
    [H,n_reg,n_reg].  Returns (A_out, A_reg) fp32."""
    P, B, D = _as3(Q)
    n_out = channels.numel()
    H = 1 if Pi_out.dim() == 2 else Pi_out.shape[0]
    lead = Q.shape[:-1]
    if out is None:
        out = (torch.empty(lead + (n_out,), device=Q.device, dtype=torch.float32),
               torch.empty(lead + (D - n_out,), device=Q.device, dtype=torch.float32))
    A_out, A_reg = out
    _check("tq_prepare_queries_split", lib().tq_prepare_queries_split(
        _dev(Q, "Q", tuple(QTYPE)), QTYPE[Q.dtype], _dev(channels, "channels", (torch.int32,)),
        _dev(Pi_out, "Pi_out", (torch.float32,)), _dev(Pi_reg, "Pi_reg", (torch.float32,)),
        _dev(A_out, "A_out", (torch.float32,)), _dev(A_reg, "A_reg", (torch.float32,)), P, H, B, D, n_out,
        _stream()))
    return A_out, A_reg


def scores_split(A_out, A_reg, out_plane, out_norm, out_codebook, out_bits, reg_plane, reg_norm,
                 reg_codebook, reg_bits, out=None):
    """Scores of the outlier-split cache: [P,B,S] (or [B,S])."""
    P, B, n_out = _as3(A_out)
    _, _, n_reg = _as3(A_reg)
    S, orow = _keys3(out_plane, P)
    S2, rrow = _keys3(reg_plane, P)
    if (S2 != S or orow * 8 != n_out * out_bits or rrow * 8 != n_reg * reg_bits
            or out_norm.numel() != P * S or reg_norm.numel() != P * S):
        raise ValueError("inconsistent split cache shapes")
    o = _scores_out(out, P, B, S, A_out)
    _check("tq_scores_split", lib().tq_scores_split(
        _dev(A_out, "A_out", (torch.float32,)), _dev(A_reg, "A_reg", (torch.float32,)),
        _dev(out_plane, "out_plane", (torch.uint8,)), _dev(out_norm, "out_norm", (torch.float16,)),
        _dev(out_codebook, "out_codebook", (torch.float32,)), out_bits,
        _dev(reg_plane, "reg_plane", (torch.uint8,)), _dev(reg_norm, "reg_norm", (torch.float16,)),
        _dev(reg_codebook, "reg_codebook", (torch.float32,)), reg_bits, _dev(o, "scores", (torch.float32,)),
        P, B, S, n_out, n_reg, _stream()))
    return o if (out is not None or A_out.dim() == 3) else o.view(B, S)


def workspace_bytes(P: int, B: int, D: int) -> int:
    return int(lib().tq_workspace_bytes(P, B, D))


def _workspace(ws, P, B, D, like):
    need = workspace_bytes(P, B, D)
    if ws is None:
        ws = torch.empty(need, device=like.device, dtype=torch.uint8)
    return ws


def solve(Q, K_idx, signs, gamma, Pi, S_mat, codebook, path="auto", workspace=None, out=None):
    """Fused query transform + scoring over an unpacked cache."""
    P, B, D = _as3(Q)
    H = 1 if Pi.dim() == 2 else Pi.shape[0]
    S, Dk = _keys3(K_idx, P)
    if Dk != D:
        raise ValueError("inconsistent key shapes")
    ws = _workspace(workspace, P, B, D, Q)
    o = _scores_out(out, P, B, S, Q)
    _check("tq_solve", lib().tq_solve(
        _dev(Q, "Q", QTYPE), QTYPE[Q.dtype], _dev(K_idx, "K_idx", (torch.uint8,)),
        _dev(signs, "signs", (torch.int8,)), _dev(gamma, "gamma", (torch.float32,)),
        _dev(Pi, "Pi", (torch.float32,)), _dev(S_mat, "S_mat", (torch.float32,)),
        _dev(codebook, "codebook", (torch.float32,)), _dev(o, "scores", (torch.float32,)),
        P, H, B, S, D, codebook.numel(), _dev(ws, "workspace", (torch.uint8,)), ws.numel(),
        PATHS[path], _stream()))
    return o if (out is not None or Q.dim() == 3) else o.view(B, S)


def solve_packed(Q, idx_plane, sign_plane, gamma_f16, Pi, S_mat, codebook, idx_bits, path="auto",
                 workspace=None, out=None):
    """Fused query transform + scoring over a bit-packed cache."""
    P, B, D = _as3(Q)
    H = 1 if Pi.dim() == 2 else Pi.shape[0]
    S, _ = _keys3(idx_plane, P)
    ws = _workspace(workspace, P, B, D, Q)
    o = _scores_out(out, P, B, S, Q)
    _check("tq_solve_packed", lib().tq_solve_packed(
        _dev(Q, "Q", QTYPE), QTYPE[Q.dtype], _dev(idx_plane, "idx_plane", (torch.uint8,)),
        _dev(sign_plane, "sign_plane", (torch.uint8,)), _dev(gamma_f16, "gamma_f16", (torch.float16,)),
        _dev(Pi, "Pi", (torch.float32,)), _dev(S_mat, "S_mat", (torch.float32,)),
        _dev(codebook, "codebook", (torch.float32,)), _dev(o, "scores", (torch.float32,)),
        P, H, B, S, D, idx_bits, _dev(ws, "workspace", (torch.uint8,)), ws.numel(),
        PATHS[path], _stream()))
    return o if (out is not None or Q.dim() == 3) else o.view(B, S)


def pack_indices(K_idx, bits, out=None):
    """uint8 codes [..., D] -> packed plane [..., D*bits/8]."""
    D = K_idx.shape[-1]
    n = K_idx.numel() // D
    o = out if out is not None else torch.empty((*K_idx.shape[:-1], D * bits // 8), device=K_idx.device, dtype=torch.uint8)
    _check("tq_pack_indices", lib().tq_pack_indices(
        _dev(K_idx, "K_idx", (torch.uint8,)), _dev(o, "idx_plane", (torch.uint8,)), n, D, bits, _stream()))
    return o


def unpack_indices(plane, D, bits, out=None):
    n = plane.numel() // (D * bits // 8)
    o = out if out is not None else torch.empty((*plane.shape[:-1], D), device=plane.device, dtype=torch.uint8)
    _check("tq_unpack_indices", lib().tq_unpack_indices(
        _dev(plane, "idx_plane", (torch.uint8,)), _dev(o, "K_idx", (torch.uint8,)), n, D, bits, _stream()))
    return o


def pack_signs(signs, out=None):
    D = signs.shape[-1]
    n = signs.numel() // D
    o = out if out is not None else torch.empty((*signs.shape[:-1], D // 8), device=signs.device, dtype=torch.uint8)
    _check("tq_pack_signs", lib().tq_pack_signs(
        _dev(signs, "signs", (torch.int8,)), _dev(o, "sign_plane", (torch.uint8,)), n, D, _stream()))
    return o


def unpack_signs(plane, D, out=None):
    n = plane.numel() // (D // 8)
    o = out if out is not None else torch.empty((*plane.shape[:-1], D), device=plane.device, dtype=torch.int8)
    _check("tq_unpack_signs", lib().tq_unpack_signs(
        _dev(plane, "sign_plane", (torch.uint8,)), _dev(o, "signs", (torch.int8,)), n, D, _stream()))
    return o


def lloyd_max_codebook(D: int, mse_bits: int, grid_points: int = 400_001, iterations: int = 300):
    """Lloyd-Max codebook (host computation in libtq), float32 numpy array of 2^mse_bits."""
    import numpy as np
    out = np.empty(1 << mse_bits, dtype=np.float32)
    _check("tq_lloyd_max_codebook", lib().tq_lloyd_max_codebook(
        D, mse_bits, grid_points, iterations, out.ctypes.data))
    return out


def haar_rotation(G):
    """Sign-fixed QR rotation of a float64 [D,D] numpy matrix (host computation in libtq)."""
    import numpy as np
    G = np.ascontiguousarray(G, dtype=np.float64)
    D = G.shape[0]
    out = np.empty((D, D), dtype=np.float32)
    _check("tq_haar_rotation", lib().tq_haar_rotation(G.ctypes.data, D, out.ctypes.data))
    return out


def compress_keys(keys, Pi, S_mat, codebook, gamma_dtype=torch.float32):
    """TurboQuant_prod compression on the GPU.  keys fp32 [P,S,D] (or [S,D]); Pi, S_mat
    [H,D,D] (or [D,D]).  Returns (K_idx uint8, signs int8, gamma fp32 or fp16)."""
    P, S, D = _as3(keys)
    H = 1 if Pi.dim() == 2 else Pi.shape[0]
    K_idx = torch.empty(keys.shape, device=keys.device, dtype=torch.uint8)
    signs = torch.empty(keys.shape, device=keys.device, dtype=torch.int8)
    gamma = torch.empty(keys.shape[:-1], device=keys.device, dtype=gamma_dtype)
    g32 = _dev(gamma, "gamma", (torch.float32,)) if gamma_dtype == torch.float32 else None
    g16 = _dev(gamma, "gamma", (torch.float16,)) if gamma_dtype == torch.float16 else None
    _check("tq_compress_keys", lib().tq_compress_keys(
        _dev(keys, "keys", (torch.float32,)), _dev(Pi, "Pi", (torch.float32,)),
        _dev(S_mat, "S_mat", (torch.float32,)), _dev(codebook, "codebook", (torch.float32,)),
        codebook.numel(), _dev(K_idx, "K_idx", (torch.uint8,)), _dev(signs, "signs", (torch.int8,)),
        g32, g16, P, H, S, D, _stream()))
    return K_idx, signs, gamma


def compress_keys_packed(keys, Pi, S_mat, codebook, idx_bits, out=None):
    """TurboQuant_prod compression on the GPU straight into the packed cache.  keys fp32
    [P,S,D] (or [S,D]); Pi, S_mat [H,D,D] (or [D,D]); codebook 2^idx_bits fp32.  Returns
    (idx_plane uint8 [..,S,D*idx_bits/8], sign_plane uint8 [..,S,D/8], gamma fp16 [..,S])."""
    P, S, D = _as3(keys)
    H = 1 if Pi.dim() == 2 else Pi.shape[0]
    lead = keys.shape[:-1]
    if out is None:
        out = (torch.empty(lead + (D * idx_bits // 8,), device=keys.device, dtype=torch.uint8),
               torch.empty(lead + (D // 8,), device=keys.device, dtype=torch.uint8),
               torch.empty(lead, device=keys.device, dtype=torch.float16))
    ip, sp, g = out
    _check("tq_compress_keys_packed", lib().tq_compress_keys_packed(
        _dev(keys, "keys", (torch.float32,)), _dev(Pi, "Pi", (torch.float32,)),
        _dev(S_mat, "S_mat", (torch.float32,)), _dev(codebook, "codebook", (torch.float32,)), idx_bits,
        _dev(ip, "idx_plane", (torch.uint8,)), _dev(sp, "sign_plane", (torch.uint8,)),
        _dev(g, "gamma", (torch.float16,)), P, H, S, D, _stream()))
    return ip, sp, g
