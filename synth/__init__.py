"""Seeded synthetic workloads for TurboQuant_prod attention scoring.

This module only draws random numbers and lays them out in the shapes of the
five workloads below.  It holds none of the method's arithmetic: no rotation,
no codebook, no quantisation, no residual, no sign sketch and no score.  The
CPU oracle (``oracle/``) and the GPU product path both take their raw inputs
from here, so that both see bit-identical draws for the same seed.

Generator: NumPy's PCG64 bit generator seeded through ``SeedSequence`` with an
entropy tuple ``(config_seed, stream, *sub_ids)``.  Streams:

* ``STREAM_KEYS``  Gaussian key draws, one sub-stream per (problem, block of
  ``KEY_BLOCK`` keys) so that any key range can be regenerated on its own.
* ``STREAM_ROT``   the Gaussian matrix whose QR factor becomes the rotation Π
  (one per KV head).
* ``STREAM_SMAT``  the Gaussian QJL projection S_mat (one per KV head).
* ``STREAM_QUERY`` the queries (one per problem).

Workload recipe (all from the pages' synthetic experiments):

* keys: g ⊙ w with g iid N(0,1) in R^D and w = 1 except w = 15 on the four
  outlier channels {3, 17, 64, 101}, then scaled to unit length in float64.
  The outlier channels are the ones the kanthi.in chapter's §5 and §8
  experiments use ("TurboQuant: Rotate-then-Quantize KV Caches at 3 Bits").
* queries: iid N(0,1), rounded to float32 (or to bfloat16, round to nearest
  even, for the prefill workload).
* S_mat: iid N(0,1) D×D, rounded to float32.
* rotation seed matrix G: iid N(0,1) D×D in float64 (the oracle and the
  product each factor it on their own).
"""
from __future__ import annotations

import dataclasses

import numpy as np

OUTLIER_CHANNELS = (3, 17, 64, 101)
OUTLIER_WEIGHT = 15.0
KEY_BLOCK = 4096

STREAM_KEYS = 1
STREAM_ROT = 2
STREAM_SMAT = 3
STREAM_QUERY = 4


@dataclasses.dataclass(frozen=True)
class Workload:
    """Shape of one scoring workload.

    P problems share nothing but the codebook; problem p uses KV head p % H
    (its own Π and S_mat).  Each problem has B queries and S keys of length D.
    ``mse_bits`` is the codebook index width (C = 2**mse_bits); the key cache
    spends one more bit per coordinate on the QJL sign.
    """

    name: str
    seed: int
    P: int
    H: int
    B: int
    S: int
    D: int
    mse_bits: int
    layout: str          # "unpacked" (uint8 idx + int8 signs), "packed" (bit planes) or
                         # "mse" (code plane + fp16 norm, the MSE-only variant, no signs) or
                         # "decode" (MSE keys and MSE values, for the fused decode) or
                         # "decode_prod" (TurboQuant_prod keys and MSE values) or
                         # "compress" (the write side: fp32 keys in, the packed cache out) or
                         # "split" (outlier split: n_out channels at mse_bits + 1 bits, the
                         # rest at mse_bits, two MSE instances with norms)
    gamma_dtype: str     # "f32" or "f16" (for "mse": the dtype of the stored norm)
    q_dtype: str         # "f32" or "bf16"
    v_bits: int = 0      # "decode_prod": bits of the MSE value codes (the keys are a
                         # TurboQuant_prod cache: mse_bits-bit codes + sign plane + fp16 gamma)
    n_out: int = 0       # "split": outlier channels

    @property
    def C(self) -> int:
        return 1 << self.mse_bits

    @property
    def keys_total(self) -> int:
        return self.P * self.S


WORKLOADS = {
    # Oracle-scale parity case.
    "c0": Workload("c0_oracle_B4_S1024", 1000, 1, 1, 4, 1024, 128, 2, "unpacked", "f32", "f32"),
    # The challenge's performance shape (riteshyadav.xyz page, "What the rearrangement saves").
    "c1": Workload("c1_challenge_B32_S32768_unpacked", 1001, 1, 1, 32, 32768, 128, 2,
                   "unpacked", "f32", "f32"),
    # Single-query decode over a bit-packed 3-bit cache (2-bit index + 1-bit sign).
    "c2": Workload("c2_decode_B1_S131072_packed3bit", 1002, 1, 1, 1, 131072, 128, 2,
                   "packed", "f16", "f32"),
    # GQA decode batch: 16 sequences x 8 KV heads, 4 query heads per KV head.
    "c3": Workload("c3_gqa_16seq_8kvh_B4_S32768_packed3bit", 1003, 128, 8, 4, 32768, 128, 2,
                   "packed", "f16", "f32"),
    # Prefill-chunk scoring over a 4-bit cache (3-bit index + 1-bit sign), bf16 queries.
    "c4": Workload("c4_prefill_B128_S262144_packed4bit", 1004, 1, 1, 128, 262144, 128, 3,
                   "packed", "f16", "bf16"),
    # MSE-only variant (no sign plane, fp16 norm), single-query decode with 3-bit codes:
    # 48 + 2 bytes per key, the same as the packed 3-bit cache of c2.
    "m1": Workload("m1_mse_decode_B1_S131072_3bit", 1005, 1, 1, 1, 131072, 128, 3,
                   "mse", "f16", "f32"),
    # Fused decode (softmax and values) over MSE keys and values, 3-bit codes each.
    "d1": Workload("d1_fused_decode_B1_S131072_k3v3", 1006, 1, 1, 1, 131072, 128, 3,
                   "decode", "f16", "f32"),
    # Fused decode over the product key cache of c2 (2-bit codes + sign + fp16 gamma: the
    # 3-bit keys of the decode page) and 3-bit MSE values.
    "d2": Workload("d2_prod_decode_B1_S131072_k3v3", 1007, 1, 1, 1, 131072, 128, 2,
                   "decode_prod", "f16", "f32", v_bits=3),
    # The GPU compressor: 32768 unit fp32 keys of D = 128 into the packed 3-bit cache of c2.
    "k1": Workload("k1_compress_S32768_D128_packed3bit", 1008, 1, 1, 1, 32768, 128, 2,
                   "compress", "f16", "f32"),
    # Outlier-split decode: 32 outlier channels at 3 bits, 96 at 2, two fp16 norms (40 B a key).
    "s1": Workload("s1_split_decode_B1_S131072_32x3_96x2", 1009, 1, 1, 1, 131072, 128, 2,
                   "split", "f16", "f32", n_out=32),
}


def _rng(*entropy: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(list(entropy))))


def unit_keys(seed: int, problem: int, start: int, count: int, D: int) -> np.ndarray:
    """Keys ``start .. start+count-1`` of one problem, float64 [count, D], unit length."""
    out = np.empty((count, D), dtype=np.float64)
    w = np.ones(D)
    for ch in OUTLIER_CHANNELS:
        if ch < D:
            w[ch] = OUTLIER_WEIGHT
    pos = start
    while pos < start + count:
        blk, off = divmod(pos, KEY_BLOCK)
        take = min(KEY_BLOCK - off, start + count - pos)
        g = _rng(seed, STREAM_KEYS, problem, blk).standard_normal((KEY_BLOCK, D))
        k = g[off:off + take] * w
        k /= np.sqrt(np.sum(k * k, axis=1, keepdims=True))
        out[pos - start:pos - start + take] = k
        pos += take
    return out


def rotation_seed_matrix(seed: int, head: int, D: int) -> np.ndarray:
    """Gaussian D×D float64 matrix whose sign-fixed QR factor is the rotation Π."""
    return _rng(seed, STREAM_ROT, head).standard_normal((D, D))


def s_matrix(seed: int, head: int, D: int) -> np.ndarray:
    """QJL projection S_mat: iid N(0,1) D×D, float32."""
    return _rng(seed, STREAM_SMAT, head).standard_normal((D, D)).astype(np.float32)


def bf16_bits_rne(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest even); returns the uint16 bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32)


def queries(seed: int, problem: int, B: int, D: int, q_dtype: str = "f32"):
    """Queries of one problem.

    Returns ``(values_f32, raw)``: ``values_f32`` holds the exact query values as
    float32 (bf16 values widened exactly), ``raw`` is what a caller passes to
    the library (float32 array, or uint16 bfloat16 bit patterns).
    """
    q = _rng(seed, STREAM_QUERY, problem).standard_normal((B, D)).astype(np.float32)
    if q_dtype == "f32":
        return q, q
    if q_dtype == "bf16":
        bits = bf16_bits_rne(q)
        return bf16_bits_to_f32(bits), bits
    raise ValueError(f"unknown query dtype {q_dtype!r}")
