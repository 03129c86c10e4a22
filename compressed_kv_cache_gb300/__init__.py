"""TurboQuant_prod attention scores from a compressed key cache, on one GB300 (sm_103a).

The work happens in libtq.so (hand-written CUDA kernels behind the C ABI of
``include/tq.h``); ``compressed_kv_cache_gb300.tq`` is its Python binding.
"""
from . import tq  # noqa: F401
from .tq import (TQError, auto_path, pack_indices, pack_signs, prepare_queries, scores,  # noqa: F401
                 scores_packed, solve, solve_packed, status_string, unpack_indices, unpack_signs,
                 workspace_bytes)
