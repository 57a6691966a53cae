"""ctypes loader for libmsa.so (the C ABI in include/msa.h).

Loading fails loudly: there is no fallback implementation of any operation."""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

OK, EINVAL, ECUDA, ENOSPC = 0, 1, 3, 4
ERR_TOPK_RANGE = 0x01
ERR_TOPK_DUP = 0x02
ERR_PAGE_RANGE = 0x04
ERR_SEQ_RANGE = 0x08
ERR_SCORE_NAN = 0x10
ERR_TIMEOUT = 0x20

#: Every symbol include/msa.h declares.
EXPORTS = ("msa_score", "msa_topk", "msa_workspace_bytes", "msa_choose_splits",
           "msa_sparse_decode", "msa_combine", "msa_get_error", "msa_strerror", "msa_version",
           "msa_sparse_decode_static", "msa_sparse_decode_select", "msa_dense_splits",
           "msa_dense_decode", "msa_score_q8", "msa_sparse_decode_q8",
           "msa_sparse_decode_select_q8", "msa_dense_decode_q8", "msa_sparse_prefill",
           "msa_sparse_prefill_select", "msa_sparse_prefill_q8", "msa_sparse_prefill_select_q8",
           "msa_score_kcache", "msa_score_kcache_q8", "msa_decode_step",
           "msa_set_input_overlap", "msa_set_union_tile", "msa_test_wait_timeout")

_lib = None
_lock = threading.Lock()


class MSAError(RuntimeError):
    def __init__(self, status: int, where: str, text: str):
        super().__init__(f"{where}: status {status} ({text})")
        self.status = status


def library_path() -> str:
    return _build.LIB


def load(path: str | None = None):
    """Load libmsa.so (built in-tree by build.build()).  Raises if it is missing."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = path or _build.LIB
        if not os.path.exists(path):
            raise ImportError(
                f"libmsa.so not found at {path}; build it with "
                "`python -m block_sparse_gqa_score_gb300.build` (needs nvcc)")
        lib = ctypes.CDLL(path)
        P, i32, i64, f32, sz = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float,
                                ctypes.c_size_t)
        lib.msa_score.argtypes = [P, P, P, P, P, i32, i32, i32, i32, i32, i64, f32, f32, P]
        lib.msa_topk.argtypes = [P, i64, i64, i64, P, P, i32, i32, i32, i32, i32, P]
        lib.msa_workspace_bytes.argtypes = [i32, i32, i32, i32]
        lib.msa_workspace_bytes.restype = sz
        lib.msa_choose_splits.argtypes = [i32, i32, i32, i32]
        lib.msa_sparse_decode.argtypes = [P, P, P, P, P, P, sz, P, i32, i32, i32, i32, i32, i64,
                                          f32, f32, f32, i32, P]
        lib.msa_combine.argtypes = [P, P, i32, i32, i32, P]
        lib.msa_sparse_decode_select.argtypes = [P, P, P, P, P, i64, i64, i64, P, P, sz, P, i32,
                                                 i32, i32, i32, i32, i64, f32, f32, f32, i32, P]
        lib.msa_sparse_decode_static.argtypes = [P, P, P, P, P, P, i32, i32, i32, i32, i32, i64,
                                                 f32, f32, f32, i32, P]
        lib.msa_dense_splits.argtypes = [i32]
        lib.msa_dense_decode.argtypes = [P, P, P, P, P, sz, P, i32, i32, i32, i32, i32, i64, f32,
                                         f32, f32, P]
        # the fp8-query variants: (q8, q_scale) in place of q
        lib.msa_score_q8.argtypes = [P, f32] + lib.msa_score.argtypes[1:]
        lib.msa_sparse_decode_q8.argtypes = [P, f32] + lib.msa_sparse_decode.argtypes[1:]
        lib.msa_sparse_decode_select_q8.argtypes = ([P, f32] +
                                                    lib.msa_sparse_decode_select.argtypes[1:])
        lib.msa_dense_decode_q8.argtypes = [P, f32] + lib.msa_dense_decode.argtypes[1:]
        # the K-only (index-K) cache scorer: msa_score's arguments
        lib.msa_score_kcache.argtypes = lib.msa_score.argtypes
        lib.msa_score_kcache_q8.argtypes = lib.msa_score_q8.argtypes
        # prefill: cu_seqlens_q after seq_lens, (B, T) in place of (B, Q)
        lib.msa_sparse_prefill.argtypes = [P, P, P, P, P, P, P, sz, P, i32, i32, i32, i32, i32,
                                           i64, f32, f32, f32, i32, P]
        lib.msa_sparse_prefill_select.argtypes = [P, P, P, P, P, P, i64, i64, i64, P, P, sz, P,
                                                  i32, i32, i32, i32, i32, i64, f32, f32, f32,
                                                  i32, P]
        lib.msa_sparse_prefill_q8.argtypes = [P, f32] + lib.msa_sparse_prefill.argtypes[1:]
        lib.msa_sparse_prefill_select_q8.argtypes = ([P, f32] +
                                                     lib.msa_sparse_prefill_select.argtypes[1:])
        # the whole step: (q, q_scale, kv, index_k, index_k_scale, ...)
        lib.msa_decode_step.argtypes = [P, f32, P, P, f32, P, P, P, P, P, sz, P, i32, i32, i32,
                                        i32, i32, i64, f32, f32, f32, i32, P]
        lib.msa_set_input_overlap.argtypes = [i32]
        lib.msa_set_union_tile.argtypes = [i32]
        lib.msa_test_wait_timeout.argtypes = [ctypes.c_ulonglong, P]
        lib.msa_get_error.argtypes = [ctypes.POINTER(ctypes.c_uint), i32]
        lib.msa_strerror.argtypes = [i32]
        lib.msa_strerror.restype = ctypes.c_char_p
        for name in ("msa_score", "msa_topk", "msa_choose_splits", "msa_sparse_decode",
                     "msa_combine", "msa_get_error", "msa_version", "msa_sparse_decode_static",
                     "msa_sparse_decode_select", "msa_dense_splits", "msa_dense_decode",
                     "msa_score_q8", "msa_sparse_decode_q8", "msa_sparse_decode_select_q8",
                     "msa_dense_decode_q8", "msa_sparse_prefill", "msa_sparse_prefill_select",
                     "msa_sparse_prefill_q8", "msa_sparse_prefill_select_q8",
                     "msa_score_kcache", "msa_score_kcache_q8", "msa_decode_step",
                     "msa_set_input_overlap", "msa_set_union_tile", "msa_test_wait_timeout"):
            getattr(lib, name).restype = i32
        _lib = lib
        return lib


def check(status: int, where: str):
    if status != OK:
        lib = load()
        raise MSAError(status, where, lib.msa_strerror(status).decode())
