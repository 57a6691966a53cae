"""CPU oracle for the block-sparse GQA decode step -- TEST INFRASTRUCTURE ONLY.

This package binds ``msa_oracle.c`` (plain C, fp64) through ctypes.  Only the
tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may
import it.  The product library never imports, links or calls anything here,
and nothing here imports the product library.

What each routine computes, and which page passage it follows, is stated in
``msa_oracle.c``.  Arrays are numpy arrays; bf16 tensors travel as their raw
16-bit patterns (``uint16``) and fp8 tensors as raw bytes (``uint8``).
"""
from __future__ import annotations

import ctypes
import fcntl
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "msa_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libmsa_oracle.so")

OK, EINVAL, ERANGE, ENAN = 0, 1, 2, 3
_STATUS = {EINVAL: "invalid argument", ERANGE: "index out of range or duplicate top-k entry",
           ENAN: "NaN input"}

_lib = None
_lock = threading.Lock()


class OracleError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"oracle {what}: status {status} ({_STATUS.get(status, '?')})")
        self.status = status


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (fp64, no fast-math) if the source is newer.

    MSA_ORACLE_LIB names an already-built library to load instead; the
    mutation test uses it to run the pins against deliberately broken copies."""
    override = os.environ.get("MSA_ORACLE_LIB")
    if override:
        return override
    os.makedirs(_OUT_DIR, exist_ok=True)

    def stale():
        return (not os.path.exists(_LIB_PATH)
                or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))

    if force or stale():
        with open(os.path.join(_OUT_DIR, ".lock"), "w") as lock:
            fcntl.flock(lock, fcntl.LOCK_EX)
            if force or stale():
                tmp = _LIB_PATH + f".tmp{os.getpid()}"
                subprocess.check_call(["gcc", "-std=c11", "-O2", "-fno-fast-math", "-Wall",
                                       "-shared", "-fPIC", "-pthread", _SRC, "-o", tmp, "-lm"])
                os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            i32, i64, f64 = ctypes.c_int, ctypes.c_int64, ctypes.c_double
            lib.orc_e4m3_to_f64.argtypes = [ctypes.c_uint8]
            lib.orc_e4m3_to_f64.restype = f64
            lib.orc_bf16_to_f64.argtypes = [ctypes.c_uint16]
            lib.orc_bf16_to_f64.restype = f64
            lib.orc_default_threads.restype = i32
            lib.orc_score.argtypes = [P, P, P, P, P, i32, i32, i32, i32, i32, i64, f64, f64, i32]
            lib.orc_score_units.argtypes = [P, P, P, P, P, P, i64, i32, i32, i32, i32, i32, i64,
                                            f64, f64, i32]
            lib.orc_score_blocks.argtypes = [P, P, P, P, P, P, i64, i32, i32, i32, i32, i32, i64,
                                             f64, f64, i32]
            lib.orc_topk.argtypes = [P, i64, i64, i64, P, P, i32, i32, i32, i32, i32]
            lib.orc_attend.argtypes = [P, P, P, P, P, P, i32, i32, i32, i32, i32, i64, i32, f64,
                                       f64, f64, i32]
            lib.orc_attend_rows.argtypes = [P, P, P, P, P, P, i64, P, i32, i32, i32, i32, i32, i64,
                                            i32, f64, f64, f64, i32]
            lib.orc_combine.argtypes = [P, P, P, i64, i32]
            for name in ("orc_score", "orc_score_units", "orc_score_blocks", "orc_topk", "orc_attend",
                         "orc_attend_rows", "orc_combine"):
                getattr(lib, name).restype = i32
            _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


def _c(a, dtype) -> np.ndarray:
    a = np.asarray(a)
    if a.dtype != dtype:
        raise TypeError(f"expected {dtype}, got {a.dtype}")
    return np.ascontiguousarray(a)


def _check(status: int, what: str):
    if status != OK:
        raise OracleError(status, what)


def default_threads() -> int:
    return int(_load().orc_default_threads())


def e4m3_to_f64(codes) -> np.ndarray:
    """Decode fp8 E4M3 codes by their bit fields."""
    lib = _load()
    codes = np.asarray(codes, dtype=np.uint8)
    table = np.array([lib.orc_e4m3_to_f64(c) for c in range(256)], dtype=np.float64)
    return table[codes]


def bf16_to_f64(bits) -> np.ndarray:
    """Decode bfloat16 bit patterns (uint16)."""
    lib = _load()
    bits = np.asarray(bits, dtype=np.uint16)
    uniq = np.unique(bits)
    vals = np.array([lib.orc_bf16_to_f64(int(u)) for u in uniq], dtype=np.float64)
    return vals[np.searchsorted(uniq, bits)]


class Problem:
    """The inputs of one decode step, as host arrays."""

    def __init__(self, q_bits, kv, block_table, seq_lens, Q, Hq, Hkv,
                 sm_scale, k_scale=1.0, v_scale=1.0):
        self.q = _c(q_bits, np.uint16)
        self.kv = _c(kv, np.uint8)
        self.block_table = _c(block_table, np.int32)
        self.seq_lens = _c(seq_lens, np.int32)
        self.B = int(self.seq_lens.shape[0])
        self.Q, self.Hq, self.Hkv = int(Q), int(Hq), int(Hkv)
        self.S = int(self.block_table.shape[1]) if self.block_table.ndim == 2 else 0
        self.NB = int(self.kv.shape[0]) if self.kv.ndim >= 1 else 0
        self.sm_scale, self.k_scale, self.v_scale = float(sm_scale), float(k_scale), float(v_scale)
        T = self.B * self.Q
        if self.q.shape != (T, self.Hq, 128):
            raise ValueError(f"q must be [T={T}, Hq={self.Hq}, 128], got {self.q.shape}")
        if self.kv.ndim != 4 or self.kv.shape[1:] != (self.Hkv, 128, 256):
            raise ValueError(f"kv must be [NB, {self.Hkv}, 128, 256], got {self.kv.shape}")
        if self.block_table.shape[0] != self.B:
            raise ValueError("block_table must have one row per request")

    @property
    def T(self) -> int:
        return self.B * self.Q


def score(p: Problem, nthreads: int = 0) -> np.ndarray:
    """Block scores [Hkv, T, S] (fp64; -inf past the current block)."""
    out = np.empty((p.Hkv, p.T, p.S), dtype=np.float64)
    st = _load().orc_score(_ptr(p.q), _ptr(p.kv), _ptr(p.block_table), _ptr(p.seq_lens), _ptr(out),
                           p.B, p.Q, p.Hq, p.Hkv, p.S, p.NB, p.sm_scale, p.k_scale, nthreads)
    _check(st, "score")
    return out


def score_units(p: Problem, units, nthreads: int = 0) -> np.ndarray:
    """Block scores of the listed (b * Hkv + g) units only; other rows are NaN."""
    units = _c(np.asarray(units, dtype=np.int64), np.int64)
    out = np.full((p.Hkv, p.T, p.S), np.nan, dtype=np.float64)
    st = _load().orc_score_units(_ptr(p.q), _ptr(p.kv), _ptr(p.block_table), _ptr(p.seq_lens),
                                 _ptr(out), _ptr(units), len(units), p.B, p.Q, p.Hq, p.Hkv, p.S,
                                 p.NB, p.sm_scale, p.k_scale, nthreads)
    _check(st, "score_units")
    return out


def score_blocks(p: Problem, triples, nthreads: int = 0) -> np.ndarray:
    """Scores of listed (b, g, n) blocks for every token of request b; other
    entries are NaN.  Returns the full [Hkv, T, S] array."""
    triples = _c(np.asarray(triples, dtype=np.int64).reshape(-1, 3), np.int64)
    out = np.full((p.Hkv, p.T, p.S), np.nan, dtype=np.float64)
    st = _load().orc_score_blocks(_ptr(p.q), _ptr(p.kv), _ptr(p.block_table), _ptr(p.seq_lens),
                                  _ptr(out), _ptr(triples), len(triples), p.B, p.Q, p.Hq, p.Hkv,
                                  p.S, p.NB, p.sm_scale, p.k_scale, nthreads)
    _check(st, "score_blocks")
    return out


def topk(scores: np.ndarray, seq_lens, Q: int, k: int = 16) -> np.ndarray:
    """Selected blocks [T, Hkv, k] from scores indexed [g, i, n] (any strides)."""
    scores = np.asarray(scores, dtype=np.float64)
    seq_lens = _c(seq_lens, np.int32)
    Hkv, T, S = scores.shape
    B = int(seq_lens.shape[0])
    if T != B * Q:
        raise ValueError("scores' token dim must be B*Q")
    st_h, st_t, st_n = (s // 8 for s in scores.strides)
    if any(s % 8 for s in scores.strides):
        raise ValueError("unaligned strides")
    out = np.empty((T, Hkv, k), dtype=np.int32)
    # pass the base of the (possibly strided) view
    base = ctypes.c_void_p(scores.__array_interface__["data"][0])
    st = _load().orc_topk(base, st_h, st_t, st_n, _ptr(seq_lens), _ptr(out), B, Q, Hkv, S, k)
    _check(st, "topk")
    return out


def attend(p: Problem, topk_idx, nthreads: int = 0) -> np.ndarray:
    """Attention over the listed blocks: [T, Hq, 128] fp64."""
    topk_idx = _c(topk_idx, np.int32)
    if topk_idx.ndim != 3 or topk_idx.shape[:2] != (p.T, p.Hkv):
        raise ValueError("topk must be [T, Hkv, k]")
    out = np.empty((p.T, p.Hq, 128), dtype=np.float64)
    st = _load().orc_attend(_ptr(p.q), _ptr(p.kv), _ptr(p.block_table), _ptr(p.seq_lens),
                            _ptr(topk_idx), _ptr(out), p.B, p.Q, p.Hq, p.Hkv, p.S, p.NB,
                            topk_idx.shape[2], p.sm_scale, p.k_scale, p.v_scale, nthreads)
    _check(st, "attend")
    return out


def attend_rows(p: Problem, topk_idx, rows, nthreads: int = 0) -> np.ndarray:
    """Attention of the listed query rows (i * Hq + h) only: [len(rows), 128]."""
    topk_idx = _c(topk_idx, np.int32)
    rows = _c(np.asarray(rows, dtype=np.int64), np.int64)
    out = np.empty((len(rows), 128), dtype=np.float64)
    st = _load().orc_attend_rows(_ptr(p.q), _ptr(p.kv), _ptr(p.block_table), _ptr(p.seq_lens),
                                 _ptr(topk_idx), _ptr(rows), len(rows), _ptr(out), p.B, p.Q, p.Hq,
                                 p.Hkv, p.S, p.NB, topk_idx.shape[2], p.sm_scale, p.k_scale,
                                 p.v_scale, nthreads)
    _check(st, "attend_rows")
    return out


def _prefill_requests(seq_lens, cu_seqlens_q):
    """(b, first token, query length) of each non-empty request of a prefill
    batch; a request's query tokens are the last q_len of its sequence."""
    seq_lens = np.asarray(seq_lens, dtype=np.int64)
    cu = np.asarray(cu_seqlens_q, dtype=np.int64)
    if cu.shape != (seq_lens.shape[0] + 1,) or cu[0] != 0 or np.any(np.diff(cu) < 0):
        raise ValueError("cu_seqlens_q must be [B + 1], ascending from 0")
    out = []
    for b in range(seq_lens.shape[0]):
        n = int(cu[b + 1] - cu[b])
        if n > seq_lens[b]:
            raise ValueError("a request's query length exceeds its sequence length")
        if n > 0:
            out.append((b, int(cu[b]), n))
    return out


def attend_prefill(q_bits, kv, block_table, seq_lens, cu_seqlens_q, topk_idx, Hq: int,
                   Hkv: int, sm_scale: float, k_scale: float = 1.0, v_scale: float = 1.0,
                   nthreads: int = 0) -> np.ndarray:
    """Sparse attention of a prefill or chunked-prefill batch, [T, Hq, 128] fp64.

    MiniMaxM3SparsePrefillMetadata on the vLLM pages: request b owns query rows
    cu_seqlens_q[b] .. cu_seqlens_q[b + 1] - 1, and they are the last q_len_b
    tokens of its seq_lens[b] (the cached context being seq_lens[b] -
    q_len_b), so local token j sits at position seq_lens[b] - q_len_b + j and
    sees pages 0 .. pos / 128, as the vLLM prefill test counts them.  Each
    request is therefore attend() of a one-request problem with Q = q_len_b."""
    q_bits = np.asarray(q_bits, dtype=np.uint16)
    topk_idx = np.asarray(topk_idx, dtype=np.int32)
    block_table = np.asarray(block_table, dtype=np.int32)
    out = np.zeros((q_bits.shape[0], Hq, 128), dtype=np.float64)
    for b, s, n in _prefill_requests(seq_lens, cu_seqlens_q):
        p = Problem(q_bits[s:s + n], kv, block_table[b:b + 1], np.asarray(seq_lens)[b:b + 1], n,
                    Hq, Hkv, sm_scale, k_scale, v_scale)
        out[s:s + n] = attend(p, topk_idx[s:s + n], nthreads)
    return out


def topk_prefill(scores: np.ndarray, seq_lens, cu_seqlens_q, k: int = 16) -> np.ndarray:
    """Per-token causal top-k of a prefill batch from scores [Hkv, T, S] (any
    strides): topk() of each request's rows with Q = q_len_b, so each token
    keeps its own current block.  Rows of empty requests do not exist; the
    returned [T, Hkv, k] is -1 where no request covers a row."""
    scores = np.asarray(scores, dtype=np.float64)
    Hkv, T, _ = scores.shape
    out = np.full((T, Hkv, k), -1, dtype=np.int32)
    for b, s, n in _prefill_requests(seq_lens, cu_seqlens_q):
        out[s:s + n] = topk(scores[:, s:s + n, :], np.asarray(seq_lens, dtype=np.int32)[b:b + 1],
                            n, k)
    return out


def combine(o, ml) -> np.ndarray:
    """Merge split-softmax parts: o [splits, rows, 128], ml [splits, rows, 2] -> [rows, 128]."""
    o = _c(np.asarray(o, dtype=np.float64), np.float64)
    ml = _c(np.asarray(ml, dtype=np.float64), np.float64)
    splits, rows = o.shape[0], o.shape[1]
    out = np.empty((rows, 128), dtype=np.float64)
    st = _load().orc_combine(_ptr(o), _ptr(ml), _ptr(out), rows, splits)
    _check(st, "combine")
    return out


def decode_step(p: Problem, k: int = 16, nthreads: int = 0):
    """Score -> select -> attend, all in the oracle. Returns (scores, topk, out)."""
    s = score(p, nthreads)
    t = topk(s, p.seq_lens, p.Q, k)
    o = attend(p, t, nthreads)
    return s, t, o
