"""Host-side tests of the C ABI: the library builds and loads, exports every
symbol include/msa.h declares, and rejects bad arguments before any launch.
No GPU is needed (validation runs before any CUDA call)."""
from __future__ import annotations

import ctypes
import os
import re

import pytest

from block_sparse_gqa_score_gb300 import _native, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "msa.h")

EINVAL, ENOSPC = _native.EINVAL, _native.ENOSPC


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _native.load()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(msa_[a-z0-9_]+)\s*\(", text)))


def test_header_and_binding_agree():
    assert _declared_functions() == sorted(_native.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name
    assert lib.msa_version() == 100


def test_status_texts(lib):
    assert lib.msa_strerror(0) == b"ok"
    assert b"invalid" in lib.msa_strerror(EINVAL)
    assert b"workspace" in lib.msa_strerror(ENOSPC)


def test_workspace_bytes(lib):
    assert lib.msa_workspace_bytes(16, 4, 64, 1) == 0
    assert lib.msa_workspace_bytes(16, 4, 64, 0) == 0
    assert lib.msa_workspace_bytes(16, 4, 64, 3) == 3 * 16 * 4 * 64 * 130 * 4
    assert lib.msa_workspace_bytes(16, 4, 64, 17) == 0
    assert lib.msa_workspace_bytes(-1, 4, 64, 2) == 0


def test_choose_splits_depends_on_shape_only(lib):
    for B, Q, Hkv in [(16, 4, 4), (32, 4, 1), (128, 1, 4), (16, 32, 4), (1, 1, 1), (2, 1, 1)]:
        s = lib.msa_choose_splits(B, Q, Hkv, 152)
        assert 1 <= s <= 16
        assert s == lib.msa_choose_splits(B, Q, Hkv, 152)
    assert lib.msa_choose_splits(1, 1, 1, 152) > 1       # a tiny batch is split
    assert lib.msa_choose_splits(128, 1, 4, 152) == 1    # 512 CTAs fill the GPU


# fake, aligned, non-null device addresses: validation must reject before use
A = ctypes.c_void_p(1 << 20)


def _score(lib, **kw):
    args = dict(q=A, kv=A, bt=A, sl=A, out=A, B=16, Q=4, Hq=64, Hkv=4, S=8, NB=100,
                sm=0.088, ks=1.0)
    args.update(kw)
    return lib.msa_score(args["q"], args["kv"], args["bt"], args["sl"], args["out"], args["B"],
                         args["Q"], args["Hq"], args["Hkv"], args["S"], args["NB"], args["sm"],
                         args["ks"], None)


@pytest.mark.parametrize("kw", [
    dict(Q=0), dict(Q=33), dict(Hq=60), dict(Hq=32), dict(Hkv=0), dict(S=0), dict(NB=0),
    dict(B=-1), dict(q=None), dict(kv=None), dict(bt=None), dict(sl=None), dict(out=None),
    dict(q=ctypes.c_void_p((1 << 20) + 8)), dict(kv=ctypes.c_void_p((1 << 20) + 4)),
    dict(sm=0.0), dict(sm=float("nan")), dict(ks=-1.0), dict(ks=float("inf")),
    dict(NB=(1 << 31) // (4 * 128)),
])
def test_score_rejects(lib, kw):
    assert _score(lib, **kw) == EINVAL


def test_qlen_bounds_follow_the_pages_dispatch_limits(lib):
    """The vLLM static-dispatch test accepts query lengths 1 and 32 and rejects
    0 and 33 (test_msa_cutlass_decode_static_dispatch)."""
    assert _score(lib, Q=0) == EINVAL and _score(lib, Q=33) == EINVAL
    # Q = 1 and 32 pass validation and only fail later for want of a device
    assert _score(lib, Q=1) != EINVAL and _score(lib, Q=32) != EINVAL


def test_empty_batch_is_a_no_op(lib):
    assert _score(lib, B=0) == 0


def _decode(lib, **kw):
    args = dict(q=A, kv=A, bt=A, sl=A, tk=A, ws=None, wsb=0, out=A, B=16, Q=4, Hq=64, Hkv=4, S=8,
                NB=100, sm=0.088, ks=1.0, vs=1.0, splits=1)
    args.update(kw)
    return lib.msa_sparse_decode(args["q"], args["kv"], args["bt"], args["sl"], args["tk"],
                                 args["ws"], args["wsb"], args["out"], args["B"], args["Q"],
                                 args["Hq"], args["Hkv"], args["S"], args["NB"], args["sm"],
                                 args["ks"], args["vs"], args["splits"], None)


@pytest.mark.parametrize("kw", [
    dict(tk=None), dict(out=None), dict(out=ctypes.c_void_p((1 << 20) + 2)), dict(splits=-1),
    dict(splits=17), dict(vs=float("nan")), dict(Q=33), dict(Hq=48),
])
def test_sparse_decode_rejects(lib, kw):
    assert _decode(lib, **kw) == EINVAL


def test_select_attend_rejects_missing_scores(lib):
    f = lib.msa_sparse_decode_select
    assert f(A, A, A, A, None, 0, 0, 1, A, None, 0, A, 16, 4, 64, 4, 8, 100, 0.088, 1.0, 1.0, 1,
             None) == EINVAL
    assert f(A, A, A, A, ctypes.c_void_p((1 << 20) + 2), 0, 0, 1, A, None, 0, A, 16, 4, 64, 4, 8,
             100, 0.088, 1.0, 1.0, 1, None) == EINVAL      # misaligned scores
    assert f(A, A, A, A, A, 0, 0, -1, A, None, 0, A, 16, 4, 64, 4, 8, 100, 0.088, 1.0, 1.0, 1,
             None) == EINVAL                               # negative stride


def test_topk_rejects(lib):
    f = lib.msa_topk
    assert f(A, 0, 0, 1, A, A, 16, 4, 4, 8, 8, None) == EINVAL       # k != 16
    assert f(A, 0, 0, 1, A, A, 16, 0, 4, 8, 16, None) == EINVAL      # Q = 0
    assert f(None, 0, 0, 1, A, A, 16, 4, 4, 8, 16, None) == EINVAL
    assert f(A, 0, 0, 1, A, None, 16, 4, 4, 8, 16, None) == EINVAL
    assert f(A, 0, 0, 1, A, A, 0, 4, 4, 8, 16, None) == 0            # empty batch


def test_combine_rejects(lib):
    f = lib.msa_combine
    assert f(A, A, 64, 64, 0, None) == EINVAL
    assert f(A, A, 64, 64, 17, None) == EINVAL
    assert f(None, A, 64, 64, 2, None) == EINVAL
    assert f(A, A, 0, 64, 2, None) == 0


def test_valid_call_without_a_device_fails_cleanly(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a device is present")
    assert _score(lib) == _native.ECUDA


def test_dense_splits_rule(lib):
    # min(16, ceil(S / 16)) splits of ceil(S / splits) blocks; ranges over 128
    # blocks (S > 2048) are not taken
    assert lib.msa_dense_splits(0) == 0
    assert lib.msa_dense_splits(1) == 1
    assert lib.msa_dense_splits(16) == 1
    assert lib.msa_dense_splits(17) == 2
    assert lib.msa_dense_splits(255) == 16
    assert lib.msa_dense_splits(2048) == 16
    assert lib.msa_dense_splits(2049) == 0


def test_dense_decode_rejects(lib):
    f = lib.msa_dense_decode
    ok = dict(q=A, kv=A, bt=A, sl=A, ws=A, wsb=1 << 30, out=A, B=16, Q=4, Hq=64, Hkv=4, S=8,
              NB=100, sm=0.088, ks=1.0, vs=1.0)

    def call(**kw):
        a = dict(ok, **kw)
        return f(a["q"], a["kv"], a["bt"], a["sl"], a["ws"], a["wsb"], a["out"], a["B"], a["Q"],
                 a["Hq"], a["Hkv"], a["S"], a["NB"], a["sm"], a["ks"], a["vs"], None)

    assert call(S=2049) == EINVAL                   # a split would span more than 128 blocks
    assert call(out=None) == EINVAL
    assert call(Q=33) == EINVAL
    assert call(vs=float("nan")) == EINVAL
    assert call(B=0) == 0                           # empty batch


def test_fp8_query_entry_points_reject_bad_scales(lib):
    for qs in (0.0, -1.0, float("inf"), float("nan")):
        assert lib.msa_score_q8(A, qs, A, A, A, A, 16, 4, 64, 4, 8, 100, 0.088, 1.0, None) == EINVAL
        assert lib.msa_sparse_decode_q8(A, qs, A, A, A, A, None, 0, A, 16, 4, 64, 4, 8, 100, 0.088,
                                        1.0, 1.0, 1, None) == EINVAL
        assert lib.msa_dense_decode_q8(A, qs, A, A, A, A, 1 << 30, A, 16, 4, 64, 4, 8, 100, 0.088,
                                       1.0, 1.0, None) == EINVAL
    assert lib.msa_sparse_decode_select_q8(A, 1.0, A, A, A, None, 0, 0, 1, A, None, 0, A, 16, 4, 64,
                                           4, 8, 100, 0.088, 1.0, 1.0, 1, None) == EINVAL


def test_prefill_rejects(lib):
    f = lib.msa_sparse_prefill
    ok = dict(kv=A, bt=A, sl=A, cu=A, tk=A, ws=None, wsb=0, out=A, B=3, T=505, Hq=64, Hkv=4,
              S=9, NB=100, sm=0.088, ks=1.0, vs=1.0, splits=1)

    def call(fn=f, q=(A,), **kw):   # q: (q,) or, for the _q8 entry, (q8, q_scale)
        a = dict(ok, **kw)
        return fn(*q, a["kv"], a["bt"], a["sl"], a["cu"], a["tk"], a["ws"], a["wsb"], a["out"],
                  a["B"], a["T"], a["Hq"], a["Hkv"], a["S"], a["NB"], a["sm"], a["ks"], a["vs"],
                  a["splits"], None)

    assert call(cu=None) == EINVAL
    assert call(cu=ctypes.c_void_p((1 << 20) + 2)) == EINVAL     # misaligned cu_seqlens_q
    assert call(tk=None) == EINVAL
    assert call(T=-1) == EINVAL
    assert call(T=(1 << 31) - 1) == EINVAL
    assert call(B=0) == EINVAL                                    # tokens but no request
    assert call(T=0) == EINVAL                                    # requests but no token
    assert call(B=0, T=0) == 0                                    # empty batch
    assert call(Hq=48) == EINVAL
    assert call(splits=17) == EINVAL
    # no query-length bound: a single request of 40000 tokens passes the host checks
    import torch
    if not torch.cuda.is_available():
        assert call(B=1, T=40000) == _native.ECUDA
    for qs in (0.0, -1.0, float("nan")):
        assert call(lib.msa_sparse_prefill_q8, (A, qs)) == EINVAL
    assert call(q=(None,)) == EINVAL
    g = lib.msa_sparse_prefill_select
    assert g(A, A, A, A, A, None, 0, 0, 1, A, None, 0, A, 3, 505, 64, 4, 9, 100, 0.088, 1.0, 1.0,
             1, None) == EINVAL                                   # no scores
    assert g(A, A, A, A, None, A, 0, 0, 1, A, None, 0, A, 3, 505, 64, 4, 9, 100, 0.088, 1.0, 1.0,
             1, None) == EINVAL                                   # no cu_seqlens_q
    assert lib.msa_sparse_prefill_select_q8(A, 0.0, A, A, A, A, A, 0, 0, 1, A, None, 0, A, 3, 505,
                                            64, 4, 9, 100, 0.088, 1.0, 1.0, 1, None) == EINVAL


def test_k_only_cache_scorer_rejects(lib):
    f = lib.msa_score_kcache
    assert f(A, None, A, A, A, 16, 4, 64, 4, 8, 100, 0.088, 1.0, None) == EINVAL   # no cache
    assert f(A, A, A, A, None, 16, 4, 64, 4, 8, 100, 0.088, 1.0, None) == EINVAL   # no scores
    assert f(A, A, A, A, A, 16, 33, 64, 4, 8, 100, 0.088, 1.0, None) == EINVAL     # qlen 33
    assert f(A, A, A, A, A, 0, 4, 64, 4, 8, 100, 0.088, 1.0, None) == 0            # empty batch
    for qs in (0.0, -1.0, float("nan")):
        assert lib.msa_score_kcache_q8(A, qs, A, A, A, A, 16, 4, 64, 4, 8, 100, 0.088, 1.0,
                                       None) == EINVAL


def test_wait_timeout_limit_checked_on_the_host(lib):
    """msa_test_wait_timeout rejects limits outside [1 us, 2 s] before anything
    reaches a device."""
    for limit in (0, 999, 2_000_000_001, 2**63):
        assert lib.msa_test_wait_timeout(limit, None) == _native.EINVAL


def test_process_wide_switches_return_the_previous_setting(lib):
    """msa_set_union_tile, msa_set_input_overlap: each returns the setting it
    replaces (any non-zero argument turns it on), and both start off."""
    for fn in (lib.msa_set_union_tile, lib.msa_set_input_overlap):
        first = fn(0)
        assert first == 0
        assert fn(7) == 0
        assert fn(1) == 1
        assert fn(0) == 1
        assert fn(0) == 0
