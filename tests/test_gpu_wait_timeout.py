"""The bounded-wait exit of the library's kernels, taken on purpose.

msa_test_wait_timeout enqueues a kernel that holds tensor memory and a bulk
copy in flight while it waits, with a short limit, on an mbarrier that nothing
completes.  The call must return, the error word must carry the timeout flag,
and the context must stay usable: an attend enqueued after it matches the
oracle and flags nothing."""
from __future__ import annotations

import ctypes
import time

import numpy as np
import pytest
import torch

import block_sparse_gqa_score_gb300 as msa
import oracle
from block_sparse_gqa_score_gb300 import _native, build
from block_sparse_gqa_score_gb300 import workloads as wl
from tests.helpers import assert_out_close, padding_rows, to_problem

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _lib():
    build.build()
    return _native.load()


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def test_wait_limit_rejects_out_of_range():
    lib = _lib()
    assert lib.msa_test_wait_timeout(10, _stream()) == _native.EINVAL
    assert lib.msa_test_wait_timeout(5_000_000_000, _stream()) == _native.EINVAL


def test_expired_wait_flags_timeout_and_leaves_context_usable():
    lib = _lib()
    torch.cuda.synchronize()
    msa.get_error(clear=True)
    limit_ns = 50_000_000                       # 50 ms
    t0 = time.perf_counter()
    assert lib.msa_test_wait_timeout(limit_ns, _stream()) == 0
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert elapsed >= limit_ns * 1e-9 * 0.9     # it waited ...
    assert elapsed < 10.0                       # ... and it returned
    assert msa.get_error(clear=True) == _native.ERR_TIMEOUT
    assert msa.get_error() == 0                 # cleared

    # the same context runs the attend as usual afterwards (tensor memory freed)
    seq_lens, Q, Hq, Hkv = [3000, 9000, 1], 4, 64, 4
    inp = wl.make_custom(seq_lens, Q, Hq, Hkv, seed=431, device=DEV, kv_std=0.5,
                         kv_scale_mode="amax")
    lists = wl.draw_topk_given(seq_lens, Q, Hkv, torch.Generator().manual_seed(3))
    out = msa.sparse_decode(inp.q, inp.kv, inp.block_table, inp.seq_lens, lists.to(DEV), Q,
                            inp.sm_scale, inp.k_scale, inp.v_scale, num_splits=3)
    ref = oracle.attend(to_problem(inp, oracle), lists.numpy())
    assert_out_close(out.float().cpu().numpy().astype(np.float64), ref,
                     padding_rows(seq_lens, Q))
    assert msa.get_error() == 0


def test_repeated_expired_waits_do_not_leak_tensor_memory():
    """Each expired wait frees its tensor memory: many in a row leave the
    512-column allocator free for the union attend, which takes all of it."""
    lib = _lib()
    msa.get_error(clear=True)
    for _ in range(8):
        assert lib.msa_test_wait_timeout(1_000_000, _stream()) == 0
    torch.cuda.synchronize()
    assert msa.get_error(clear=True) == _native.ERR_TIMEOUT
    prev = msa.set_union_tile(True)
    try:
        seq_lens, Q, Hq, Hkv = [5000, 700], 4, 64, 4
        inp = wl.make_custom(seq_lens, Q, Hq, Hkv, seed=432, device=DEV, kv_std=0.5,
                             kv_scale_mode="amax")
        lists = wl.draw_topk_given(seq_lens, Q, Hkv, torch.Generator().manual_seed(5))
        out = msa.sparse_decode(inp.q, inp.kv, inp.block_table, inp.seq_lens, lists.to(DEV), Q,
                                inp.sm_scale, inp.k_scale, inp.v_scale, num_splits=2)
        ref = oracle.attend(to_problem(inp, oracle), lists.numpy())
        assert_out_close(out.float().cpu().numpy().astype(np.float64), ref,
                         padding_rows(seq_lens, Q))
        assert msa.get_error() == 0
    finally:
        msa.set_union_tile(prev)
