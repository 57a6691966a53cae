"""msa_sparse_decode_static: the allocation-free entry point, for callers that
only hold the step's inputs and outputs and cannot allocate device memory (no
workspace from their host interface, no cudaMalloc on their hot path).

It is checked through the C ABI against msa_sparse_decode on the same inputs,
on two calls in a row (the scratch array keeps the previous call's contents,
which must not leak into the next result).  This file sorts last so that a
run stopping at its first failure has already run every other test."""
from __future__ import annotations

import ctypes

import numpy as np
import pytest
import torch

from block_sparse_gqa_score_gb300 import _native, build
from block_sparse_gqa_score_gb300 import workloads as wl
from tests.helpers import OUT_MAX_ABS, OUT_MEAN_ABS

pytestmark = pytest.mark.gpu
DEV = "cuda"
STATIC_SCRATCH_BYTES = 4 << 20


def _lib():
    build.build()
    return _native.load()


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _call_static(lib, inp, topk, out, splits):
    return lib.msa_sparse_decode_static(
        inp.q.data_ptr(), inp.kv.data_ptr(), inp.block_table.data_ptr(), inp.seq_lens.data_ptr(),
        topk.data_ptr(), out.data_ptr(), inp.batch, inp.qlen, inp.num_q_heads, inp.num_kv_heads,
        inp.stride, inp.num_blocks, inp.sm_scale, inp.k_scale, inp.v_scale, splits, _stream())


def _call_with_workspace(lib, inp, topk, out, splits):
    need = lib.msa_workspace_bytes(inp.batch, inp.qlen, inp.num_q_heads, splits)
    ws = torch.empty(max(need, 16), dtype=torch.uint8, device=DEV)
    st = lib.msa_sparse_decode(
        inp.q.data_ptr(), inp.kv.data_ptr(), inp.block_table.data_ptr(), inp.seq_lens.data_ptr(),
        topk.data_ptr(), ws.data_ptr(), need, out.data_ptr(), inp.batch, inp.qlen,
        inp.num_q_heads, inp.num_kv_heads, inp.stride, inp.num_blocks, inp.sm_scale, inp.k_scale,
        inp.v_scale, splits, _stream())
    torch.cuda.synchronize()
    return st


def _close(a: torch.Tensor, b: torch.Tensor):
    d = (a.float() - b.float()).abs()
    assert torch.isfinite(a.float()).all()
    assert d.max().item() <= OUT_MAX_ABS and d.mean().item() <= OUT_MEAN_ABS


CASES = [
    # seq_lens, qlen, Hq, Hkv, splits (0 = library's choice)
    ([2048, 3000], 1, 16, 1, 0),
    ([700, 20000, 5, 9000], 4, 64, 4, 3),
]


def test_static_scratch_matches_workspace_path_on_two_calls_in_a_row():
    lib = _lib()
    for seq_lens, Q, Hq, Hkv, splits in CASES:
        inp = wl.make_custom(seq_lens, Q, Hq, Hkv, seed=211, device=DEV, kv_std=0.5,
                             kv_scale_mode="amax")
        topk = wl.draw_topk_given(seq_lens, Q, Hkv, torch.Generator().manual_seed(3)).to(DEV)
        want = torch.empty_like(inp.q)
        assert _call_with_workspace(lib, inp, topk, want, splits or
                                    lib.msa_choose_splits(inp.batch, Q, Hkv,
                                    torch.cuda.get_device_properties(0).multi_processor_count)) == 0
        for _ in range(2):
            got = torch.full_like(inp.q, float("nan"))
            assert _call_static(lib, inp, topk, got, splits) == 0
            torch.cuda.synchronize()
            _close(got, want)


def test_static_scratch_rejects_shapes_beyond_its_size():
    lib = _lib()
    inp = wl.make_custom([4096] * 16, 32, 64, 4, seed=212, device=DEV)
    topk = wl.draw_topk_given(inp.seq_lens_list, 32, 4, torch.Generator().manual_seed(1)).to(DEV)
    out = torch.zeros_like(inp.q)
    need = lib.msa_workspace_bytes(16, 32, 64, 16)
    assert need > STATIC_SCRATCH_BYTES
    assert _call_static(lib, inp, topk, out, 16) == _native.ENOSPC
    assert torch.count_nonzero(out).item() == 0           # nothing was enqueued
    assert _call_static(lib, inp, topk, out, 1) == 0      # one split needs no scratch
    torch.cuda.synchronize()
    ref = torch.empty_like(inp.q)
    assert _call_with_workspace(lib, inp, topk, ref, 1) == 0
    _close(out, ref)
