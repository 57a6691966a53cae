"""Stream order of the library calls (include/msa.h, "Stream order"): with the
default setting a call reads the inputs that kernels enqueued just before it on
the same stream wrote, with no synchronisation in between.

Each test fills the input buffers with stale values, then enqueues on one
stream: a kernel that spins for about a millisecond, in-place writes of the
final q, seq_lens, current K|V pages (and top-k lists), and the library call.
The result must be the oracle's on the final inputs."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import block_sparse_gqa_score_gb300 as msa
import oracle
from block_sparse_gqa_score_gb300 import workloads as wl
from tests.helpers import assert_out_close, assert_scores_close, to_problem

pytestmark = pytest.mark.gpu
DEV = "cuda"
SPIN_CYCLES = 2_000_000


@pytest.fixture(autouse=True)
def _default_order():
    prev = msa.set_input_overlap(False)
    msa.get_error(clear=True)
    yield
    msa.set_input_overlap(prev)


def _np(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def _current_pages(inp):
    """Physical pages of each request's current (last) block."""
    bt = inp.block_table.cpu()
    return torch.tensor([int(bt[b, (L - 1) // 128]) for b, L in enumerate(inp.seq_lens_list)
                         if L > 0], dtype=torch.long)


def _stale_copies(inp, seed):
    """Stale q, seq_lens and current pages, and the final values to write."""
    g = torch.Generator(device=DEV).manual_seed(seed)
    final = {"q": inp.q.clone(), "seq_lens": inp.seq_lens.clone(),
             "pages": inp.kv[_current_pages(inp).to(DEV)].clone()}
    stale_q = torch.randn(inp.q.shape, generator=g, device=DEV).to(torch.bfloat16)
    # shorter sequences (the tokens being appended not yet counted)
    stale_lens = torch.clamp(inp.seq_lens - 3, min=1)
    stale_pages = torch.randint(0, 0x7E, final["pages"].shape, generator=g, device=DEV,
                                dtype=torch.int32).to(torch.uint8)
    return final, stale_q, stale_lens, stale_pages


def _write_final_after_spin(inp, final, pages_idx):
    torch.cuda._sleep(SPIN_CYCLES)
    inp.q.copy_(final["q"])
    inp.seq_lens.copy_(final["seq_lens"])
    inp.kv.index_copy_(0, pages_idx, final["pages"])


@pytest.mark.parametrize("seq_lens,Q,Hq,Hkv", [
    ([3000, 9000, 700, 5000], 4, 64, 4),
    ([2050, 60000, 300], 2, 16, 1),        # 469 blocks: selection fused into the attend
    ([70000, 66000], 1, 16, 1),            # 547 blocks: the selector kernel, then the attend
])
def test_decode_step_reads_inputs_written_just_before(seq_lens, Q, Hq, Hkv):
    inp = wl.make_custom(seq_lens, Q, Hq, Hkv, seed=301, device=DEV, kv_std=0.5,
                         kv_scale_mode="amax")
    s_ref, t_ref, o_ref = oracle.decode_step(to_problem(inp, oracle))
    final, stale_q, stale_lens, stale_pages = _stale_copies(inp, 302)
    pages_idx = _current_pages(inp).to(DEV)
    bufs = msa.DecodeBuffers.allocate(len(seq_lens), Q, Hq, Hkv, inp.stride, DEV)
    for _ in range(2):      # the second round runs after a finished step on the same buffers
        inp.q.copy_(stale_q)
        inp.seq_lens.copy_(stale_lens)
        inp.kv.index_copy_(0, pages_idx, stale_pages)
        bufs.out.fill_(float("nan"))
        torch.cuda.synchronize()
        _write_final_after_spin(inp, final, pages_idx)
        scores, topk, out = msa.decode_step(inp.q, inp.kv, inp.block_table, inp.seq_lens, Q,
                                            inp.sm_scale, inp.k_scale, inp.v_scale, buffers=bufs)
        torch.cuda.synchronize()
        assert_scores_close(scores.cpu().numpy().astype(np.float64), s_ref)
        assert np.array_equal(topk.cpu().numpy(), t_ref)
        assert_out_close(_np(out), o_ref)
    assert msa.get_error() == 0


def test_separate_calls_read_inputs_written_just_before():
    """msa_score, msa_topk and msa_sparse_decode called one by one, each right
    after writes of its own inputs (the top-k lists for the attend)."""
    seq_lens, Q, Hq, Hkv = [4000, 12000, 900], 4, 64, 4
    inp = wl.make_custom(seq_lens, Q, Hq, Hkv, seed=303, device=DEV, kv_std=0.5,
                         kv_scale_mode="amax")
    p = to_problem(inp, oracle)
    s_ref = oracle.score(p)
    given = wl.draw_topk_given(seq_lens, Q, Hkv, torch.Generator().manual_seed(5))
    o_ref = oracle.attend(p, given.numpy())
    final, stale_q, stale_lens, stale_pages = _stale_copies(inp, 304)
    pages_idx = _current_pages(inp).to(DEV)
    inp.q.copy_(stale_q)
    inp.seq_lens.copy_(stale_lens)
    inp.kv.index_copy_(0, pages_idx, stale_pages)
    torch.cuda.synchronize()
    _write_final_after_spin(inp, final, pages_idx)
    scores = msa.score(inp.q, inp.kv, inp.block_table, inp.seq_lens, Q, inp.sm_scale, inp.k_scale)
    torch.cuda._sleep(SPIN_CYCLES)
    scores_view = scores.clone()     # a torch kernel between the scorer and the selector
    topk = msa.topk(scores_view, inp.seq_lens, Q)
    lists = torch.full_like(topk, -1)
    torch.cuda._sleep(SPIN_CYCLES)
    lists.copy_(given.to(DEV))
    out = msa.sparse_decode(inp.q, inp.kv, inp.block_table, inp.seq_lens, lists, Q, inp.sm_scale,
                            inp.k_scale, inp.v_scale, num_splits=3)
    torch.cuda.synchronize()
    assert_scores_close(scores.cpu().numpy().astype(np.float64), s_ref)
    assert np.array_equal(topk.cpu().numpy(),
                          oracle.topk(scores.cpu().numpy().astype(np.float64),
                                      np.array(seq_lens, dtype=np.int32), Q))
    assert_out_close(_np(out), o_ref)
    assert msa.get_error() == 0
