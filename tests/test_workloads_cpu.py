"""The seeded input generators (shared by the CUDA path and the oracle):
the structure each input promises, checked on the CPU."""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

from block_sparse_gqa_score_gb300 import workloads as wl


def test_paged_layout_is_a_permutation_with_zero_tails():
    seq_lens = [300, 0, 129, 4000, 1]
    bt, nb = wl.paged_layout(seq_lens, torch.Generator().manual_seed(1), min_stride=40)
    pages = [math.ceil(L / 128) for L in seq_lens]
    assert nb == sum(pages) and bt.shape == (5, 40)
    used = torch.cat([bt[b, :n] for b, n in enumerate(pages)])
    assert sorted(used.tolist()) == list(range(nb))            # every page once
    for b, n in enumerate(pages):
        assert torch.all(bt[b, n:] == 0)


@pytest.mark.parametrize("q_lens,seq_lens", [([4, 4, 4], [3000, 100, 20000]),
                                             ([300, 0, 77, 1], [300, 50, 1100, 70000])])
def test_drawn_lists_hold_the_current_block_and_distinct_earlier_ones(q_lens, seq_lens):
    t = wl.draw_topk_varlen(q_lens, seq_lens, 2, torch.Generator().manual_seed(2)).numpy()
    assert t.shape == (sum(q_lens), 2, 16)
    i = 0
    for L, n in zip(seq_lens, q_lens):
        for j in range(n):
            pos = L - n + j
            for g in range(2):
                row = t[i, g]
                kept = row[row >= 0]
                assert np.all(row[len(kept):] == -1)           # -1 only at the tail
                cur = pos // 128
                assert len(kept) == min(16, cur + 1)
                assert kept[-1] == cur and np.all(np.diff(kept) > 0)
            i += 1


def test_uniform_lengths_draw_the_same_lists_as_the_varlen_drawer():
    a = wl.draw_topk_given([3000, 900], 3, 2, torch.Generator().manual_seed(3))
    b = wl.draw_topk_varlen([3, 3], [3000, 900], 2, torch.Generator().manual_seed(3))
    assert torch.equal(a, b)


def test_all_visible_lists_cover_every_visible_page():
    # request 0: 129 tokens with a 2-token chunk (positions 127 and 128);
    # request 1: a single token (position 0)
    t = wl.all_visible_lists_varlen([2, 1], [129, 1], 1, 4).numpy()
    for i, pos in enumerate([127, 128, 0]):
        row = t[i, 0]
        assert row.tolist() == list(range(pos // 128 + 1)) + [-1] * (3 - pos // 128)


def test_prefill_inputs_offsets_and_rejects():
    inp = wl.make_prefill([3, 0, 5], [10, 4, 700], 16, 1, seed=4)
    assert inp.cu_seqlens_q.tolist() == [0, 3, 3, 8]
    assert inp.tokens == 8 and tuple(inp.q.shape) == (8, 16, 128)
    assert inp.q_lens == [3, 0, 5] and inp.qlen == 0
    with pytest.raises(ValueError):
        wl.make_prefill([11], [10], 16, 1, seed=4)


def test_inputs_are_seeded_and_layers_differ():
    a = wl.make_inputs("tiny_b2_q1_h16kv1_2k3k", layer=0)
    b = wl.make_inputs("tiny_b2_q1_h16kv1_2k3k", layer=0)
    c = wl.make_inputs("tiny_b2_q1_h16kv1_2k3k", layer=1)
    assert torch.equal(a.q, b.q) and torch.equal(a.kv, b.kv)
    assert torch.equal(a.block_table, b.block_table)
    assert a.seq_lens_list == c.seq_lens_list                 # lengths: per workload
    assert not torch.equal(a.kv, c.kv)                        # values: per layer
