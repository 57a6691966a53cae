"""The sparse attend of decode steps with several query tokens per request,
which shares each page among a request's tokens (one pass over the union of a
4-token tile's lists).  Every case is compared element by element with the
oracle's attend on the same lists: lists of one request that are identical,
disjoint or partly overlapping, lists without the current block, tokens whose
positions straddle a block boundary, partial tiles (Q = 2, 3, 5, 7), padding
rows, split counts from 1 to more than the union has pages, an fp8 query,
the whole step against the per-token step, and a CUDA graph replayed after
its inputs change."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import block_sparse_gqa_score_gb300 as msa
import oracle
from block_sparse_gqa_score_gb300 import workloads as wl
from tests.helpers import assert_out_close, padding_rows, to_problem

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(autouse=True)
def _union_mode():
    prev = msa.set_union_tile(True)
    msa.get_error(clear=True)
    yield
    msa.set_union_tile(prev)


def _np(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def _lists(seq_lens, Q, Hkv, pattern, gen):
    """[T, Hkv, 16] lists of one overlap pattern between a request's tokens."""
    out = torch.full((len(seq_lens) * Q, Hkv, 16), -1, dtype=torch.int32)
    for b, L in enumerate(seq_lens):
        curs = [(L - Q + j) // 128 if L - Q + j >= 0 else -1 for j in range(Q)]
        c0 = min(c for c in curs if c >= 0) if any(c >= 0 for c in curs) else -1
        for g in range(Hkv):
            shared = torch.randperm(c0 + 1, generator=gen)[:16].tolist() if c0 >= 0 else []
            for j in range(Q):
                cur = curs[j]
                if cur < 0:
                    continue
                if pattern == "identical":          # the same blocks for every token
                    ids = shared
                elif pattern == "disjoint":         # block n only for token n % Q
                    ids = [n for n in range(cur + 1) if n % Q == j][-16:]
                elif pattern == "no_current":       # earlier blocks only, drawn per token
                    ids = torch.randperm(cur, generator=gen)[:16].tolist() if cur > 0 else []
                else:                               # partly overlapping: half shared
                    own = torch.randperm(cur + 1, generator=gen)[:8].tolist()
                    ids = list(dict.fromkeys([cur] + own + shared))[:16]
                ids = sorted(ids)
                out[b * Q + j, g, :len(ids)] = torch.tensor(ids, dtype=torch.int32)
    return out


PATTERNS = ["identical", "disjoint", "overlap", "no_current"]


@pytest.mark.parametrize("pattern", PATTERNS)
@pytest.mark.parametrize("Q", [2, 4, 7])
def test_union_attend_list_patterns(pattern, Q):
    seq_lens = [3000, 130 + Q, 9000, 1410, Q - 1, 700]   # 1410 - 4 straddles blocks 10 | 11
    Hq, Hkv = 64, 4
    inp = wl.make_custom(seq_lens, Q, Hq, Hkv, seed=401, device=DEV, kv_std=0.5,
                         kv_scale_mode="amax")
    lists = _lists(seq_lens, Q, Hkv, pattern, torch.Generator().manual_seed(Q))
    ref = oracle.attend(to_problem(inp, oracle), lists.numpy())
    for splits in (1, 2, 5):
        out = msa.sparse_decode(inp.q, inp.kv, inp.block_table, inp.seq_lens, lists.to(DEV), Q,
                                inp.sm_scale, inp.k_scale, inp.v_scale, num_splits=splits)
        assert_out_close(_np(out), ref, padding_rows(seq_lens, Q))
    assert msa.get_error() == 0


@pytest.mark.parametrize("Q,splits", [(3, 1), (4, 16), (5, 3), (32, 1)])
def test_union_attend_drawn_lists_and_splits(Q, splits):
    """Drawn lists (the current block and 15 earlier ones per token), short
    and padding rows, more splits than some unions have pages."""
    seq_lens = [40000, 300, 0, 2, 17000]
    Hq, Hkv = 32, 2
    inp = wl.make_custom(seq_lens, Q, Hq, Hkv, seed=402, device=DEV, kv_std=0.5,
                         kv_scale_mode="amax")
    lists = wl.draw_topk_given(seq_lens, Q, Hkv, torch.Generator().manual_seed(9))
    out = msa.sparse_decode(inp.q, inp.kv, inp.block_table, inp.seq_lens, lists.to(DEV), Q,
                            inp.sm_scale, inp.k_scale, inp.v_scale, num_splits=splits)
    ref = oracle.attend(to_problem(inp, oracle), lists.numpy())
    assert_out_close(_np(out), ref, padding_rows(seq_lens, Q))
    assert msa.get_error() == 0


def test_union_select_mode_matches_given_lists():
    """Selecting inside the kernel (one warp per token) gives the selector's
    lists and the same bits as attending those lists."""
    seq_lens, Q, Hq, Hkv = [5000, 33000, 129, 260], 4, 64, 4
    inp = wl.make_custom(seq_lens, Q, Hq, Hkv, seed=403, device=DEV, kv_std=0.5,
                         kv_scale_mode="amax")
    scores = msa.score(inp.q, inp.kv, inp.block_table, inp.seq_lens, Q, inp.sm_scale,
                       inp.k_scale)
    for splits in (1, 3):
        tk, out = msa.sparse_decode_select(inp.q, inp.kv, inp.block_table, inp.seq_lens, scores,
                                           Q, inp.sm_scale, inp.k_scale, inp.v_scale,
                                           num_splits=splits)
        want = oracle.topk(scores.cpu().numpy().astype(np.float64),
                           np.array(seq_lens, dtype=np.int32), Q)
        assert np.array_equal(tk.cpu().numpy(), want)
        sep = msa.sparse_decode(inp.q, inp.kv, inp.block_table, inp.seq_lens, tk, Q,
                                inp.sm_scale, inp.k_scale, inp.v_scale, num_splits=splits)
        assert torch.equal(out, sep)
        assert_out_close(_np(out), oracle.attend(to_problem(inp, oracle), want))
    assert msa.get_error() == 0


def test_union_flags_bad_entries_per_token():
    """A bad entry in one token's list is skipped for that token only."""
    seq_lens, Q, Hq, Hkv = [2000, 5000], 4, 16, 1
    inp = wl.make_custom(seq_lens, Q, Hq, Hkv, seed=404, device=DEV)
    lists = wl.draw_topk_given(seq_lens, Q, Hkv, torch.Generator().manual_seed(2))
    bad = lists.clone()
    bad[1, 0, 3] = 10_000          # beyond token 1's current block
    bad[6, 0, 5] = bad[6, 0, 4]    # listed twice by token 6
    clean = bad.clone()
    clean[1, 0, 3] = -1
    clean[6, 0, 5] = -1
    out = msa.sparse_decode(inp.q, inp.kv, inp.block_table, inp.seq_lens, bad.to(DEV), Q,
                            inp.sm_scale, inp.k_scale, inp.v_scale, num_splits=2)
    flags = msa.get_error()
    assert flags & msa._native.ERR_TOPK_RANGE and flags & msa._native.ERR_TOPK_DUP
    ref = oracle.attend(to_problem(inp, oracle), clean.numpy())
    assert_out_close(_np(out), ref)


def _fp8(inp):
    """The query quantised per tensor (scale = amax / 448) and the oracle
    problem for it: the fp8 codes as bf16 (exact) with sm_scale * q_scale."""
    from tests.helpers import q_bits
    qf = inp.q.float()
    q_scale = float(qf.abs().max()) / 448.0
    q8 = (qf / q_scale).to(torch.float8_e4m3fn)
    p = oracle.Problem(q_bits(q8.to(torch.bfloat16)), inp.kv.cpu().numpy(),
                       inp.block_table.cpu().numpy(), inp.seq_lens.cpu().numpy(), inp.qlen,
                       inp.num_q_heads, inp.num_kv_heads, inp.sm_scale * q_scale, inp.k_scale,
                       inp.v_scale)
    return q8, q_scale, p


def test_union_fp8_query_matches_oracle():
    """An fp8 query (value q8 * q_scale) through the union tile: the whole step
    (selection inside the union kernel) and the attend on given lists."""
    seq_lens, Q, Hq, Hkv = [7000, 260, 15000, 3], 4, 64, 4
    inp = wl.make_custom(seq_lens, Q, Hq, Hkv, seed=405, device=DEV, kv_std=0.5,
                         kv_scale_mode="amax")
    q8, qs, p = _fp8(inp)
    scores, tk, out = msa.decode_step(q8, inp.kv, inp.block_table, inp.seq_lens, Q, inp.sm_scale,
                                      inp.k_scale, inp.v_scale, q_scale=qs)
    s_gpu = _np(scores)
    assert np.array_equal(tk.cpu().numpy(),
                          oracle.topk(s_gpu, np.array(seq_lens, dtype=np.int32), Q))
    assert_out_close(_np(out), oracle.attend(p, tk.cpu().numpy()), padding_rows(seq_lens, Q))
    given = wl.draw_topk_given(seq_lens, Q, Hkv, torch.Generator().manual_seed(6))
    out2 = msa.sparse_decode(q8, inp.kv, inp.block_table, inp.seq_lens, given.to(DEV), Q,
                             inp.sm_scale, inp.k_scale, inp.v_scale, num_splits=3, q_scale=qs)
    assert_out_close(_np(out2), oracle.attend(p, given.numpy()), padding_rows(seq_lens, Q))
    assert msa.get_error() == 0


def test_union_step_agrees_with_the_per_token_step():
    """The whole step with and without the union tile: the same scores and
    lists (the scorer and selector are shared), outputs that both match the
    oracle."""
    seq_lens, Q, Hq, Hkv = [9000, 4100, 20000, 128], 4, 64, 4
    inp = wl.make_custom(seq_lens, Q, Hq, Hkv, seed=406, device=DEV, kv_std=0.5,
                         kv_scale_mode="amax")
    s_u, tk_u, out_u = msa.decode_step(inp.q, inp.kv, inp.block_table, inp.seq_lens, Q,
                                       inp.sm_scale, inp.k_scale, inp.v_scale)
    msa.set_union_tile(False)
    s_t, tk_t, out_t = msa.decode_step(inp.q, inp.kv, inp.block_table, inp.seq_lens, Q,
                                       inp.sm_scale, inp.k_scale, inp.v_scale)
    assert torch.equal(s_u, s_t)
    assert torch.equal(tk_u, tk_t)
    ref = oracle.attend(to_problem(inp, oracle), tk_t.cpu().numpy())
    assert_out_close(_np(out_u), ref, padding_rows(seq_lens, Q))
    assert_out_close(_np(out_t), ref, padding_rows(seq_lens, Q))
    assert msa.get_error() == 0


def test_union_graph_replay_after_inputs_change():
    """The union attend captured once in a CUDA graph (fixed split count and
    workspace), replayed after the lengths, the lists and the query change in
    place: the oracle's result on the new inputs."""
    Q, Hq, Hkv, splits = 4, 32, 2, 2
    lens_a, lens_b = [9000, 3000, 12000], [4000, 12800, 131]
    inp = wl.make_custom(lens_a, Q, Hq, Hkv, seed=407, device=DEV, kv_std=0.5, min_stride=110)
    lists = wl.draw_topk_given(lens_a, Q, Hkv, torch.Generator().manual_seed(7)).to(DEV)
    out = torch.empty_like(inp.q)
    ws = torch.empty(msa.workspace_bytes(3, Q, Hq, splits) or 1, dtype=torch.uint8, device=DEV)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        msa.sparse_decode(inp.q, inp.kv, inp.block_table, inp.seq_lens, lists, Q, inp.sm_scale,
                          inp.k_scale, inp.v_scale, out=out, num_splits=splits, workspace=ws)
        with torch.cuda.graph(graph, stream=s):
            msa.sparse_decode(inp.q, inp.kv, inp.block_table, inp.seq_lens, lists, Q,
                              inp.sm_scale, inp.k_scale, inp.v_scale, out=out,
                              num_splits=splits, workspace=ws)
    torch.cuda.synchronize()
    inp.seq_lens.copy_(torch.tensor(lens_b, dtype=torch.int32))
    lists.copy_(wl.draw_topk_given(lens_b, Q, Hkv, torch.Generator().manual_seed(8)))
    inp.q.copy_(torch.randn(inp.q.shape, generator=torch.Generator().manual_seed(9)).to(inp.q))
    torch.cuda.synchronize()
    graph.replay()
    torch.cuda.synchronize()
    p = to_problem(inp, oracle)
    assert_out_close(_np(out), oracle.attend(p, lists.cpu().numpy()), padding_rows(lens_b, Q))
    assert msa.get_error() == 0
