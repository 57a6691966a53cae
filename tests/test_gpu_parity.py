"""Parity of the CUDA path (through the C ABI) with the CPU oracle on the same
seeded inputs.  Bar: top-k bit-exact given identical scores; scores within
relative 1e-3; bf16 outputs within max-abs 2e-2 and mean-abs 2e-3, padding rows
exactly zero."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import block_sparse_gqa_score_gb300 as msa
import oracle
from block_sparse_gqa_score_gb300 import workloads as wl
from tests.helpers import (assert_out_close, assert_scores_close, index_problem, padding_rows,
                           prefill_oracle, q_bits, to_problem)

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(autouse=True)
def _clean_error_word():
    msa.get_error(clear=True)
    yield


def _np(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64) if t.dtype == torch.bfloat16 \
        else t.detach().cpu().numpy()


# The vLLM interleaved-cache test's shapes: seq_lens [257, 513] x pairs with
# qlen in {1, 2, 3, 4, 8}, tp1 (64/4) and tp4 (16/1) head geometries, then the
# ragged update [129, 385]; plus short, padding and long rows of our own.
SMALL_CASES = [
    ([257, 513] * 2, 1, 64, 4),
    ([257, 513] * 2, 2, 64, 4),
    ([257, 513] * 2, 3, 64, 4),
    ([257, 513] * 2, 4, 16, 1),
    ([257, 513] * 2, 8, 64, 4),
    ([129, 385] * 2, 4, 64, 4),
    ([0, 2, 3, 130, 2048, 2049], 4, 16, 1),       # padding rows, page boundaries
    ([3000, 5000, 4100], 1, 32, 2),
    ([2500, 700], 32, 16, 1),                     # qlen at its upper bound
    ([6000, 1], 5, 64, 4),
    ([9000, 300], 16, 32, 2),                     # 256 query rows: one full MMA N
    ([5000, 17, 4500], 17, 16, 1),                # 272 rows: two MMA units of 9 + 8 tokens
]


@pytest.mark.parametrize("seq_lens,Q,Hq,Hkv", SMALL_CASES)
def test_score_matches_oracle(seq_lens, Q, Hq, Hkv):
    inp = wl.make_custom(seq_lens, Q, Hq, Hkv, seed=101, device=DEV, kv_std=0.5,
                         kv_scale_mode="amax", min_stride=3)
    gpu = msa.score(inp.q, inp.kv, inp.block_table, inp.seq_lens, Q, inp.sm_scale, inp.k_scale)
    ref = oracle.score(to_problem(inp, oracle))
    assert_scores_close(_np(gpu).astype(np.float64), ref)
    assert msa.get_error() == 0


@pytest.mark.parametrize("seq_lens,Q,Hq,Hkv", SMALL_CASES)
def test_topk_bit_exact_given_gpu_scores(seq_lens, Q, Hq, Hkv):
    inp = wl.make_custom(seq_lens, Q, Hq, Hkv, seed=102, device=DEV, min_stride=3)
    scores = msa.score(inp.q, inp.kv, inp.block_table, inp.seq_lens, Q, inp.sm_scale)
    got = msa.topk(scores, inp.seq_lens, Q)
    want = oracle.topk(_np(scores).astype(np.float64), np.array(seq_lens, dtype=np.int32), Q)
    assert np.array_equal(_np(got), want)


@pytest.mark.parametrize("S,cur_lo", [(40, 17), (300, 200), (3000, 2500)])
def test_topk_ties_and_strides(S, cur_lo):
    """Integer-valued scores force ties; the buffer is stored [Hkv, S, T] and
    read through its transposed view (arbitrary strides); S = 3000 exercises
    rows longer than the selector's shared-memory cache."""
    g = torch.Generator().manual_seed(S)
    B, Q, Hkv = 3, 4, 2
    seq_lens = torch.randint(cur_lo * 128, S * 128 - 4, (B,), generator=g).to(torch.int32)
    phys = torch.randint(-4, 5, (Hkv, S, B * Q), generator=g).float()
    phys[0, 5, :] = -0.0
    phys[1, 7, :] = 0.0
    scores = phys.to(DEV).transpose(1, 2)           # [Hkv, T, S] view
    got = msa.topk(scores, seq_lens.to(DEV), Q)
    want = oracle.topk(phys.double().numpy().transpose(0, 2, 1), seq_lens.numpy(), Q)
    assert np.array_equal(_np(got), want)


ATTEND_CASES = SMALL_CASES + [([20000, 9000, 40000], 4, 64, 4), ([70000], 2, 16, 1)]


@pytest.mark.parametrize("seq_lens,Q,Hq,Hkv", ATTEND_CASES)
@pytest.mark.parametrize("splits", [1, 3])
def test_attend_matches_oracle(seq_lens, Q, Hq, Hkv, splits):
    inp = wl.make_custom(seq_lens, Q, Hq, Hkv, seed=103, device=DEV, kv_std=0.5,
                         kv_scale_mode="amax")
    gen = torch.Generator().manual_seed(7)
    topk = wl.draw_topk_given(seq_lens, Q, Hkv, gen)
    out = msa.sparse_decode(inp.q, inp.kv, inp.block_table, inp.seq_lens, topk.to(DEV), Q,
                            inp.sm_scale, inp.k_scale, inp.v_scale, num_splits=splits)
    ref = oracle.attend(to_problem(inp, oracle), topk.numpy())
    assert_out_close(_np(out), ref, padding_rows(seq_lens, Q))
    assert msa.get_error() == 0


def test_attend_pages_all_visible_topk_graph_replay():
    """The vLLM test's flow: all-visible top-k for [257, 513], then ragged
    [129, 385] written in place, captured in a CUDA graph and replayed after
    the lengths change back."""
    Q, Hq, Hkv = 4, 64, 4
    lens_a, lens_b = [257, 513] * 8, [129, 385] * 8
    inp = wl.make_custom(lens_a, Q, Hq, Hkv, seed=104, device=DEV, kv_std=0.25)
    topk = wl.all_visible_topk(lens_a, Q, Hkv).to(DEV)
    out = torch.empty_like(inp.q)
    ws = torch.empty(msa.workspace_bytes(16, Q, Hq, 2) or 1, dtype=torch.uint8, device=DEV)

    def run():
        msa.sparse_decode(inp.q, inp.kv, inp.block_table, inp.seq_lens, topk, Q, inp.sm_scale,
                          out=out, num_splits=2, workspace=ws)

    run()
    assert_out_close(_np(out), oracle.attend(to_problem(inp, oracle), topk.cpu().numpy()))
    inp.seq_lens.copy_(torch.tensor(lens_b, dtype=torch.int32))
    topk.copy_(wl.all_visible_topk(lens_b, Q, Hkv))
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        run()                               # warm-up on the capture stream
        with torch.cuda.graph(graph, stream=s):
            run()
    torch.cuda.synchronize()
    inp.seq_lens.copy_(torch.tensor(lens_a, dtype=torch.int32))
    topk.copy_(wl.all_visible_topk(lens_a, Q, Hkv))
    out.zero_()
    graph.replay()
    torch.cuda.synchronize()
    inp.seq_lens_list = lens_a
    assert_out_close(_np(out), oracle.attend(to_problem(inp, oracle), topk.cpu().numpy()))


def test_split_counts_agree():
    inp = wl.make_custom([30000, 12000, 50000, 999], 4, 64, 4, seed=105, device=DEV)
    topk = wl.draw_topk_given(inp.seq_lens_list, 4, 4, torch.Generator().manual_seed(1)).to(DEV)
    outs = [msa.sparse_decode(inp.q, inp.kv, inp.block_table, inp.seq_lens, topk, 4,
                              inp.sm_scale, num_splits=s).float() for s in (1, 2, 5, 16)]
    for o in outs[1:]:
        assert (o - outs[0]).abs().max().item() <= 4e-3


def test_combine_matches_oracle():
    T, Hq, splits = 6, 32, 5
    g = torch.Generator().manual_seed(3)
    rows = T * Hq
    o = torch.randn((splits, rows, 128), generator=g, dtype=torch.float64)
    m = torch.randn((splits, rows), generator=g, dtype=torch.float64) * 4
    l = torch.rand((splits, rows), generator=g, dtype=torch.float64) * 10
    l[1, :7] = 0.0                          # empty parts
    m[1, :7] = -float("inf")
    l[:, 9] = 0.0                           # a row with every part empty
    m[:, 9] = -float("inf")
    ml = torch.stack([m, l], dim=-1)
    # a part whose maximum is NaN (l > 0) carries no softmax state: the merge
    # skips it, i.e. its row equals the merge with that part marked empty
    ml_nan = ml.clone()
    ml_nan[2, 11, 0] = float("nan")
    ml_ref = ml.clone()
    ml_ref[2, 11, 1] = 0.0
    ws = torch.cat([o.float().reshape(-1), ml_nan.float().reshape(-1)]).to(DEV)
    got = msa.combine(ws, T, Hq, splits)
    want = oracle.combine(o.float().double().numpy(), ml_ref.float().double().numpy())
    g = _np(got).reshape(rows, 128)
    # the merged rows are rounded to bf16 (8 significant bits): half an ulp is
    # 2^-9 relative; allow 2^-8 relative plus fp32 noise
    assert np.all(np.abs(g - want) <= 2.0 ** -8 * np.abs(want) + 1e-4)
    assert np.all(g[9] == 0)


def test_decode_step_tiny_workload_end_to_end():
    inp = wl.make_inputs("tiny_b2_q1_h16kv1_2k3k", device=DEV)
    scores, topk, out = msa.decode_step(inp.q, inp.kv, inp.block_table, inp.seq_lens, inp.qlen,
                                        inp.sm_scale, inp.k_scale, inp.v_scale)
    p = to_problem(inp, oracle)
    s_ref, t_ref, o_ref = oracle.decode_step(p)
    assert_scores_close(_np(scores).astype(np.float64), s_ref)
    assert np.array_equal(_np(topk), t_ref)
    assert_out_close(_np(out), o_ref)
    assert msa.get_error() == 0


def test_bad_indices_are_flagged_and_skipped():
    seq_lens = [1000, 600]
    inp = wl.make_custom(seq_lens, 1, 16, 1, seed=106, device=DEV)
    good = wl.all_visible_topk(seq_lens, 1, 1)
    bad = good.clone()
    bad[0, 0, 8] = 9          # cur is 7: out of range
    bad[1, 0, 5] = 2          # duplicate of slot 2
    out = msa.sparse_decode(inp.q, inp.kv, inp.block_table, inp.seq_lens, bad.to(DEV), 1,
                            inp.sm_scale)
    flags = msa.get_error()
    assert flags & msa._native.ERR_TOPK_RANGE and flags & msa._native.ERR_TOPK_DUP
    assert_out_close(_np(out), oracle.attend(to_problem(inp, oracle), good.numpy()))
    bt = inp.block_table.clone()
    bt[1, 1] = inp.num_blocks + 5
    msa.sparse_decode(inp.q, inp.kv, bt, inp.seq_lens, good.to(DEV), 1, inp.sm_scale)
    assert msa.get_error() & msa._native.ERR_PAGE_RANGE
    msa.score(inp.q, inp.kv, bt, inp.seq_lens, 1, inp.sm_scale)
    assert msa.get_error() & msa._native.ERR_PAGE_RANGE
    long = inp.seq_lens.clone()
    long[0] = inp.stride * 128 + 1
    msa.topk(torch.zeros((1, 2, inp.stride), device=DEV), long, 1)
    assert msa.get_error() & msa._native.ERR_SEQ_RANGE


@pytest.mark.parametrize("seq_lens,Q,Hq,Hkv", SMALL_CASES)
def test_select_attend_matches_the_separate_stages(seq_lens, Q, Hq, Hkv):
    """msa_sparse_decode_select selects inside the attend kernel: the lists are
    bit-exact against the oracle given the GPU's scores, and the output has the
    same bits as msa_sparse_decode on those lists."""
    inp = wl.make_custom(seq_lens, Q, Hq, Hkv, seed=107, device=DEV, kv_std=0.5,
                         kv_scale_mode="amax", min_stride=3)
    scores = msa.score(inp.q, inp.kv, inp.block_table, inp.seq_lens, Q, inp.sm_scale, inp.k_scale)
    splits = 3 if Q == 8 else 0
    tk, out = msa.sparse_decode_select(inp.q, inp.kv, inp.block_table, inp.seq_lens, scores, Q,
                                       inp.sm_scale, inp.k_scale, inp.v_scale, num_splits=splits)
    want = oracle.topk(_np(scores).astype(np.float64), np.array(seq_lens, dtype=np.int32), Q)
    assert np.array_equal(_np(tk), want)
    sep = msa.sparse_decode(inp.q, inp.kv, inp.block_table, inp.seq_lens, tk, Q, inp.sm_scale,
                            inp.k_scale, inp.v_scale, num_splits=splits)
    assert torch.equal(out, sep)
    assert msa.get_error() == 0


@pytest.mark.parametrize("S,cur_lo", [(40, 17), (300, 200), (700, 600)])
def test_select_attend_ties_and_strides(S, cur_lo):
    """Tie-heavy integer scores read through a transposed view; S = 700 takes
    the selector's path for rows longer than 512 candidates."""
    g = torch.Generator().manual_seed(S + 1)
    B, Q, Hq, Hkv = 3, 4, 32, 2
    seq_lens = torch.randint(cur_lo * 128, S * 128 - 4, (B,), generator=g).tolist()
    inp = wl.make_custom(seq_lens, Q, Hq, Hkv, seed=108, device=DEV, min_stride=S)
    assert inp.stride == S
    phys = torch.randint(-4, 5, (Hkv, S, B * Q), generator=g).float()
    phys[0, 5, :] = -0.0
    phys[1, 7, :] = 0.0
    scores = phys.to(DEV).transpose(1, 2)           # [Hkv, T, S] view
    tk, out = msa.sparse_decode_select(inp.q, inp.kv, inp.block_table, inp.seq_lens, scores, Q,
                                       inp.sm_scale)
    want = oracle.topk(phys.double().numpy().transpose(0, 2, 1), np.array(seq_lens, dtype=np.int32), Q)
    assert np.array_equal(_np(tk), want)
    sep = msa.sparse_decode(inp.q, inp.kv, inp.block_table, inp.seq_lens, tk, Q, inp.sm_scale)
    assert torch.equal(out, sep)
    assert msa.get_error() == 0


def test_attend_lists_without_the_current_block():
    """Lists that leave out the current block: the attend loads that block's
    page speculatively before it sees the list, and must then discard it (and
    start stage 0 over); the output must still match the oracle."""
    seq_lens, Q, Hq, Hkv = [3000, 9000, 17000, 700], 4, 64, 4
    inp = wl.make_custom(seq_lens, Q, Hq, Hkv, seed=109, device=DEV, kv_std=0.5,
                         kv_scale_mode="amax")
    topk = wl.draw_topk_given(seq_lens, Q, Hkv, torch.Generator().manual_seed(9))
    for i in range(len(seq_lens) * Q):
        b, j = divmod(i, Q)
        pos = seq_lens[b] - Q + j
        if pos < 0:
            continue
        cur = pos // 128
        row = topk[i]
        row[row == cur] = -1                          # drop the current block ...
        if i % 3 == 0 and cur >= 1:
            row[0, 0] = cur - 1 if (row[0] != cur - 1).all() else row[0, 0]  # ... some rows vary
    for splits in (1, 3):
        out = msa.sparse_decode(inp.q, inp.kv, inp.block_table, inp.seq_lens, topk.to(DEV), Q,
                                inp.sm_scale, inp.k_scale, inp.v_scale, num_splits=splits)
        ref = oracle.attend(to_problem(inp, oracle), topk.numpy())
        assert_out_close(_np(out), ref, padding_rows(seq_lens, Q))
        assert msa.get_error() == 0


DENSE_CASES = [
    ([2048, 3000], 1, 16, 1),                     # the tiny workload's shapes
    ([129, 385, 0, 7], 4, 64, 4),                 # units of 2, 4, 0 and 1 blocks, padding rows
    ([0, 2, 3, 130, 2048, 2049], 4, 16, 1),       # page boundaries
    ([2500, 700], 32, 16, 1),                     # qlen at its upper bound
    ([20000, 9000, 40000], 4, 64, 4),             # uneven units: 313 blocks in 16 parts, 71 in fewer
    ([70000], 2, 16, 1),                          # blocks past the prologue's table copy
    ([262144], 1, 16, 1),                         # the longest table: 16 splits of 128 blocks
    # lengths from 1 to 260000 tokens and a padding request: the units share
    # one CTA per SM by their blocks, from one part to the workspace's sixteen
    ([1, 131072, 0, 5000, 260000, 128, 129], 3, 32, 2),
    # more (request, tile, KV head) units than SMs: one CTA each
    ([1000 + 37 * b for b in range(40)], 8, 32, 2),
]


@pytest.mark.parametrize("seq_lens,Q,Hq,Hkv", DENSE_CASES)
def test_dense_decode_matches_oracle(seq_lens, Q, Hq, Hkv):
    """Dense decode against the oracle's attend over every visible block."""
    inp = wl.make_custom(seq_lens, Q, Hq, Hkv, seed=110, device=DEV, kv_std=0.5,
                         kv_scale_mode="amax")
    out = msa.dense_decode(inp.q, inp.kv, inp.block_table, inp.seq_lens, Q, inp.sm_scale,
                           inp.k_scale, inp.v_scale)
    lists = wl.all_visible_lists(seq_lens, Q, Hkv, inp.stride)
    ref = oracle.attend(to_problem(inp, oracle), lists.numpy())
    assert_out_close(_np(out), ref, padding_rows(seq_lens, Q))
    assert msa.get_error() == 0


@pytest.mark.parametrize("Q", [1, 4])
def test_dense_decode_equals_sparse_decode_on_short_rows(Q):
    """With at most 16 visible blocks per row, dense decode and the sparse
    attend over all-visible lists attend the same keys.  With one token per
    request both run one CTA per token over the same pages in the same order:
    the same bits.  With several, the sparse attend shares each page between
    the request's tokens (accumulating in another order): within the output
    tolerance of each other and of the oracle."""
    seq_lens, Hq, Hkv = [257, 513, 2048, 1, 0], 64, 4
    inp = wl.make_custom(seq_lens, Q, Hq, Hkv, seed=111, device=DEV, kv_std=0.5)
    dense = msa.dense_decode(inp.q, inp.kv, inp.block_table, inp.seq_lens, Q, inp.sm_scale,
                             inp.k_scale, inp.v_scale)
    topk = wl.all_visible_topk(seq_lens, Q, Hkv).to(DEV)
    sparse = msa.sparse_decode(inp.q, inp.kv, inp.block_table, inp.seq_lens, topk, Q,
                               inp.sm_scale, inp.k_scale, inp.v_scale, num_splits=1)
    if Q == 1:
        assert torch.equal(dense, sparse)
    else:
        ref = oracle.attend(to_problem(inp, oracle), topk.cpu().numpy())
        assert_out_close(_np(dense), ref, padding_rows(seq_lens, Q))
        assert_out_close(_np(sparse), ref, padding_rows(seq_lens, Q))
        assert_out_close(_np(sparse), _np(dense))
    assert msa.get_error() == 0


def test_dense_decode_graph_replay_after_lengths_change():
    """Captured once, replayed after seq_lens change (split count fixed by the
    table's stride): still the oracle's result."""
    Q, Hq, Hkv = 2, 32, 2
    lens_a, lens_b = [9000, 3000, 12000], [4000, 12800, 130]
    inp = wl.make_custom(lens_a, Q, Hq, Hkv, seed=112, device=DEV, kv_std=0.5, min_stride=100)
    out = torch.empty_like(inp.q)
    ws = torch.empty(msa.workspace_bytes(3, Q, Hq, msa.dense_splits(inp.stride)) or 1,
                     dtype=torch.uint8, device=DEV)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        msa.dense_decode(inp.q, inp.kv, inp.block_table, inp.seq_lens, Q, inp.sm_scale,
                         inp.k_scale, inp.v_scale, out=out, workspace=ws)
        with torch.cuda.graph(graph, stream=s):
            msa.dense_decode(inp.q, inp.kv, inp.block_table, inp.seq_lens, Q, inp.sm_scale,
                             inp.k_scale, inp.v_scale, out=out, workspace=ws)
    torch.cuda.synchronize()
    inp.seq_lens.copy_(torch.tensor(lens_b, dtype=torch.int32))
    torch.cuda.synchronize()
    graph.replay()
    torch.cuda.synchronize()
    ref = oracle.attend(to_problem(inp, oracle),
                        wl.all_visible_lists(lens_b, Q, Hkv, inp.stride).numpy())
    assert_out_close(_np(out), ref, padding_rows(lens_b, Q))
    assert msa.get_error() == 0


def _fp8_query(inp):
    """The query quantised per tensor (scale = amax / 448, as vLLM's
    scaled_fp8_quant with a dynamic scale), and the oracle problem for it: the
    fp8 codes as bf16 (exact) with sm_scale * q_scale."""
    qf = inp.q.float()
    q_scale = float(qf.abs().max()) / 448.0
    q8 = (qf / q_scale).to(torch.float8_e4m3fn)
    p = oracle.Problem(q_bits(q8.to(torch.bfloat16)), inp.kv.cpu().numpy(),
                       inp.block_table.cpu().numpy(), inp.seq_lens.cpu().numpy(), inp.qlen,
                       inp.num_q_heads, inp.num_kv_heads, inp.sm_scale * q_scale, inp.k_scale,
                       inp.v_scale)
    return q8, q_scale, p


FP8Q_CASES = [([257, 513] * 2, 4, 64, 4), ([0, 2, 3, 130, 2048, 2049], 4, 16, 1),
              ([2500, 700], 32, 16, 1), ([20000, 9000], 4, 64, 4)]


@pytest.mark.parametrize("seq_lens,Q,Hq,Hkv", FP8Q_CASES)
def test_fp8_query_matches_oracle(seq_lens, Q, Hq, Hkv):
    """msa_*_q8: an fp8 query of value q8 * q_scale through the scorer, the
    fused select-then-attend step, the attend on given lists and dense decode."""
    inp = wl.make_custom(seq_lens, Q, Hq, Hkv, seed=113, device=DEV, kv_std=0.5,
                         kv_scale_mode="amax")
    q8, qs, p = _fp8_query(inp)
    scores, tk, out = msa.decode_step(q8, inp.kv, inp.block_table, inp.seq_lens, Q, inp.sm_scale,
                                      inp.k_scale, inp.v_scale, q_scale=qs)
    s_gpu = _np(scores).astype(np.float64)
    assert_scores_close(s_gpu, oracle.score(p))
    assert np.array_equal(_np(tk), oracle.topk(s_gpu, np.array(seq_lens, dtype=np.int32), Q))
    assert_out_close(_np(out), oracle.attend(p, _np(tk)), padding_rows(seq_lens, Q))
    given = wl.draw_topk_given(seq_lens, Q, Hkv, torch.Generator().manual_seed(5))
    out2 = msa.sparse_decode(q8, inp.kv, inp.block_table, inp.seq_lens, given.to(DEV), Q,
                             inp.sm_scale, inp.k_scale, inp.v_scale, num_splits=2, q_scale=qs)
    assert_out_close(_np(out2), oracle.attend(p, given.numpy()), padding_rows(seq_lens, Q))
    out3 = msa.dense_decode(q8, inp.kv, inp.block_table, inp.seq_lens, Q, inp.sm_scale,
                            inp.k_scale, inp.v_scale, q_scale=qs)
    lists = wl.all_visible_lists(seq_lens, Q, Hkv, inp.stride).numpy()
    assert_out_close(_np(out3), oracle.attend(p, lists), padding_rows(seq_lens, Q))
    assert msa.get_error() == 0


# Every query length the scorer has its own instantiation for (the length
# compiled in), and a generic one on each side of them, bf16 and fp8: the
# two-CTA kernels up to qlen 7, the one-CTA kernels from qlen 8.
SCORE_QLENS = [(q, fp8) for q in (1, 2, 3, 4, 5, 6, 7, 8, 9, 16, 17, 32) for fp8 in (False, True)]


@pytest.mark.parametrize("Q,fp8", SCORE_QLENS)
def test_score_every_compiled_query_length(Q, fp8):
    """Scores against the oracle for each query length the scorer compiles in
    (and generic neighbours), with a bf16 or an fp8 query; rows straddle a
    unit boundary near the start of a CTA's range (short and long requests)."""
    seq_lens, Hq, Hkv = [700, 5000, 129, 2300], 32, 2
    inp = wl.make_custom(seq_lens, Q, Hq, Hkv, seed=140 + Q, device=DEV, kv_std=0.5,
                         kv_scale_mode="amax")
    if fp8:
        q8, qs, p = _fp8_query(inp)
        gpu = msa.score(q8, inp.kv, inp.block_table, inp.seq_lens, Q, inp.sm_scale, inp.k_scale,
                        q_scale=qs)
    else:
        p = to_problem(inp, oracle)
        gpu = msa.score(inp.q, inp.kv, inp.block_table, inp.seq_lens, Q, inp.sm_scale,
                        inp.k_scale)
    assert_scores_close(_np(gpu).astype(np.float64), oracle.score(p))
    assert msa.get_error() == 0


def test_dense_decode_skips_and_flags_a_bad_page():
    """A block-table entry out of range in dense decode: that block is skipped
    and MSA_ERR_PAGE_RANGE set; the rest equals the oracle over every other
    visible block (the current block's and an earlier block's entries)."""
    seq_lens, Q, Hq, Hkv = [9000, 3000], 2, 32, 2
    inp = wl.make_custom(seq_lens, Q, Hq, Hkv, seed=114, device=DEV, kv_std=0.5)
    for b, n in [(0, 20), (1, (seq_lens[1] - 1) // 128)]:   # an earlier block; a current one
        bt = inp.block_table.clone()
        bt[b, n] = inp.num_blocks + 3
        out = msa.dense_decode(inp.q, inp.kv, bt, inp.seq_lens, Q, inp.sm_scale, inp.k_scale,
                               inp.v_scale)
        assert msa.get_error() & msa._native.ERR_PAGE_RANGE
        lists = wl.all_visible_lists(seq_lens, Q, Hkv, inp.stride)
        sub = lists[b * Q:(b + 1) * Q]                # a view: the skipped block goes
        sub[sub == n] = -1
        assert_out_close(_np(out), oracle.attend(to_problem(inp, oracle), lists.numpy()),
                         padding_rows(seq_lens, Q))


def test_fp8_query_select_attend_with_splits():
    """The fused select-then-attend step with an fp8 query and two splits
    equals the separate selector and attend on the same query."""
    seq_lens, Q, Hq, Hkv = [20000, 9000, 300], 4, 64, 4
    inp = wl.make_custom(seq_lens, Q, Hq, Hkv, seed=115, device=DEV, kv_std=0.5,
                         kv_scale_mode="amax")
    q8, qs, p = _fp8_query(inp)
    scores = msa.score(q8, inp.kv, inp.block_table, inp.seq_lens, Q, inp.sm_scale, inp.k_scale,
                       q_scale=qs)
    tk, out = msa.sparse_decode_select(q8, inp.kv, inp.block_table, inp.seq_lens, scores, Q,
                                       inp.sm_scale, inp.k_scale, inp.v_scale, num_splits=2,
                                       q_scale=qs)
    tk2 = msa.topk(scores, inp.seq_lens, Q)
    assert torch.equal(tk, tk2)
    sep = msa.sparse_decode(q8, inp.kv, inp.block_table, inp.seq_lens, tk2, Q, inp.sm_scale,
                            inp.k_scale, inp.v_scale, num_splits=2, q_scale=qs)
    assert torch.equal(out, sep)
    assert_out_close(_np(out), oracle.attend(p, _np(tk)), padding_rows(seq_lens, Q))
    assert msa.get_error() == 0


# ----------------------------------------------------------------------------- prefill

# The vLLM prefill test's batch in both head geometries (q_lens [300, 128, 77]
# over seq_lens [300, 640, 1100]: a fresh prompt, then two chunks over cached
# context), chunks over long contexts, and an empty request with a 70k one.
PREFILL_CASES = [
    ([300, 128, 77], [300, 640, 1100], 64, 4),
    ([300, 128, 77], [300, 640, 1100], 16, 1),
    ([64, 1, 200, 33], [20000, 9000, 5000, 33], 64, 4),
    ([5, 0, 7, 1], [500, 300, 900, 70000], 16, 1),
]


@pytest.mark.parametrize("q_lens,seq_lens,Hq,Hkv", PREFILL_CASES)
@pytest.mark.parametrize("splits", [1, 3])
def test_prefill_matches_oracle(q_lens, seq_lens, Hq, Hkv, splits):
    inp = wl.make_prefill(q_lens, seq_lens, Hq, Hkv, seed=121, device=DEV, kv_std=0.5,
                          kv_scale_mode="amax")
    topk = wl.draw_topk_varlen(q_lens, seq_lens, Hkv, torch.Generator().manual_seed(12))
    out = msa.sparse_prefill(inp.q, inp.kv, inp.block_table, inp.seq_lens, inp.cu_seqlens_q,
                             topk.to(DEV), inp.sm_scale, inp.k_scale, inp.v_scale,
                             num_splits=splits)
    assert_out_close(_np(out), prefill_oracle(inp, oracle, topk))
    assert msa.get_error() == 0


def test_prefill_fp8_query_all_visible_pages():
    """The vLLM prefill test's flow: fp8 query with q_scale, k_scale 0.5 and
    v_scale 2.0, every causally visible page listed, ending with the token's
    own page."""
    q_lens, seq_lens = [300, 128, 77], [300, 640, 1100]
    for Hq, Hkv in [(64, 4), (16, 1)]:
        inp = wl.make_prefill(q_lens, seq_lens, Hq, Hkv, seed=122, device=DEV, kv_std=0.25,
                              fp8_query=True)
        inp.k_scale, inp.v_scale = 0.5, 2.0
        topk = wl.all_visible_lists_varlen(q_lens, seq_lens, Hkv, 16)
        out = msa.sparse_prefill(inp.q, inp.kv, inp.block_table, inp.seq_lens,
                                 inp.cu_seqlens_q, topk.to(DEV), inp.sm_scale, inp.k_scale,
                                 inp.v_scale, q_scale=inp.q_scale)
        assert_out_close(_np(out), prefill_oracle(inp, oracle, topk))
        assert msa.get_error() == 0


@pytest.mark.parametrize("splits", [1, 2])
def test_prefill_with_equal_lengths_is_bit_identical_to_decode(splits):
    """Equal query lengths put prefill tokens at the decode positions, and both
    entry points then run one CTA per token over the same pages (the default
    decode attend): the same bits."""
    seq_lens, Q, Hq, Hkv = [20000, 9000, 300, 4100], 8, 64, 4
    inp = wl.make_custom(seq_lens, Q, Hq, Hkv, seed=123, device=DEV, kv_std=0.5)
    topk = wl.draw_topk_given(seq_lens, Q, Hkv, torch.Generator().manual_seed(13)).to(DEV)
    cu = torch.arange(len(seq_lens) + 1, dtype=torch.int32, device=DEV) * Q
    dec = msa.sparse_decode(inp.q, inp.kv, inp.block_table, inp.seq_lens, topk, Q, inp.sm_scale,
                            num_splits=splits)
    pre = msa.sparse_prefill(inp.q, inp.kv, inp.block_table, inp.seq_lens, cu, topk,
                             inp.sm_scale, num_splits=splits)
    assert torch.equal(dec, pre)
    scores = msa.score(inp.q, inp.kv, inp.block_table, inp.seq_lens, Q, inp.sm_scale)
    tk_d, dec_s = msa.sparse_decode_select(inp.q, inp.kv, inp.block_table, inp.seq_lens, scores,
                                           Q, inp.sm_scale, num_splits=splits)
    tk_p, pre_s = msa.sparse_prefill_select(inp.q, inp.kv, inp.block_table, inp.seq_lens, cu,
                                            scores, inp.sm_scale, num_splits=splits)
    assert torch.equal(tk_d, tk_p) and torch.equal(dec_s, pre_s)
    assert msa.get_error() == 0


@pytest.mark.parametrize("S", [40, 700])
def test_prefill_select_per_token_topk(S):
    """Per-token causal top-16 from tie-heavy integer scores read through a
    transposed view: lists bit-exact against the oracle, output identical to
    msa_sparse_prefill on those lists.  S = 700 takes the selector's path for
    rows longer than 512 candidates."""
    g = torch.Generator().manual_seed(S + 3)
    q_lens = [150, 0, 9, 1]
    seq_lens = [S * 128 - 7, 200, (S - 30) * 128, 300]
    inp = wl.make_prefill(q_lens, seq_lens, 32, 2, seed=124, device=DEV, min_stride=S)
    T = inp.tokens
    phys = torch.randint(-4, 5, (2, S, T), generator=g).float()
    scores = phys.to(DEV).transpose(1, 2)                  # [Hkv, T, S] view
    tk, out = msa.sparse_prefill_select(inp.q, inp.kv, inp.block_table, inp.seq_lens,
                                        inp.cu_seqlens_q, scores, inp.sm_scale, num_splits=2)
    want = oracle.topk_prefill(phys.double().numpy().transpose(0, 2, 1), seq_lens,
                               inp.cu_seqlens_q.cpu().numpy())
    assert np.array_equal(_np(tk), want)
    sep = msa.sparse_prefill(inp.q, inp.kv, inp.block_table, inp.seq_lens, inp.cu_seqlens_q, tk,
                             inp.sm_scale, num_splits=2)
    assert torch.equal(out, sep)
    assert msa.get_error() == 0


def test_prefill_flags_inconsistent_batches():
    """Tokens past cu_seqlens_q[B] and a request whose query is longer than
    its sequence are flagged MSA_ERR_SEQ_RANGE and written as zero rows; every
    other row is still the oracle's."""
    q_lens, seq_lens, Hq, Hkv = [40, 9, 30], [3000, 9, 700], 16, 1
    inp = wl.make_prefill(q_lens, seq_lens, Hq, Hkv, seed=125, device=DEV, kv_std=0.5)
    topk = wl.draw_topk_varlen(q_lens, seq_lens, Hkv, torch.Generator().manual_seed(14))
    ref = prefill_oracle(inp, oracle, topk)
    # cu_seqlens_q ends 10 tokens early: the last request has 20 query tokens
    # (positions 680 .. 699), and the 10 rows after it belong to no request
    cu = inp.cu_seqlens_q.clone()
    cu[-1] -= 10
    out = _np(msa.sparse_prefill(inp.q, inp.kv, inp.block_table, inp.seq_lens, cu, topk.to(DEV),
                                 inp.sm_scale, num_splits=2))
    assert msa.get_error() & msa._native.ERR_SEQ_RANGE
    assert np.all(out[69:] == 0.0)
    short = oracle.attend_prefill(q_bits(inp.q[:69]), inp.kv.cpu().numpy(),
                                  inp.block_table.cpu().numpy(), inp.seq_lens.cpu().numpy(),
                                  cu.cpu().numpy(), topk[:69].numpy(), Hq, Hkv, inp.sm_scale)
    assert_out_close(out[:69], short)
    assert np.array_equal(short[:49], ref[:49])
    # request 1 claims more query tokens than its sequence holds
    sl = inp.seq_lens.clone()
    sl[1] = 5
    out = _np(msa.sparse_prefill(inp.q, inp.kv, inp.block_table, sl, inp.cu_seqlens_q,
                                 topk.to(DEV), inp.sm_scale))
    assert msa.get_error() & msa._native.ERR_SEQ_RANGE
    z = np.zeros(inp.tokens, dtype=bool)
    z[40:49] = True
    assert np.all(out[z] == 0.0)
    assert_out_close(out[~z], ref[~z])


# ----------------------------------------------------------------------------- index-K cache

@pytest.mark.parametrize("seq_lens,Q,Hq,Hkv", [([257, 513] * 2, 4, 64, 4),
                                               ([0, 2, 3, 130, 2048, 2049], 4, 16, 1),
                                               ([2500, 700], 32, 16, 1),
                                               ([9000, 300], 16, 32, 2)])
def test_score_on_a_k_only_cache(seq_lens, Q, Hq, Hkv):
    """msa_score_kcache: scores on a K-only [NB, Hkv, 128, 128] cache are
    bit-identical to msa_score on a packed cache holding the same K bytes (any
    V), for a bf16 and an fp8 query, and match the oracle."""
    inp = wl.make_custom(seq_lens, Q, Hq, Hkv, seed=131, device=DEV, kv_std=0.5,
                         kv_scale_mode="amax", min_stride=3)
    k_only = inp.kv[..., :128].contiguous()
    got = msa.score(inp.q, k_only, inp.block_table, inp.seq_lens, Q, inp.sm_scale, inp.k_scale)
    want = msa.score(inp.q, inp.kv, inp.block_table, inp.seq_lens, Q, inp.sm_scale, inp.k_scale)
    assert torch.equal(got, want)
    inp.index_k, inp.index_k_scale = k_only, inp.k_scale
    assert_scores_close(_np(got).astype(np.float64), oracle.score(index_problem(inp, oracle)))
    q8, qs, _ = _fp8_query(inp)
    got8 = msa.score(q8, k_only, inp.block_table, inp.seq_lens, Q, inp.sm_scale, inp.k_scale,
                     q_scale=qs)
    want8 = msa.score(q8, inp.kv, inp.block_table, inp.seq_lens, Q, inp.sm_scale, inp.k_scale,
                      q_scale=qs)
    assert torch.equal(got8, want8)
    assert msa.get_error() == 0


def test_decode_step_scores_on_the_index_cache():
    """decode_step(index_k=...): blocks selected from scores on a separate
    K-only cache, attended on the K|V cache; the selection is bit-exact
    against the oracle's given the GPU's scores, the scores and the output
    match the oracle."""
    seq_lens, Q, Hq, Hkv = [20000, 9000, 300, 4100], 4, 64, 4
    inp = wl.make_custom(seq_lens, Q, Hq, Hkv, seed=132, device=DEV, kv_std=0.5,
                         kv_scale_mode="amax")
    inp.index_k, inp.index_k_scale = wl.draw_index_k(
        inp.num_blocks, Hkv, torch.Generator(device=DEV).manual_seed(133), DEV, std=0.5,
        scale_mode="amax")
    scores, tk, out = msa.decode_step(inp.q, inp.kv, inp.block_table, inp.seq_lens, Q,
                                      inp.sm_scale, inp.k_scale, inp.v_scale,
                                      index_k=inp.index_k, index_k_scale=inp.index_k_scale)
    s = _np(scores).astype(np.float64)
    assert_scores_close(s, oracle.score(index_problem(inp, oracle)))
    want = oracle.topk(s, np.array(seq_lens, dtype=np.int32), Q)
    assert np.array_equal(_np(tk), want)
    assert_out_close(_np(out), oracle.attend(to_problem(inp, oracle), want),
                     padding_rows(seq_lens, Q))
    assert msa.get_error() == 0


@pytest.mark.parametrize("B", [100, 1100])
def test_prefill_many_requests(B):
    """More requests than a warp has lanes: the token -> request search takes
    two (100 requests) and three (1100) rounds.  Ragged query lengths with
    empty requests and fresh prompts."""
    g = torch.Generator().manual_seed(B)
    seq_lens = torch.randint(1, 3000, (B,), generator=g).tolist()
    q_lens = [min(L, int(n)) for L, n in zip(seq_lens, torch.randint(0, 6, (B,), generator=g))]
    q_lens[3] = seq_lens[3]                                  # a whole prompt
    inp = wl.make_prefill(q_lens, seq_lens, 16, 1, seed=126, device=DEV, kv_std=0.5)
    topk = wl.draw_topk_varlen(q_lens, seq_lens, 1, torch.Generator().manual_seed(15))
    out = msa.sparse_prefill(inp.q, inp.kv, inp.block_table, inp.seq_lens, inp.cu_seqlens_q,
                             topk.to(DEV), inp.sm_scale, num_splits=2)
    assert_out_close(_np(out), prefill_oracle(inp, oracle, topk))
    assert msa.get_error() == 0


@pytest.mark.parametrize("B,Q,Hq,Hkv", [(1100, 1, 16, 1), (300, 4, 32, 2), (200, 8, 16, 1)])
def test_step_with_many_requests(B, Q, Hq, Hkv):
    """Batches of hundreds of short requests (empty ones among them): the
    scorer's prefix sum over the requests then takes several requests per
    thread (and, at qlen 8, runs in the one-CTA-per-SM shape), the pages of a
    CTA span many requests, and most rows have fewer than 16 candidates."""
    gen = np.random.default_rng(B + Q)
    seq_lens = [int(x) for x in gen.integers(0, 2600, size=B)]
    seq_lens[:5] = [0, 1, 128, 129, 2048]
    inp = wl.make_custom(seq_lens, Q, Hq, Hkv, seed=121 + Q, device=DEV, kv_std=0.5,
                         kv_scale_mode="amax")
    scores, tk, out = msa.decode_step(inp.q, inp.kv, inp.block_table, inp.seq_lens, Q,
                                      inp.sm_scale, inp.k_scale, inp.v_scale)
    p = to_problem(inp, oracle)
    s_gpu = _np(scores).astype(np.float64)
    assert_scores_close(s_gpu, oracle.score(p))
    assert np.array_equal(_np(tk), oracle.topk(s_gpu, np.array(seq_lens, dtype=np.int32), Q))
    assert_out_close(_np(out), oracle.attend(p, _np(tk)), padding_rows(seq_lens, Q))
    assert msa.get_error() == 0
