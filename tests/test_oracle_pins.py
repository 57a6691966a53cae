"""Pins of the CPU oracle against facts fixed outside it: library decoders,
closed forms, brute force, invariances and the pages' own helper rules.

None of these tests needs a GPU."""
from __future__ import annotations

import itertools
import math

import numpy as np
import pytest
import torch

import oracle
from block_sparse_gqa_score_gb300 import workloads as wl
from tests.helpers import (dense_reference, prefill_oracle, q_bits, read_golden_rows,
                           to_problem)

D = 128
PAGE = 128


# ----------------------------------------------------------------------------- decoders

def test_e4m3_decode_exhaustive_vs_torch():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_to_f64(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    # spot values of the OCP E4M3 format
    assert ours[0x7E] == 448.0 and ours[0xFE] == -448.0
    assert ours[0x01] == 2.0 ** -9 and ours[0x08] == 2.0 ** -6
    assert ours[0x38] == 1.0 and ours[0xB8] == -1.0
    assert np.isnan(ours[0x7F]) and np.isnan(ours[0xFF])
    assert nan.sum() == 2


def test_bf16_decode_exhaustive_vs_torch():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = oracle.bf16_to_f64(bits)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])


# ----------------------------------------------------------------------------- attend

DENSE_CASES = [
    # seq_lens, Q, Hq, Hkv  (every row sees <= 16 pages, so top-k = all pages)
    ([257, 513], 4, 16, 1),
    ([2048, 129, 1, 300], 1, 16, 1),
    ([129, 385, 256], 3, 8, 2),        # G = 4 with two KV heads: group mapping
    ([2, 5, 130], 4, 8, 4),            # rows with pos < 0 (L < Q)
]


@pytest.mark.parametrize("seq_lens,Q,Hq,Hkv", DENSE_CASES)
def test_attend_equals_dense_when_topk_covers_all(seq_lens, Q, Hq, Hkv):
    inp = wl.make_custom(seq_lens, Q, Hq, Hkv, seed=11, kv_std=0.7, kv_scale_mode="amax")
    assert inp.k_scale != 1.0 and inp.v_scale != 1.0
    topk = wl.all_visible_topk(seq_lens, Q, Hkv)
    p = to_problem(inp, oracle)
    ours = oracle.attend(p, topk.numpy())
    ref, _ = dense_reference(inp)
    np.testing.assert_allclose(ours, ref.numpy(), rtol=0, atol=1e-12)


def test_attend_sparse_selection_equals_masked_dense():
    seq_lens = [3000, 2100]
    inp = wl.make_custom(seq_lens, 2, 16, 2, seed=5)
    gen = torch.Generator().manual_seed(3)
    topk = wl.draw_topk_given(seq_lens, 2, 2, gen)
    ours = oracle.attend(to_problem(inp, oracle), topk.numpy())
    ref, _ = dense_reference(inp, topk)
    np.testing.assert_allclose(ours, ref.numpy(), rtol=0, atol=1e-12)


def test_attend_constant_values_give_that_constant():
    inp = wl.make_custom([700, 2500, 64], 2, 16, 2, seed=7)
    inp.kv[..., D:] = 0x3C                      # every V element = 1.5
    inp.v_scale = 0.75
    gen = torch.Generator().manual_seed(1)
    topk = wl.draw_topk_given(inp.seq_lens_list, 2, 2, gen)
    out = oracle.attend(to_problem(inp, oracle), topk.numpy())
    np.testing.assert_allclose(out, np.full_like(out, 1.5 * 0.75), rtol=0, atol=1e-12)


def test_attend_single_key_returns_that_value():
    inp = wl.make_custom([1, 1], 1, 16, 1, seed=9)
    inp.v_scale = 1.25
    topk = wl.all_visible_topk([1, 1], 1, 1)
    out = oracle.attend(to_problem(inp, oracle), topk.numpy())
    for b in range(2):
        page = int(inp.block_table[b, 0])
        v = torch.from_numpy(inp.kv[page, 0, 0, D:].numpy()).view(torch.float8_e4m3fn)
        v = v.to(torch.float64).numpy() * 1.25
        for h in range(16):
            np.testing.assert_allclose(out[b, h], v, rtol=0, atol=1e-12)


def test_attend_two_keys_logistic_closed_form():
    # Q = 2: row j = 0 sees one key (pos 0), row j = 1 sees both (pos 1)
    inp = wl.make_custom([2], 2, 16, 1, seed=13)
    p = to_problem(inp, oracle)
    out = oracle.attend(p, wl.all_visible_topk([2], 2, 1).numpy())
    page = int(inp.block_table[0, 0])
    kv = torch.from_numpy(inp.kv[page, 0, :2].numpy()).view(torch.float8_e4m3fn).to(torch.float64)
    K, V = kv[:, :D].numpy(), kv[:, D:].numpy()
    qf = inp.q.to(torch.float64).numpy()
    for h in range(16):
        np.testing.assert_allclose(out[0, h], V[0], rtol=0, atol=1e-12)
        a = inp.sm_scale * float(qf[1, h] @ K[0])
        b = inp.sm_scale * float(qf[1, h] @ K[1])
        sig = lambda x: 1.0 / (1.0 + math.exp(-x))  # noqa: E731
        want = sig(a - b) * V[0] + sig(b - a) * V[1]
        np.testing.assert_allclose(out[1, h], want, rtol=0, atol=1e-12)


def test_attend_physical_page_permutation_is_bit_exact():
    inp = wl.make_custom([1000, 2000], 3, 16, 2, seed=21)
    gen = torch.Generator().manual_seed(2)
    topk = wl.draw_topk_given(inp.seq_lens_list, 3, 2, gen).numpy()
    base = oracle.attend(to_problem(inp, oracle), topk)
    nb = inp.kv.shape[0]
    perm = torch.randperm(nb, generator=gen)            # new location of physical page p
    kv2 = torch.empty_like(inp.kv)
    kv2[perm] = inp.kv
    bt2 = perm.to(torch.int32)[inp.block_table.long()]
    p2 = oracle.Problem(q_bits(inp.q), kv2.numpy(), bt2.numpy(), inp.seq_lens.numpy(), 3, 16, 2,
                        inp.sm_scale, inp.k_scale, inp.v_scale)
    assert np.array_equal(oracle.attend(p2, topk), base)


def test_attend_invariant_to_topk_list_order():
    inp = wl.make_custom([2500, 3100], 2, 16, 1, seed=23)
    gen = torch.Generator().manual_seed(4)
    topk = wl.draw_topk_given(inp.seq_lens_list, 2, 1, gen)
    topk[0, 0, 5] = -1                                   # a hole inside the list
    base = oracle.attend(to_problem(inp, oracle), topk.numpy())
    shuffled = topk.clone()
    for i in range(shuffled.shape[0]):
        shuffled[i, 0] = shuffled[i, 0, torch.randperm(16, generator=gen)]
    out = oracle.attend(to_problem(inp, oracle), shuffled.numpy())
    np.testing.assert_allclose(out, base, rtol=0, atol=1e-12)


def test_attend_padding_rows_are_zero():
    inp = wl.make_custom([0, 300, 2], 4, 16, 1, seed=25)
    topk = wl.all_visible_topk(inp.seq_lens_list, 4, 1)
    out = oracle.attend(to_problem(inp, oracle), topk.numpy())
    assert np.all(out[0:4] == 0.0)          # seq_len 0
    assert np.all(out[8:10] == 0.0)         # L = 2, Q = 4: j = 0, 1 have pos < 0
    assert np.all(np.abs(out[4:8]).sum(axis=-1) > 0)
    assert np.all(np.abs(out[10:12]).sum(axis=-1) > 0)


def test_attend_rejects_bad_topk_entries():
    inp = wl.make_custom([300], 1, 16, 1, seed=27)
    p = to_problem(inp, oracle)
    bad = wl.all_visible_topk([300], 1, 1).numpy().copy()
    bad[0, 0, 3] = 3                                    # cur is 2
    with pytest.raises(oracle.OracleError) as e:
        oracle.attend(p, bad)
    assert e.value.status == oracle.ERANGE
    dup = wl.all_visible_topk([300], 1, 1).numpy().copy()
    dup[0, 0, 3] = 1
    with pytest.raises(oracle.OracleError):
        oracle.attend(p, dup)
    bt_bad = inp.block_table.clone()
    bt_bad[0, 1] = inp.kv.shape[0]
    p2 = oracle.Problem(q_bits(inp.q), inp.kv.numpy(), bt_bad.numpy(), inp.seq_lens.numpy(), 1,
                        16, 1, inp.sm_scale)
    with pytest.raises(oracle.OracleError):
        oracle.attend(p2, wl.all_visible_topk([300], 1, 1).numpy())


def test_attend_rows_matches_full():
    inp = wl.make_custom([900, 1500], 2, 16, 2, seed=29)
    gen = torch.Generator().manual_seed(5)
    topk = wl.draw_topk_given(inp.seq_lens_list, 2, 2, gen).numpy()
    p = to_problem(inp, oracle)
    full = oracle.attend(p, topk).reshape(-1, D)
    rows = np.array([0, 5, 17, 33, 63], dtype=np.int64)
    assert np.array_equal(oracle.attend_rows(p, topk, rows), full[rows])


# ----------------------------------------------------------------------------- score

@pytest.mark.parametrize("seq_lens,Q,Hq,Hkv", DENSE_CASES + [([3000, 1900], 2, 16, 2)])
def test_score_equals_max_of_dense_logits(seq_lens, Q, Hq, Hkv):
    inp = wl.make_custom(seq_lens, Q, Hq, Hkv, seed=31, kv_std=0.5, kv_scale_mode="amax")
    ours = oracle.score(to_problem(inp, oracle))
    _, ref = dense_reference(inp)
    fin = np.isfinite(ref.numpy())
    assert np.array_equal(np.isfinite(ours), fin)
    assert np.all(ours[~fin] == -np.inf)
    np.testing.assert_allclose(ours[fin], ref.numpy()[fin], rtol=0, atol=1e-12)


def test_score_single_key_closed_form():
    inp = wl.make_custom([1], 1, 16, 1, seed=33)
    inp.k_scale = 0.5
    s = oracle.score(to_problem(inp, oracle))
    page = int(inp.block_table[0, 0])
    k0 = torch.from_numpy(inp.kv[page, 0, 0, :D].numpy()).view(torch.float8_e4m3fn)
    k0 = k0.to(torch.float64).numpy() * 0.5
    qf = inp.q.to(torch.float64).numpy()[0]
    want = max(inp.sm_scale * float(qf[h] @ k0) for h in range(16))
    assert s.shape == (1, 1, 1)
    assert abs(s[0, 0, 0] - want) <= 1e-12 * max(1.0, abs(want))


def test_score_padding_rows_and_future_blocks_are_minus_inf():
    inp = wl.make_custom([0, 200, 2], 4, 16, 1, seed=35, min_stride=4)
    s = oracle.score(to_problem(inp, oracle))
    assert np.all(s[:, 0:4] == -np.inf)
    assert np.all(s[:, 8:10] == -np.inf)                 # pos < 0
    assert np.all(np.isfinite(s[:, 4:8, :2])) and np.all(s[:, 4:8, 2:] == -np.inf)
    assert np.all(np.isfinite(s[:, 10:12, 0])) and np.all(s[:, 10:12, 1:] == -np.inf)


# ----------------------------------------------------------------------------- select

def _brute_force_select(scores_row: np.ndarray, cur: int, k: int = 16):
    """The unique subset X of 0..cur-1 with |X| = k-1 such that every chosen x
    beats every unchosen y in the order (score desc, index asc)."""
    best = None
    for X in itertools.combinations(range(cur), k - 1):
        Xs = set(X)
        ok = all((scores_row[x], -x) > (scores_row[y], -y)
                 for x in X for y in range(cur) if y not in Xs)
        if ok:
            assert best is None, "selection must be unique"
            best = sorted(X)
    assert best is not None
    return best + [cur]


@pytest.mark.parametrize("cur", [15, 16, 17, 18, 20])
def test_select_matches_brute_force_with_ties(cur):
    rng = np.random.default_rng(cur)
    T, S = 3, cur + 3
    seq_lens = np.array([cur * PAGE + 1 + 3], dtype=np.int32)     # pos = cur*128 + j
    scores = rng.integers(-3, 4, size=(1, T, S)).astype(np.float64)  # many ties
    got = oracle.topk(scores, seq_lens, T)
    for j in range(T):
        pos = int(seq_lens[0]) - T + j
        c = pos // PAGE
        assert c == cur
        want = _brute_force_select(scores[0, j], c) if c + 1 > 16 else list(range(c + 1))
        want = want + [-1] * (16 - len(want))
        assert got[j, 0].tolist() == want


def test_select_short_rows_keep_everything_and_padding_rows_are_empty():
    seq_lens = np.array([0, 5 * PAGE, 2], dtype=np.int32)
    scores = np.random.default_rng(0).normal(size=(2, 12, 8))
    got = oracle.topk(scores, seq_lens, 4)
    assert np.all(got[0:4] == -1)
    for j in range(4):                       # pos = 636 + j -> cur 4 for j < 4
        assert got[4 + j, 0].tolist() == [0, 1, 2, 3, 4] + [-1] * 11
    assert np.all(got[8:10] == -1)           # pos < 0
    assert np.all(got[10:12, :, 0] == 0) and np.all(got[10:12, :, 1:] == -1)


def test_select_reads_arbitrary_strides():
    rng = np.random.default_rng(7)
    Hkv, T, S = 2, 6, 40
    seq_lens = np.array([39 * PAGE + 2, 30 * PAGE + 50], dtype=np.int32)
    phys = rng.normal(size=(Hkv, S, T))                 # [head, block, token] storage
    view = phys.transpose(0, 2, 1)                      # read as [head, token, block]
    a = oracle.topk(view, seq_lens, 3)
    b = oracle.topk(np.ascontiguousarray(view), seq_lens, 3)
    assert np.array_equal(a, b)


def test_select_golden_make_topk_rows():
    """The pages' _make_topk rows for seq_lens [257, 513], Q = 4 (every row sees
    at most 16 pages, so the selector must keep all of them ascending)."""
    gold = read_golden_rows("make_topk_257_513_q4.txt")
    seq_lens = np.array([257, 513], dtype=np.int32)
    scores = np.random.default_rng(1).normal(size=(1, 8, 5))
    got = oracle.topk(scores, seq_lens, 4)
    assert np.array_equal(got[:, 0, :], gold[:, 1:])
    assert np.array_equal(gold[:, 1:], wl.all_visible_topk([257, 513], 4, 1)[:, 0].numpy())


def test_kv_layout_golden_strides():
    gold = read_golden_rows("kv_cache_stride_hnd.txt")
    for hkv, *strides in gold.tolist():
        kv, _, _ = wl.draw_kv(3, hkv, torch.Generator().manual_seed(0), "cpu")
        assert list(kv.stride()) == strides


# ----------------------------------------------------------------------------- combine

def _part(z: np.ndarray, V: np.ndarray):
    """(o, m, l) of one key subset in the documented split format."""
    if len(z) == 0:
        return np.zeros(D), -np.inf, 0.0
    z2 = z * math.log2(math.e)
    m = z2.max()
    w = np.exp2(z2 - m)
    return w @ V, m, w.sum()


def test_combine_of_disjoint_parts_equals_softmax_over_union():
    rng = np.random.default_rng(3)
    rows, n = 5, 300
    parts = [(0, 90), (90, 90), (90, 200), (200, 300)]     # includes an empty part
    o = np.zeros((len(parts), rows, D))
    ml = np.zeros((len(parts), rows, 2))
    want = np.zeros((rows, D))
    for r in range(rows):
        z = rng.normal(scale=3.0, size=n)
        V = rng.normal(size=(n, D))
        want[r] = torch.softmax(torch.from_numpy(z), 0).numpy() @ V
        for s, (a, b) in enumerate(parts):
            o[s, r], ml[s, r, 0], ml[s, r, 1] = _part(z[a:b], V[a:b])
    got = oracle.combine(o, ml)
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-12)


def test_combine_all_empty_is_zero():
    o = np.zeros((3, 2, D))
    ml = np.zeros((3, 2, 2))
    ml[..., 0] = -np.inf
    assert np.all(oracle.combine(o, ml) == 0.0)


# ----------------------------------------------------------------------------- whole step

def test_decode_step_on_tiny_workload_is_consistent():
    inp = wl.make_inputs("tiny_b2_q1_h16kv1_2k3k")
    p = to_problem(inp, oracle)
    s, t, o = oracle.decode_step(p)
    # request 0 sees exactly 16 pages: all kept, ascending
    assert t[0, 0].tolist() == list(range(16))
    # request 1 (L = 3000, cur = 23): current block last, 15 others
    row = t[1, 0].tolist()
    assert row[-1] == 23 and len(set(row)) == 16 and row == sorted(row)
    kept = set(row[:-1])
    worst_kept = min(s[0, 1, n] for n in kept)
    best_dropped = max(s[0, 1, n] for n in range(23) if n not in kept)
    assert worst_kept >= best_dropped
    ref, _ = dense_reference(inp, torch.from_numpy(t))
    np.testing.assert_allclose(o, ref.numpy(), rtol=0, atol=1e-12)


def test_score_blocks_matches_full_scores():
    inp = wl.make_custom([3000, 1500], 3, 32, 2, seed=37)
    p = to_problem(inp, oracle)
    full = oracle.score(p)
    triples = [(0, 1, 23), (1, 0, 0), (1, 1, 11), (0, 0, 5), (1, 0, 20)]
    part = oracle.score_blocks(p, triples)
    for b, g, n in triples:
        rows = slice(b * 3, b * 3 + 3)
        assert np.array_equal(part[g, rows, n], full[g, rows, n])


# ----------------------------------------------------------------------------- prefill

# The vLLM prefill test's batch: q_lens [300, 128, 77] over seq_lens
# [300, 640, 1100] (a fresh prompt, then two chunks over cached context), plus
# an empty request and single-token chunks of our own.
PREFILL_CASES = [
    ([300, 128, 77], [300, 640, 1100], 16, 1),
    ([5, 0, 1, 40], [700, 300, 129, 40], 8, 2),
]


@pytest.mark.parametrize("q_lens,seq_lens,Hq,Hkv", PREFILL_CASES)
def test_prefill_equals_dense_causal_attention(q_lens, seq_lens, Hq, Hkv):
    """With every visible page listed (the prefill test's lists), prefill
    attention is plain causal attention: token j of request b sees keys
    0 .. seq_len - q_len + j of its own sequence."""
    inp = wl.make_prefill(q_lens, seq_lens, Hq, Hkv, seed=21, kv_std=0.7, kv_scale_mode="amax")
    topk = wl.all_visible_lists_varlen(q_lens, seq_lens, Hkv, 16)
    ours = prefill_oracle(inp, oracle, topk)
    ref, _ = dense_reference(inp)
    np.testing.assert_allclose(ours, ref.numpy(), rtol=0, atol=1e-12)


def test_prefill_sparse_lists_equal_masked_dense():
    q_lens, seq_lens = [33, 2, 64], [3000, 2100, 64]
    inp = wl.make_prefill(q_lens, seq_lens, 16, 2, seed=22)
    topk = wl.draw_topk_varlen(q_lens, seq_lens, 2, torch.Generator().manual_seed(4))
    ours = prefill_oracle(inp, oracle, topk)
    ref, _ = dense_reference(inp, topk)
    np.testing.assert_allclose(ours, ref.numpy(), rtol=0, atol=1e-12)


def test_prefill_token_equals_one_token_decode_at_its_position():
    """Causality: a prefill token at position pos gives what a one-token
    decode step of the same sequence cut at pos + 1 gives."""
    q_lens, seq_lens = [20, 7], [1500, 260]
    inp = wl.make_prefill(q_lens, seq_lens, 16, 1, seed=23)
    topk = wl.draw_topk_varlen(q_lens, seq_lens, 1, torch.Generator().manual_seed(5))
    full = prefill_oracle(inp, oracle, topk)
    qb = q_bits(inp.q)
    kv = inp.kv.numpy()
    bt = inp.block_table.numpy()
    for i, (b, j) in enumerate([(0, 0), (0, 11), (0, 19), (1, 0), (1, 6)]):
        row = sum(q_lens[:b]) + j
        pos = seq_lens[b] - q_lens[b] + j
        p = oracle.Problem(qb[row:row + 1], kv, bt[b:b + 1], np.array([pos + 1], np.int32), 1,
                           16, 1, inp.sm_scale, inp.k_scale, inp.v_scale)
        one = oracle.attend(p, topk[row:row + 1].numpy())
        assert np.array_equal(one[0], full[row])


def test_prefill_with_equal_lengths_is_the_decode_step():
    seq_lens, Q = [900, 400, 1300], 6
    inp = wl.make_custom(seq_lens, Q, 16, 2, seed=24)
    topk = wl.draw_topk_given(seq_lens, Q, 2, torch.Generator().manual_seed(6))
    dec = oracle.attend(to_problem(inp, oracle), topk.numpy())
    pre = oracle.attend_prefill(q_bits(inp.q), inp.kv.numpy(), inp.block_table.numpy(),
                                inp.seq_lens.numpy(), np.arange(4, dtype=np.int32) * Q,
                                topk.numpy(), 16, 2, inp.sm_scale, inp.k_scale, inp.v_scale)
    assert np.array_equal(dec, pre)
    scores = np.random.default_rng(1).integers(-3, 4, (2, 3 * Q, 11)).astype(np.float64)
    want = oracle.topk(scores, np.array(seq_lens, np.int32), Q)
    got = oracle.topk_prefill(scores, seq_lens, np.arange(4) * Q)
    assert np.array_equal(got, want)


def test_prefill_topk_keeps_each_tokens_own_block():
    """Each token of a chunk keeps its own current block, whatever the scores."""
    seq_lens, q_lens = [3 * PAGE + 10, 20 * PAGE], [2 * PAGE, 3]
    cu = np.array([0, 2 * PAGE, 2 * PAGE + 3])
    scores = np.zeros((1, int(cu[-1]), 20))
    t = oracle.topk_prefill(scores, seq_lens, cu)
    for b in range(2):
        for j in range(q_lens[b]):
            pos = seq_lens[b] - q_lens[b] + j
            row = t[cu[b] + j, 0]
            kept = row[row >= 0]
            assert kept[-1] == pos // PAGE
            want = min(pos // PAGE + 1, 16)
            assert len(kept) == want and len(set(kept.tolist())) == want


def test_prefill_rejects_inconsistent_lengths():
    inp = wl.make_prefill([4], [10], 16, 1, seed=25)
    topk = np.zeros((4, 1, 16), np.int32) - 1
    with pytest.raises(ValueError):
        oracle.attend_prefill(q_bits(inp.q), inp.kv.numpy(), inp.block_table.numpy(),
                              np.array([3], np.int32), np.array([0, 4]), topk, 16, 1, 1.0)
    with pytest.raises(ValueError):
        oracle.attend_prefill(q_bits(inp.q), inp.kv.numpy(), inp.block_table.numpy(),
                              np.array([10, 10], np.int32), np.array([0, 5, 4]), topk, 16, 1,
                              1.0)


# ----------------------------------------------------------------------------- index-K cache

def test_score_ignores_the_value_half():
    """The scores depend on the K half of each page row only: replacing every
    V byte leaves them bit-identical (the premise of scoring on a K-only
    cache laid into the K halves of a packed one)."""
    inp = wl.make_custom([3000, 700], 4, 16, 2, seed=31, kv_std=0.5, kv_scale_mode="amax")
    ref = oracle.score(to_problem(inp, oracle))
    other = inp.kv.clone()
    other[..., D:] = torch.randint(0, 0x7F, other[..., D:].shape, dtype=torch.uint8)
    inp.kv = other
    assert np.array_equal(oracle.score(to_problem(inp, oracle)), ref)
