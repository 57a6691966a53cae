"""Shared test helpers: host copies of step inputs for the oracle, and an
independent dense attention written with torch library ops."""
from __future__ import annotations

import math
import os

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
PAGE = 128
D = 128


def q_bits(q: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> uint16 bit patterns (host)."""
    return q.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def to_problem(inp, oracle):
    """The oracle's problem for these inputs.  An fp8 query (value q * q_scale)
    goes in as its codes decoded to bf16 (exact: every e4m3 value is a bf16
    value) with sm_scale * q_scale."""
    q, sm_scale = inp.q, inp.sm_scale
    if q.dtype != torch.bfloat16:
        q, sm_scale = q.to(torch.bfloat16), inp.sm_scale * inp.q_scale
    return oracle.Problem(q_bits(q), inp.kv.detach().cpu().numpy(),
                          inp.block_table.detach().cpu().numpy(),
                          inp.seq_lens.detach().cpu().numpy(), inp.qlen, inp.num_q_heads,
                          inp.num_kv_heads, sm_scale, inp.k_scale, inp.v_scale)


def prefill_oracle(inp, oracle, topk, nthreads: int = 0) -> np.ndarray:
    """oracle.attend_prefill on prefill inputs (an fp8 query as in to_problem)."""
    q, sm_scale = inp.q, inp.sm_scale
    if q.dtype != torch.bfloat16:
        q, sm_scale = q.to(torch.bfloat16), inp.sm_scale * inp.q_scale
    topk = topk.cpu().numpy() if isinstance(topk, torch.Tensor) else topk
    return oracle.attend_prefill(q_bits(q), inp.kv.detach().cpu().numpy(),
                                 inp.block_table.detach().cpu().numpy(),
                                 inp.seq_lens.detach().cpu().numpy(),
                                 inp.cu_seqlens_q.detach().cpu().numpy(), topk,
                                 inp.num_q_heads, inp.num_kv_heads, sm_scale, inp.k_scale,
                                 inp.v_scale, nthreads)


def index_problem(inp, oracle):
    """The oracle's problem for scoring on the inputs' K-only (index-K) cache:
    a packed cache whose K halves are the index-K bytes (V halves zero; the
    scorer reads no V), with k_scale = index_k_scale."""
    q, sm_scale = inp.q, inp.sm_scale
    if q.dtype != torch.bfloat16:
        q, sm_scale = q.to(torch.bfloat16), inp.sm_scale * inp.q_scale
    k = inp.index_k.detach().cpu().numpy()
    kv = np.zeros(k.shape[:3] + (2 * D,), dtype=np.uint8)
    kv[..., :D] = k
    return oracle.Problem(q_bits(q), kv, inp.block_table.detach().cpu().numpy(),
                          inp.seq_lens.detach().cpu().numpy(), inp.qlen, inp.num_q_heads,
                          inp.num_kv_heads, sm_scale, inp.index_k_scale, inp.v_scale)


def request_problem(inp, oracle, b: int):
    """The oracle's problem for request b of a prefill batch alone (Q = its
    query length, so its tokens sit at the last positions of its sequence)."""
    q, sm_scale = inp.q, inp.sm_scale
    if q.dtype != torch.bfloat16:
        q, sm_scale = q.to(torch.bfloat16), inp.sm_scale * inp.q_scale
    s0, n = sum(inp.q_lens[:b]), inp.q_lens[b]
    return oracle.Problem(q_bits(q[s0:s0 + n]), inp.kv.detach().cpu().numpy(),
                          inp.block_table[b:b + 1].detach().cpu().numpy(),
                          inp.seq_lens[b:b + 1].detach().cpu().numpy(), n, inp.num_q_heads,
                          inp.num_kv_heads, sm_scale, inp.k_scale, inp.v_scale)


def read_golden_rows(name: str) -> np.ndarray:
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            rows.append([int(v) for v in line.split()])
    return np.array(rows, dtype=np.int64)


def fp8_to_f64(kv_bytes: torch.Tensor) -> torch.Tensor:
    """Decode fp8 bytes with torch's own float8_e4m3fn conversion."""
    return kv_bytes.cpu().view(torch.float8_e4m3fn).to(torch.float64)


def dense_reference(inp, topk=None):
    """Causal attention written with torch ops in fp64: for each request and KV
    head, gather the logical key/value sequence through the block table, form
    softmax(q K^T * sm_scale + causal mask) V over the listed pages (all
    visible pages when topk is None).  Also returns, per (g, token, block), the
    max over the group's heads of the visible logits (the block score)."""
    B = len(inp.seq_lens_list)
    # one query length per request (prefill inputs), else qlen for every request
    q_lens = list(inp.q_lens) if inp.q_lens is not None else [inp.qlen] * B
    first = np.concatenate([[0], np.cumsum(q_lens)]).astype(int)
    Hq, Hkv = inp.num_q_heads, inp.num_kv_heads
    G = Hq // Hkv
    S = inp.stride
    kvf = fp8_to_f64(inp.kv)
    K_all = kvf[..., :D] * inp.k_scale
    V_all = kvf[..., D:] * inp.v_scale
    q = inp.q.cpu().to(torch.float64)
    if inp.q.dtype != torch.bfloat16:     # fp8 query codes, value q * q_scale
        q = q * inp.q_scale
    bt = inp.block_table.cpu()
    T = int(first[-1])
    out = torch.zeros((T, Hq, D), dtype=torch.float64)
    scores = torch.full((Hkv, T, S), -math.inf, dtype=torch.float64)
    for b, L in enumerate(inp.seq_lens_list):
        n_pages = math.ceil(L / PAGE)
        if n_pages == 0:
            continue
        pages = bt[b, :n_pages].long()
        for g in range(Hkv):
            K = K_all[pages, g].reshape(n_pages * PAGE, D)
            V = V_all[pages, g].reshape(n_pages * PAGE, D)
            Q = q_lens[b]
            for j in range(Q):
                i = int(first[b]) + j
                pos = L - Q + j
                if pos < 0:
                    continue
                qs = q[i, g * G:(g + 1) * G]                     # [G, D]
                logits = (qs @ K.T) * inp.sm_scale               # [G, n_pages*128]
                key_idx = torch.arange(n_pages * PAGE)
                visible = key_idx <= pos
                if topk is not None:
                    sel = torch.zeros(n_pages, dtype=torch.bool)
                    for n in topk[i, g].tolist():
                        if n >= 0:
                            sel[n] = True
                    visible = visible & sel[key_idx // PAGE]
                masked = logits.masked_fill(~visible, -math.inf)
                blk = masked.reshape(G, n_pages, PAGE).amax(dim=(0, 2))
                scores[g, i, :n_pages] = blk
                if visible.any():
                    p = torch.softmax(masked, dim=-1)
                    out[i, g * G:(g + 1) * G] = p @ V
    return out, scores


# Tolerances of the decode step (fp32 block scores; bf16 outputs).
SCORE_REL = 1e-3        # |gpu - ref| <= SCORE_REL * max(1, |ref|) on finite scores
OUT_MAX_ABS = 2e-2      # bf16 outputs vs the fp64 oracle, max over all elements
OUT_MEAN_ABS = 2e-3     # ... and mean over all elements


def assert_scores_close(gpu: np.ndarray, ref: np.ndarray, mask: np.ndarray | None = None):
    """Scores: -inf exactly where the oracle has -inf, relative 1e-3 elsewhere."""
    if mask is None:
        mask = np.ones(ref.shape, dtype=bool)
    g, r = gpu[mask], ref[mask]
    inf = np.isneginf(r)
    assert np.array_equal(np.isneginf(g), inf), "-inf pattern differs"
    fin = ~inf
    assert np.all(np.isfinite(g[fin]))
    err = np.abs(g[fin] - r[fin]) / np.maximum(1.0, np.abs(r[fin]))
    assert err.size == 0 or err.max() <= SCORE_REL, f"score rel err {err.max():.3e}"


def assert_out_close(gpu: np.ndarray, ref: np.ndarray, zero_rows: np.ndarray | None = None):
    """bf16 outputs: max-abs <= 2e-2 and mean-abs <= 2e-3; padding rows exactly 0."""
    gpu = np.asarray(gpu, dtype=np.float64)
    d = np.abs(gpu - ref)
    assert np.all(np.isfinite(gpu)), "non-finite output"
    assert d.max() <= OUT_MAX_ABS, f"max abs err {d.max():.3e}"
    assert d.mean() <= OUT_MEAN_ABS, f"mean abs err {d.mean():.3e}"
    if zero_rows is not None and zero_rows.any():
        assert np.all(gpu[zero_rows] == 0.0), "padding rows must be exactly zero"


def padding_rows(seq_lens, qlen: int) -> np.ndarray:
    """[T] bool: query tokens with pos = seq_len - qlen + j < 0."""
    rows = []
    for L in seq_lens:
        for j in range(qlen):
            rows.append(L - qlen + j < 0)
    return np.array(rows, dtype=bool)
