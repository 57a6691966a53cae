"""Seeded synthetic inputs for the sparse-decode step.

This module only draws inputs: shapes, page layouts, random values and, for
the attend-only workload, a given top-k list.  It holds none of the step's
arithmetic (no scoring, selection or attention), so both the CUDA path and the
CPU oracle can be fed from it.

Layouts follow the vLLM MiniMax-M3 sparse attention pages:
  * q: bf16 [T, Hq, 128], token i = b * Q + j (request-major), as
    MiniMaxM3SparseTritonImpl.forward views the query.
  * kv: fp8 e4m3 [NB, Hkv, 128, 256]; K in the first 128 bytes of a token row,
    V in the last 128 (MiniMaxM3SparseBackend.get_kv_cache_shape, HND order).
  * block_table: int32 [B, S]; each request's logical pages scattered over a
    random permutation of the physical pages, zero-filled past its last page
    (test_minimax_m3_msa_cutlass_sparse_decode.py, _make_paged_layout).
  * seq_lens: int32 [B].
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

HEAD_DIM = 128
PAGE = 128
TOPK = 16
FP8_MAX = 448.0


@dataclass
class Workload:
    """Description of one synthetic workload (sizes and value recipe)."""
    name: str
    batch: int
    qlen: int
    num_q_heads: int
    num_kv_heads: int
    seq_lens: str            # recipe tag, see _draw_seq_lens
    seed: int
    kv_std: float = 1.0
    kv_scale_mode: str = "unit"   # "unit": scale 1; "amax": scale = amax / 448 per side
    key_outlier_frac: float = 0.0
    key_outlier_mult: float = 1.0
    topk_given: bool = False      # attend-only: draw the top-k list instead of scoring
    dense: bool = False           # dense decode: every visible block, no scoring or list
    fp8_query: bool = False       # q quantised to fp8 e4m3 with a per-tensor scale
    pad_frac: float = 0.0         # fraction of requests with seq_len 0
    seq_args: dict = field(default_factory=dict)
    # chunked prefill: request b's query is its last q_len_b tokens, q_len_b
    # drawn uniformly in [lo, hi] (at most seq_len), each token with its own
    # drawn top-k list (then qlen is unused)
    prefill_q: tuple | None = None
    # the scorer reads a separate K-only (index-K) cache on the same pages
    index_k: bool = False

    @property
    def tokens(self) -> int:
        if self.prefill_q is not None:
            raise ValueError("a prefill workload's token count depends on its draws")
        return self.batch * self.qlen

    def describe(self) -> dict:
        d = {"workload": self.name, "batch": self.batch, "decode_query_len": self.qlen,
             "num_q_heads": self.num_q_heads, "num_kv_heads": self.num_kv_heads,
             "head_dim": HEAD_DIM, "page": PAGE, "topk": TOPK, "seq_lens": self.seq_lens,
             "pipeline": ("dense attend+combine" if self.dense else "attend+combine"
                          if self.topk_given else "score+topk+attend+combine"),
             "query": "fp8 e4m3, per-tensor scale amax/448" if self.fp8_query else "bf16"}
        if self.index_k:
            d["scorer_keys"] = "separate K-only index cache [NB, Hkv, 128, 128], fp8"
        if self.prefill_q is not None:
            del d["decode_query_len"]
            d["prefill_query_lens"] = f"uniform {self.prefill_q[0]}-{self.prefill_q[1]}"
            d["pipeline"] = "prefill attend (msa_sparse_prefill), given per-token top-k"
        return d


WORKLOADS = {
    w.name: w for w in [
        Workload("tiny_b2_q1_h16kv1_2k3k", 2, 1, 16, 1, "fixed", seed=1001,
                 seq_args={"values": [2048, 3000]}),
        Workload("b16_q4_h64kv4_8k-32k", 16, 4, 64, 4, "uniform", seed=1002, kv_std=0.5,
                 kv_scale_mode="amax", seq_args={"lo": 8192, "hi": 32768}),
        Workload("b32_q4_h16kv1_64k-128k_attend", 32, 4, 16, 1, "uniform", seed=1003,
                 topk_given=True, seq_args={"lo": 65536, "hi": 131072}),
        Workload("b128_q1_h64kv4_lognormal16k_pad10", 128, 1, 64, 4, "lognormal", seed=1004,
                 pad_frac=0.10, seq_args={"median": 16384, "sigma": 0.75, "lo": 1024,
                                          "hi": 65536}),
        Workload("b16_q32_h64kv4_256k_outliers", 16, 32, 64, 4, "fixed", seed=1005,
                 key_outlier_frac=0.05, key_outlier_mult=8.0,
                 seq_args={"values": [262144] * 16}),
        # the qlen-32 workload on 2 requests: the same kernels at a size a
        # full profiler capture can take (about 1 GB on the device)
        Workload("b2_q32_h64kv4_256k_outliers", 2, 32, 64, 4, "fixed", seed=1008,
                 key_outlier_frac=0.05, key_outlier_mult=8.0,
                 seq_args={"values": [262144] * 2}),
        # the same model's dense layers (every visible block) on the batch-16
        # decode shapes
        Workload("dense_b16_q4_h64kv4_8k-32k", 16, 4, 64, 4, "uniform", seed=1006, kv_std=0.5,
                 kv_scale_mode="amax", dense=True, seq_args={"lo": 8192, "hi": 32768}),
        # the batch-16 step with the query quantised to fp8 per tensor, the form
        # the vLLM CUTLASS decode takes (query_fp8, q_scale)
        Workload("b16_q4_h64kv4_8k-32k_fp8q", 16, 4, 64, 4, "uniform", seed=1007, kv_std=0.5,
                 kv_scale_mode="amax", fp8_query=True, seq_args={"lo": 8192, "hi": 32768}),
        # the batch-16 step with the blocks scored on a separate K-only cache
        # (index-K sub-pages) instead of the attend's K
        Workload("b16_q4_h64kv4_8k-32k_indexk", 16, 4, 64, 4, "uniform", seed=1010, kv_std=0.5,
                 kv_scale_mode="amax", index_k=True, seq_args={"lo": 8192, "hi": 32768}),
        # chunked prefill on the same model: 4 requests of 8k-32k tokens, each
        # with a 1k-2k query chunk at its end, every token with its own list
        Workload("prefill_b4_chunk1k-2k_h64kv4_8k-32k", 4, 0, 64, 4, "uniform", seed=1009,
                 kv_std=0.5, kv_scale_mode="amax", topk_given=True, prefill_q=(1024, 2048),
                 seq_args={"lo": 8192, "hi": 32768}),
    ]
}

#: The workload the headline benchmark line is quoted on.
HEADLINE = "b16_q4_h64kv4_8k-32k"


def _draw_seq_lens(w: Workload, gen: torch.Generator) -> list[int]:
    a = w.seq_args
    if w.seq_lens == "fixed":
        vals = list(a["values"])
        if len(vals) != w.batch:
            raise ValueError("fixed seq_lens must list one length per request")
    elif w.seq_lens == "uniform":
        vals = torch.randint(a["lo"], a["hi"] + 1, (w.batch,), generator=gen).tolist()
    elif w.seq_lens == "lognormal":
        z = torch.randn((w.batch,), generator=gen, dtype=torch.float64)
        vals = torch.exp(math.log(a["median"]) + a["sigma"] * z).round().clamp(a["lo"], a["hi"])
        vals = [int(v) for v in vals.tolist()]
    else:
        raise ValueError(w.seq_lens)
    if w.pad_frac > 0:
        n_pad = int(round(w.pad_frac * w.batch))
        pad = torch.randperm(w.batch, generator=gen)[:n_pad].tolist()
        for b in pad:
            vals[b] = 0
    return [int(v) for v in vals]


def paged_layout(seq_lens: list[int], gen: torch.Generator, min_stride: int = 1):
    """block_table [B, S] over a shuffled pool of NB = sum(ceil(L/128)) pages."""
    pages = [math.ceil(L / PAGE) for L in seq_lens]
    nb = sum(pages)
    stride = max(max(pages) if pages else 0, min_stride)
    bt = torch.zeros((len(seq_lens), stride), dtype=torch.int32)
    perm = torch.randperm(max(nb, 1), generator=gen).to(torch.int32)
    off = 0
    for b, n in enumerate(pages):
        bt[b, :n] = perm[off:off + n]
        off += n
    return bt, nb


def _to_fp8(x: torch.Tensor) -> torch.Tensor:
    """Saturating cast to float8_e4m3fn, returned as raw bytes."""
    return x.clamp(-FP8_MAX, FP8_MAX).to(torch.float8_e4m3fn).view(torch.uint8)


def draw_kv(nb: int, hkv: int, gen: torch.Generator, device, std: float = 1.0,
            scale_mode: str = "unit", outlier_frac: float = 0.0, outlier_mult: float = 1.0):
    """Packed K|V pages [NB, Hkv, 128, 256] as fp8 bytes, plus (k_scale, v_scale).

    K and V are drawn N(0, std^2) in bf16.  With scale_mode "amax" each side is
    divided by its own per-tensor scale amax/448 before the saturating cast.
    A seeded fraction of key rows (per page row and KV head) is multiplied by
    outlier_mult before quantising."""
    nb = max(nb, 1)
    shape = (nb, hkv, PAGE, HEAD_DIM)
    k = torch.randn(shape, generator=gen, device=device, dtype=torch.bfloat16)
    v = torch.randn(shape, generator=gen, device=device, dtype=torch.bfloat16)
    if std != 1.0:
        k.mul_(std)
        v.mul_(std)
    if outlier_frac > 0:
        rows = torch.rand((nb, hkv, PAGE, 1), generator=gen, device=device) < outlier_frac
        k = torch.where(rows, k * outlier_mult, k)
    if scale_mode == "amax":
        k_scale = float(k.abs().max().float()) / FP8_MAX
        v_scale = float(v.abs().max().float()) / FP8_MAX
    elif scale_mode == "unit":
        k_scale = v_scale = 1.0
    else:
        raise ValueError(scale_mode)
    kv = torch.empty((nb, hkv, PAGE, 2 * HEAD_DIM), dtype=torch.uint8, device=device)
    kv[..., :HEAD_DIM] = _to_fp8(k.float() / k_scale)
    kv[..., HEAD_DIM:] = _to_fp8(v.float() / v_scale)
    return kv, k_scale, v_scale


def draw_index_k(nb: int, hkv: int, gen: torch.Generator, device, std: float = 1.0,
                 scale_mode: str = "unit"):
    """A K-only cache [NB, Hkv, 128, 128] as fp8 bytes plus its scale, drawn
    like draw_kv's K half (N(0, std^2) in bf16, per-tensor scale 1 or
    amax/448, saturating cast)."""
    k = torch.randn((max(nb, 1), hkv, PAGE, HEAD_DIM), generator=gen, device=device,
                    dtype=torch.bfloat16)
    if std != 1.0:
        k.mul_(std)
    if scale_mode == "amax":
        scale = float(k.abs().max().float()) / FP8_MAX
    elif scale_mode == "unit":
        scale = 1.0
    else:
        raise ValueError(scale_mode)
    return _to_fp8(k.float() / scale), scale


def draw_topk_varlen(q_lens: list[int], seq_lens: list[int], hkv: int, gen: torch.Generator):
    """Attend-only input: per (token, KV head), the token's current block plus
    up to 15 distinct blocks drawn uniformly from the earlier ones, ascending,
    -1 padded.  Request b's q_lens[b] tokens are the last ones of its
    seq_lens[b], rows request-major; rows with no visible token are all -1."""
    out = torch.full((sum(q_lens), hkv, TOPK), -1, dtype=torch.int32)
    i = 0
    for L, qlen in zip(seq_lens, q_lens):
        for j in range(qlen):
            visible = L - qlen + j + 1          # tokens this query row may see
            if visible > 0:
                cur = (visible - 1) // PAGE
                for g in range(hkv):
                    if cur + 1 <= TOPK:
                        ids = list(range(cur + 1))
                    else:
                        pick = torch.randperm(cur, generator=gen)[:TOPK - 1]
                        ids = sorted(pick.tolist()) + [cur]
                    out[i, g, :len(ids)] = torch.tensor(ids, dtype=torch.int32)
            i += 1
    return out


def draw_topk_given(seq_lens: list[int], qlen: int, hkv: int, gen: torch.Generator):
    """draw_topk_varlen with qlen tokens for every request."""
    return draw_topk_varlen([qlen] * len(seq_lens), seq_lens, hkv, gen)


def all_visible_lists_varlen(q_lens: list[int], seq_lens: list[int], hkv: int, width: int):
    """Every visible page ascending, -1 padded to `width` columns, for request
    b's q_lens[b] last tokens: the lists that make the sparse attend dense (the
    vLLM prefill test's lists while a row sees at most 16 pages)."""
    out = torch.full((sum(q_lens), hkv, width), -1, dtype=torch.int32)
    i = 0
    for L, qlen in zip(seq_lens, q_lens):
        for j in range(qlen):
            visible = L - qlen + j + 1
            if visible > 0:
                n = math.ceil(visible / PAGE)
                if n > width:
                    raise ValueError("more visible pages than columns")
                out[i, :, :n] = torch.arange(n, dtype=torch.int32)
            i += 1
    return out


def all_visible_lists(seq_lens: list[int], qlen: int, hkv: int, width: int):
    """all_visible_lists_varlen with qlen tokens for every request."""
    return all_visible_lists_varlen([qlen] * len(seq_lens), seq_lens, hkv, width)


def all_visible_topk(seq_lens: list[int], qlen: int, hkv: int):
    """Every visible page ascending, -1 padded: the top-k the vLLM test file's
    _make_topk builds (valid only while a row sees at most 16 pages)."""
    B = len(seq_lens)
    out = torch.full((B * qlen, hkv, TOPK), -1, dtype=torch.int32)
    for b, L in enumerate(seq_lens):
        for j in range(qlen):
            visible = L - qlen + j + 1
            if visible <= 0:
                continue
            n = math.ceil(visible / PAGE)
            if n > TOPK:
                raise ValueError("more than 16 visible pages")
            out[b * qlen + j, :, :n] = torch.arange(n, dtype=torch.int32)
    return out


@dataclass
class StepInputs:
    """One layer's inputs, on `device`."""
    q: torch.Tensor            # bf16 [T, Hq, 128], or fp8 e4m3 of value q * q_scale
    kv: torch.Tensor           # uint8 [NB, Hkv, 128, 256] (fp8 e4m3 bytes)
    block_table: torch.Tensor  # int32 [B, S]
    seq_lens: torch.Tensor     # int32 [B]
    seq_lens_list: list
    k_scale: float
    v_scale: float
    sm_scale: float
    qlen: int
    num_q_heads: int
    num_kv_heads: int
    topk: torch.Tensor | None = None   # int32 [T, Hkv, 16] when given
    q_scale: float = 1.0               # per-tensor scale of an fp8 q
    # a prefill batch: request b's q_lens[b] query tokens are the last ones of
    # its seq_lens[b] (context seq_lens[b] - q_lens[b] tokens already cached),
    # rows cu_seqlens_q[b] .. cu_seqlens_q[b + 1] - 1; qlen is then 0
    q_lens: list | None = None
    cu_seqlens_q: torch.Tensor | None = None   # int32 [B + 1]
    # a separate K-only cache the scorer reads (index-K sub-pages), same pages
    index_k: torch.Tensor | None = None        # uint8 [NB, Hkv, 128, 128] (fp8 e4m3 bytes)
    index_k_scale: float = 1.0

    @property
    def batch(self) -> int:
        return len(self.seq_lens_list)

    @property
    def tokens(self) -> int:
        return sum(self.q_lens) if self.q_lens is not None else self.batch * self.qlen

    @property
    def num_blocks(self) -> int:
        return int(self.kv.shape[0])

    @property
    def stride(self) -> int:
        return int(self.block_table.shape[1])


def make_inputs(w: Workload | str, device="cpu", layer: int = 0,
                seq_lens: list[int] | None = None) -> StepInputs:
    """Draw one layer of workload `w` (seeded by the workload seed and `layer`).

    Request lengths depend on the seed only, so every layer of a workload has
    the same lengths and block-table shape; values and page permutations
    differ per layer."""
    if isinstance(w, str):
        w = WORKLOADS[w]
    gen_host = torch.Generator().manual_seed(w.seed)
    if seq_lens is None:
        seq_lens = _draw_seq_lens(w, gen_host)
    if w.prefill_q is not None:
        lo, hi = w.prefill_q
        q_lens = torch.randint(lo, hi + 1, (len(seq_lens),), generator=gen_host).tolist()
        q_lens = [min(n, L) for n, L in zip(q_lens, seq_lens)]
        inp = make_prefill(q_lens, seq_lens, w.num_q_heads, w.num_kv_heads,
                           seed=w.seed * 1000 + layer, device=device, kv_std=w.kv_std,
                           kv_scale_mode=w.kv_scale_mode, fp8_query=w.fp8_query)
        inp.topk = draw_topk_varlen(q_lens, seq_lens, w.num_kv_heads,
                                    torch.Generator().manual_seed(w.seed * 1000 + layer + 5)
                                    ).to(inp.q.device)
        return inp
    gen_host = torch.Generator().manual_seed(w.seed * 1000 + layer)
    bt, nb = paged_layout(seq_lens, gen_host)
    dev = torch.device(device)
    gen_dev = torch.Generator(device=dev).manual_seed(w.seed * 1000 + layer + 17)
    kv, k_scale, v_scale = draw_kv(nb, w.num_kv_heads, gen_dev, dev, std=w.kv_std,
                                   scale_mode=w.kv_scale_mode, outlier_frac=w.key_outlier_frac,
                                   outlier_mult=w.key_outlier_mult)
    q = torch.randn((w.tokens, w.num_q_heads, HEAD_DIM), generator=gen_dev, device=dev,
                    dtype=torch.bfloat16)
    topk = None
    if w.topk_given:
        topk = draw_topk_given(seq_lens, w.qlen, w.num_kv_heads, gen_host).to(dev)
    q_scale = 1.0
    if w.fp8_query:   # per-tensor dynamic scale: the largest magnitude maps to 448
        qf = q.float()
        q_scale = float(qf.abs().max()) / FP8_MAX
        q = (qf / q_scale).to(torch.float8_e4m3fn)
    index_k, index_k_scale = None, 1.0
    if w.index_k:
        index_k, index_k_scale = draw_index_k(nb, w.num_kv_heads, gen_dev, dev, std=w.kv_std,
                                              scale_mode=w.kv_scale_mode)
    return StepInputs(q=q, kv=kv, block_table=bt.to(dev),
                      seq_lens=torch.tensor(seq_lens, dtype=torch.int32, device=dev),
                      seq_lens_list=list(seq_lens), k_scale=k_scale, v_scale=v_scale,
                      sm_scale=HEAD_DIM ** -0.5, qlen=w.qlen, num_q_heads=w.num_q_heads,
                      num_kv_heads=w.num_kv_heads, topk=topk, q_scale=q_scale,
                      index_k=index_k, index_k_scale=index_k_scale)


def make_custom(seq_lens: list[int], qlen: int, num_q_heads: int, num_kv_heads: int,
                seed: int, device="cpu", kv_std: float = 1.0, kv_scale_mode: str = "unit",
                key_outlier_frac: float = 0.0, key_outlier_mult: float = 1.0,
                min_stride: int = 1, q_std: float = 1.0) -> StepInputs:
    """Inputs of arbitrary small shape, for tests."""
    gen_host = torch.Generator().manual_seed(seed)
    bt, nb = paged_layout(seq_lens, gen_host, min_stride=min_stride)
    dev = torch.device(device)
    gen_dev = torch.Generator(device=dev).manual_seed(seed + 17)
    kv, k_scale, v_scale = draw_kv(nb, num_kv_heads, gen_dev, dev, std=kv_std,
                                   scale_mode=kv_scale_mode, outlier_frac=key_outlier_frac,
                                   outlier_mult=key_outlier_mult)
    q = torch.randn((len(seq_lens) * qlen, num_q_heads, HEAD_DIM), generator=gen_dev,
                    device=dev, dtype=torch.bfloat16)
    if q_std != 1.0:
        q = (q.float() * q_std).to(torch.bfloat16)
    return StepInputs(q=q, kv=kv, block_table=bt.to(dev),
                      seq_lens=torch.tensor(seq_lens, dtype=torch.int32, device=dev),
                      seq_lens_list=list(seq_lens), k_scale=k_scale, v_scale=v_scale,
                      sm_scale=HEAD_DIM ** -0.5, qlen=qlen, num_q_heads=num_q_heads,
                      num_kv_heads=num_kv_heads)


def make_prefill(q_lens: list[int], seq_lens: list[int], num_q_heads: int, num_kv_heads: int,
                 seed: int, device="cpu", kv_std: float = 1.0, kv_scale_mode: str = "unit",
                 min_stride: int = 1, fp8_query: bool = False) -> StepInputs:
    """Seeded inputs of a prefill or chunked-prefill batch (the vLLM prefill
    test's recipe: q ~ N(0, 1) in bf16, K and V as draw_kv, pages scattered by
    paged_layout): request b's q_lens[b] query tokens are the last ones of its
    seq_lens[b], as MiniMaxM3SparsePrefillMetadata describes them.  With
    fp8_query the query is quantised per tensor (scale amax / 448)."""
    if len(q_lens) != len(seq_lens) or any(q < 0 or q > L for q, L in zip(q_lens, seq_lens)):
        raise ValueError("need one q_len per request with 0 <= q_len <= seq_len")
    gen_host = torch.Generator().manual_seed(seed)
    bt, nb = paged_layout(seq_lens, gen_host, min_stride=min_stride)
    dev = torch.device(device)
    gen_dev = torch.Generator(device=dev).manual_seed(seed + 17)
    kv, k_scale, v_scale = draw_kv(nb, num_kv_heads, gen_dev, dev, std=kv_std,
                                   scale_mode=kv_scale_mode)
    q = torch.randn((sum(q_lens), num_q_heads, HEAD_DIM), generator=gen_dev, device=dev,
                    dtype=torch.bfloat16)
    q_scale = 1.0
    if fp8_query:
        qf = q.float()
        q_scale = float(qf.abs().max()) / FP8_MAX
        q = (qf / q_scale).to(torch.float8_e4m3fn)
    cu = [0]
    for n in q_lens:
        cu.append(cu[-1] + n)
    return StepInputs(q=q, kv=kv, block_table=bt.to(dev),
                      seq_lens=torch.tensor(seq_lens, dtype=torch.int32, device=dev),
                      seq_lens_list=list(seq_lens), k_scale=k_scale, v_scale=v_scale,
                      sm_scale=HEAD_DIM ** -0.5, qlen=0, num_q_heads=num_q_heads,
                      num_kv_heads=num_kv_heads, q_scale=q_scale, q_lens=list(q_lens),
                      cu_seqlens_q=torch.tensor(cu, dtype=torch.int32, device=dev))
