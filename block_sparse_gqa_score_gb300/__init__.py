"""GB300-native (sm_103a) block-sparse GQA decode over a paged fp8 KV cache.

One decode step of MiniMax-M3-style indexer-selected sparse attention, as the
vLLM MiniMax-M3 sparse attention pages and TensorRT-LLM PR #17171 describe it:

  score()          each block's largest visible scaled q.k over a KV head's query heads
  topk()           top-16 blocks (current block kept, ties to the lower index)
  sparse_decode()  split-K attention over the selected pages (+ merge)
  sparse_prefill() the same attend for prefill batches (one query length per
                   request, cu_seqlens_q)
  combine()        merge of split-K partials
  decode_step()    the three stages back to back on one stream

Every function here only checks and marshals torch tensors into the C ABI of
libmsa.so (include/msa.h); all arithmetic runs in that library's CUDA kernels.
There is no CPU fallback: if the library is missing, calls raise.

Tensor layouts (see include/msa.h): q bf16 [T, Hq, 128] with T = B * qlen
request-major; kv fp8 e4m3 [num_blocks, Hkv, 128, 256] (K bytes 0..127, V bytes
128..255), given as uint8 or float8_e4m3fn; block_table int32 [B, S];
seq_lens int32 [B]; scores fp32 [Hkv, T, S]; topk int32 [T, Hkv, 16].
"""
from __future__ import annotations

import ctypes
import math
from dataclasses import dataclass

import torch

from . import _native
from ._native import MSAError  # noqa: F401

HEAD_DIM = 128
PAGE_SIZE = 128
TOPK = 16
GROUP = 16
MAX_QLEN = 32

__all__ = ["score", "topk", "sparse_decode", "sparse_decode_select", "sparse_prefill",
           "sparse_prefill_select", "dense_decode", "dense_splits",
           "combine", "decode_step",
           "fused_selection", "FUSED_MAX_BLOCKS", "workspace_bytes",
           "choose_splits", "get_error", "set_input_overlap", "set_union_tile", "DecodeBuffers",
           "MSAError"]


def _lib():
    return _native.load()


def _stream(device: torch.device, stream) -> ctypes.c_void_p:
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return ctypes.c_void_p(s.cuda_stream)


def _need(t: torch.Tensor, name: str, dtypes, device=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype not in dtypes:
        raise TypeError(f"{name} must have dtype in {dtypes}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if device is not None and t.device != device:
        raise ValueError(f"{name} must be on {device}")


_KV_DTYPES = (torch.uint8, torch.float8_e4m3fn)


_FP8_Q = getattr(torch, "float8_e4m3fn", None)


def _geometry(q, kv, block_table, seq_lens, qlen: int | None, k_only_ok: bool = False):
    """Shapes of a step's inputs; q must hold B * qlen tokens (qlen None: any).
    k_only_ok: kv may also be a K-only cache [num_blocks, Hkv, 128, 128]."""
    _need(q, "q", (torch.bfloat16,) + ((_FP8_Q,) if _FP8_Q is not None else ()))
    dev = q.device
    _need(kv, "kv", _KV_DTYPES, dev)
    _need(block_table, "block_table", (torch.int32,), dev)
    _need(seq_lens, "seq_lens", (torch.int32,), dev)
    if kv.dim() != 4 or kv.shape[2] != PAGE_SIZE or not (
            kv.shape[3] == 2 * HEAD_DIM or (k_only_ok and kv.shape[3] == HEAD_DIM)):
        raise ValueError("kv must be [num_blocks, Hkv, 128, 256]"
                         + (" (or a K-only [num_blocks, Hkv, 128, 128])" if k_only_ok else ""))
    if q.dim() != 3 or q.shape[2] != HEAD_DIM:
        raise ValueError("q must be [T, Hq, 128]")
    if block_table.dim() != 2 or seq_lens.dim() != 1 or block_table.shape[0] != seq_lens.shape[0]:
        raise ValueError("block_table must be [B, S] and seq_lens [B]")
    B, S = block_table.shape
    Hkv = kv.shape[1]
    Hq = q.shape[1]
    if qlen is not None and q.shape[0] != B * qlen:
        raise ValueError(f"q has {q.shape[0]} tokens, expected B*qlen = {B * qlen}")
    return dev, int(B), int(S), int(Hq), int(Hkv), int(kv.shape[0])


def workspace_bytes(batch: int, qlen: int, num_q_heads: int, num_splits: int) -> int:
    return int(_lib().msa_workspace_bytes(batch, qlen, num_q_heads, num_splits))


def choose_splits(batch: int, qlen: int, num_kv_heads: int, sm_count: int | None = None) -> int:
    if sm_count is None:
        sm_count = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    return int(_lib().msa_choose_splits(batch, qlen, num_kv_heads, sm_count))


def _fp8(q, q_scale: float) -> bool:
    """Whether q is an fp8 query (then its value is q * q_scale)."""
    if q.dtype == torch.bfloat16:
        return False
    if not (q_scale > 0 and math.isfinite(q_scale)):
        raise ValueError("an fp8 query needs a finite q_scale > 0")
    return True


def score(q, kv, block_table, seq_lens, qlen: int, sm_scale: float, k_scale: float = 1.0,
          scores: torch.Tensor | None = None, stream=None, q_scale: float = 1.0) -> torch.Tensor:
    """Block scores fp32 [Hkv, T, S] (msa_score; msa_score_q8 for an fp8 q of
    value q * q_scale).  `kv` may be the packed K|V cache [NB, Hkv, 128, 256]
    or a K-only (index-K) cache [NB, Hkv, 128, 128] (msa_score_kcache)."""
    dev, B, S, Hq, Hkv, NB = _geometry(q, kv, block_table, seq_lens, qlen, k_only_ok=True)
    if scores is None:
        scores = torch.empty((Hkv, B * qlen, S), dtype=torch.float32, device=dev)
    _need(scores, "scores", (torch.float32,), dev)
    if tuple(scores.shape) != (Hkv, B * qlen, S):
        raise ValueError("scores must be [Hkv, T, S]")
    args = (kv.data_ptr(), block_table.data_ptr(), seq_lens.data_ptr(), scores.data_ptr(), B, qlen,
            Hq, Hkv, S, NB, float(sm_scale), float(k_scale), _stream(dev, stream))
    k_only = kv.shape[3] == HEAD_DIM
    if _fp8(q, q_scale):
        f = _lib().msa_score_kcache_q8 if k_only else _lib().msa_score_q8
        st = f(q.data_ptr(), float(q_scale), *args)
    else:
        f = _lib().msa_score_kcache if k_only else _lib().msa_score
        st = f(q.data_ptr(), *args)
    _native.check(st, "msa_score")
    return scores


def topk(scores: torch.Tensor, seq_lens: torch.Tensor, qlen: int, k: int = TOPK,
         out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Selected blocks int32 [T, Hkv, 16] (msa_topk).  `scores` is indexed
    [g, i, n] and may be any strided view (e.g. a transpose of [Hkv, S, T])."""
    if not (isinstance(scores, torch.Tensor) and scores.is_cuda and scores.dtype == torch.float32):
        raise TypeError("scores must be a CUDA float32 tensor")
    dev = scores.device
    _need(seq_lens, "seq_lens", (torch.int32,), dev)
    Hkv, T, S = scores.shape
    B = seq_lens.shape[0]
    if T != B * qlen:
        raise ValueError("scores' token dim must be B*qlen")
    if out is None:
        out = torch.empty((T, Hkv, k), dtype=torch.int32, device=dev)
    _need(out, "out", (torch.int32,), dev)
    sh, stt, sn = scores.stride()
    st = _lib().msa_topk(scores.data_ptr(), sh, stt, sn, seq_lens.data_ptr(), out.data_ptr(), B,
                         qlen, Hkv, S, k, _stream(dev, stream))
    _native.check(st, "msa_topk")
    return out


def sparse_decode(q, kv, block_table, seq_lens, topk_idx, qlen: int, sm_scale: float,
                  k_scale: float = 1.0, v_scale: float = 1.0, out: torch.Tensor | None = None,
                  num_splits: int = 0, workspace: torch.Tensor | None = None,
                  stream=None, q_scale: float = 1.0) -> torch.Tensor:
    """Attention over the selected pages, bf16 [T, Hq, 128] (msa_sparse_decode;
    with more than one split the merge runs on the same stream)."""
    dev, B, S, Hq, Hkv, NB = _geometry(q, kv, block_table, seq_lens, qlen)
    _need(topk_idx, "topk", (torch.int32,), dev)
    if tuple(topk_idx.shape) != (B * qlen, Hkv, TOPK):
        raise ValueError("topk must be [T, Hkv, 16]")
    if out is None:
        out = torch.empty(q.shape, dtype=torch.bfloat16, device=dev)
    _need(out, "out", (torch.bfloat16,), dev)
    splits = num_splits if num_splits > 0 else choose_splits(B, qlen, Hkv)
    need = workspace_bytes(B, qlen, Hq, splits)
    if need and (workspace is None or workspace.numel() * workspace.element_size() < need):
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    args = (kv.data_ptr(), block_table.data_ptr(), seq_lens.data_ptr(), topk_idx.data_ptr(), ws_ptr,
            ws_bytes, out.data_ptr(), B, qlen, Hq, Hkv, S, NB, float(sm_scale), float(k_scale),
            float(v_scale), splits, _stream(dev, stream))
    if _fp8(q, q_scale):
        st = _lib().msa_sparse_decode_q8(q.data_ptr(), float(q_scale), *args)
    else:
        st = _lib().msa_sparse_decode(q.data_ptr(), *args)
    _native.check(st, "msa_sparse_decode")
    return out


def dense_splits(stride: int) -> int:
    """Split count of dense_decode for a block table of `stride` columns (0:
    longer than dense_decode takes)."""
    return int(_lib().msa_dense_splits(int(stride)))


def dense_decode(q, kv, block_table, seq_lens, qlen: int, sm_scale: float, k_scale: float = 1.0,
                 v_scale: float = 1.0, out: torch.Tensor | None = None,
                 workspace: torch.Tensor | None = None, stream=None,
                 q_scale: float = 1.0) -> torch.Tensor:
    """Attention over every visible block, bf16 [T, Hq, 128] (msa_dense_decode;
    with more than one split the merge runs on the same stream)."""
    dev, B, S, Hq, Hkv, NB = _geometry(q, kv, block_table, seq_lens, qlen)
    if out is None:
        out = torch.empty(q.shape, dtype=torch.bfloat16, device=dev)
    _need(out, "out", (torch.bfloat16,), dev)
    splits = dense_splits(S)
    if splits == 0:
        raise ValueError("dense_decode takes block tables of at most 2048 columns")
    need = workspace_bytes(B, qlen, Hq, splits)
    if need and (workspace is None or workspace.numel() * workspace.element_size() < need):
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    args = (kv.data_ptr(), block_table.data_ptr(), seq_lens.data_ptr(), ws_ptr, ws_bytes,
            out.data_ptr(), B, qlen, Hq, Hkv, S, NB, float(sm_scale), float(k_scale),
            float(v_scale), _stream(dev, stream))
    if _fp8(q, q_scale):
        st = _lib().msa_dense_decode_q8(q.data_ptr(), float(q_scale), *args)
    else:
        st = _lib().msa_dense_decode(q.data_ptr(), *args)
    _native.check(st, "msa_dense_decode")
    return out


#: Rows of at most this many candidate blocks are selected inside the attend
#: kernel (the selector keeps them in registers there); longer rows go through
#: the selector kernel, which holds up to 2048 candidates in registers.
FUSED_MAX_BLOCKS = 512


def fused_selection(stride: int) -> bool:
    """Whether decode_step selects inside the attend kernel for a block table of
    `stride` columns (the longest possible row)."""
    return stride <= FUSED_MAX_BLOCKS


def sparse_decode_select(q, kv, block_table, seq_lens, scores, qlen: int, sm_scale: float,
                         k_scale: float = 1.0, v_scale: float = 1.0,
                         topk_out: torch.Tensor | None = None, out: torch.Tensor | None = None,
                         num_splits: int = 0, workspace: torch.Tensor | None = None,
                         stream=None, q_scale: float = 1.0):
    """Selection and attention in one kernel (msa_sparse_decode_select): the
    top-16 blocks of every (token, KV head) row are selected from `scores`
    (any strides, as msa_topk) and attended.  Returns (topk [T, Hkv, 16], out)."""
    dev, B, S, Hq, Hkv, NB = _geometry(q, kv, block_table, seq_lens, qlen)
    # any strided view, as for topk()
    if not (isinstance(scores, torch.Tensor) and scores.is_cuda and scores.dtype == torch.float32
            and scores.device == dev):
        raise TypeError("scores must be a float32 tensor on q's device")
    if scores.dim() != 3 or scores.shape[0] != Hkv or scores.shape[1] != B * qlen \
            or scores.shape[2] < S:
        raise ValueError("scores must be [Hkv, T, >= S]")
    if topk_out is None:
        topk_out = torch.empty((B * qlen, Hkv, TOPK), dtype=torch.int32, device=dev)
    _need(topk_out, "topk_out", (torch.int32,), dev)
    if out is None:
        out = torch.empty(q.shape, dtype=torch.bfloat16, device=dev)
    _need(out, "out", (torch.bfloat16,), dev)
    splits = num_splits if num_splits > 0 else choose_splits(B, qlen, Hkv)
    need = workspace_bytes(B, qlen, Hq, splits)
    if need and (workspace is None or workspace.numel() * workspace.element_size() < need):
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    sh, st, sn = scores.stride()
    args = (kv.data_ptr(), block_table.data_ptr(), seq_lens.data_ptr(), scores.data_ptr(), sh, st,
            sn, topk_out.data_ptr(), ws_ptr, ws_bytes, out.data_ptr(), B, qlen, Hq, Hkv, S, NB,
            float(sm_scale), float(k_scale), float(v_scale), splits, _stream(dev, stream))
    if _fp8(q, q_scale):
        status = _lib().msa_sparse_decode_select_q8(q.data_ptr(), float(q_scale), *args)
    else:
        status = _lib().msa_sparse_decode_select(q.data_ptr(), *args)
    _native.check(status, "msa_sparse_decode_select")
    return topk_out, out


def _prefill_geometry(q, kv, block_table, seq_lens, cu_seqlens_q):
    """Shapes of a prefill-style batch: q holds T tokens, request b owning
    tokens cu_seqlens_q[b] .. cu_seqlens_q[b + 1] - 1."""
    dev, B, S, Hq, Hkv, NB = _geometry(q, kv, block_table, seq_lens, None)
    _need(cu_seqlens_q, "cu_seqlens_q", (torch.int32,), dev)
    if tuple(cu_seqlens_q.shape) != (B + 1,):
        raise ValueError("cu_seqlens_q must be [B + 1]")
    return dev, B, int(q.shape[0]), S, Hq, Hkv, NB


def _prefill_splits(T: int, Hq: int, Hkv: int, num_splits: int, workspace, dev):
    # one CTA per token: the single-token rule, choose_splits(T, 1, ...)
    splits = num_splits if num_splits > 0 else choose_splits(max(T, 1), 1, Hkv)
    need = workspace_bytes(max(T, 1), 1, Hq, splits)
    if need and (workspace is None or workspace.numel() * workspace.element_size() < need):
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    return splits, ws_ptr, ws_bytes


def sparse_prefill(q, kv, block_table, seq_lens, cu_seqlens_q, topk_idx, sm_scale: float,
                   k_scale: float = 1.0, v_scale: float = 1.0, out: torch.Tensor | None = None,
                   num_splits: int = 0, workspace: torch.Tensor | None = None, stream=None,
                   q_scale: float = 1.0) -> torch.Tensor:
    """Sparse attend of a prefill or chunked-prefill batch (msa_sparse_prefill):
    request b's query tokens are q[cu_seqlens_q[b] : cu_seqlens_q[b + 1]], the
    last ones of its seq_lens[b]; each token attends its own list
    topk_idx [T, Hkv, 16].  Returns bf16 [T, Hq, 128]."""
    dev, B, T, S, Hq, Hkv, NB = _prefill_geometry(q, kv, block_table, seq_lens, cu_seqlens_q)
    _need(topk_idx, "topk", (torch.int32,), dev)
    if tuple(topk_idx.shape) != (T, Hkv, TOPK):
        raise ValueError("topk must be [T, Hkv, 16]")
    if out is None:
        out = torch.empty(q.shape, dtype=torch.bfloat16, device=dev)
    _need(out, "out", (torch.bfloat16,), dev)
    splits, ws_ptr, ws_bytes = _prefill_splits(T, Hq, Hkv, num_splits, workspace, dev)
    args = (kv.data_ptr(), block_table.data_ptr(), seq_lens.data_ptr(), cu_seqlens_q.data_ptr(),
            topk_idx.data_ptr(), ws_ptr, ws_bytes, out.data_ptr(), B, T, Hq, Hkv, S, NB,
            float(sm_scale), float(k_scale), float(v_scale), splits, _stream(dev, stream))
    if _fp8(q, q_scale):
        st = _lib().msa_sparse_prefill_q8(q.data_ptr(), float(q_scale), *args)
    else:
        st = _lib().msa_sparse_prefill(q.data_ptr(), *args)
    _native.check(st, "msa_sparse_prefill")
    return out


def sparse_prefill_select(q, kv, block_table, seq_lens, cu_seqlens_q, scores, sm_scale: float,
                          k_scale: float = 1.0, v_scale: float = 1.0,
                          topk_out: torch.Tensor | None = None, out: torch.Tensor | None = None,
                          num_splits: int = 0, workspace: torch.Tensor | None = None,
                          stream=None, q_scale: float = 1.0):
    """Per-token causal top-16 selected from `scores` [Hkv, T, >= S] (any
    strides) and attended, for a prefill-style batch
    (msa_sparse_prefill_select).  Returns (topk [T, Hkv, 16], out)."""
    dev, B, T, S, Hq, Hkv, NB = _prefill_geometry(q, kv, block_table, seq_lens, cu_seqlens_q)
    if not (isinstance(scores, torch.Tensor) and scores.is_cuda and scores.dtype == torch.float32
            and scores.device == dev):
        raise TypeError("scores must be a float32 tensor on q's device")
    if scores.dim() != 3 or scores.shape[0] != Hkv or scores.shape[1] != T \
            or scores.shape[2] < S:
        raise ValueError("scores must be [Hkv, T, >= S]")
    if topk_out is None:
        topk_out = torch.empty((T, Hkv, TOPK), dtype=torch.int32, device=dev)
    _need(topk_out, "topk_out", (torch.int32,), dev)
    if out is None:
        out = torch.empty(q.shape, dtype=torch.bfloat16, device=dev)
    _need(out, "out", (torch.bfloat16,), dev)
    splits, ws_ptr, ws_bytes = _prefill_splits(T, Hq, Hkv, num_splits, workspace, dev)
    sh, st, sn = scores.stride()
    args = (kv.data_ptr(), block_table.data_ptr(), seq_lens.data_ptr(), cu_seqlens_q.data_ptr(),
            scores.data_ptr(), sh, st, sn, topk_out.data_ptr(), ws_ptr, ws_bytes, out.data_ptr(),
            B, T, Hq, Hkv, S, NB, float(sm_scale), float(k_scale), float(v_scale), splits,
            _stream(dev, stream))
    if _fp8(q, q_scale):
        status = _lib().msa_sparse_prefill_select_q8(q.data_ptr(), float(q_scale), *args)
    else:
        status = _lib().msa_sparse_prefill_select(q.data_ptr(), *args)
    _native.check(status, "msa_sparse_prefill_select")
    return topk_out, out


def combine(workspace: torch.Tensor, tokens: int, num_q_heads: int, num_splits: int,
            out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Merge split-K partials (layout of msa_workspace_bytes) into bf16 [T, Hq, 128]."""
    if not (isinstance(workspace, torch.Tensor) and workspace.is_cuda):
        raise TypeError("workspace must be a CUDA tensor")
    dev = workspace.device
    if out is None:
        out = torch.empty((tokens, num_q_heads, HEAD_DIM), dtype=torch.bfloat16, device=dev)
    _need(out, "out", (torch.bfloat16,), dev)
    st = _lib().msa_combine(workspace.data_ptr(), out.data_ptr(), tokens, num_q_heads, num_splits,
                            _stream(dev, stream))
    _native.check(st, "msa_combine")
    return out


@dataclass
class DecodeBuffers:
    """Preallocated outputs and workspace of one decode step (reusable, and
    stable addresses for CUDA-graph capture)."""
    scores: torch.Tensor
    topk: torch.Tensor
    out: torch.Tensor
    workspace: torch.Tensor | None
    num_splits: int

    @staticmethod
    def allocate(batch: int, qlen: int, num_q_heads: int, num_kv_heads: int, stride: int,
                 device, num_splits: int = 0) -> "DecodeBuffers":
        T = batch * qlen
        splits = num_splits if num_splits > 0 else choose_splits(batch, qlen, num_kv_heads)
        need = workspace_bytes(batch, qlen, num_q_heads, splits)
        ws = torch.empty(need, dtype=torch.uint8, device=device) if need else None
        return DecodeBuffers(
            scores=torch.empty((num_kv_heads, T, stride), dtype=torch.float32, device=device),
            topk=torch.empty((T, num_kv_heads, TOPK), dtype=torch.int32, device=device),
            out=torch.empty((T, num_q_heads, HEAD_DIM), dtype=torch.bfloat16, device=device),
            workspace=ws, num_splits=splits)


def decode_step(q, kv, block_table, seq_lens, qlen: int, sm_scale: float, k_scale: float = 1.0,
                v_scale: float = 1.0, buffers: DecodeBuffers | None = None, stream=None,
                q_scale: float = 1.0, index_k: torch.Tensor | None = None,
                index_k_scale: float | None = None):
    """One decode step in one library call (msa_decode_step): score, then
    selection + attention on one stream, no host sync -- in one kernel
    (msa_sparse_decode_select) while rows have at most FUSED_MAX_BLOCKS
    candidate blocks, else msa_topk then msa_sparse_decode (-> combine when
    split).  With `index_k` (a K-only cache [NB, Hkv, 128, 128] on the same
    block table, scale index_k_scale, default k_scale) the blocks are scored
    on it instead of kv's K halves.  Returns (scores, topk, out)."""
    dev, B, S, Hq, Hkv, NB = _geometry(q, kv, block_table, seq_lens, qlen)
    if buffers is None:
        buffers = DecodeBuffers.allocate(B, qlen, Hq, Hkv, S, dev)
    if index_k is not None:
        _need(index_k, "index_k", _KV_DTYPES, dev)
        if (index_k.dim() != 4 or index_k.shape[1] != Hkv or index_k.shape[2] != PAGE_SIZE
                or index_k.shape[3] != HEAD_DIM or index_k.shape[0] != NB):
            raise ValueError("index_k must be [num_blocks, Hkv, 128, 128]")
    bf = buffers
    _need(bf.scores, "scores", (torch.float32,), dev)
    _need(bf.topk, "topk", (torch.int32,), dev)
    _need(bf.out, "out", (torch.bfloat16,), dev)
    if (tuple(bf.scores.shape) != (Hkv, B * qlen, S) or tuple(bf.topk.shape) != (B * qlen, Hkv, TOPK)
            or tuple(bf.out.shape) != tuple(q.shape)):
        raise ValueError("buffers do not match the step's shapes")
    ws = bf.workspace
    ws_ptr = ws.data_ptr() if ws is not None else None
    ws_bytes = ws.numel() * ws.element_size() if ws is not None else 0
    fp8 = _fp8(q, q_scale)
    ik_scale = (k_scale if index_k_scale is None else index_k_scale) if index_k is not None else 0.0
    st = _lib().msa_decode_step(
        q.data_ptr(), float(q_scale) if fp8 else 0.0, kv.data_ptr(),
        index_k.data_ptr() if index_k is not None else None, float(ik_scale),
        block_table.data_ptr(), seq_lens.data_ptr(), bf.scores.data_ptr(), bf.topk.data_ptr(),
        ws_ptr, ws_bytes, bf.out.data_ptr(), B, qlen, Hq, Hkv, S, NB, float(sm_scale),
        float(k_scale), float(v_scale), bf.num_splits, _stream(dev, stream))
    _native.check(st, "msa_decode_step")
    return bf.scores, bf.topk, bf.out


def set_union_tile(enable: bool) -> bool:
    """msa_set_union_tile: attend sparse decode steps of two or more tokens per
    request over the union of each 4-token tile's lists, loading each shared
    page once (pays off when a request's tokens list mostly the same blocks).
    Off by default; dense decode always works this way.  Returns the previous
    setting."""
    return bool(_lib().msa_set_union_tile(1 if enable else 0))


def set_input_overlap(enable: bool) -> bool:
    """msa_set_input_overlap: let the first kernel of every library call start
    before the previous kernel on its stream has finished (only safe when that
    kernel wrote none of the call's inputs, e.g. another library call).  Off
    by default.  Returns the previous setting."""
    return bool(_lib().msa_set_input_overlap(1 if enable else 0))


def get_error(clear: bool = True) -> int:
    """The device's sticky MSA_ERR_* bits (synchronises the device)."""
    flags = ctypes.c_uint(0)
    _native.check(_lib().msa_get_error(ctypes.byref(flags), 1 if clear else 0), "msa_get_error")
    return int(flags.value)
