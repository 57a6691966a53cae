#!/usr/bin/env python3
"""Benchmark of the sparse-decode step (score -> select -> attend -> merge).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME]

Prints ONE JSON line.  A step is one pass of the whole decode step for one
layer's batch: msa_score, then msa_sparse_decode_select (the block selection
and the attend in one kernel; + msa_combine when split).  Inputs are synthetic and resident in HBM before the timed region; the
layers rotate over independent KV pools whose total size is >= 4x the L2, so
no step finds its inputs in L2.  The timed region is a CUDA-graph replay of
the K steps (kernels only), bracketed by CUDA events on the launch stream.
Each kernel's own duration (for the roofline figures) is taken right after it
from a graph of that kernel's launches alone.  value = query tokens / s (per
layer, all ranks).

--impl reference times the CPU oracle (the only reference implementation of
this method available here) on the host cores: each step runs the oracle's
whole pipeline for one (request, KV head) unit of the same workload.

Under torchrun each rank runs an independent replica on its own GPU (the step
has no exchange); rank 0 prints the max-over-ranks timing.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = "sparse-decode query-tokens/s per layer"
UNIT = "tokens/s"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_SUSTAINED_TFLOPS = 1700.0   # sustained dense bf16 GEMM rate of a GB300, when unmeasured
PROFILES = os.path.join(ROOT, "profiles")


# ----------------------------------------------------------------------------- helpers

def _args():
    from block_sparse_gqa_score_gb300 import workloads as wl
    ap = argparse.ArgumentParser(
        description="One JSON line: query tokens/s per layer of a workload's step, with the "
                    "dominant kernel's roofline, the end-to-end figure and the CPU oracle's.")
    ap.add_argument("--gpus", type=int, default=1,
                    help="ranks, one GPU each (N > 1: launched under torchrun, replicas)")
    ap.add_argument("--steps", type=int, default=2000, help="timed steps")
    ap.add_argument("--warmup", type=int, default=50, help="untimed warm-up steps (at least 3 for a valid measurement)")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours",
                    help="ours: the CUDA library; reference: the fp64 CPU oracle, one "
                         "(request, KV head) unit per step")
    ap.add_argument("--workload", default=None, choices=sorted(wl.WORKLOADS),
                    help=f"default: {wl.HEADLINE}")
    ap.add_argument("--no-e2e", action="store_true",
                    help="skip the end-to-end measurement (host copies, public API)")
    ap.add_argument("--no-cpu-baseline", action="store_true",
                    help="skip timing the CPU oracle beside the line")
    ap.add_argument("--input-overlap", action="store_true",
                    help="msa_set_input_overlap(1) for the timed steps: each step's first kernel "
                         "may start while the previous step's last kernel finishes (valid here: "
                         "that kernel writes none of the step's inputs); default off")
    ap.add_argument("--union-tile", action="store_true",
                    help="msa_set_union_tile(1): attend each request's 4-token tiles over the union "
                         "of their lists (default: one CTA per token)")
    ap.add_argument("--graph-chunk", type=int, default=250,
                    help="steps captured per CUDA graph in the timed region")
    return ap.parse_args()


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return rank, world, local


def _barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def _max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def _fp8_tensor_peak():
    """Dense fp8 tensor peak in TFLOP/s: the measured sustained bf16 GEMM rate
    (the kernels are timed in long back-to-back loops) times 2, the nominal
    fp8 / bf16 ratio (4.5 / 2.25 PFLOP/s)."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return 2.0 * float(d["bf16_tflops_sustained"]), "measured (bf16 sustained x 2)"
    except Exception:
        return 2.0 * FALLBACK_BF16_SUSTAINED_TFLOPS, "fallback (bf16 sustained x 2)"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled in the background; the
    samples that arrive between mark_start() and mark_stop() are kept."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int, period_ms: int = 20):
        self.samples = []
        self.t0 = self.t1 = None
        self.proc = None
        try:
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            target = uuid if uuid.startswith("GPU-") else f"GPU-{uuid}"
        except Exception:
            target = os.environ.get("CUDA_VISIBLE_DEVICES", "0").split(",")[device_index]
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", target, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", f"-lms", str(period_ms)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), line.strip()))

    def mark_start(self):
        self.t0 = time.time()

    def mark_stop(self):
        self.t1 = time.time()

    def summary(self):
        if self.proc is not None:
            time.sleep(0.05)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        inside = [s for t, s in self.samples if self.t0 <= t <= self.t1]
        where = "timed region"
        if not inside:   # timed region shorter than the sampling period
            inside = [s for t, s in self.samples if t >= self.t0 - 0.5][:3]
            where = "nearest samples (timed region shorter than the sampling period)"
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for s in inside:
            parts = [p.strip() for p in s.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
                power.append(float(parts[2]))
            except ValueError:
                continue
            for name, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None,
                "reasons": sorted(reasons), "samples": len(sm), "window": where}


def _code_only(src: str) -> str:
    """A CUDA source without its comments and blank space: what the compiler
    sees, so that an edit to a comment leaves a kernel's digest unchanged."""
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    src = re.sub(r"//[^\n]*", "", src)
    return "\n".join(line.strip() for line in src.splitlines() if line.strip())


def _source_digest(*names) -> str:
    """Digest of a kernel's sources (code only), recorded with each ncu summary
    under profiles/: a summary whose digest differs describes other code."""
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "block_sparse_gqa_score_gb300", "csrc", n)) as f:
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


KERNEL_SOURCES = {"attend": ("msa_attend.cu", "msa_union.cu", "msa_device.cuh", "msa_tcgen05.cuh",
                             "msa_launch.h", "msa_select.cuh"),
                  "score": ("msa_score.cu", "msa_device.cuh", "msa_tcgen05.cuh", "msa_launch.h"),
                  "topk": ("msa_topk.cu", "msa_device.cuh", "msa_launch.h", "msa_select.cuh")}


def _traffic_from_profiles(stage: str, workload: str):
    """DRAM bytes per launch recorded from an ncu capture in profiles/, or None
    when absent or taken on different kernel source."""
    path = os.path.join(PROFILES, f"{stage}_kernel_{workload}.txt")
    if not os.path.exists(path):
        return None
    fields = {}
    with open(path) as f:
        for line in f:
            if ":" in line and not line.startswith("#"):
                k, v = line.split(":", 1)
                fields[k.strip()] = v.strip()
    if fields.get("source_digest") != _source_digest(*KERNEL_SOURCES[stage]):
        return None
    try:
        return float(fields["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


# ----------------------------------------------------------------------------- work accounting

def _work(inp, topk_cpu: np.ndarray | None, reads_lists: bool = True):
    """Algorithmic bytes per launch of each stage, and the scorer's useful flops."""
    B, Hq, Hkv, S = inp.batch, inp.num_q_heads, inp.num_kv_heads, inp.stride
    # query tokens per request (one length per request in a prefill batch)
    q_lens = inp.q_lens if inp.q_lens is not None else [inp.qlen] * B
    first = np.concatenate([[0], np.cumsum(q_lens)]).astype(int)
    T = int(first[-1])
    pages = [math.ceil(L / 128) for L in inp.seq_lens_list]
    q_bytes = T * Hq * 128 * inp.q.element_size()   # bf16, or an fp8 query
    out_bytes = T * Hq * 128 * 2
    score = sum(pages) * Hkv * 16384 + q_bytes + Hkv * T * S * 4 + B * S * 4
    cand = 0
    for b, L in enumerate(inp.seq_lens_list):
        Q = q_lens[b]
        for j in range(Q):
            pos = L - Q + j
            if pos >= 0:
                cur = pos // 128
                cand += cur if cur + 1 > 16 else 0
    topk = cand * Hkv * 4 + T * Hkv * 16 * 4
    # the scorer's products: every visible page-head's 128 keys against its
    # group's 16 heads x Q tokens, 128-dim dot products
    score_flops = sum(n * Q for n, Q in zip(pages, q_lens)) * Hkv * 2.0 * 128 * 128 * 16
    union = per_token = 0
    if topk_cpu is not None:
        for b in range(B):
            rows = topk_cpu[first[b]:first[b + 1]]      # [q_len, Hkv, 16]
            for g in range(Hkv):
                ids = rows[:, g, :]
                ids = ids[ids >= 0]
                union += len(np.unique(ids))
                per_token += len(ids)
    attend = union * 32768 + q_bytes + out_bytes + (T * Hkv * 16 * 4 if reads_lists else 0)
    return {"score": score, "topk": topk, "attend": attend, "union_pages": union,
            "token_pages": per_token, "attend_kv_bytes": union * 32768, "score_flops": score_flops}


# ----------------------------------------------------------------------------- reference arm

def run_reference(args, rank, world):
    if rank != 0:
        return
    import oracle
    from block_sparse_gqa_score_gb300 import workloads as wl
    name = args.workload or wl.HEADLINE
    w = wl.WORKLOADS[name]
    inp = wl.make_inputs(w, device="cpu")
    p = _problem(inp, oracle)
    cores = oracle.default_threads()
    units = [(b, g) for b in range(inp.batch) for g in range(inp.num_kv_heads)
             if inp.seq_lens_list[b] > 0]

    given = _given_lists(w, inp)
    p_score = _score_problem(inp, oracle, p) if p is not None else None

    def step(k):
        b, g = units[k % len(units)]
        _oracle_unit(p, inp, oracle, b, g, cores, given, p_score)
        return _unit_tokens(inp, b)

    for k in range(args.warmup):
        step(k)
    t0 = time.perf_counter()
    tokens = 0.0
    for k in range(args.steps):
        tokens += step(args.warmup + k)
    dt = time.perf_counter() - t0
    v = tokens / dt
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * dt / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": w.describe(),
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": "one (request, KV head) unit per step, round robin: "
                                       + ("attention of its query rows x 16 heads over the "
                                          "given top-k" if w.topk_given else
                                          "attention of its query rows x 16 heads over every "
                                          "visible block" if w.dense else
                                          "scores of all its visible blocks, selection of its "
                                          "query rows, attention of its query rows x 16 heads")
                                       + "; counted as its query tokens / Hkv"},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def _given_lists(w, inp):
    """The lists the oracle attends over when it does not select them: the
    drawn top-k (attend-only workloads) or every visible block (dense decode)."""
    if w.topk_given:
        return inp.topk.cpu().numpy()
    if w.dense:
        from block_sparse_gqa_score_gb300 import workloads as wl
        return wl.all_visible_lists(inp.seq_lens_list, inp.qlen, inp.num_kv_heads,
                                    inp.stride).numpy()
    return None


def _problem(inp, oracle, b=None):
    """The oracle's problem: the whole batch, or (a prefill batch) request b
    alone with Q = its query length, so that its tokens sit at the last
    positions of its sequence."""
    # an fp8 query (value q * q_scale): its codes as bf16 (exact) with sm_scale * q_scale
    q, sm_scale = inp.q, inp.sm_scale
    if q.dtype != torch.bfloat16:
        q, sm_scale = q.to(torch.bfloat16), inp.sm_scale * inp.q_scale
    bits = q.cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    bt, sl, Q = inp.block_table.cpu().numpy(), inp.seq_lens.cpu().numpy(), inp.qlen
    if inp.q_lens is not None:
        if b is None:
            return None   # built per request by _oracle_unit
        s0, Q = sum(inp.q_lens[:b]), inp.q_lens[b]
        bits, bt, sl = bits[s0:s0 + Q], bt[b:b + 1], sl[b:b + 1]
    return oracle.Problem(bits, inp.kv.cpu().numpy(), bt, sl, Q, inp.num_q_heads,
                          inp.num_kv_heads, sm_scale, inp.k_scale, inp.v_scale)


def _score_problem(inp, oracle, p):
    """The problem the oracle scores on: p itself, or (a workload with a K-only
    index cache) p's query over a packed cache whose K halves are the index-K
    bytes, with the index cache's scale."""
    if inp.index_k is None:
        return p
    k = inp.index_k.cpu().numpy()
    kv = np.zeros(k.shape[:3] + (256,), dtype=np.uint8)
    kv[..., :128] = k
    return oracle.Problem(p.q, kv, p.block_table, p.seq_lens, p.Q, p.Hq, p.Hkv, p.sm_scale,
                          inp.index_k_scale, p.v_scale)


def _unit_tokens(inp, b) -> float:
    """Query tokens one (request, KV head) unit stands for: its request's / Hkv."""
    Q = inp.q_lens[b] if inp.q_lens is not None else inp.qlen
    return Q / inp.num_kv_heads


def _oracle_unit(p, inp, oracle, b, g, nthreads, topk_given=None, p_score=None):
    """The oracle's whole pipeline for one (request, KV head) unit."""
    Q, G = inp.qlen, inp.num_q_heads // inp.num_kv_heads
    if inp.q_lens is not None:
        # a prefill request: its own problem, its rows of the given lists
        s0, Q = sum(inp.q_lens[:b]), inp.q_lens[b]
        rows = [j * inp.num_q_heads + g * G + h for j in range(Q) for h in range(G)]
        oracle.attend_rows(_problem(inp, oracle, b), topk_given[s0:s0 + Q], rows, nthreads)
        return
    L = inp.seq_lens_list[b]
    cur = (L - 1) // 128
    if topk_given is None:
        triples = [(b, g, n) for n in range(cur + 1)]
        s = oracle.score_blocks(p_score if p_score is not None else p, triples, nthreads)
        sub = np.where(np.isnan(s[g:g + 1, b * Q:(b + 1) * Q]), -np.inf,
                       s[g:g + 1, b * Q:(b + 1) * Q])
        t = oracle.topk(sub, np.array([L], dtype=np.int32), Q)       # [Q, 1, 16]
        full = np.full((inp.tokens, inp.num_kv_heads, 16), -1, dtype=np.int32)
        full[b * Q:(b + 1) * Q, g] = t[:, 0]
    else:
        full = topk_given
    rows = [(b * Q + j) * inp.num_q_heads + g * G + h for j in range(Q) for h in range(G)]
    oracle.attend_rows(p, full, rows, nthreads)


def cpu_baseline(inp, w, lists, budget_s: float = 12.0):
    """The oracle timed on this host on a bounded sample of the workload."""
    import oracle
    p = _problem(inp, oracle)
    cores = oracle.default_threads()
    units = [(b, g) for b in range(inp.batch) for g in range(inp.num_kv_heads)
             if inp.seq_lens_list[b] > 0]
    p_score = _score_problem(inp, oracle, p) if p is not None else None
    done, tokens = 0, 0.0
    t0 = time.perf_counter()
    for b, g in units:
        _oracle_unit(p, inp, oracle, b, g, cores, lists, p_score)
        done += 1
        tokens += _unit_tokens(inp, b)
        if time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    # the same units on one thread, for a few seconds
    done1, tokens1 = 0, 0.0
    t1 = time.perf_counter()
    for b, g in units[:done]:
        _oracle_unit(p, inp, oracle, b, g, 1, lists, p_score)
        done1 += 1
        tokens1 += _unit_tokens(inp, b)
        if time.perf_counter() - t1 > budget_s / 4:
            break
    dt1 = time.perf_counter() - t1
    what = ("prefill attend, given per-token top-k" if w.prefill_q else
            "attend only, given top-k" if w.topk_given else "dense attend, every visible block"
            if w.dense else "score, select, attend")
    sample = (f"{done} of {len(units)} (request, KV head) units of layer 0, each the whole "
              f"oracle pipeline ({what})")
    return {"value": tokens / dt, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": sample, "seconds": dt,
            "one_core": {"value": tokens1 / dt1, "units": done1, "seconds": dt1}}


# ----------------------------------------------------------------------------- our arm

def run_ours(args, rank, world, local):
    import block_sparse_gqa_score_gb300 as msa
    from block_sparse_gqa_score_gb300 import build as msa_build
    from block_sparse_gqa_score_gb300 import workloads as wl

    msa_build.build()
    msa._native.load()
    msa.set_input_overlap(args.input_overlap)
    msa.set_union_tile(args.union_tile)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    name = args.workload or wl.HEADLINE
    w = wl.WORKLOADS[name]
    props = torch.cuda.get_device_properties(dev)
    l2 = getattr(props, "L2_cache_size", 128 << 20) or (128 << 20)

    # layers: independent KV pools, total >= 4x L2, at least 2
    first = wl.make_inputs(w, device=dev, layer=0)
    layer_bytes = (first.kv.numel() + first.q.numel() * 2
                   + (first.index_k.numel() if first.index_k is not None else 0))
    n_layers = max(2, math.ceil(4 * l2 / max(layer_bytes, 1)))
    layers = [first] + [wl.make_inputs(w, device=dev, layer=l) for l in range(1, n_layers)]
    T = first.tokens   # every layer has the same request and query lengths
    # buffers and splits sized by tokens: B requests of qlen, or T prefill tokens
    tb, tq = (T, 1) if w.prefill_q else (w.batch, w.qlen)
    splits = msa.choose_splits(tb, tq, w.num_kv_heads, props.multi_processor_count)
    if w.dense:   # the split count of dense decode follows the block table's stride
        splits = max(msa.dense_splits(inp.stride) for inp in layers)
    bufs = [msa.DecodeBuffers.allocate(tb, tq, w.num_q_heads, w.num_kv_heads, inp.stride, dev,
                                       splits) for inp in layers]
    stream = torch.cuda.Stream(dev)

    def stage_calls(l):
        inp, bf = layers[l], bufs[l]
        if w.prefill_q:
            return [lambda: None, lambda: None,
                    lambda: msa.sparse_prefill(inp.q, inp.kv, inp.block_table, inp.seq_lens,
                                               inp.cu_seqlens_q, inp.topk, inp.sm_scale,
                                               inp.k_scale, inp.v_scale, out=bf.out,
                                               num_splits=bf.num_splits, workspace=bf.workspace,
                                               q_scale=inp.q_scale)]
        if w.dense:
            return [lambda: None, lambda: None,
                    lambda: msa.dense_decode(inp.q, inp.kv, inp.block_table, inp.seq_lens,
                                             inp.qlen, inp.sm_scale, inp.k_scale, inp.v_scale,
                                             out=bf.out, workspace=bf.workspace,
                                             q_scale=inp.q_scale)]
        if w.topk_given:
            return [lambda: None, lambda: None,
                    lambda: msa.sparse_decode(inp.q, inp.kv, inp.block_table, inp.seq_lens,
                                              inp.topk, inp.qlen, inp.sm_scale, inp.k_scale,
                                              inp.v_scale, out=bf.out, num_splits=bf.num_splits,
                                              workspace=bf.workspace, q_scale=inp.q_scale)]
        # the blocks are scored on the K-only index cache when the workload has one
        keys, k_sc = ((inp.kv, inp.k_scale) if inp.index_k is None
                      else (inp.index_k, inp.index_k_scale))
        score_call = lambda: msa.score(inp.q, keys, inp.block_table, inp.seq_lens, inp.qlen,
                                       inp.sm_scale, k_sc, scores=bf.scores,
                                       q_scale=inp.q_scale)
        if fused:   # the selection runs inside the attend kernel (msa_sparse_decode_select)
            return [score_call, lambda: None,
                    lambda: msa.sparse_decode_select(inp.q, inp.kv, inp.block_table,
                                                     inp.seq_lens, bf.scores, inp.qlen,
                                                     inp.sm_scale, inp.k_scale, inp.v_scale,
                                                     topk_out=bf.topk, out=bf.out,
                                                     num_splits=bf.num_splits,
                                                     workspace=bf.workspace,
                                                     q_scale=inp.q_scale)]
        return [score_call,
                lambda: msa.topk(bf.scores, inp.seq_lens, inp.qlen, out=bf.topk),
                lambda: msa.sparse_decode(inp.q, inp.kv, inp.block_table, inp.seq_lens, bf.topk,
                                          inp.qlen, inp.sm_scale, inp.k_scale, inp.v_scale,
                                          out=bf.out, num_splits=bf.num_splits,
                                          workspace=bf.workspace, q_scale=inp.q_scale)]

    def step_call(l):
        """One whole step through the public API: msa_decode_step (score, then
        selection and attend in one library call), or the attend alone."""
        inp, bf = layers[l], bufs[l]
        if attend_only:
            stage_calls(l)[2]()
            return
        msa.decode_step(inp.q, inp.kv, inp.block_table, inp.seq_lens, inp.qlen, inp.sm_scale,
                        inp.k_scale, inp.v_scale, buffers=bf, q_scale=inp.q_scale,
                        index_k=inp.index_k, index_k_scale=inp.index_k_scale)

    attend_only = w.topk_given or w.dense
    fused = (not attend_only) and msa.fused_selection(first.stride)
    launches_per_step = (1 if attend_only else (2 if fused else 3)) + (1 if splits > 1 else 0)

    # warm-up (eager), then the per-layer work figures from the real top-k lists
    msa.get_error(clear=True)
    with torch.cuda.stream(stream):
        for k in range(args.warmup):
            step_call(k % n_layers)
    torch.cuda.synchronize(dev)
    flags = msa.get_error(clear=True)
    works = []
    for inp, bf in zip(layers, bufs):
        lists = _given_lists(w, inp)
        works.append(_work(inp, lists if lists is not None else bf.topk.cpu().numpy(),
                           reads_lists=not w.dense))

    # the timed region: CUDA-graph replays of `chunk` steps, kernels only
    chunk = max(1, min(args.steps, args.graph_chunk))
    graphs = []
    mode = "cuda-graph"

    def capture(nsteps, which=None):
        """A graph of `nsteps` whole steps, or of one stage's launches alone
        (`which`: its index in stage_calls), replayed as a chain of library
        calls with the input overlap on (each launch follows another of the
        same kernel, which writes none of its inputs)."""
        g = torch.cuda.CUDAGraph()
        prev = msa.set_input_overlap(which is not None or args.input_overlap)
        try:
            with torch.cuda.graph(g, stream=stream):
                for k in range(nsteps):
                    if which is None:
                        step_call(k % n_layers)
                    else:
                        stage_calls(k % n_layers)[which]()
        finally:
            msa.set_input_overlap(prev)
        return g

    try:
        full, rem = divmod(args.steps, chunk)
        if full:
            graphs.append((capture(chunk), full))
        if rem:
            graphs.append((capture(rem), 1))
    except Exception as e:  # pragma: no cover - depends on the torch build
        mode = f"eager ({type(e).__name__})"
        graphs = []

    clocks = ClockSampler(local)
    time.sleep(0.2)
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    _barrier(world)
    torch.cuda.synchronize(dev)
    clocks.mark_start()
    # One untimed pass of each graph (its upload), enqueued right before the
    # timed replays so that the GPU goes from it into the timed region without
    # idling: after the sampler's start-up pause a 20-step region otherwise
    # began on an idle GPU and measured 4.6 us per step slower than 2000 steps.
    with torch.cuda.stream(stream):
        for g, _n in graphs:
            g.replay()
    start.record(stream)
    with torch.cuda.stream(stream):              # replays launch on the current stream
        if graphs:
            for g, reps in graphs:
                for _ in range(reps):
                    g.replay()
        else:
            for k in range(args.steps):
                step_call(k % n_layers)
    stop.record(stream)
    torch.cuda.synchronize(dev)
    clocks.mark_stop()
    _barrier(world)
    total_ms = _max_over_ranks(start.elapsed_time(stop), world)
    flags |= msa.get_error(clear=True)

    # Per-kernel durations: right after the timed region, each stage's launches
    # of the same steps (same layer rotation) replayed alone as a CUDA graph and
    # timed with CUDA events on the launch stream.  Event nodes between the
    # stages of the timed graph would themselves add several microseconds per
    # boundary, so the timed region carries none; the stage durations add up
    # to the step time within a few percent (reported as stage_sum_vs_step).
    stage_names = ("score", "topk", "attend")
    avg_ms = {k: 0.0 for k in stage_names}
    reps_stage = min(args.steps, chunk)
    for s_i, k in enumerate(stage_names):
        if (k == "topk" and fused) or (attend_only and k != "attend"):
            continue   # fused: the selection is part of the attend kernel
        try:
            g = capture(reps_stage, which=s_i) if graphs else None
        except Exception:  # pragma: no cover
            g = None
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            if g is not None:
                g.replay()       # upload, straight into the timed replay (no idle gap)
            a.record(stream)
            if g is not None:
                g.replay()
            else:
                for j in range(reps_stage):
                    stage_calls(j % n_layers)[s_i]()
            b.record(stream)
        b.synchronize()
        avg_ms[k] = _max_over_ranks(a.elapsed_time(b), world) / reps_stage
    # the attend on its own (msa_sparse_decode over the lists the step selected),
    # the kernel the gathered-KV figure is defined on
    attend_alone_ms = avg_ms["attend"]
    if fused:
        def plain(l):
            inp, bf = layers[l], bufs[l]
            msa.sparse_decode(inp.q, inp.kv, inp.block_table, inp.seq_lens, bf.topk, inp.qlen,
                              inp.sm_scale, inp.k_scale, inp.v_scale, out=bf.out,
                              num_splits=bf.num_splits, workspace=bf.workspace,
                              q_scale=inp.q_scale)
        g = None
        if graphs:
            g = torch.cuda.CUDAGraph()
            prev = msa.set_input_overlap(True)    # a chain of attend launches, as above
            try:
                with torch.cuda.graph(g, stream=stream):
                    for j in range(reps_stage):
                        plain(j % n_layers)
            finally:
                msa.set_input_overlap(prev)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            if g is not None:
                g.replay()       # upload, straight into the timed replay
            a.record(stream)
            if g is not None:
                g.replay()
            else:
                for j in range(reps_stage):
                    plain(j % n_layers)
            b.record(stream)
        b.synchronize()
        attend_alone_ms = _max_over_ranks(a.elapsed_time(b), world) / reps_stage
    flags |= msa.get_error(clear=True)
    value = world * T * args.steps / (total_ms / 1e3)
    peak, peak_kind = _peaks()
    mean_work = {k: sum(x[k] for x in works) / len(works) for k in works[0]}
    stages = {}
    for k in ("score", "topk", "attend"):
        if (attend_only and k != "attend") or (k == "topk" and fused):
            continue
        # fused: the attend kernel also selects (reads the candidates, writes the lists)
        work_k = mean_work[k] + (mean_work["topk"] if k == "attend" and fused else 0)
        gbs = work_k / (avg_ms[k] / 1e3) / 1e9 if avg_ms[k] > 0 else None
        stages[k] = {"ms": avg_ms[k], "algorithmic_bytes": work_k, "GB/s": gbs,
                     "frac_of_hbm": (gbs / peak) if gbs else None}
    if fused:
        stages["attend"]["includes"] = "block selection (msa_sparse_decode_select)"
    tpeak, tpeak_kind = _fp8_tensor_peak()
    if "score" in stages and avg_ms["score"] > 0:
        tf = mean_work["score_flops"] / (avg_ms["score"] / 1e3) / 1e12
        stages["score"].update({"algorithmic_tflop": mean_work["score_flops"] / 1e12,
                                "TFLOP/s": tf, "frac_of_fp8_tensor": tf / tpeak})
    dominant = max(stages, key=lambda k: stages[k]["ms"])
    d = stages[dominant]
    note = ("achieved = algorithmic {} per launch / mean launch duration (CUDA events around a "
            "graph of that kernel's launches of the timed steps, replayed after the timed region)")
    # the scorer's intensity is 32 Q flop per K byte: above the fp8 ridge point
    # (peak flops / peak bytes) its roofline is the tensor peak
    if (dominant == "score" and mean_work["score_flops"] / mean_work["score"]
            > tpeak * 1e12 / (peak * 1e9)):
        roofline = {"bound": "tensor", "kernel": "score_kernel", "achieved": d["TFLOP/s"],
                    "peak": tpeak, "unit": "TFLOP/s", "frac": d["frac_of_fp8_tensor"],
                    "traffic": _traffic_from_profiles(dominant, name), "peak_kind": tpeak_kind,
                    "note": f"of {tpeak_kind}; " + note.format("flops (useful products; the "
                            "exact bf16 query as two fp8 parts doubles the executed MMA work)")}
    else:
        # the attend stage runs union_attend_kernel for dense decode (qlen >= 2)
        # and with msa_set_union_tile(1)
        union = dominant == "attend" and ((w.dense and w.qlen >= 2) or
                                          (args.union_tile and w.qlen >= 2 and not w.prefill_q))
        roofline = {"bound": "hbm", "kernel": "union_attend_kernel" if union else f"{dominant}_kernel",
                    "achieved": d["GB/s"],
                    "peak": peak, "unit": "GB/s", "frac": d["frac_of_hbm"],
                    "traffic": _traffic_from_profiles(dominant, name), "peak_kind": peak_kind,
                    "note": f"of {peak_kind}; " + note.format("bytes")}
    gathered = {"GB/s": mean_work["attend_kv_bytes"] / (attend_alone_ms / 1e3) / 1e9,
                "kernel": ("union_attend_kernel over every visible block (msa_dense_decode)"
                           if w.dense else "attend_kernel on each token's list "
                           "(msa_sparse_prefill)" if w.prefill_q else
                           "attend_kernel on the step's lists (msa_sparse_decode)"),
                "ms": attend_alone_ms,
                "union_pages_per_step": mean_work["union_pages"],
                "token_pages_per_step": mean_work["token_pages"]}
    gathered["frac_of_hbm"] = gathered["GB/s"] / peak
    # what the kernel's CTAs load (each token's own pages; pages shared by a
    # request's tokens come again, mostly from L2) per second
    gathered["token_pages_GB/s"] = mean_work["token_pages"] * 32768 / (attend_alone_ms / 1e3) / 1e9
    if fused:
        gathered["fused_select_attend_frac_of_hbm"] = (
            mean_work["attend_kv_bytes"] / (avg_ms["attend"] / 1e3) / 1e9 / peak)

    line = {"impl": "ours", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": total_ms / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "fp8e4m3 MMA operands, f32 accumulate and softmax", "data": "synthetic",
            "config": dict(w.describe(), layers_rotated=n_layers,
                           l2_policy=f"inputs larger than L2: {n_layers} independent layers "
                                     f"({layer_bytes * n_layers / 1e9:.2f} GB) rotated",
                           splits=splits, timing=mode, parallelism=f"replicas x{world}",
                           input_overlap=bool(args.input_overlap),
                           union_tile=bool(args.union_tile)),
            "roofline": roofline, "stages": stages, "attend_gathered_kv": gathered,
            "stage_sum_vs_step": sum(avg_ms.values()) / (total_ms / args.steps),
            "gpu_launches": launches_per_step * args.steps, "error_flags": flags}
    line["clocks"] = clocks.summary()

    if rank == 0 and not args.no_e2e:
        line["e2e"] = _e2e(msa, w, layers, bufs, stream, dev, world, args)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        inp0 = layers[0]
        # None (a scoring workload): the oracle scores and selects as well
        line["cpu_baseline"] = cpu_baseline(_to_cpu(inp0), w, _given_lists(w, inp0))
    if rank == 0:
        print(json.dumps(line))


def _to_cpu(inp):
    import copy
    c = copy.copy(inp)
    c.q, c.kv, c.block_table, c.seq_lens = (inp.q.cpu(), inp.kv.cpu(), inp.block_table.cpu(),
                                            inp.seq_lens.cpu())
    c.topk = inp.topk.cpu() if inp.topk is not None else None
    if inp.index_k is not None:
        c.index_k = inp.index_k.cpu()
    if inp.cu_seqlens_q is not None:
        c.cu_seqlens_q = inp.cu_seqlens_q.cpu()
    return c


def _e2e(msa, w, layers, bufs, stream, dev, world, args):
    """The same metric through the public Python API, with each step's inputs
    (q, seq_lens, block_table, and the given top-k for attend-only workloads)
    copied from pinned host memory and the output copied back to pinned host
    memory; the KV cache is resident model state.  The steps (copies and API
    calls) are captured once into a CUDA graph, as a serving loop would, with
    the copies double-buffered on a second stream, and the graph is replayed in
    the timed region; if capture fails the same calls run eagerly."""
    n_layers = len(layers)
    # each layer's step inputs packed in one pinned buffer (q, seq_lens,
    # block_table[, top-k], each 256-byte aligned), copied with one transfer
    # into a device buffer of the same layout that the API calls view

    def layout(inp):
        parts = [("q", inp.q), ("seq_lens", inp.seq_lens), ("block_table", inp.block_table)]
        if w.prefill_q:
            parts.append(("cu_seqlens_q", inp.cu_seqlens_q))
        if w.topk_given:
            parts.append(("topk", inp.topk))
        offs, off = {}, 0
        for name, t in parts:
            offs[name] = (off, t)
            off += (t.numel() * t.element_size() + 255) // 256 * 256
        return offs, off

    host, dev_in, views = [], [], []
    for inp in layers:
        offs, nbytes = layout(inp)
        hbuf = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
        dbuf = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        v = {}
        for name, (off, t) in offs.items():
            n = t.numel() * t.element_size()
            hbuf[off:off + n].copy_(t.cpu().contiguous().view(-1).view(torch.uint8))
            v[name] = dbuf[off:off + n].view(t.dtype).view(t.shape)
        host.append({"in": hbuf, "out": torch.empty(inp.q.shape, dtype=torch.bfloat16).pin_memory()})
        dev_in.append(dbuf)
        views.append(v)
    h2d_bytes = sum(t.numel() * t.element_size() for _, t in layout(layers[0])[0].values())
    d2h_bytes = host[0]["out"].numel() * 2
    steps = min(args.steps, 500)

    copy_stream = torch.cuda.Stream(dev)

    def h2d(k):
        l = k % n_layers
        dev_in[l].copy_(host[l]["in"], non_blocking=True)

    def compute(k):
        l = k % n_layers
        inp, bf, v = layers[l], bufs[l], views[l]
        if w.prefill_q:
            msa.sparse_prefill(v["q"], inp.kv, v["block_table"], v["seq_lens"], v["cu_seqlens_q"],
                               v["topk"], inp.sm_scale, inp.k_scale, inp.v_scale, out=bf.out,
                               num_splits=bf.num_splits, workspace=bf.workspace,
                               q_scale=inp.q_scale)
        elif w.topk_given:
            msa.sparse_decode(v["q"], inp.kv, v["block_table"], v["seq_lens"], v["topk"],
                              inp.qlen, inp.sm_scale, inp.k_scale, inp.v_scale, out=bf.out,
                              num_splits=bf.num_splits, workspace=bf.workspace,
                              q_scale=inp.q_scale)
        elif w.dense:
            msa.dense_decode(v["q"], inp.kv, v["block_table"], v["seq_lens"], inp.qlen,
                             inp.sm_scale, inp.k_scale, inp.v_scale, out=bf.out,
                             workspace=bf.workspace, q_scale=inp.q_scale)
        else:
            msa.decode_step(v["q"], inp.kv, v["block_table"], v["seq_lens"], inp.qlen,
                            inp.sm_scale, inp.k_scale, inp.v_scale, buffers=bf,
                            q_scale=inp.q_scale, index_k=inp.index_k,
                            index_k_scale=inp.index_k_scale)

    def d2h(k):
        l = k % n_layers
        host[l]["out"].copy_(bufs[l].out, non_blocking=True)

    out_stream = torch.cuda.Stream(dev)

    def run(nsteps):
        """Every step's copies and API calls.  Step k+1's inputs are copied on
        one side stream while step k's kernels run, and step k's output is read
        back on another; a layer's device buffers are reused only after the
        step that last read or wrote them."""
        done = [torch.cuda.Event() for _ in range(nsteps)]     # step k's kernels done
        landed = [torch.cuda.Event() for _ in range(nsteps)]   # step k's inputs on the device
        read = [torch.cuda.Event() for _ in range(nsteps)]     # step k's output read back
        with torch.cuda.stream(copy_stream):
            copy_stream.wait_stream(stream)
            h2d(0)
            landed[0].record(copy_stream)
        out_stream.wait_stream(stream)
        for k in range(nsteps):
            if k + 1 < nsteps:
                with torch.cuda.stream(copy_stream):
                    if k + 1 - n_layers >= 0:
                        copy_stream.wait_event(done[k + 1 - n_layers])
                    h2d(k + 1)
                    landed[k + 1].record(copy_stream)
            stream.wait_event(landed[k])
            if k - n_layers >= 0:
                stream.wait_event(read[k - n_layers])
            with torch.cuda.stream(stream):
                compute(k)
            done[k].record(stream)
            with torch.cuda.stream(out_stream):
                out_stream.wait_event(done[k])
                d2h(k)
                read[k].record(out_stream)
        stream.wait_stream(copy_stream)
        stream.wait_stream(out_stream)

    mode = ("public Python API captured in a CUDA graph; each step's input copy and output "
            "read-back on side streams, overlapping the neighbouring steps' kernels")
    graph = None
    with torch.cuda.stream(stream):
        run(min(args.warmup, 20) or 1)
        torch.cuda.synchronize(dev)
        try:
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=stream):
                run(steps)
            graph.replay()                      # upload
            torch.cuda.synchronize(dev)
        except Exception as e:  # pragma: no cover - depends on the torch build
            graph = None
            mode = f"public Python API, eager launches ({type(e).__name__} in capture)"
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        if graph is not None:
            graph.replay()
        else:
            run(steps)
        b.record()
        torch.cuda.synchronize(dev)
    ms = a.elapsed_time(b)
    return {"value": world * layers[0].tokens * steps / (ms / 1e3), "unit": UNIT,
            "h2d_bytes_per_step": h2d_bytes, "d2h_bytes_per_step": d2h_bytes, "steps": steps,
            "ms_per_step": ms / steps, "path": mode}


def main():
    args = _args()
    rank, world, local = _dist()
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_ours(args, rank, world, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
