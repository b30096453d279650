#!/usr/bin/env python3
"""Benchmark of the MSA forward pass (index selection + sparse attention).

One step = one msa_forward call (every stage of the hot path: plan, index
scores with fused top-k, schedule, Main Branch, combine -- or, for decode
workloads, the index scan, top-k, split attention and combine) over one batch
of seeded synthetic inputs already resident in HBM.

Default workload: prefill_128k (one causal sequence of 131072 queries, 64/4
heads, head dim 128, d_idx 128, block 128, k 16) -- the "prefill at 128K" of
the metric.  The same JSON line carries a nested ``decode`` record for
decode_1m (8 sequences decoding against 1,048,576-token caches), the metric's
"decode at 1M", measured in the same process after the prefill arrays are
freed.  Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--decode-workload NAME|none]
                  [--impl msa|reference]

Under torchrun (N > 1) every rank runs its own copy of the workload on its own
GPU (weak scaling, no data-path collective); the reported time is the max over
ranks.  ``--impl reference`` times the CPU oracle (the plain reference
implementation of the method) on the host cores, on a bounded sample of the
same workload, and reports the same metric.

The CPU-baseline leg times the oracle on a position-stratified sample of the
workload's query rows; the same oracle outputs are compared with the GPU's
rows of the timed step and reported as ``parity``.
"""
from __future__ import annotations

import argparse
import hashlib
import re
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "MSA prefill query-tok/s & decode tok/s at 128K/1M ctx; % of TC/HBM roofline"
L2_BYTES = 129 * 1024 * 1024


class L2Guard:
    """Keeps one timed step from finding the previous step's inputs in L2.  Inputs of at least twice the L2 size
    cannot stay resident across a step (each step streams all of them), so nothing is done between steps;
    smaller inputs are evicted by writing a buffer larger than L2 between steps, outside the timed brackets.
    The flush buffer is not used for large inputs because its dirty lines are written back to HBM inside the
    next timed step (about 20 us for the 129 MB of L2), a cost no real step pays."""

    def __init__(self, x, dev):
        self.input_bytes = sum(t.numel() * t.element_size() for t in (x.q, x.k, x.v, x.q_idx, x.k_idx))
        self.flush = None
        if self.input_bytes < 2 * L2_BYTES:
            self.flush = torch.empty(max(2 * L2_BYTES, 256 << 20) // 4, dtype=torch.float32, device=dev)

    def __call__(self):
        if self.flush is not None:
            self.flush.zero_()

    def describe(self) -> str:
        gb = self.input_bytes / 1e9
        if self.flush is None:
            return f"inputs larger than L2 ({gb:.2f} GB read per step, L2 129 MB): no flush between steps"
        return f"inputs of {gb:.2f} GB (under twice L2): a 258 MB buffer is written between timed steps"


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def max_over_ranks(value: float, device=None) -> float:
    """Largest value over all ranks (the slowest replica's time); identity without a process group."""
    if not (torch.distributed.is_available() and torch.distributed.is_initialized()):
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device or "cpu")
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ algorithmic work
def algorithmic_work(x, idx: torch.Tensor):
    """Per-stage algorithmic FLOPs / bytes of one step (from the actual selection)."""
    cfg = x.cfg
    G = cfg.hq // cfg.hkv
    dev = idx.device
    cu_q = x.cu_q.long().to(dev)
    cu_k = x.cu_k.long().to(dev)
    seq = torch.repeat_interleave(torch.arange(len(x.seqs), device=dev), (cu_q[1:] - cu_q[:-1]))
    t = torch.arange(x.total_q, device=dev) - cu_q[seq]
    pos = (cu_k[seq + 1] - cu_k[seq]) - (cu_q[seq + 1] - cu_q[seq]) + t          # [T]
    # index: 2 * d_idx FLOPs per (query, group, causal key)
    index_flops = float(2 * cfg.d_idx * cfg.hkv * (pos + 1).double().sum().item())
    # Main Branch: tokens attended per (query, group)
    b = idx.long()
    valid = b >= 0
    start = b * 128
    ntok_blk = torch.clamp(pos[:, None, None] - start + 1, min=0, max=128) * valid
    ntok = ntok_blk.sum(dim=2)                                                     # [T, Hkv]
    attn_flops = float(4 * cfg.head_dim * G * ntok.double().sum().item())
    n_slots = int(valid.sum().item())
    # K/V bytes the Main Branch must read at least once: each selected block's K and V rows
    kv_bytes_selected = float(2 * 2 * cfg.head_dim * ntok.double().sum().item())  # per (query,group) reads
    k_idx_bytes = float(2 * cfg.d_idx * (pos + 1).double().sum().item()) if cfg.is_decode else None
    # combine: read every valid partial (G x 128 bf16 + G fp32 LSE + G fp32 log weight), write O and LSE
    combine_bytes = float(n_slots * G * (cfg.head_dim * 2 + 8) + x.total_q * cfg.hq * (cfg.head_dim * 2 + 4) +
                          x.total_q * cfg.hkv * cfg.topk * 4)
    T, D = x.total_q, cfg.head_dim
    q_bytes = float(T * cfg.hq * D * 2)
    o_bytes = float(T * cfg.hq * (D * 2 + 4))
    # Main Branch HBM bytes of the KV-outer design with per-slot partials: Q read once, each (sequence, key block,
    # group) that any query selected read once (K and V), every partial O (bf16) + LSE + log weight written by the
    # attention and read back by the combine, O and LSE written
    seq = torch.repeat_interleave(torch.arange(len(x.seqs), device=dev), (cu_q[1:] - cu_q[:-1]))
    keyed = torch.where(valid, (seq[:, None, None] * (1 << 40) + b * cfg.hkv +
                                torch.arange(cfg.hkv, device=dev)[None, :, None]), torch.full_like(b, -1))
    n_blocks_sel = int(torch.unique(keyed[valid]).numel())
    main_bytes = (q_bytes + n_blocks_sel * 2.0 * 128 * D * 2 + 2.0 * n_slots * G * (D * 2 + 8) + o_bytes)
    decode_bytes = None
    if cfg.is_decode:
        decode_bytes = (k_idx_bytes + kv_bytes_selected + q_bytes + float(T * cfg.hkv * cfg.d_idx * 2) + o_bytes +
                        float(T * cfg.hkv * cfg.topk * 4))
    return {"index_flops": index_flops, "attn_flops": attn_flops, "n_slots": n_slots,
            "kv_bytes_selected": kv_bytes_selected, "k_idx_bytes": k_idx_bytes,
            "combine_bytes": combine_bytes, "ntok_total": float(ntok.double().sum().item()),
            "main_branch_model_bytes": main_bytes, "decode_step_bytes": decode_bytes}


# ------------------------------------------------------------------ clocks
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"msa_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.fh.close()
        return False

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return None
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            f = [c.strip() for c in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------ traffic record from ncu
def code_only(text: str) -> str:
    """C/CUDA source without comments, blank lines and indentation: what the compiler sees, so that a
    comment edit keeps a traffic record that a code change invalidates."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(" ".join(line.split()) for line in text.splitlines() if line.strip())


def kernel_source_hash(name: str, read=None) -> str:
    """Hash of a kernel file's code and of common.cuh's (comments and layout ignored)."""
    read = read or (lambda rel: open(os.path.join(ROOT, rel), encoding="utf-8").read())
    h = hashlib.sha256()
    for rel in (f"block_sparse_attention_05_gb300/csrc/{name}", "block_sparse_attention_05_gb300/csrc/common.cuh"):
        h.update(code_only(read(rel)).encode())
    return h.hexdigest()[:16]


def ncu_traffic(workload: str, kernel_file: str, x):
    """DRAM bytes per launch of the dominant kernel from the committed ncu record (profiles/traffic.txt, JSON),
    scaled from the captured case to this one by the record's unit (queries for prefill, cached keys for
    decode); None when absent or taken on a different version of the kernel."""
    p = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(p):
        return None
    try:
        rec = json.load(open(p)).get(workload)
    except (ValueError, OSError):
        return None
    if not rec or rec.get("source") != kernel_file or rec.get("source_hash") != kernel_source_hash(kernel_file):
        return None
    units_now = {"total_q": x.total_q, "total_k": x.total_k}[rec["units_kind"]]
    return rec["dram_bytes"] / rec["units"] * units_now


def step_spacing(gaps_ms):
    """Summary of the times between consecutive steps' completions (ms): a stalled step stands out against
    the median."""
    g = np.asarray(gaps_ms, dtype=np.float64)
    med = float(np.median(g))
    return {"median": med, "min": float(g.min()), "max": float(g.max()), "over_2x_median": int((g > 2 * med).sum())}


# ------------------------------------------------------------------ CPU oracle timing (+ parity of its rows)
def host_copy(x):
    return dict(cu_q=x.cu_q.cpu(), cu_k=x.cu_k.cpu(), q=x.q.cpu(), k=x.k.cpu(), v=x.v.cpu(),
                q_idx=x.q_idx.cpu(), k_idx=x.k_idx.cpu())


def stratified_rows(total: int, n: int, seed: int) -> np.ndarray:
    """n query rows, one drawn uniformly from each of n equal strata of [0, total) (all rows when n >= total)."""
    if n >= total:
        return np.arange(total, dtype=np.int32)
    rng = np.random.default_rng(seed)
    edges = np.linspace(0, total, n + 1).astype(np.int64)
    return np.array([rng.integers(edges[j], max(edges[j] + 1, edges[j + 1])) for j in range(n)], np.int32)


def oracle_rate(x, budget_s: float, max_rows: int = 100000, seed: int = 0, host=None):
    """Query rows per second of the CPU oracle on a position-stratified sample of the workload's rows.
    Returns (rate, rows, seconds, cores, sampled row indices, the oracle's outputs for them)."""
    import oracle
    host = host or host_copy(x)
    cfg = x.cfg
    ncores = os.cpu_count() or 1

    def run(rows):
        t0 = time.perf_counter()
        out = oracle.forward(host["cu_q"], host["cu_k"], host["q"], host["k"], host["v"], host["q_idx"],
                             host["k_idx"], block=cfg.block, topk=cfg.topk, rows=rows)
        return time.perf_counter() - t0, out

    n0 = min(x.total_q, max(ncores, 8))
    rows = stratified_rows(x.total_q, n0, seed)
    t, out = run(rows)
    n = int(min(x.total_q, max_rows, max(n0, n0 * budget_s / max(t, 1e-6))))
    if n > n0:
        rows = stratified_rows(x.total_q, n, seed + 1)
        t, out = run(rows)
    return len(rows) / t, len(rows), t, ncores, rows, out


NEAR_TIE = 1e-5


def parity_of_rows(rows, ref, idx, o, lse, group):
    """The GPU's outputs on the oracle's sampled rows against the oracle's: index rows that differ outside
    the near-tie exemption, the near-tie count (a property of the data), the rows the exemption excused
    (near-tie and differing: bounded by 0.1 %), and O / LSE errors over the non-exempt rows."""
    r = torch.from_numpy(rows.astype(np.int64)).to(idx.device)
    gi = idx[r].cpu().numpy()
    go = o[r].float().cpu().numpy().astype(np.float64)
    gl = lse[r].cpu().numpy().astype(np.float64)
    tie = ref["gap"] < NEAR_TIE
    differ = (gi != ref["idx"]).any(axis=-1)
    mism = differ & ~tie
    excused = differ & tie
    ok = np.repeat(~tie, group, axis=1)
    err = np.abs(go - ref["o"])[ok]
    lerr = np.abs(gl - ref["lse"])[ok]
    n_pairs = int(tie.size)
    return {"rows_checked": int(len(rows)), "query_group_rows": n_pairs, "mismatches": int(mism.sum()),
            "near_tie_rows": int(tie.sum()), "near_tie_rate": float(tie.sum()) / max(n_pairs, 1),
            "excused_rows": int(excused.sum()), "excused_rate": float(excused.sum()) / max(n_pairs, 1),
            "o_max_err": float(err.max()) if err.size else 0.0, "o_mean_err": float(err.mean()) if err.size else 0.0,
            "lse_max_err": float(lerr.max()) if lerr.size else 0.0,
            "tolerance": {"o_max": 1e-2, "o_mean": 1e-3, "lse_max": 1e-3, "excused_rate": 1e-3},
            "rows": "position-stratified sample of the CPU-baseline leg; GPU outputs of the last timed step"}


# ------------------------------------------------------------------ one workload
def measure(msa, cfg, steps, warmup, args, dev, world, rank):
    """Times `steps` msa_forward steps of `cfg` (device-resident inputs), then the end-to-end arm, the CPU
    oracle baseline and the parity of its rows.  Returns the record (rank 0) and the kernel launch count."""
    unit = "tok/s" if cfg.is_decode else "query tok/s"
    x = workloads.generate(cfg, device=dev)
    prob = msa.Problem(x.cu_q, x.cu_k, x.total_q, x.total_k, x.max_q, x.max_k, cfg.hq, cfg.hkv, cfg.d_idx,
                       cfg.topk)
    ws = msa.workspace(prob, msa.Op.FORWARD)
    idx = torch.empty((x.total_q, cfg.hkv, cfg.topk), dtype=torch.int32, device=dev)
    o = torch.empty_like(x.q)
    lse = torch.empty((x.total_q, cfg.hq), dtype=torch.float32, device=dev)
    flush = L2Guard(x, dev)
    timer = msa.StageTimer()

    def step():
        msa.msa_forward(prob, x.q, x.k, x.v, x.q_idx, x.k_idx, idx=idx, o=o, lse=lse, ws=ws)

    for _ in range(warmup):
        flush()
        step()
    torch.cuda.synchronize()
    flags = msa.msa_read_device_status(ws)
    if flags:
        raise RuntimeError(f"device status flags {flags} after warm-up")

    # ---------------- timed region (device-resident inputs): the steps are enqueued back to back, each
    # bracketed by CUDA events on the library's stream, with the L2 guard between them outside the brackets
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    launches0 = msa.kernel_launch_count()
    with ClockSampler(dev.index) as clk:
        for i in range(steps):
            flush()
            starts[i].record()
            step()
            ends[i].record()
        torch.cuda.synchronize()
    launches = msa.kernel_launch_count() - launches0
    if world > 1:
        torch.distributed.barrier()
    if msa.msa_read_device_status(ws):
        raise RuntimeError("device status flags raised during the timed steps")
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]

    # ---------------- per-stage times: a second pass with the library's stage events (one step at a time)
    stage_ms = {s: [] for s in msa.STAGES}
    with timer:
        for i in range(min(steps, 50)):
            flush()
            step()
            torch.cuda.synchronize()
            for k, v in timer.elapsed_ms().items():
                stage_ms[k].append(v)
    ms = sum(step_ms) / len(step_ms)
    ms = max_over_ranks(ms, dev)
    units_per_gpu = x.total_q
    value = units_per_gpu * world / (ms / 1000.0)

    # ---------------- roofline of the dominant kernel
    peaks = measured_peaks()
    work = algorithmic_work(x, idx)
    stage_mean = {k: sum(v) / len(v) for k, v in stage_ms.items() if v}
    dominant = max(stage_mean, key=stage_mean.get)
    kernel_file = {"index": "decode.cu" if cfg.is_decode else "index_score.cu",
                   "attn": "decode.cu" if cfg.is_decode else "sparse_attn.cu",
                   "combine": "combine.cu", "topk": "topk.cu", "schedule": "schedule.cu", "plan": "plan.cu"}
    if dominant == "attn" and not cfg.is_decode:
        bound, unit_r, amount, peak = "tensor", "TFLOP/s", work["attn_flops"], peaks["bf16_tflops"]
    elif dominant == "index" and not cfg.is_decode:
        bound, unit_r, amount, peak = "tensor", "TFLOP/s", work["index_flops"], peaks["bf16_tflops"]
    elif dominant == "index":
        bound, unit_r, amount, peak = "hbm", "GB/s", work["k_idx_bytes"], peaks["hbm_gbs"]
    elif dominant == "combine":
        bound, unit_r, amount, peak = "hbm", "GB/s", work["combine_bytes"], peaks["hbm_gbs"]
    else:
        bound, unit_r, amount, peak = "hbm", "GB/s", work["kv_bytes_selected"], peaks["hbm_gbs"]
    achieved = amount / (stage_mean[dominant] * 1e-3) / (1e12 if unit_r == "TFLOP/s" else 1e9)
    traffic = ncu_traffic(cfg.name, kernel_file[dominant], x)
    roofline = {"bound": bound, "kernel": dominant, "achieved": achieved, "peak": peak, "unit": unit_r,
                "frac": achieved / peak, "traffic": traffic,
                "peak_source": f"{peaks['source']} ({'bf16 burst' if bound == 'tensor' else 'HBM copy'})"}
    stages = {}
    for k, v in stage_mean.items():
        e = {"ms": v, "share": v / ms}
        if k == "index" and not cfg.is_decode:
            e["tflops"] = work["index_flops"] / (v * 1e-3) / 1e12
            e["frac_of_tc_peak"] = e["tflops"] / peaks["bf16_tflops"]
        if k == "index" and cfg.is_decode:
            e["gbs"] = work["k_idx_bytes"] / (v * 1e-3) / 1e9
            e["frac_of_hbm_peak"] = e["gbs"] / peaks["hbm_gbs"]
        if k == "attn" and not cfg.is_decode:
            e["tflops"] = work["attn_flops"] / (v * 1e-3) / 1e12
            e["frac_of_tc_peak"] = e["tflops"] / peaks["bf16_tflops"]
        if k == "attn" and cfg.is_decode:
            e["gbs"] = work["kv_bytes_selected"] / (v * 1e-3) / 1e9
        if k == "combine":
            e["gbs"] = work["combine_bytes"] / (v * 1e-3) / 1e9
            e["frac_of_hbm_peak"] = e["gbs"] / peaks["hbm_gbs"]
        stages[k] = e
    extra = {}
    if not cfg.is_decode and "attn" in stage_mean and "combine" in stage_mean:
        # the Main Branch as the sparse-attention gate measures it: its FLOPs over the attention and
        # combine time together, beside the bound that the HBM bytes of this design put on it
        t_ac = (stage_mean["attn"] + stage_mean["combine"]) * 1e-3
        tf = work["attn_flops"] / t_ac / 1e12
        bound_tf = work["attn_flops"] / (work["main_branch_model_bytes"] / (peaks["hbm_gbs"] * 1e9)) / 1e12
        extra["sparse_attention"] = {
            "stages": "attn + combine", "ms": t_ac * 1e3, "tflops": tf, "frac_of_tc_peak": tf / peaks["bf16_tflops"],
            "traffic_model_bytes": work["main_branch_model_bytes"],
            "traffic_model_bound_tflops": min(bound_tf, peaks["bf16_tflops"]),
            "traffic_model_bound_frac": min(1.0, bound_tf / peaks["bf16_tflops"]),
            "traffic_model": "HBM bytes of the design: Q read once, per-slot partial O (bf16) + LSE + log weight "
                             "written and read back once, O and LSE written; bound = FLOPs / (bytes / HBM peak)"}
    if cfg.is_decode:
        gbs = work["decode_step_bytes"] / (ms * 1e-3) / 1e9
        extra["whole_step"] = {"bytes": work["decode_step_bytes"], "gbs": gbs,
                               "frac_of_hbm_peak": gbs / peaks["hbm_gbs"],
                               "bytes_are": "K_idx scan + selected K/V + q, q_idx read; o, lse, idx written"}

    # ---------------- end to end through the C ABI with host buffers
    # Every step copies its inputs in from pinned host memory and its outputs back, inside the timed
    # region.  Two buffer sets: step n+1's inputs go in (one copy stream) and step n-1's outputs come back
    # (another) while step n computes on the library's stream.
    # Decode keeps the KV cache (k, v, k_idx) resident on the device as state: a step brings in the new
    # token's q and q_idx and its own k, v and k_idx rows, which are appended into the cache on the device.
    e2e = None
    if not args.no_e2e:
        nbuf = 2
        if cfg.is_decode:
            rows = (x.cu_k[1:].long() - 1)                       # cache row of each sequence's new token
            names = ("q", "q_idx", "k_new", "v_new", "k_idx_new")
            src = {"q": x.q, "q_idx": x.q_idx, "k_new": x.k[rows], "v_new": x.v[rows], "k_idx_new": x.k_idx[rows]}
        else:
            names = ("q", "k", "v", "q_idx", "k_idx", "cu_q", "cu_k")
            src = {n: getattr(x, n) for n in names}
        host_in = {n: src[n].cpu().pin_memory() for n in names}
        dev_in = [{n: torch.empty_like(src[n]) for n in names} for _ in range(nbuf)]
        if cfg.is_decode:
            for d in dev_in:  # the resident cache and sequence layout are shared by both buffer sets
                d.update(k=x.k, v=x.v, k_idx=x.k_idx, cu_q=x.cu_q, cu_k=x.cu_k)
        dev_out = [dict(idx=torch.empty_like(idx), o=torch.empty_like(o), lse=torch.empty_like(lse))
                   for _ in range(nbuf)]
        host_out = [{n: torch.empty(t.shape, dtype=t.dtype).pin_memory() for n, t in d.items()} for d in dev_out]
        probs = [msa.Problem(dev_in[i]["cu_q"], dev_in[i]["cu_k"], x.total_q, x.total_k, x.max_q, x.max_k,
                             cfg.hq, cfg.hkv, cfg.d_idx, cfg.topk) for i in range(nbuf)]
        h2d = sum(t.numel() * t.element_size() for t in host_in.values())
        d2h = sum(t.numel() * t.element_size() for t in host_out[0].values())
        s_comp = torch.cuda.current_stream()
        s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
        ev_in = [torch.cuda.Event() for _ in range(nbuf)]
        ev_done = [torch.cuda.Event() for _ in range(nbuf)]
        ev_out = [torch.cuda.Event() for _ in range(nbuf)]

        def e2e_step(n):
            bi = n % nbuf
            with torch.cuda.stream(s_in):
                if n >= nbuf:
                    s_in.wait_event(ev_done[bi])  # step n-2 has finished reading these inputs
                for name in names:
                    dev_in[bi][name].copy_(host_in[name], non_blocking=True)
                ev_in[bi].record(s_in)
            s_comp.wait_event(ev_in[bi])
            if n >= nbuf:
                s_comp.wait_event(ev_out[bi])  # step n-2's outputs have been copied out
            if cfg.is_decode:  # append the new token's rows to the resident cache
                x.k.index_copy_(0, rows, dev_in[bi]["k_new"])
                x.v.index_copy_(0, rows, dev_in[bi]["v_new"])
                x.k_idx.index_copy_(0, rows, dev_in[bi]["k_idx_new"])
            d = dev_out[bi]
            msa.msa_forward(probs[bi], dev_in[bi]["q"], dev_in[bi]["k"], dev_in[bi]["v"], dev_in[bi]["q_idx"],
                            dev_in[bi]["k_idx"], idx=d["idx"], o=d["o"], lse=d["lse"], ws=ws)
            ev_done[bi].record(s_comp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_done[bi])
                for name in ("idx", "o", "lse"):
                    host_out[bi][name].copy_(d[name], non_blocking=True)
                ev_out[bi].record(s_out)

        for n in range(2 * nbuf):
            e2e_step(n)
        torch.cuda.synchronize()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(s_comp)
        s_in.wait_event(t0)
        s_out.wait_event(t0)
        done = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        for n in range(steps):
            e2e_step(n + 2 * nbuf)
            done[n].record(s_comp)  # this step's compute has finished
        for ev in ev_out:
            s_comp.wait_event(ev)  # every step's outputs are back in host memory
        t1.record(s_comp)
        t1.synchronize()
        e2e_ms = t0.elapsed_time(t1) / steps
        e2e_ms = max_over_ranks(e2e_ms, dev)
        # spacing of consecutive steps' compute completions: a host copy that stalls shows as one long step
        gaps = [t0.elapsed_time(done[0])] + [done[i - 1].elapsed_time(done[i]) for i in range(1, steps)]
        e2e = {"value": units_per_gpu * world / (e2e_ms / 1000.0), "unit": unit, "ms_per_step": e2e_ms,
               "steps": steps, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "step_spacing_ms": step_spacing(gaps),
               "overlap": "two buffer sets: step n+1's inputs in and step n-1's outputs out during step n"}
        if cfg.is_decode:
            e2e["inputs"] = "q, q_idx and the new token's k, v, k_idx rows (appended on the device); KV cache resident"
        del dev_in, dev_out, host_in, host_out

    # ---------------- CPU oracle baseline (rank 0, N = 1 only), and the parity of its rows
    cpu, parity = None, None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rate, n, t, cores, rows, ref = oracle_rate(x, budget_s=args.cpu_budget)
        cpu = {"value": rate, "unit": unit, "cores": cores, "kind": "oracle",
               "sample": f"{n} position-stratified query rows of {cfg.name} (all groups and heads), {t:.1f} s"}
        parity = parity_of_rows(rows, ref, idx, o, lse, cfg.hq // cfg.hkv)

    rec = None
    if rank == 0:
        rec = {"workload": f"{cfg.name}: {cfg.description}", "value": value, "unit": unit, "steps": steps,
               "warmup": warmup, "ms_per_step": ms, "l2": flush.describe(), "seqs": len(x.seqs), "total_q": x.total_q,
               "total_k": x.total_k, "roofline": roofline, **extra, "stages": stages, "cpu_baseline": cpu,
               "parity": parity, "e2e": e2e, "gpu_launches": launches, "clocks": clk.summary(),
               "work": {"index_flops": work["index_flops"], "attn_flops": work["attn_flops"],
                        "selected_slots": work["n_slots"], "attended_tokens": work["ntok_total"]}}
    del x, ws, idx, o, lse, flush
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return rec


# ------------------------------------------------------------------ index prologue
def measure_prologue(msa, cfg, steps, warmup, dev, d_model=3072):
    """Times msa_index_prologue (hidden states -> Q_idx and the new tokens' K_idx rows) on the workload's tokens
    with synthetic weights: CUDA events around each launch on the library's stream, inputs larger than L2."""
    x = workloads.generate(cfg, device=dev)
    prob = msa.Problem(x.cu_q, x.cu_k, x.total_q, x.total_k, x.max_q, x.max_k, cfg.hq, cfg.hkv, cfg.d_idx,
                       cfg.topk)
    pin = workloads.prologue_inputs(x.total_q, cfg.hkv, cfg.d_idx, d_model=d_model, device=dev)
    ws = msa.workspace(prob, msa.Op.INDEX_PROLOGUE)
    q_idx = torch.empty_like(x.q_idx)
    for _ in range(warmup):
        msa.msa_index_prologue(prob, pin.x, pin.w_q, pin.w_k, pin.gamma_q, pin.gamma_k, x.k_idx, q_idx=q_idx, ws=ws)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for a, b in ev:
        a.record()
        msa.msa_index_prologue(prob, pin.x, pin.w_q, pin.w_k, pin.gamma_q, pin.gamma_k, x.k_idx, q_idx=q_idx, ws=ws)
        b.record()
    torch.cuda.synchronize()
    if msa.msa_read_device_status(ws):
        raise RuntimeError("device status flags raised by the index prologue")
    ms = sum(a.elapsed_time(b) for a, b in ev) / steps
    flops = 2.0 * x.total_q * (cfg.hkv + 1) * cfg.d_idx * d_model
    tf = flops / (ms * 1e-3) / 1e12
    peaks = measured_peaks()
    rec = {"workload": f"{cfg.name} tokens, d_model {d_model}, {cfg.hkv} index query heads + 1 key head of "
                       f"{cfg.d_idx}", "ms": ms, "flops": flops, "tflops": tf,
           "frac_of_tc_peak": tf / peaks["bf16_tflops"], "peak_source": f"{peaks['source']} (bf16 burst)",
           "steps": steps, "data": "synthetic hidden states and weights (seeded)"}
    del x, pin, ws, q_idx
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return rec


# ------------------------------------------------------------------ fp8 K/V
def measure_fp8(msa, cfg, steps, warmup, dev):
    """The same step with fp8 (E4M3, per-block scales) K and V for the Main Branch (msa_forward_fp8), after one
    msa_quantize_kv_fp8 of the workload's K and V (timed separately): step time, stage times and, for decode,
    the Main Branch's K/V bytes per second (one byte per element)."""
    x = workloads.generate(cfg, device=dev)
    prob = msa.Problem(x.cu_q, x.cu_k, x.total_q, x.total_k, x.max_q, x.max_k, cfg.hq, cfg.hkv, cfg.d_idx,
                       cfg.topk)
    qws = msa.workspace(prob, msa.Op.QUANTIZE_KV_FP8)
    k8, v8, ks, vs = msa.msa_quantize_kv_fp8(prob, x.k, x.v, ws=qws)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    msa.msa_quantize_kv_fp8(prob, x.k, x.v, k8=k8, v8=v8, k_scale=ks, v_scale=vs, ws=qws)
    b.record()
    torch.cuda.synchronize()
    quant_ms = a.elapsed_time(b)
    ws = msa.workspace(prob, msa.Op.FORWARD_FP8)
    idx = torch.empty((x.total_q, cfg.hkv, cfg.topk), dtype=torch.int32, device=dev)
    o = torch.empty_like(x.q)
    lse = torch.empty((x.total_q, cfg.hq), dtype=torch.float32, device=dev)
    flush = L2Guard(x, dev)

    def step():
        msa.msa_forward_fp8(prob, x.q, k8, v8, ks, vs, x.q_idx, x.k_idx, idx=idx, o=o, lse=lse, ws=ws)

    for _ in range(warmup):
        flush()
        step()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for s_, e_ in ev:
        flush()
        s_.record()
        step()
        e_.record()
    torch.cuda.synchronize()
    if msa.msa_read_device_status(ws):
        raise RuntimeError("device status flags raised by the fp8 forward")
    ms = sum(s_.elapsed_time(e_) for s_, e_ in ev) / steps
    timer = msa.StageTimer()
    stage = {}
    with timer:
        for _ in range(min(steps, 20)):
            flush()
            step()
            torch.cuda.synchronize()
            for k_, v_ in timer.elapsed_ms().items():
                stage[k_] = stage.get(k_, 0.0) + v_ / min(steps, 20)
    work = algorithmic_work(x, idx)
    peaks = measured_peaks()
    unit = "tok/s" if cfg.is_decode else "query tok/s"
    rec = {"workload": f"{cfg.name}, fp8 K/V", "value": x.total_q / (ms * 1e-3), "unit": unit, "ms_per_step": ms,
           "steps": steps, "stages_ms": stage, "quantize_ms": quant_ms,
           "quantize_gbs": 3.0 * x.total_k * cfg.hkv * cfg.head_dim * 2 / (quant_ms * 1e-3) / 1e9}
    if "attn" in stage:
        if cfg.is_decode:
            kv8 = work["kv_bytes_selected"] / 2  # one byte per K and V element
            rec["attn_kv_gbs"] = kv8 / (stage["attn"] * 1e-3) / 1e9
            rec["attn_kv_bytes"] = kv8
        else:
            rec["attn_tflops"] = work["attn_flops"] / (stage["attn"] * 1e-3) / 1e12
            rec["attn_frac_of_tc_peak"] = rec["attn_tflops"] / peaks["bf16_tflops"]
    if cfg.d_idx == 128:
        rec["fp8_index"] = measure_fp8_index(msa, x, prob, k8, v8, ks, vs, idx, ws, flush, steps, warmup, peaks)
    del x, ws, idx, o, lse, flush, k8, v8, ks, vs, qws
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return rec


def measure_fp8_index(msa, x, prob, k8, v8, ks, vs, idx_bf16_index, ws, flush, steps, warmup, peaks):
    """The all-fp8 step (msa_forward_fp8_index: E4M3 Q_idx / K_idx as well as K / V) after one
    msa_quantize_index_fp8 of the workload's index inputs (timed separately), with the same L2 guard as
    the other steps.  Also how far its selection departs from the bf16 index's (informational: a quantized
    index selects other blocks; its parity is against the oracle over the same codes, in the tests)."""
    cfg = x.cfg
    qws = msa.workspace(prob, msa.Op.QUANTIZE_INDEX_FP8)
    q8, qsc, kk8, ksc = msa.msa_quantize_index_fp8(prob, x.q_idx, x.k_idx, ws=qws)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    msa.msa_quantize_index_fp8(prob, x.q_idx, x.k_idx, q8, qsc, kk8, ksc, ws=qws)
    b.record()
    torch.cuda.synchronize()
    quant_ms = a.elapsed_time(b)
    idx = torch.empty_like(idx_bf16_index)  # ws: the fp8 K/V step's workspace (op MSA_OP_FORWARD_FP8)
    o = torch.empty_like(x.q)
    lse = torch.empty((x.total_q, cfg.hq), dtype=torch.float32, device=x.q.device)

    def step():
        msa.msa_forward_fp8_index(prob, x.q, k8, v8, ks, vs, q8, qsc, kk8, ksc, idx=idx, o=o, lse=lse, ws=ws)

    for _ in range(warmup):
        flush()
        step()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for s_, e_ in ev:
        flush()
        s_.record()
        step()
        e_.record()
    torch.cuda.synchronize()
    if msa.msa_read_device_status(ws):
        raise RuntimeError("device status flags raised by the all-fp8 forward")
    ms = sum(s_.elapsed_time(e_) for s_, e_ in ev) / steps
    timer = msa.StageTimer()
    stage = {}
    n_st = min(steps, 20)
    with timer:
        for _ in range(n_st):
            flush()
            step()
            torch.cuda.synchronize()
            for k_, v_ in timer.elapsed_ms().items():
                stage[k_] = stage.get(k_, 0.0) + v_ / n_st
    work = algorithmic_work(x, idx)
    unit = "tok/s" if cfg.is_decode else "query tok/s"
    rec = {"workload": f"{cfg.name}, fp8 K/V and fp8 index", "value": x.total_q / (ms * 1e-3), "unit": unit,
           "ms_per_step": ms, "steps": steps, "stages_ms": stage, "quantize_index_ms": quant_ms}
    same = (idx == idx_bf16_index).all(dim=-1)
    a_ = idx_bf16_index.long()
    b_ = idx.long()
    inter = ((a_[..., :, None] == b_[..., None, :]) & (a_[..., :, None] >= 0)).any(dim=-1).sum(dim=-1)
    n_sel = (a_ >= 0).sum(dim=-1).clamp(min=1)
    rec["selection_vs_bf16_index"] = {"rows_identical": float(same.float().mean().item()),
                                      "mean_overlap": float((inter.float() / n_sel.float()).mean().item())}
    if "index" in stage:
        if cfg.is_decode:
            kb = work["k_idx_bytes"] / 2 + 4.0 * x.total_k / 128  # one byte per code, one fp32 scale per block
            rec["index_gbs"] = kb / (stage["index"] * 1e-3) / 1e9
            rec["index_frac_of_hbm_peak"] = rec["index_gbs"] / peaks["hbm_gbs"]
            rec["index_bytes"] = kb
        else:
            rec["index_tflops"] = work["index_flops"] / (stage["index"] * 1e-3) / 1e12
            rec["index_frac_of_fp8_peak"] = rec["index_tflops"] / (2.0 * peaks["bf16_tflops"])
            rec["fp8_peak_source"] = "2 x the measured bf16 burst (the nominal fp8 / bf16 ratio)"
    del qws, q8, qsc, kk8, ksc, idx, o, lse
    return rec


# ------------------------------------------------------------------ main
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default="prefill_128k", choices=sorted(workloads.CONFIGS))
    ap.add_argument("--decode-workload", default="decode_1m", choices=sorted(workloads.CONFIGS) + ["none"],
                    help="decode workload measured after the main one, reported as the nested 'decode' record")
    ap.add_argument("--decode-steps", type=int, default=2500,
                    help="timed steps of the nested decode record (about 1 s at decode_1m)")
    ap.add_argument("--impl", default="msa", choices=["msa", "reference"])
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-prologue", action="store_true", help="skip the index prologue measurement")
    ap.add_argument("--no-fp8", action="store_true", help="skip the fp8 K/V measurements")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    world, rank, local = dist_env()
    cfg = workloads.get(args.workload)
    unit = "tok/s" if cfg.is_decode else "query tok/s"

    if args.impl == "reference":
        if rank != 0:
            return 0
        # inputs are drawn on the GPU when there is one (only to make them; the timed work is the oracle's)
        x = workloads.generate(cfg, device="cuda" if torch.cuda.is_available() else "cpu")
        host = host_copy(x)
        per_step = []
        rows_done = 0
        cores = os.cpu_count() or 1
        budget = max(2.0, 60.0 / max(1, args.steps + args.warmup))
        for i in range(args.warmup + args.steps):
            rate, n, t, cores, _, _ = oracle_rate(x, budget_s=budget, seed=2 * i, host=host)
            if i >= args.warmup:
                per_step.append((n, t))
                rows_done += n
        tot_t = sum(t for _, t in per_step)
        value = rows_done / tot_t
        line = {"impl": "reference", "metric": METRIC, "value": value, "unit": unit, "n_gpus": args.gpus,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000 * tot_t / len(per_step),
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic",
                "config": {"workload": f"{cfg.name}: {cfg.description}", "seqs": len(x.seqs),
                           "total_q": x.total_q, "total_k": x.total_k,
                           "sample": "rows per step, position-stratified"},
                "cpu_baseline": {"value": value, "unit": unit, "cores": cores, "kind": "oracle",
                                 "sample": f"{rows_done} query rows of {cfg.name} over {args.steps} steps"},
                "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return 0

    import block_sparse_attention_05_gb300 as msa

    if world > 1:
        torch.cuda.set_device(local)
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())

    main_rec = measure(msa, cfg, args.steps, args.warmup, args, dev, world, rank)
    pro_rec = None
    if not cfg.is_decode and not args.no_prologue:
        pro_rec = measure_prologue(msa, cfg, max(args.steps, 10), args.warmup, dev)
    dec_rec = None
    fp8_rec = {}
    if not args.no_fp8:
        fp8_rec[cfg.name] = measure_fp8(msa, cfg, args.steps, args.warmup, dev)
    if args.decode_workload != "none" and args.decode_workload != args.workload:
        dcfg = workloads.get(args.decode_workload)
        dec_rec = measure(msa, dcfg, args.decode_steps, args.warmup, args, dev, world, rank)
        if not args.no_fp8:
            fp8_rec[dcfg.name] = measure_fp8(msa, dcfg, args.decode_steps, args.warmup, dev)

    if rank == 0:
        m = main_rec
        line = {
            "metric": METRIC, "value": m["value"] * 1.0, "unit": unit, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": m["ms_per_step"], "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": m["workload"], "seqs": m["seqs"], "total_q": m["total_q"],
                       "total_k": m["total_k"],
                       "l2": m["l2"],
                       "parallelism": "replicas" if world > 1 else "single"},
            "roofline": m["roofline"],
        }
        for key in ("sparse_attention", "whole_step"):
            if key in m:
                line[key] = m[key]
        line.update({"stages": m["stages"], "cpu_baseline": m["cpu_baseline"], "parity": m["parity"],
                     "e2e": m["e2e"], "gpu_launches": m["gpu_launches"], "clocks": m["clocks"], "work": m["work"]})
        if pro_rec is not None:
            line["index_prologue"] = pro_rec
        if fp8_rec:
            line["fp8_kv"] = fp8_rec
        if dec_rec is not None:
            dec_rec = dict(dec_rec)
            dec_rec["value"] = dec_rec["value"] * 1.0
            line["decode"] = dec_rec
        print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
