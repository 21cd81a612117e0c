#!/usr/bin/env python3
"""Benchmark: split-K decode attention on one GB300 (replicas for N > 1).

Default workload: Llama-3-8B-shaped GQA decode (batch 64, 32 q / 8 KV heads,
head_dim 128, ragged kv_len uniform in [512, 8192], paged cache with page
128 and a seeded random page permutation, bf16, auto split-K).  One step is
one attn_decode call (partition kernel + split-K reduce) over that batch.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload llama3|long_context|mla|mla_mtp|sparse_mla|mixed|few_token|tiny]

Prints one JSON line (rank 0).  The metric is achieved HBM bandwidth:
algorithmic bytes per call (visible K + V, plus q, out and lse) over the
device time per call, with the KV cache resident in HBM.  The KV cache
(>= 1.1 GB) is larger than L2 (129 MB), so consecutive calls cannot hit in
L2; no flush is needed between them.

--impl reference times the fp64 CPU oracle (the only reference there is) on
the host cores, on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = ("decode-attn achieved HBM GB/s (% of GB300 peak) and µs/call, "
          "GQA 32q/8kv d128")
FALLBACK_HBM_GBS = 6800.0
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "traffic.json")
_CSRC = "split_flash_decoding_gb300/csrc/"
KERNEL_SOURCES = {
    "gqa_decode_tc": [_CSRC + f for f in ("gqa_decode_tc.cu", "gqa_items.cuh", "tc.cuh",
                                          "ptx.cuh", "launch.h")],
    "gqa_decode": [_CSRC + f for f in ("gqa_decode.cu", "ptx.cuh", "launch.h")],
    "mla_decode": [_CSRC + f for f in ("mla_decode.cu", "tc.cuh", "ptx.cuh", "launch.h")],
    "tile_attention": [_CSRC + f for f in ("tile_attention.cu", "tc.cuh", "ptx.cuh",
                                           "launch.h")],
    "tile_attention_pair": [_CSRC + f for f in ("tile_attention_pair.cu", "tc.cuh", "ptx.cuh",
                                                "launch.h")],
}


# The kernel that dominates each workload's call (the library decides the
# route; this only names the kernel whose counters the profiles hold).
DOMINANT_KERNEL = {
    "llama3": "gqa_decode_tc", "long_context": "gqa_decode_tc", "few_token": "gqa_decode_tc",
    "tiny": "gqa_decode", "mla": "mla_decode", "mla_mtp": "mla_decode",
    "sparse_mla": "mla_decode", "mixed": "tile_attention",
}


def dominant_kernel(workload: str, partitions: int = 0) -> str:
    if workload == "mixed" and partitions == -2:      # two Q tiles per CTA pair, on request
        return "tile_attention_pair"
    return DOMINANT_KERNEL[workload]


def workload_config(w, world: int) -> dict:
    """The workload description both arms print under "config"."""
    return {
        "workload": w.name,
        "batch": w.batch, "num_q_rows": w.rows, "num_q_heads": w.num_q_heads,
        "num_kv_heads": w.num_kv_heads, "head_dim": w.dim_qk, "dim_v": w.dim_v,
        "page_size": w.page_size, "total_kv_tokens": sum(w.kv_len_host),
        "max_kv_len": w.max_kv_len, "max_q_len": w.max_q_len, "causal": bool(w.causal),
        "algorithmic_bytes_per_call": algorithmic_bytes(w),
        "flops_per_call": algorithmic_flops(w),
        "l2": "inputs larger than L2: the KV cache read every step exceeds 129 MB; no flush",
        "parallelism": f"replicas x{world}",
    }


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=4000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="llama3",
                    choices=["llama3", "long_context", "mla", "mla_mtp", "sparse_mla", "mixed",
                             "few_token", "tiny"])
    ap.add_argument("--partitions", type=int, default=0, help="0 = planner's choice")
    ap.add_argument("--batch", type=int, default=0,
                    help="override the batch of the llama3 / mla workloads (profiling captures)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    return ap.parse_args()


# ---------------------------------------------------------------------------
# helpers
# ---------------------------------------------------------------------------

def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured", d
    except Exception:
        return FALLBACK_HBM_GBS, "fallback", {}


def source_hash(kernel: str) -> str:
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from a committed ncu capture, if it was taken on
    the current kernel source; else None."""
    try:
        with open(PROFILE_TRAFFIC) as f:
            d = json.load(f)
        e = d[kernel][workload]
        if e.get("source_hash") == source_hash(kernel):
            return float(e["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.idx = device_index
        self.proc = None
        self.lines = []
        self.t_marks = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(self.idx), "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.reader = threading.Thread(target=self._read, daemon=True)
            self.reader.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self):
        self.t_marks.append(time.time())

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        rows = []
        for t, line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((t, float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        t0, t1 = (self.t_marks + [0, 0])[:2]
        window = [r for r in rows if t0 <= r[0] <= t1 + 0.2] or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in window for i, v in enumerate(r[3])
                          if v.strip().lower() == "active"})
        return {"sm_mhz": statistics.median(r[1] for r in window),
                "sm_max_mhz": max(r[2] for r in window), "reasons": reasons,
                "samples": len(window)}


def build_workload(name: str, device, batch: int = 0):
    from split_flash_decoding_gb300 import workloads as W
    if name == "llama3":
        return W.llama3_8b_decode(device=device, **({"batch": batch} if batch else {}))
    if name == "long_context":
        return W.long_context_decode(device=device)
    if name == "mla":
        return W.deepseek_v3_mla_decode(device=device, **({"batch": batch} if batch else {}))
    if name == "mla_mtp":
        return W.deepseek_v3_mtp_decode(device=device, **({"batch": batch} if batch else {}))
    if name == "sparse_mla":
        return W.deepseek_v32_sparse_mla_decode(device=device,
                                                **({"batch": batch} if batch else {}))
    if name == "mixed":
        return W.mixed_prefill_decode(device=device)
    if name == "few_token":
        return W.few_token_decode(device=device, **({"batch": batch} if batch else {}))
    if name == "tiny":
        return W.tiny_decode(device=device)
    raise ValueError(name)


def algorithmic_bytes(w) -> int:
    """Visible K + V bytes (each byte once per call), q, out and lse; for
    sparse top-k also the 4-byte index of every key read."""
    hkv = w.num_kv_heads
    total_keys = sum(w.kv_len_host)
    if w.is_mla:
        kv = total_keys * w.dim_qk * 2                 # V is a prefix of K
    else:
        kv = total_keys * hkv * (w.dim_qk + w.dim_v) * 2
    if w.indices is not None:
        kv += total_keys * 4
    q = w.q.numel() * 2
    o = w.rows * w.num_q_heads * w.dim_v * 2
    lse = w.rows * w.num_q_heads * 4
    return kv + q + o + lse


def visible_pairs(w) -> int:
    """(row, key) pairs the mask lets through, summed over sequences."""
    if w.q_row_offsets_host is None:
        return sum(w.kv_len_host)
    total = 0
    o = w.q_row_offsets_host
    for b, L in enumerate(w.kv_len_host):
        n = o[b + 1] - o[b]
        if not w.causal:
            total += n * L
        else:
            # row i sees min(L, L - n + i + 1) keys (at least 0)
            for i in range(n):
                total += max(0, min(L, L - n + i + 1))
    return total


def algorithmic_flops(w) -> int:
    return visible_pairs(w) * w.num_q_heads * 2 * (w.dim_qk + w.dim_v)


def roofline_bound(flops: float, nbytes: float, tensor_tflops: float, hbm_gbs: float) -> str:
    """Whichever roof the algorithmic intensity reaches first: FLOP per byte
    above the ridge (tensor peak / HBM peak) is tensor-bound."""
    ridge = tensor_tflops * 1e12 / (hbm_gbs * 1e9)
    return "tensor" if flops / nbytes > ridge else "hbm"


def max_over_ranks(values, dist, device=None):
    """Element-wise max of per-rank timings (host-side bookkeeping only; the
    attention path itself has no collective)."""
    import torch
    vals = torch.tensor([float(v) for v in values], dtype=torch.float64)
    if dist is not None:
        t = vals.to(device) if device is not None else vals
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        vals = t.cpu()
    return [float(x) for x in vals]


def whole_job_value(world: int, bytes_per_rank: int, ms_per_step: float) -> float:
    """Weak scaling: every rank processes its own copy of the workload, so
    the job moves world * bytes per step in the slowest rank's time."""
    return world * bytes_per_rank / (ms_per_step * 1e-3) / 1e9


# ---------------------------------------------------------------------------
# the reference arm: the fp64 CPU oracle on the host cores
# ---------------------------------------------------------------------------

def oracle_sample_time(w, k_host, v_host, seqs, threads=None):
    """Run the oracle on every (query row, head) of the listed sequences;
    returns (seconds, bytes those sequences account for, threads)."""
    import numpy as np
    import oracle
    offs = w.q_row_offsets_host
    rows, heads = [], []
    n_rows = 0
    for b in seqs:
        for r in (range(offs[b], offs[b + 1]) if offs is not None else (b,)):
            n_rows += 1
            for h in range(w.num_q_heads):
                rows.append(r)
                heads.append(h)
    threads = threads or os.cpu_count() or 1
    if w.indices is not None:
        kk = oracle.KV.sparse(k_host, w.indices.cpu())
    elif w.page_table is not None:
        kk = oracle.KV.paged(k_host, w.page_table.cpu())
    else:
        kk = oracle.KV.contiguous(k_host)
    vv = kk if v_host is None else (oracle.KV.paged(v_host, w.page_table.cpu())
                                    if w.page_table is not None else oracle.KV.contiguous(v_host))
    sink = None if w.sink is None else w.sink.cpu()
    t0 = time.perf_counter()
    if rows:
        oracle.attention(w.q.cpu(), kk, vv, w.kv_len.cpu(), group=w.group, scale=w.scale,
                         dim_v=w.dim_v, sink=sink, causal=w.causal,
                         q_row_offsets=None if w.q_row_offsets is None else w.q_row_offsets.cpu(),
                         sample=(np.array(rows), np.array(heads)), threads=threads)
    dt = time.perf_counter() - t0
    hkv = w.num_kv_heads
    per_key = (w.dim_qk * 2) if w.is_mla else hkv * (w.dim_qk + w.dim_v) * 2
    if w.indices is not None:
        per_key += 4
    nbytes = sum(w.kv_len_host[b] * per_key for b in seqs)
    nbytes += n_rows * w.num_q_heads * (w.dim_qk * 2 + w.dim_v * 2 + 4)
    return dt, nbytes, threads


def host_copies(w):
    import torch
    k_host = w.k_cache.cpu()
    v_host = None if w.v_cache is None else w.v_cache.cpu()
    torch.cuda.synchronize()
    return k_host, v_host


def choose_sample(w, k_host, v_host, budget_s):
    """Sequences (in seed order) whose oracle time fits the budget."""
    t1, _, _ = oracle_sample_time(w, k_host, v_host, [0])
    per_key = t1 / max(1, w.kv_len_host[0])
    seqs, est = [], 0.0
    for b, L in enumerate(w.kv_len_host):
        c = per_key * max(L, 1)
        if seqs and est + c > budget_s:
            break
        seqs.append(b)
        est += c
    return seqs


def run_reference(args, rank, world):
    import torch
    if rank != 0:
        return
    torch.cuda.set_device(0)
    w = build_workload(args.workload, torch.device("cuda", 0), args.batch)
    k_host, v_host = host_copies(w)
    total_budget = 150.0
    per_step = total_budget / max(1, args.steps + args.warmup)
    seqs = choose_sample(w, k_host, v_host, per_step)
    for _ in range(args.warmup):
        oracle_sample_time(w, k_host, v_host, seqs)
    secs, nbytes, threads = 0.0, 0, 1
    for _ in range(args.steps):
        dt, nb, threads = oracle_sample_time(w, k_host, v_host, seqs)
        secs += dt
        nbytes += nb
    value = nbytes / secs / 1e9
    sample = (f"all (row, head) pairs of sequences {seqs[0]}..{seqs[-1]} "
              f"({len(seqs)} of {w.batch}) per step")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(secs / max(1, args.steps) * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(w, world),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

def run_ours(args, rank, world, dist):
    import torch
    from split_flash_decoding_gb300 import attn
    local = int(os.environ.get("LOCAL_RANK", rank))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = build_workload(args.workload, dev, args.batch)
    stream = torch.cuda.Stream(device=dev)

    sparse = w.indices is not None
    span = w.indices.shape[1] if sparse else w.max_kv_len
    P, ws_bytes = attn.attn_plan_partitions(w.batch, w.rows, w.num_q_heads, w.num_kv_heads,
                                            w.dim_v, span, args.partitions,
                                            max_q_len=w.max_q_len)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device=dev)
    out = torch.empty((w.rows, w.num_q_heads, w.dim_v), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((w.rows, w.num_q_heads), dtype=torch.float32, device=dev)

    # The binding plans again from its num_partitions; 0 there is its own
    # automatic choice, so the balanced MLA split goes in as its request.
    Pc = attn.ATTN_PARTITIONS_BALANCED if (w.is_mla and P == 0) else P

    def call(q=w.q, kv_len=w.kv_len, page_table=w.page_table, o=out, l=lse, indices=w.indices,
             offs=w.q_row_offsets):
        if sparse:
            attn.attn_mla_decode_sparse(q, w.k_cache, indices, kv_len, scale=w.scale,
                                        dim_v=w.dim_v, sink=w.sink, num_partitions=Pc,
                                        workspace=ws, out=o, lse=l, stream=stream)
        elif w.is_mla and offs is not None:
            attn.attn_mla_decode_rows(q, w.k_cache, kv_len, offs, scale=w.scale,
                                      max_kv_len=w.max_kv_len, causal=w.causal, dim_v=w.dim_v,
                                      page_table=page_table, sink=w.sink, num_partitions=Pc,
                                      workspace=ws, out=o, lse=l, stream=stream)
        elif w.is_mla:
            attn.attn_mla_decode(q, w.k_cache, kv_len, scale=w.scale, max_kv_len=w.max_kv_len,
                                 dim_v=w.dim_v, page_table=page_table, sink=w.sink,
                                 num_partitions=Pc, workspace=ws, out=o, lse=l, stream=stream)
        else:
            attn.attn_decode(q, w.k_cache, w.v_cache, kv_len, group=w.group, scale=w.scale,
                             max_kv_len=w.max_kv_len, page_table=page_table, sink=w.sink,
                             q_row_offsets=offs, max_q_len=w.max_q_len,
                             causal=w.causal, num_partitions=Pc, workspace=ws, out=o, lse=l,
                             stream=stream)

    # one kernel for P = 1, the tile kernels (one Q tile or the pair) and
    # the on-chip merge (P = 2 or 4 on the head_dim-128 GQA path); decode +
    # reduce otherwise (P slices, the balanced GQA or MLA split)
    tile_path = args.workload == "mixed"
    on_chip = not w.is_mla and w.dim_qk == 128 and P in (2, 4)
    launches_per_call = 1 if P == 1 or tile_path or on_chip else 2
    nbytes = algorithmic_bytes(w)
    flops = algorithmic_flops(w)

    clocks = ClockSampler(local)
    if rank == 0:
        clocks.start()
    with torch.cuda.stream(stream):
        for _ in range(max(3, args.warmup)):
            call()
    torch.cuda.synchronize(dev)
    attn.attn_device_error_flags(clear=True)

    # ---- device-timed region: inputs resident in HBM ----
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize(dev)
    clocks.mark()
    t_begin = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_begin.record(stream)
    for i in range(args.steps):
        starts[i].record(stream)
        call()
        ends[i].record(stream)
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    clocks.mark()
    if dist is not None:
        dist.barrier()
    total_ms = t_begin.elapsed_time(t_end)
    per_call_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    flags = attn.attn_device_error_flags(clear=True)
    if flags:
        raise RuntimeError(f"device error flags {flags:#x} during the timed region")

    # ---- end to end through the public API, host buffers ----
    e2e_steps = max(1, min(args.steps, 200))
    q_host = w.q.cpu().pin_memory()
    kvl_host = w.kv_len.cpu().pin_memory()
    pt_host = None if w.page_table is None else w.page_table.cpu().pin_memory()
    out_host = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    lse_host = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
    q_dev = torch.empty_like(w.q)
    kvl_dev = torch.empty_like(w.kv_len)
    pt_dev = None if pt_host is None else torch.empty_like(w.page_table)
    idx_host = None if w.indices is None else w.indices.cpu().pin_memory()
    idx_dev = None if idx_host is None else torch.empty_like(w.indices)
    h2d = q_host.numel() * 2 + kvl_host.numel() * 4 + (0 if pt_host is None else pt_host.numel() * 4)
    h2d += 0 if idx_host is None else idx_host.numel() * 4
    offs_host = None if w.q_row_offsets is None else w.q_row_offsets.cpu().pin_memory()
    offs_dev = None if offs_host is None else torch.empty_like(w.q_row_offsets)
    h2d += 0 if offs_host is None else offs_host.numel() * 4
    d2h = out_host.numel() * 2 + lse_host.numel() * 4

    def e2e_step():
        with torch.cuda.stream(stream):
            q_dev.copy_(q_host, non_blocking=True)
            kvl_dev.copy_(kvl_host, non_blocking=True)
            if pt_dev is not None:
                pt_dev.copy_(pt_host, non_blocking=True)
            if idx_dev is not None:
                idx_dev.copy_(idx_host, non_blocking=True)
            if offs_dev is not None:
                offs_dev.copy_(offs_host, non_blocking=True)
            call(q=q_dev, kv_len=kvl_dev, page_table=pt_dev, indices=idx_dev, offs=offs_dev)
            out_host.copy_(out, non_blocking=True)
            lse_host.copy_(lse, non_blocking=True)
        stream.synchronize()

    for _ in range(3):
        e2e_step()
    if dist is not None:
        dist.barrier()
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        e2e_step()
    e2e_s = (time.perf_counter() - t0) / e2e_steps
    if dist is not None:
        dist.barrier()
    clocks.stop()

    # ---- max over ranks ----
    mean_call_ms = sum(per_call_ms) / len(per_call_ms)
    total_ms, mean_call_ms, e2e_s = max_over_ranks([total_ms, mean_call_ms, e2e_s], dist, dev)
    if rank != 0:
        return

    ms_per_step = total_ms / args.steps
    value = whole_job_value(world, nbytes, ms_per_step)
    peak, peak_kind, peaks = measured_peaks()
    achieved = nbytes / (mean_call_ms * 1e-3) / 1e9
    tflops = flops / (mean_call_ms * 1e-3) / 1e12
    tensor_peak = float(peaks.get("bf16_tflops", 1900.0))
    kernel_key = dominant_kernel(args.workload, args.partitions)
    traffic = profiled_traffic(kernel_key, w.name)
    cpu = None
    if not args.no_cpu_baseline:
        # About 10-20 s of host work: a prefix of the batch sized to ~10 s,
        # repeated until 10 s have been spent (the whole batch may fit).
        k_host, v_host = host_copies(w)
        seqs = choose_sample(w, k_host, v_host, 10.0)
        dt, nb, reps = 0.0, 0, 0
        while dt < 10.0 and reps < 1000:
            d1, n1, threads = oracle_sample_time(w, k_host, v_host, seqs)
            dt += d1
            nb += n1
            reps += 1
        d1, n1, _ = oracle_sample_time(w, k_host, v_host, seqs[:1], threads=1)
        cpu = {"value": round(nb / dt / 1e9, 4), "unit": "GB/s", "cores": threads,
               "kind": "oracle",
               "sample": f"fp64 oracle over every (row, head) of sequences "
                         f"{seqs[0]}..{seqs[-1]} ({len(seqs)} of {w.batch}) x {reps} "
                         f"repetitions, {nb / 1e6:.1f} MB of K/V/q/out, {dt:.1f} s",
               "single_thread": {"value": round(n1 / d1 / 1e9, 4), "unit": "GB/s",
                                 "sample": f"sequence {seqs[0]}, one thread, {d1:.2f} s"}}
    # The bound is whichever roof the algorithmic intensity reaches first:
    # FLOP per byte above the ridge (tensor peak / HBM peak) is tensor-bound.
    ridge = tensor_peak * 1e12 / (peak * 1e9)
    if roofline_bound(flops, nbytes, tensor_peak, peak) == "tensor":
        # e.g. causal prefill tiles (about 9x past the ridge), MLA with draft rows
        roofline = {"bound": "tensor", "achieved": round(tflops, 2), "peak": tensor_peak,
                    "unit": "TFLOP/s", "frac": round(tflops / tensor_peak, 4),
                    "traffic": traffic, "peak_source": "measured bf16_tflops (burst)",
                    "kernel": f"{kernel_key} (with its split-K reduce launch where there is "
                              "one, one call), CUDA events per call on the launch stream",
                    "intensity_flop_per_byte": round(flops / nbytes, 1), "ridge": round(ridge, 1)}
    else:
        roofline = {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak,
                    "unit": "GB/s", "frac": round(achieved / peak, 4), "traffic": traffic,
                    "peak_source": f"{peak_kind} hbm_gbs",
                    "kernel": f"{kernel_key} (with its split-K reduce launch where there is "
                              "one, one call), CUDA events per call on the launch stream",
                    "intensity_flop_per_byte": round(flops / nbytes, 1), "ridge": round(ridge, 1)}
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 5),
        "us_per_call": round(ms_per_step * 1e3, 2),
        "us_per_call_median": round(statistics.median(per_call_ms) * 1e3, 2),
        "hbm_frac": round(value / world / peak, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": workload_config(w, world),
        "plan": {"num_partitions": P, "workspace_bytes": ws_bytes,
                 "note": "num_partitions 0: the balanced MLA split; -1: the balanced GQA split; -2: two Q tiles per CTA pair"},
        "clocks": clocks.summary(),
        "e2e": {"value": round(world * nbytes / e2e_s / 1e9, 2), "unit": "GB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "us_per_step": round(e2e_s * 1e6, 2),
                "note": "public Python API per step: H2D of q, kv_len and the page table "
                        "(or the top-k indices) from pinned memory, the decode call, D2H of "
                        "out and lse, stream sync; KV cache resident"},
        "gpu_launches": launches_per_call * args.steps,
        "roofline": roofline,
        "cpu_baseline": cpu,
        "tensor": {"achieved_tflops": round(tflops, 2), "peak_tflops": tensor_peak,
                   "frac": round(tflops / tensor_peak, 4),
                   "note": "algorithmic FLOPs (visible pairs x 2 x (d_qk + d_v) per head) "
                           "over the per-call time; only meaningful for the tensor-core paths"},
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    dist = None
    if world > 1:
        import torch
        import torch.distributed as tdist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", rank)))
        tdist.init_process_group("nccl")
        dist = tdist
    try:
        run_ours(args, rank, world, dist)
    finally:
        if dist is not None:
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
