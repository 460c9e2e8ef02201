#!/usr/bin/env python
"""Benchmark of sparse MLA decode (SFA) + lse merge on GB300.

One step = one full pass of the path over one batch of synthetic inputs:
index resolution, latent-row gather, QK^T, online softmax, P.V, epilogue, and
(for sharded workloads) the lse merge of the shard partials.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl ours|reference]

Prints one JSON line (rank 0).  Under torchrun (N > 1) every rank runs the same
workload on its own GPU (replicas: weak scaling, no data-path collective); the
reported time is the max over ranks and `value` aggregates all ranks' work.
"""
from __future__ import annotations

import argparse
import dataclasses
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

from deepseek_sparse_mla_sfa_gb300 import workloads  # noqa: E402

METRIC = "sparse MLA decode TFLOP/s and gather GB/s (h=128, top_k=2048); % of roofline"
UNIT = "TFLOP/s"
L2_FLUSH_BYTES = 256 << 20
ROW_BYTES = 576 * 2
FLOPS_PER_ROW_HEAD = 2 * (576 + 512)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


class L2Scrub:
    """Evicts the L2 before a timed call: a 256 MiB write, so that no input of the call
    stays resident, then a 256 MiB read of a buffer that is never written, so that the L2
    is left holding clean lines and the timed call does not pay for writing back the
    scrub's own dirty lines (about 126 MB of them after the write alone)."""

    def __init__(self, dev):
        self.dirty = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
        self.clean = torch.zeros(L2_FLUSH_BYTES // 8, dtype=torch.int64, device=dev)

    def __call__(self):
        self.dirty.zero_()
        self.clean.max()


def hold_device(cycles: int = 200_000):
    """Keep the device busy (~0.1 ms spin, outside the timed events) while the host enqueues
    the timed call, so that the events bracket device time and not host launch latency."""
    torch.cuda._sleep(cycles)


def accounting(inp: workloads.Inputs):
    """Algorithmic work of one step: FLOPs and bytes per kernel (the method's own work:
    only the selected rows count; softmax exponentials are not FLOPs)."""
    w = inp.w
    T, h, n = w.T, w.h, w.n_splits
    i = torch.arange(w.Q, device=inp.topk_idx.device).repeat(w.B)
    L = inp.seq_lens.long().repeat_interleave(w.Q) - (w.Q - 1 - i)
    idx = inp.topk_idx.long()
    k_valid = ((idx >= 0) & (idx < L.unsqueeze(1))).sum(dim=1)
    kv_total = int(k_valid.sum())
    flops = FLOPS_PER_ROW_HEAD * h * kv_total
    gather = kv_total * ROW_BYTES
    q_b = T * h * 576 * 2
    idx_b = T * w.top_k * 4
    res_b = T * h * 513 * 4
    decode_b = gather + q_b + idx_b + (res_b if n == 1 else n * res_b)
    merge_b = n * res_b + res_b if n > 1 else 0
    return {"k_valid_total": kv_total, "flops": flops, "gather_bytes": gather,
            "decode_bytes": decode_b, "merge_bytes": merge_b, "total_bytes": decode_b + merge_b}


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while the timed loop runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.tmp = None

    def start(self):
        try:
            self.tmp = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=self.tmp, stderr=subprocess.DEVNULL)
            self.t0 = time.time()
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self, t_begin, t_end):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.tmp.flush()
        self.tmp.seek(0)
        rows = [r.strip().split(",") for r in self.tmp.read().splitlines() if r.strip()]
        self.tmp.close()
        os.unlink(self.tmp.name)
        sm, smax, reasons, power = [], None, set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                smax = float(r[2])
                power.append(float(r[3]))
            except ValueError:
                continue
            for nm, v in zip(names, r[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm),
                "power_w_max": max(power) if power else None}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    """The largest of every rank's x (the slowest rank's time sets the job's time)."""
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def rank_workload(w: workloads.Workload, rank: int) -> workloads.Workload:
    """The batch rank `rank` decodes: the same shapes as `w`, its own tokens (seed
    offset by the rank), so N ranks process N independent batches (weak scaling)."""
    return dataclasses.replace(w, seed=w.seed + 1000 * rank) if rank else w


def job_value(flops_per_rank: float, ms: float, world: int) -> float:
    """Whole-job TFLOP/s: every rank's work over the slowest rank's step time."""
    return world * flops_per_rank / (ms * 1e-3) / 1e12


def cpu_model() -> str:
    """The host CPU's model name, as the kernel reports it (empty when unknown)."""
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                key, _, val = line.partition(":")
                if key.strip().lower() in ("model name", "cpu model", "hardware") and val.strip():
                    return val.strip()
    except OSError:
        pass
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    return ""


def cpu_oracle_leg(inp, acc, target_s=15.0, max_tokens=None):
    """Time the fp64 oracle, as it stands, on the host cores over a bounded sample of
    the workload (whole tokens, all heads, all shards).  Returns (line dict, elapsed)."""
    import numpy as np
    import oracle
    w = inp.w
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    prob = oracle.Problem(inp.q, inp.kv, inp.block_table, inp.seq_lens, inp.topk_idx, w.Q, w.scale)
    L = (prob.seq_lens.repeat(w.Q) - (w.Q - 1 - np.tile(np.arange(w.Q), w.B))).astype(np.int64)
    kval = ((prob.topk_idx >= 0) & (prob.topk_idx < L[:, None])).sum(axis=1)

    def run(tokens):
        t = np.repeat(tokens, w.h).astype(np.int32)
        hh = np.tile(np.arange(w.h), len(tokens)).astype(np.int32)
        t0 = time.perf_counter()
        if w.n_splits > 1:
            n = w.n_splits
            r = np.tile(np.arange(n), len(t)).astype(np.int32)
            op, lp = oracle.decode_sampled(prob, np.repeat(t, n), np.repeat(hh, n), shards=r,
                                           n_splits=n, nthreads=cores)
            oracle.merge(op.reshape(len(t), n, -1).transpose(1, 0, 2), lp.reshape(len(t), n).T)
        else:
            oracle.decode_sampled(prob, t, hh, nthreads=cores)
        return time.perf_counter() - t0

    t1 = run(np.array([0]))
    n_tok = max(1, min(w.T, int(target_s / max(t1, 1e-6))))
    if max_tokens:
        n_tok = min(n_tok, max_tokens)
    tokens = np.linspace(0, w.T - 1, n_tok).round().astype(np.int64)
    tokens = np.unique(tokens)
    el = run(tokens)
    flops = FLOPS_PER_ROW_HEAD * w.h * int(kval[tokens].sum())
    val = flops / el / 1e12
    return {"value": val, "unit": UNIT, "cores": cores, "kind": "oracle", "cpu_model": cpu_model(),
            "sample": f"{len(tokens)} of {w.T} query tokens of {w.name}, all {w.h} heads"
                      f"{', all %d shards + merge' % w.n_splits if w.n_splits > 1 else ''}; "
                      f"{el:.2f} s fp64 on {cores} host threads"}, el


def run_reference(args, world, rank):
    if rank != 0:
        return
    w = workloads.CONFIGS[args.config]
    inp = workloads.make(w, device="cuda" if torch.cuda.is_available() else "cpu")
    acc = accounting(inp)
    per_step = max(2.0, 60.0 / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        cpu_oracle_leg(inp, acc, target_s=min(per_step, 5.0))
    vals, tot = [], 0.0
    line_cb = None
    for _ in range(args.steps):
        cb, el = cpu_oracle_leg(inp, acc, target_s=per_step)
        vals.append(cb["value"])
        tot += el
        line_cb = cb
    value = statistics.mean(vals) if vals else 0.0
    if line_cb is not None:
        line_cb = dict(line_cb, value=value)   # this run's own value, over all its steps
    line = {"metric": METRIC, "value": value, "unit": UNIT, "impl": "reference",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * tot / max(1, args.steps), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "Q": w.Q, "h": w.h, "S": w.S,
                       "top_k": w.top_k, "n_splits": w.n_splits},
            "cpu_baseline": line_cb,
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_ours(args, world, rank, local):
    import deepseek_sparse_mla_sfa_gb300 as sfa
    w = rank_workload(workloads.CONFIGS[args.config], rank)
    peaks = load_peaks()
    inp = workloads.make(w, device="cuda")
    acc = accounting(inp)
    T, h, n = w.T, w.h, w.n_splits
    dev = inp.q.device
    out = torch.empty((T, h, 512), dtype=torch.float32, device=dev)
    lse = torch.empty((T, h), dtype=torch.float32, device=dev)
    op = torch.empty((n, T, h, 512), dtype=torch.float32, device=dev) if n > 1 else None
    lp = torch.empty((n, T, h), dtype=torch.float32, device=dev) if n > 1 else None
    wsb = sfa.workspace_bytes(w.B, w.Q, h, w.top_k, n)
    ws = torch.empty(max(wsb, 1), dtype=torch.uint8, device=dev)
    flush = L2Scrub(dev)
    n_dec, tc_path = sfa.decode_launches(w.B, w.Q, h, w.top_k, w.block_size, n, merge=False)
    launches_per_step = n_dec + (1 if n > 1 else 0)

    def step(evs=None):
        if evs:
            evs[0].record()
        if n > 1:
            sfa.decode(inp.q, inp.kv, inp.block_table, inp.seq_lens, inp.topk_idx, w.scale,
                       n_splits=n, Q=w.Q, merge=False, out_part=op, lse_part=lp, workspace=ws)
            if evs:
                evs[1].record()
            sfa.lse_merge(op, lp, out=out, lse=lse)
            if evs:
                evs[2].record()
        else:
            sfa.decode(inp.q, inp.kv, inp.block_table, inp.seq_lens, inp.topk_idx, w.scale,
                       n_splits=1, Q=w.Q, out=out, lse=lse, workspace=ws)
            if evs:
                evs[1].record()

    for _ in range(args.warmup):
        flush()
        step()
    torch.cuda.synchronize()
    if sfa.last_device_status() != 0:
        raise RuntimeError("device status error during warm-up")

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    t_begin = time.time()
    for k in range(args.steps):
        flush()                      # scrub L2 between timed steps (outside the events)
        hold_device()                      # the host enqueues the step while the device spins
        step(evs[k])
    torch.cuda.synchronize()
    barrier(world)
    t_end = time.time()
    clk = clocks.stop(t_begin, t_end)
    dec_ms = [e[0].elapsed_time(e[1]) for e in evs]
    # a single-shard step is the decode launch alone (no merge event is recorded)
    mrg_ms = [e[1].elapsed_time(e[2]) if n > 1 else 0.0 for e in evs]
    step_ms = [a + b for a, b in zip(dec_ms, mrg_ms)]
    local_ms = sum(step_ms) / max(1, len(step_ms))
    ms = max_over_ranks(local_ms, world)
    dec_avg = sum(dec_ms) / max(1, len(dec_ms))
    mrg_avg = sum(mrg_ms) / max(1, len(mrg_ms))

    value = job_value(acc["flops"], ms, world)
    gather_gbs = acc["gather_bytes"] / (ms * 1e-3) / 1e9
    alg_gbs = acc["total_bytes"] / (ms * 1e-3) / 1e9
    roof_s = max(acc["flops"] / (peaks["bf16_tflops"] * 1e12), acc["total_bytes"] / (peaks["hbm_gbs"] * 1e9))
    dominant = "decode" if dec_avg >= mrg_avg else "lse_merge"
    dom_ms = dec_avg if dominant == "decode" else mrg_avg
    dom_bytes = acc["decode_bytes"] if dominant == "decode" else acc["merge_bytes"]
    achieved = dom_bytes / (dom_ms * 1e-3) / 1e9
    traffic = read_traffic(dominant, tc_path, w.name)

    # end to end through the host-buffer entry point: H2D of the step's inputs, decode,
    # D2H of out + lse, all inside the timed region
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(sfa, inp, args.steps, flush)
    cpu = None
    if world == 1 and rank == 0 and not args.no_cpu_baseline:
        cpu, _ = cpu_oracle_leg(inp, acc, target_s=15.0)
    next_rows = None if args.no_next_rows else measure_next_rows(sfa, inp, peaks, flush)
    configs = None
    if not args.no_configs and rank == 0:
        mine = {"decode_us": dec_avg * 1e3, "merge_us": mrg_avg * 1e3 if n > 1 else None, "step_us": ms * 1e3}
        configs = measure_configs(sfa, peaks, flush, w.name, mine, acc, steps=max(10, min(args.steps, 30)))

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "median_ms_per_step": statistics.median(step_ms),
        "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "Q": w.Q, "h": w.h, "S": w.S, "top_k": w.top_k,
                   "n_splits": n, "block_size": w.block_size, "seed": w.seed,
                   "l2": "flushed between timed steps (256 MiB write, then 256 MiB read of another buffer; outside the timed events)",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "gather_gbs": gather_gbs, "algorithmic_gbs": alg_gbs,
        "pct_of_roofline": 100.0 * roof_s / (ms * 1e-3),
        "roofline_time_us": roof_s * 1e6,
        # the step's tensor work against the measured bf16 peaks: the burst figure for a
        # kernel timed alone, the seconds-long sustained figure beside it
        "tensor": {"tflops": value / world,
                   "frac_of_burst": value / world / peaks["bf16_tflops"],
                   "frac_of_sustained": value / world / peaks["bf16_tflops_sustained"],
                   "peak_burst": peaks["bf16_tflops"], "peak_sustained": peaks["bf16_tflops_sustained"]},
        "kernel_path": {3: "tcgen05 stacked-half", 2: "tcgen05 small-head", 1: "tcgen05 CTA pair",
                        0: "cuda-core"}[tc_path],
        "kernels": {"decode_ms": dec_avg, "lse_merge_ms": mrg_avg if n > 1 else None},
        "roofline": {"bound": "hbm", "kernel": dominant, "achieved": achieved,
                     "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
                     "traffic": traffic, "peak_source": peaks["source"] + " (hbm copy)"},
        "e2e": e2e,
        "cpu_baseline": cpu,
        "gpu_launches": launches_per_step * args.steps,
        "next_rows": next_rows,
        "configs": configs,
        "clocks": clk,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


def measure_next_rows(sfa, inp, peaks, flush):
    """The rows after the decode step at this workload's shapes, each timed alone with CUDA
    events on the launching stream (L2 scrubbed before each launch):
      kv_write - the T new tokens' latent rows scattered into the cache at their slots;
      uv_proj  - the W_UV up-projection of the decode output (synthetic weights);
      topk     - the indexer's top-k selection producing this workload's index lists from
                 seeded N(0, 1) scores over each sequence's cache (causal range per token);
      lse_merge - the shard merge at the 8-shard long-context shape (8 x 32 tokens x 128
                 heads of fp32 partials), which a single-shard step does not run."""
    w = inp.w
    dev = inp.q.device
    T, h = w.T, w.h
    g = torch.Generator(device="cpu").manual_seed(w.seed + 99)
    num_slots = inp.kv.shape[0] * inp.kv.shape[1]
    slots = torch.randperm(num_slots, generator=g)[:T].to(torch.int32).to(dev)
    rows = torch.randn((T, 576), generator=g).to(torch.bfloat16).to(dev)
    kv_copy = inp.kv  # written in place: the rows land in slots no decode of this run reads again
    out = torch.randn((T, h, 512), generator=g).to(dev) * 0.3
    w_uv = (torch.randn((h, 512, 128), generator=g) / 512 ** 0.5).to(torch.bfloat16).to(dev)
    y = torch.empty((T, h, 128), dtype=torch.bfloat16, device=dev)
    S = int(inp.seq_lens.max())
    scores = workloads.indexer_scores(T, S, dev, seed=w.seed + 98)
    idx = torch.empty((T, w.top_k), dtype=torch.int32, device=dev)

    def timed(fn, n):
        # the L2 scrub before each call also keeps the stream busy while the host enqueues
        # the call, so the events bracket device time only
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        evs = []
        for _ in range(n):
            flush()
            hold_device()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            evs.append((e0, e1))
        torch.cuda.synchronize()
        return sum(a.elapsed_time(b) for a, b in evs) / n * 1e-3   # seconds

    t_kv = timed(lambda: sfa.kv_write(kv_copy, slots, rows), 30)
    t_uv = timed(lambda: sfa.uv_proj(out, w_uv, y), 30)
    t_tk = timed(lambda: sfa.topk(scores, w.top_k, seq_lens=inp.seq_lens, Q=w.Q, S=S, out=idx), 30)
    lw = workloads.CONFIGS["long_dcp"]
    m_rows = lw.T * lw.h
    op = torch.randn((lw.n_splits, lw.T, lw.h, 512), generator=g).to(dev)
    lp = (torch.randn((lw.n_splits, lw.T, lw.h), generator=g) * 3.0).to(dev)
    mo = torch.empty((lw.T, lw.h, 512), dtype=torch.float32, device=dev)
    ml = torch.empty((lw.T, lw.h), dtype=torch.float32, device=dev)
    t_mg = timed(lambda: sfa.lse_merge(op, lp, out=mo, lse=ml), 30)
    if sfa.last_device_status() != 0:
        raise RuntimeError("device status error in the next-row kernels")
    kv_bytes = T * 1152 * 2 + T * 4
    uv_bytes = T * h * 512 * 4 + h * 512 * 128 * 2 + T * h * 128 * 2
    uv_flops = 2 * T * h * 512 * 128
    uv_gbs = uv_bytes / t_uv / 1e9
    # algorithmic bytes: each token's candidate scores read once, its list written once
    L = (inp.seq_lens.to(torch.int64).repeat_interleave(w.Q)
         - (w.Q - 1 - torch.arange(T, device=dev) % w.Q)).clamp(0, S)
    tk_bytes = int(L.sum()) * 4 + T * w.top_k * 4
    tk_gbs = tk_bytes / t_tk / 1e9
    mg_bytes = (lw.n_splits + 1) * m_rows * 513 * 4
    mg_gbs = mg_bytes / t_mg / 1e9
    return {
        "kv_write": {"us": t_kv * 1e6, "rows": T, "bytes": kv_bytes, "GB/s": kv_bytes / t_kv / 1e9,
                     "note": "latency-bound at this size (one 1152-byte row per warp)"},
        "uv_proj": {"us": t_uv * 1e6, "shape": f"[{T},{h},512] x [{h},512,128]", "TFLOP/s": uv_flops / t_uv / 1e12,
                    "roofline": {"bound": "hbm", "achieved": uv_gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                 "frac": uv_gbs / peaks["hbm_gbs"], "bytes": uv_bytes}},
        "topk": {"us": t_tk * 1e6, "shape": f"[{T},{S}] -> [{T},{w.top_k}]",
                 "roofline": {"bound": "hbm", "achieved": tk_gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                              "frac": tk_gbs / peaks["hbm_gbs"], "bytes": tk_bytes}},
        "lse_merge": {"us": t_mg * 1e6, "shape": f"[{lw.n_splits},{lw.T},{lw.h},512] -> [{lw.T},{lw.h},512]",
                      "roofline": {"bound": "hbm", "achieved": mg_gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                   "frac": mg_gbs / peaks["hbm_gbs"], "bytes": mg_bytes}},
    }


# the headline shape with 16 heads: the small-head kernel's gather-bound case
SMALL_HEAD = workloads.Workload("sfa_h16", B=64, Q=1, h=16, S=32768, top_k=2048, n_splits=1,
                                index_kind="uniform", seed=1234 + 6)


def roofline_of(acc, peaks):
    """Roofline time of one step: the slower of the tensor work at the measured bf16 peak
    and the algorithmic bytes at the measured HBM bandwidth."""
    t_tensor = acc["flops"] / (peaks["bf16_tflops"] * 1e12)
    t_hbm = acc["total_bytes"] / (peaks["hbm_gbs"] * 1e9)
    return max(t_tensor, t_hbm), ("tensor" if t_tensor > t_hbm else "hbm")


def measure_configs(sfa, peaks, flush, measured_name, measured, measured_acc, steps=20):
    """Every workload's step (decode, plus the lse merge when it is sharded) timed alone
    with CUDA events on the launching stream, L2 scrubbed before each step, with its
    algorithmic bytes and FLOPs (the same accounting as the headline) and its fraction of
    the roofline.  The workload the headline step already timed is reported from that
    measurement."""
    res = {}
    todo = [(n, w) for n, w in workloads.CONFIGS.items() if n in ("tiny", "dense", "sfa_h128", "mtp", "long_dcp")]
    todo.append(("sfa_h16", SMALL_HEAD))
    for name, w in todo:
        if name == measured_name:
            acc, times = measured_acc, dict(measured)
        else:
            inp = workloads.make(w, device="cuda")
            acc = accounting(inp)
            n, T, h = w.n_splits, w.T, w.h
            dev = inp.q.device
            out = torch.empty((T, h, 512), dtype=torch.float32, device=dev)
            lse = torch.empty((T, h), dtype=torch.float32, device=dev)
            op = torch.empty((n, T, h, 512), dtype=torch.float32, device=dev) if n > 1 else None
            lp = torch.empty((n, T, h), dtype=torch.float32, device=dev) if n > 1 else None

            def step(evs=None):
                if evs:
                    evs[0].record()
                if n > 1:
                    sfa.decode(inp.q, inp.kv, inp.block_table, inp.seq_lens, inp.topk_idx, w.scale,
                               n_splits=n, Q=w.Q, merge=False, out_part=op, lse_part=lp)
                    if evs:
                        evs[1].record()
                    sfa.lse_merge(op, lp, out=out, lse=lse)
                    if evs:
                        evs[2].record()
                else:
                    sfa.decode(inp.q, inp.kv, inp.block_table, inp.seq_lens, inp.topk_idx, w.scale,
                               n_splits=1, Q=w.Q, out=out, lse=lse)
                    if evs:
                        evs[1].record()

            for _ in range(3):
                flush()
                step()
            torch.cuda.synchronize()
            evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
            for k in range(steps):
                flush()
                hold_device()
                step(evs[k])
            torch.cuda.synchronize()
            if sfa.last_device_status() != 0:
                raise RuntimeError(f"device status error in workload {name}")
            dec = statistics.mean(e[0].elapsed_time(e[1]) for e in evs) * 1e3
            mrg = statistics.mean(e[1].elapsed_time(e[2]) for e in evs) * 1e3 if n > 1 else 0.0
            times = {"decode_us": dec, "merge_us": mrg if n > 1 else None,
                     "step_us": dec + (mrg if n > 1 else 0.0)}
            del inp, out, lse, op, lp
            torch.cuda.empty_cache()
        step_s = times["step_us"] * 1e-6
        roof_s, bound = roofline_of(acc, peaks)
        entry = {"B": w.B, "Q": w.Q, "h": w.h, "S": w.S, "top_k": w.top_k, "n_splits": w.n_splits,
                 **{k: v for k, v in times.items()},
                 "flops": acc["flops"], "algorithmic_bytes": acc["total_bytes"],
                 "gather_bytes": acc["gather_bytes"],
                 "TFLOP/s": acc["flops"] / step_s / 1e12,
                 "algorithmic_GB/s": acc["total_bytes"] / step_s / 1e9,
                 "roofline_us": roof_s * 1e6, "bound": bound, "frac": roof_s / step_s}
        if name == "tiny":
            entry["bound"] = "latency"
            entry["note"] = "a few KB of work: launch latency, not bandwidth, sets the time"
        if name == "sfa_h16":
            entry["note"] = ("not one of the five workloads: the headline shape with 16 heads, "
                             "where the step is a gather with little arithmetic per byte")
        entry["kernel"] = {3: "tcgen05 stacked-half", 2: "tcgen05 small-head", 1: "tcgen05 CTA pair",
                           0: "cuda-core"}[
            sfa.decode_launches(w.B, w.Q, w.h, w.top_k, w.block_size, w.n_splits)[1]]
        res[name] = entry
    return res


def read_traffic(kernel: str, tc_path: int, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if the kernel's sources (its
    .cu file, the host entry points and every header) still match the capture."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(path):
        return None
    from deepseek_sparse_mla_sfa_gb300 import build as _b
    src = {"decode": {3: "sfa_stack.cu", 2: "sfa_narrow.cu", 1: "sfa_tc.cu", 0: "sfa_simt.cu"}[int(tc_path)],
           "lse_merge": "sfa_merge.cu"}.get(kernel)
    if src is None:
        return None
    src_hash = _b.source_hash([src, "sfa_api.cu"])
    for line in open(path):
        parts = line.split()
        if len(parts) >= 4 and not line.startswith("#"):
            k, wl, h, b = parts[:4]
            if k == kernel and wl == workload and h == src_hash:
                return float(b)
    return None


def run_e2e(sfa, inp, steps, flush):
    """The step end to end: pinned host q / block_table / seq_lens / topk_idx in, out and
    lse back to pinned host memory, the cache resident in HBM.  Timed through the serving
    loop's call, a HostPlan (the sfa_decode_host step captured once, launched every step),
    and for reference through sfa_decode_host enqueued call by call."""
    w = inp.w
    pin = lambda t: t.cpu().contiguous().pin_memory()
    q_h, bt_h, sl_h, idx_h = pin(inp.q), pin(inp.block_table), pin(inp.seq_lens), pin(inp.topk_idx)
    out_h = torch.empty((w.T, w.h, 512), dtype=torch.float32).pin_memory()
    lse_h = torch.empty((w.T, w.h), dtype=torch.float32).pin_memory()
    nbytes = sfa.decode_host_staging_bytes(w.B, w.Q, w.h, w.top_k, inp.max_blocks, w.n_splits)
    staging = torch.empty(nbytes, dtype=torch.uint8, device=inp.q.device)
    direct = lambda: sfa.decode_host(q_h, inp.kv, bt_h, sl_h, idx_h, w.scale, w.n_splits, w.Q,
                                     out_h, lse_h, staging)
    plan = sfa.HostPlan(q_h, inp.kv, bt_h, sl_h, idx_h, w.scale, w.n_splits, w.Q, out_h, lse_h, staging)

    def timed(call):
        for _ in range(3):
            call()
        torch.cuda.synchronize()
        tot = 0.0
        for _ in range(steps):
            flush()
            torch.cuda.synchronize()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record()
            call()
            e1.record()
            e1.synchronize()
            tot += e0.elapsed_time(e1)
        return tot / max(1, steps)

    ms = timed(plan.launch)
    ms_direct = timed(direct)
    plan.close()
    acc = accounting(inp)
    h2d = sum(t.numel() * t.element_size() for t in (q_h, bt_h, sl_h, idx_h))
    d2h = out_h.numel() * 4 + lse_h.numel() * 4
    return {"value": acc["flops"] / (ms * 1e-3) / 1e12, "unit": UNIT, "ms_per_step": ms,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "api": "HostPlan.launch: the sfa_decode_host step captured once as a CUDA graph "
                   "(pinned host buffers, device-resident cache)",
            "direct_call_ms_per_step": ms_direct}


def spawn_ranks(n: int):
    """Re-run this command as n replica ranks (one per GPU) under torch.distributed.run on
    this node, rendezvous on 127.0.0.1; rank 0 prints the line."""
    import socket
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n}",
           "--master-addr=127.0.0.1", f"--master-port={port}", os.path.abspath(__file__), *sys.argv[1:]]
    sys.exit(subprocess.call(cmd))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", default=workloads.HEADLINE, choices=sorted(workloads.CONFIGS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-next-rows", action="store_true",
                    help="skip timing the kv_write / uv_proj / topk / lse_merge rows around the decode step")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip timing the other workloads (the line's `configs` object)")
    ap.add_argument("--batch", type=int, default=0,
                    help="override the workload's B (smaller cases for profiler captures)")
    ap.add_argument("--seq-len", type=int, default=0,
                    help="override the workload's S (smaller caches for profiler captures)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.batch or args.seq_len:
        base = workloads.CONFIGS[args.config]
        S = args.seq_len or base.S
        w = dataclasses.replace(base, B=args.batch or base.B, S=S, S_min=min(base.S_min, S) if base.S_min else 0,
                                top_k=min(base.top_k, S),
                                name=f"{args.config}_b{args.batch or base.B}_s{S}")
        workloads.CONFIGS[w.name] = w
        args.config = w.name
    world_env = int(os.environ.get("WORLD_SIZE", "1"))
    if args.gpus > 1 and world_env == 1 and "LOCAL_RANK" not in os.environ:
        # N replicas asked for without a launcher: start one rank per GPU through torchrun
        spawn_ranks(args.gpus)
        return
    if world_env > 1 and args.gpus != world_env:
        sys.exit(f"bench.py: --gpus {args.gpus} does not match WORLD_SIZE={world_env} of the launcher")
    if args.impl == "reference":
        # the reference arm is the CPU oracle: rank 0 alone runs it, the other ranks exit
        # without work, and no GPU or process group is needed
        run_reference(args, world_env, int(os.environ.get("RANK", "0")))
        return
    world, rank, local = dist_setup()
    try:
        run_ours(args, world, rank, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
