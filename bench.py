#!/usr/bin/env python3
"""Benchmark of single-token MLA decode (split-KV) on GB300.

One step = one ``mla_decode`` call (one kernel launch: split-KV attention with the
log-sum-exp merge fused in) over one batch of seeded synthetic inputs already resident
in HBM.  Between timed calls a 256 MiB buffer is written to flush the 129 MB L2
(cold-cache timing, as the pages' own timing harness does), then a second 256 MiB
buffer is read so that the flush's dirty lines are written back before the timed call
starts instead of during it.  Prints ONE JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config I] [--impl ours|reference]

``--impl reference`` times the CPU fp64 oracle on the host cores on a bounded sample of
the same workload (the only other place this script runs the oracle).
Under torchrun (N > 1) every rank decodes its own replica of the workload (the batch is
sharded, no collective on the data path) and rank 0 reports the aggregate.
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

METRIC = "MLA decode \u00b5s/call and KV-cache HBM GB/s (fraction of 8 TB/s) per config"
DEFAULT_CONFIG = 2          # fp8-e4m3, batch 64 x 8192 tokens, split-KV + combine
FLUSH_BYTES = 256 << 20


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", type=int, default=DEFAULT_CONFIG)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the per-workload timings of all five workloads")
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--cpu-seconds", type=float, default=60.0,
                    help="--impl reference: total oracle time over all warm-up and timed steps")
    ap.add_argument("--quick", action="store_true",
                    help="timed steps only (no clock soak, e2e or CPU baseline); for profiler runs")
    ap.add_argument("--q-len", type=int, default=1,
                    help="with --page-size: query tokens per sequence (mla_decode_paged_multi when > 1)")
    ap.add_argument("--batch", type=int, default=0,
                    help="with --quick: the workload with this many sequences instead (a smaller case for profilers)")
    ap.add_argument("--page-size", type=int, default=0, choices=[0, 1, 2, 4, 8, 16, 32, 64, 128],
                    help="with --quick: store the workload's cache in shuffled pages of this many rows "
                         "and time mla_decode_paged")
    return ap.parse_args()


def max_over_ranks(values, ws, device=None):
    """Element-wise maximum of `values` over all ranks (a job takes as long as its slowest
    rank).  Identity for a single process."""
    if ws <= 1:
        return [float(v) for v in values]
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def job_gbs(kv_bytes_per_rank, ws, ms):
    """Whole-job KV GB/s: every rank decodes its own replica of the workload in `ms`."""
    return kv_bytes_per_rank * ws / (ms * 1e-3) / 1e9


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def kernel_source_hash() -> str:
    """Hash of the split kernel's translation unit: mla_split.cu and the headers it includes
    (the device code the committed ncu counters were taken on; the host-only sources of the
    library do not enter)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "mla_attention_decode_splitkv_gb300", "csrc")
    for name in ("mla_internal.h", "mla_split.cu", "ptx.cuh"):
        h.update(name.encode())
        h.update(open(os.path.join(csrc, name), "rb").read())
    return h.hexdigest()[:16]


def ncu_traffic(workload: str):
    """DRAM bytes per split-kernel launch from the committed ncu summary, if it was taken on
    the current kernel source; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    try:
        d = json.load(open(path))
        ent = d.get(workload)
        if ent and ent.get("kernel_source_hash") == kernel_source_hash():
            return float(ent["dram_bytes_per_launch"])
    except Exception:
        return None
    return None


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 100 ms while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


def oracle_sample_rate(inp, budget_s: float, max_rows: int = None):
    """Times the CPU oracle on whole batch rows (copied to the host) for about budget_s
    seconds of wall time.  Returns (GB/s of KV bytes, seconds, rows, threads)."""
    import numpy as np  # noqa: F401
    import oracle
    from mla_attention_decode_splitkv_gb300 import synth

    ip = inp.kv_indptr.cpu().tolist()
    B = len(ip) - 1
    order = list(range(B))
    threads = oracle.max_threads()
    # first, one row to size the sample
    rows, total_bytes, t_total = 0, 0, 0.0
    row_bytes = synth.KV_ROW_BYTES[inp.kv_dtype]
    scale_cpu = None if inp.kv_scale is None else inp.kv_scale
    while rows < B and (max_rows is None or rows < max_rows):
        take = 1 if rows == 0 else max(1, min(B - rows, threads,
                                              int((budget_s - t_total) / max(t_total / rows, 1e-3) * threads)))
        sel = order[rows:rows + take]
        lens = [ip[b + 1] - ip[b] for b in sel]
        q = inp.q[sel].cpu()
        kv = __import__("torch").cat([inp.kv[ip[b]:ip[b + 1]] for b in sel]).cpu()
        sc = None
        if inp.kv_dtype == synth.KV_FP8:
            sc = scale_cpu.cpu()
        elif inp.kv_dtype == synth.KV_MXFP4:
            sc = __import__("torch").cat([scale_cpu[ip[b]:ip[b + 1]] for b in sel]).cpu()
        sub_ip = synth.indptr_from_lengths(lens)
        t0 = time.perf_counter()
        oracle.decode(q, kv, sc, sub_ip, inp.kv_dtype, nthreads=threads)
        t_total += time.perf_counter() - t0
        rows += take
        total_bytes += sum(lens) * row_bytes
        if t_total >= budget_s:
            break
    return total_bytes / t_total / 1e9, t_total, rows, threads


def run_reference(args, ws, rank):
    if rank != 0:
        return
    import torch
    from mla_attention_decode_splitkv_gb300 import synth
    spec = synth.CONFIGS[args.config]
    inp = synth.make_config(args.config, device="cpu", keep_src=False) if spec.batch * (spec.kv_len or 4096) <= 600000 \
        else synth.make_config(args.config, device="cuda" if torch.cuda.is_available() else "cpu", keep_src=False)
    per_step_budget = max(0.05, args.cpu_seconds / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        oracle_sample_rate(inp, per_step_budget / 4, max_rows=1)
    rates, secs, nrows = [], 0.0, 0
    threads = 1
    for _ in range(args.steps):
        r, t, n, threads = oracle_sample_rate(inp, per_step_budget)
        rates.append(r)
        secs += t
        nrows += n
    value = statistics.mean(rates)
    kv_bytes = inp.kv_bytes()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": kv_bytes / (value * 1e9) * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_dict(spec, inp),
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": f"{nrows} whole batch rows over {args.steps} steps ({secs:.1f} s of oracle time); "
                                   f"ms_per_step extrapolates to the full batch"},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def measure_workload(pkg, index, dev, steps, flush_l2, with_oracle=True):
    """One workload of the five, in the library's own launch configuration: cold calls (L2
    flushed before each), back-to-back warm calls, the split kernel's own time (library
    events), KV GB/s and its fraction of the measured HBM peak, the ncu traffic ratio when
    the committed counters match this kernel source, and the largest error against the
    CPU oracle over a few sampled batch rows."""
    import numpy as np
    import torch
    from mla_attention_decode_splitkv_gb300 import synth

    spec = synth.CONFIGS[index]
    inp = synth.make_config(index, device=dev, keep_src=False)
    B = inp.batch
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    ns = pkg.resolve_splits(spec.num_splits, B, inp.rows // B, sms, spec.kv_dtype)
    pkg.reserve_workspace(pkg.workspace_slots(B, ns, sms))
    out = torch.empty((B, 16, 512), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream(dev)

    def call():
        rc = pkg.mla_decode(inp.q, inp.kv, inp.kv_scale, inp.kv_indptr, out, B, ns, spec.kv_dtype, stream)
        if rc != pkg.MLA_OK:
            raise pkg.MLAError(rc, "mla_decode")

    for _ in range(3):
        call()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for i in range(steps):
        flush_l2(i)
        evs[i][0].record(stream)
        call()
        evs[i][1].record(stream)
    torch.cuda.synchronize()
    cold_us = [a.elapsed_time(b) * 1e3 for a, b in evs]
    # the same cold calls again, with the library's own events around its kernel
    pkg.profile_begin()
    for i in range(steps):
        flush_l2(i)
        call()
    torch.cuda.synchronize()
    split_ms_sum, _, ncalls = pkg.profile_end()
    wevs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for a, b in wevs:
        a.record(stream)
        call()
        b.record(stream)
    torch.cuda.synchronize()
    warm_us = [a.elapsed_time(b) * 1e3 for a, b in wevs]
    if pkg.device_status(clear=True) != pkg.MLA_OK:
        raise RuntimeError(f"kernel reported a pipeline timeout on {spec.name}")
    kv_bytes = inp.kv_bytes()
    kernel_us = split_ms_sum / max(1, ncalls) * 1e3
    peak, _ = peaks()
    res = {"workload": spec.name, "num_splits": ns, "kv_bytes_per_call": kv_bytes,
           "cold_us_median": statistics.median(cold_us), "warm_us_median": statistics.median(warm_us),
           "kernel_us": kernel_us, "gbs": kv_bytes / (statistics.median(cold_us) * 1e-6) / 1e9,
           "kernel_gbs": kv_bytes / (kernel_us * 1e-6) / 1e9}
    res["frac_of_measured_peak"] = res["kernel_gbs"] / peak
    tr = ncu_traffic(spec.name)
    res["traffic_ratio"] = None if tr is None else tr / kv_bytes
    if with_oracle:
        import oracle
        ip = inp.kv_indptr.cpu().tolist()
        rows = sorted({0, B - 1} | set(np.random.default_rng(index).choice(B, size=min(B, 2), replace=False).tolist()))
        worst = 0.0
        got_all = out.float().cpu().numpy()
        for b in rows:
            kv_rows = inp.kv[ip[b]:ip[b + 1]].cpu()
            scale = None if inp.kv_scale is None else (
                inp.kv_scale[ip[b]:ip[b + 1]].cpu() if spec.kv_dtype == synth.KV_MXFP4 else inp.kv_scale.cpu())
            o, _ = oracle.attend(inp.q[b].cpu(), kv_rows, scale, spec.kv_dtype, 0, ip[b + 1] - ip[b])
            worst = max(worst, float(np.abs(got_all[b] - o).max()))
        res["max_abs_err_vs_oracle"] = worst
        res["oracle_rows_checked"] = len(rows)
        # the CPU oracle's own rate on this workload (whole batch rows, about 1.5 s of wall time)
        r, t, n, threads = oracle_sample_rate(inp, 1.5)
        res["cpu_oracle"] = {"gbs": r, "cores": threads, "rows": n, "seconds": t}
    del inp, out
    torch.cuda.empty_cache()
    return res


def config_dict(spec, inp):
    """The workload, the same for both arms (the GPU arm's launch shape is in its `launch` key)."""
    from mla_attention_decode_splitkv_gb300 import synth
    lens = inp.lens
    return {"workload": spec.name, "batch": spec.batch,
            "kv_len": spec.kv_len if spec.kv_len else f"ragged U[1,8192], mean {sum(lens) / len(lens):.0f}",
            "kv_dtype": synth.DTYPE_NAMES[spec.kv_dtype],
            "heads": 16, "head_dim": 576, "v_dim": 512, "kv_bytes_per_call": inp.kv_bytes(),
            "l2": "flushed between timed calls (256 MiB write, then 256 MiB read to retire the dirty lines)",
            "headline": "value and roofline are this workload's; the metric is per workload, and all five "
                        "(in their own launch configurations) are in per_config"}


def main():
    args = parse()
    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if args.impl == "ours" else "gloo")
    if args.impl == "reference":
        run_reference(args, ws, rank)
        return

    import torch
    import mla_attention_decode_splitkv_gb300 as pkg
    from mla_attention_decode_splitkv_gb300 import build as pkg_build
    from mla_attention_decode_splitkv_gb300 import synth

    pkg_build.build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    spec = synth.CONFIGS[args.config]
    if args.batch:
        if not args.quick:
            raise SystemExit("--batch is a --quick measurement")
        import dataclasses
        spec = dataclasses.replace(spec, name=f"{spec.name}_batch{args.batch}", batch=args.batch)
        lens = ([spec.kv_len] * spec.batch if spec.kv_len else synth.ragged_lengths(spec.batch, 8192, spec.seed))
        inp = synth.make_inputs(spec.batch, lens, spec.kv_dtype, spec.seed, device=dev, keep_src=False)
    else:
        inp = synth.make_config(args.config, device=dev, keep_src=False)
    B = inp.batch
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    ns = pkg.resolve_splits(spec.num_splits, B, inp.rows // B, sms, spec.kv_dtype)
    paged = None
    if args.q_len > 1 and not args.page_size:
        raise SystemExit("--q-len > 1 needs --page-size")
    if args.page_size:
        if not args.quick:
            raise SystemExit("--page-size is a --quick measurement")
        if args.q_len > 1:
            ns = 0          # the library's multi-query default (uniform splits over the query-token pairs)
        paged = synth.to_paged(inp, args.page_size, seed=spec.seed + 7).to(dev)
        if args.q_len > 1:
            mq, mqo = synth.make_queries([args.q_len] * B, seed=spec.seed + 8, device=dev)
        kv_bytes = inp.kv_bytes()
        inp.kv = None                    # free the contiguous copy
        torch.cuda.empty_cache()
    pkg.reserve_workspace(pkg.workspace_slots(B * max(1, args.q_len), ns, sms))
    out = torch.empty((B * max(1, args.q_len), 16, 512), dtype=torch.bfloat16, device=dev)
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    evict = torch.ones(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    evict_sum = torch.empty((), dtype=torch.float32, device=dev)

    def flush_l2(i):
        flush.fill_(float(i))
        torch.sum(evict, dim=0, out=evict_sum)
    stream = torch.cuda.current_stream(dev)

    def call():
        if paged is not None and args.q_len > 1:
            rc = pkg.mla_decode_paged_multi(mq, mqo, B * args.q_len, paged.kv, paged.kv_scale, paged.page_indptr,
                                            paged.page_indices, paged.last_page_len, args.page_size, out, B, ns,
                                            spec.kv_dtype, stream)
        elif paged is not None:
            rc = pkg.mla_decode_paged(paged.q, paged.kv, paged.kv_scale, paged.page_indptr, paged.page_indices,
                                      paged.last_page_len, args.page_size, out, B, ns, spec.kv_dtype, stream)
        else:
            rc = pkg.mla_decode(inp.q, inp.kv, inp.kv_scale, inp.kv_indptr, out, B, ns, spec.kv_dtype, stream)
        if rc != pkg.MLA_OK:
            raise pkg.MLAError(rc, "mla_decode")

    for _ in range(max(3, args.warmup)):
        call()
    torch.cuda.synchronize()
    sampler = ClockSampler(local if "CUDA_VISIBLE_DEVICES" not in os.environ else 0)
    if not args.quick:
        sampler.start()
        t_soak = time.perf_counter()
        while time.perf_counter() - t_soak < 0.6:      # load the GPU so clock samples exist
            for _ in range(20):
                call()
            torch.cuda.synchronize()
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for i in range(args.steps):
        flush_l2(i)
        evs[i][0].record(stream)
        call()
        evs[i][1].record(stream)
    torch.cuda.synchronize()
    # second pass, same pattern, with the library's own events around its split kernel
    pkg.profile_begin()
    for i in range(args.steps):
        flush_l2(i)
        call()
    torch.cuda.synchronize()
    split_ms_sum, call_ms_sum, ncalls = pkg.profile_end()
    # warm calls (no flush between them), each timed on its own, for the latency medians
    # (not in --quick runs, whose launch sequence the profiler commands count on)
    n_warm = 0 if args.quick else max(20, args.steps)
    wevs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_warm)]
    for a, b in wevs:
        a.record(stream)
        call()
        b.record(stream)
    torch.cuda.synchronize()
    warm_us = [a.elapsed_time(b) * 1e3 for a, b in wevs]
    if ws > 1:
        torch.distributed.barrier()
    clocks = sampler.stop()
    step_ms = [a.elapsed_time(b) for a, b in evs]
    ms = statistics.mean(step_ms)
    split_ms = split_ms_sum / max(1, ncalls)
    if pkg.device_status(clear=True) != pkg.MLA_OK:
        raise RuntimeError("kernel reported a pipeline timeout during the benchmark")
    if args.quick:
        if rank == 0:
            kvb = kv_bytes if paged is not None else inp.kv_bytes()
            print(json.dumps({"workload": spec.name, "page_size": args.page_size, "q_len": args.q_len,
                              "num_splits": ns,
                              "us_per_call": ms * 1e3, "split_kernel_us": split_ms * 1e3,
                              "kv_bytes_per_call": kvb, "split_gbs": kvb / (split_ms * 1e-3) / 1e9}), flush=True)
        return

    # ---- end to end: host (pinned) inputs -> device, decode, output -> host, every step
    q_h = inp.q.cpu().pin_memory()
    kv_h = inp.kv.cpu().pin_memory()
    sc_h = None if inp.kv_scale is None else inp.kv_scale.cpu().pin_memory()
    ip_h = inp.kv_indptr.cpu().pin_memory()
    out_h = torch.empty((B, 16, 512), dtype=torch.bfloat16).pin_memory()
    q_d, kv_d = torch.empty_like(inp.q), torch.empty_like(inp.kv)
    sc_d = None if sc_h is None else torch.empty_like(inp.kv_scale)
    ip_d = torch.empty_like(inp.kv_indptr)
    h2d = q_h.numel() * 2 + kv_h.numel() * kv_h.element_size() + (0 if sc_h is None else sc_h.numel() * sc_h.element_size()) \
        + ip_h.numel() * 4
    d2h = out_h.numel() * 2

    def e2e_step():
        q_d.copy_(q_h, non_blocking=True)
        kv_d.copy_(kv_h, non_blocking=True)
        if sc_d is not None:
            sc_d.copy_(sc_h, non_blocking=True)
        ip_d.copy_(ip_h, non_blocking=True)
        rc = pkg.mla_decode(q_d, kv_d, sc_d, ip_d, out, B, ns, spec.kv_dtype, stream)
        if rc != pkg.MLA_OK:
            raise pkg.MLAError(rc, "mla_decode")
        out_h.copy_(out, non_blocking=True)

    e2e_step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.e2e_steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / args.e2e_steps
    assert torch.equal(out_h, out.cpu())

    # ---- aggregate over ranks (max time)
    ms, split_ms, e2e_ms = max_over_ranks([ms, split_ms, e2e_ms], ws, dev)
    if rank != 0:
        return
    kv_bytes = inp.kv_bytes()
    value = job_gbs(kv_bytes, ws, ms)
    peak, peak_kind = peaks()
    achieved = kv_bytes / (split_ms * 1e-3) / 1e9
    launches_per_call = 1          # the split kernel; the merge runs inside it
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms, "us_per_call": ms * 1e3, "frac_of_8tbs": value / ws / 8000.0,
        "latency_us": {"cold_median": statistics.median(step_ms) * 1e3, "warm_median": statistics.median(warm_us),
                       "cold_calls": len(step_ms), "warm_calls": len(warm_us)},
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": {0: "bf16", 1: "e4m3", 2: "e4m3"}[spec.kv_dtype],
        "data": "synthetic (seeded N(0,1) q and KV, stored per the workload's cache encoding)",
        "config": config_dict(spec, inp),
        "launch": {"num_splits": (f"{ns} per sequence (uniform)" if ns else "balanced (persistent, one CTA per SM)")
                                 + ("" if spec.num_splits is not None else ", chosen by mla_decode_pick_splits")},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "peak_kind": f"{peak_kind} (burst copy)", "kernel": "mla_split_kernel",
                     "split_kernel_us": split_ms * 1e3, "algorithmic_bytes_per_launch": kv_bytes,
                     "traffic": ncu_traffic(spec.name)},
        "e2e": {"value": job_gbs(kv_bytes, ws, e2e_ms), "unit": "GB/s", "ms_per_step": e2e_ms,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": args.steps * launches_per_call,
        "clocks": clocks,
    }
    if not args.no_cpu_baseline:
        r, t, n, threads = oracle_sample_rate(inp, 12.0)
        line["cpu_baseline"] = {"value": r, "unit": "GB/s", "cores": threads, "kind": "oracle",
                                "sample": f"{n} whole batch rows of the workload ({t:.1f} s)"}
    if not args.no_per_config:
        # The metric is per workload: every one of the five, in its own launch configuration.
        del inp, q_d, kv_d, q_h, kv_h
        torch.cuda.empty_cache()
        line["per_config"] = [measure_workload(pkg, i, dev, max(10, min(args.steps, 30)), flush_l2,
                                               with_oracle=not args.no_cpu_baseline)
                              for i in range(len(synth.CONFIGS))]
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
