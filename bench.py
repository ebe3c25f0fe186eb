"""Benchmark: paged-KV split-KV decode attention on one GB300.

One step = one decode op (stage 1 + merge) over the workload's batch, timed
with CUDA events on the launching stream after an L2 flush (a 512 MB write,
then a 512 MB read that pushes the dirty lines out) that sits outside the
events. The default workload is the long-context GQA
decode at 64K tokens (batch 1, 16 query heads over 2 KV heads, d 256, page
16, random page order); --workload picks another.

Prints one JSON line (rank 0). value = algorithmic KV bytes of one op /
device time per op (GB/s); ms_per_step is that device time. e2e repeats the
op through the C ABI from pinned host buffers (q and page table in, out and
lse back) with the copies inside the events; the KV cache stays resident in
HBM like model weights. roofline = the stage-1 kernel's algorithmic bytes /
its own event-timed duration against the measured HBM copy bandwidth.
cpu_baseline = the fp64 oracle on this host's cores, on a bounded sample.

--impl reference times the oracle itself as the reference arm.
Under torchrun (N > 1) every rank runs its own replica (no collective in
the op); value sums the ranks' bytes over the slowest rank's time.
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
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode-attention µs/op and achieved HBM GB/s (% of GB300 peak) at 1 GPU"
FLUSH_BYTES = 512 << 20
FALLBACK_HBM_GBS = 6800.0


def workload(name: str):
    """A named workload; a trailing "_q<n>" asks for n query tokens per request
    (multi-token decode, causal among them) on the same cache."""
    from paged_kv_cache_plan_gb300 import workloads as W
    q_len = 1
    base, sep, tail = name.rpartition("_q")
    if sep and tail.isdigit():
        name, q_len = base, int(tail)
    if name.startswith("gqa_long_"):
        return W.gqa_long(int(name.split("_")[-1].rstrip("k")) * 1024, q_len=q_len)
    if name == "gqa_tiny":
        return W.gqa_tiny(q_len=q_len)
    if name.startswith("mla16_b"):
        return W.mla16(int(name[len("mla16_b"):]), q_len=q_len)
    if name.startswith("mla_h"):
        h, b = name[len("mla_h"):].split("_b")
        return W.mla_many(int(h), int(b), q_len=q_len)
    if name.startswith("gqa_varlen_"):
        return W.gqa_varlen(name[len("gqa_varlen_"):], q_len=q_len)
    raise SystemExit(f"unknown workload {name}")


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def recorded_traffic(kernel_src: str, workload_name: str):
    """DRAM bytes per stage-1 launch from the committed ncu summary, if it was
    taken on the current kernel source; else None."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    try:
        with open(path) as f:
            rec = json.load(f)
        sha = hashlib.sha256(open(kernel_src, "rb").read()).hexdigest()[:16]
        ent = rec.get(workload_name)
        if ent and ent.get("source_sha") == sha:
            return float(ent["bytes_per_launch"])
    except Exception:
        pass
    return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons while the timed loop runs."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.2)
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in getattr(self, "lines", []):
            f = [x.strip() for x in l.split(",")]
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
                for n, v in zip(names, f[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
            except (ValueError, IndexError):
                continue
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_init():
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64,
                     device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def oracle_sample_rate(case, budget_s: float, threads: int):
    """Oracle GB/s (the op's KV bytes per second) on the case truncated to
    the first n tokens of each request, n sized to the time budget."""
    import oracle
    from paged_kv_cache_plan_gb300 import workloads as W
    import torch

    def truncated(n):
        lens = torch.clamp(case.seq_lens, max=n).to(torch.int32)
        c = W.DecodeCase(case.name, case.q, case.k_pages, case.v_pages, case.page_table, lens,
                         case.heads, case.kv_heads, case.head_dim, case.head_dim_v,
                         case.page_size, case.k_row_pitch, case.v_row_pitch, case.scale,
                         case.dtype, case.mla, 0, 0, {}, case.q_len)
        return c

    def op_bytes(c):
        if case.mla:
            return int(c.seq_lens.sum()) * case.k_row_pitch * 2
        return int(c.seq_lens.sum()) * case.kv_heads * (case.head_dim + case.head_dim_v) * 2

    def run(c):
        P = oracle.problem(**W.oracle_problem_kwargs(c))
        t0 = time.perf_counter()
        oracle.decode(P, c.q, c.k_pages, c.v_pages, c.page_table, c.seq_lens, threads=threads)
        return time.perf_counter() - t0

    maxL = int(case.seq_lens.max())
    n = min(maxL, 256)
    dt = run(truncated(n))
    while dt < budget_s / 4 and n < maxL:
        n = min(maxL, n * 4)
        dt = run(truncated(n))
    c = truncated(n)
    reps, total, t_end = 0, 0.0, time.perf_counter() + budget_s
    while True:
        total += run(c)
        reps += 1
        if time.perf_counter() >= t_end:
            break
    gbs = op_bytes(c) * reps / total / 1e9
    sample = (f"{c.name}: first {n} of {maxL} tokens per request, all "
              f"{case.batch * case.q_len * case.heads} (request, token, head) rows, {reps} runs, "
              f"fp64 oracle on {threads} threads")
    return gbs, total / reps, sample, n


def reference_arm(args, world, rank):
    """The oracle as the reference arm: each step a bounded sample."""
    if rank != 0:
        return
    case = workload(args.workload)
    import oracle
    oracle.build()
    threads = os.cpu_count() or 1
    per_step = max(0.02, min(1.0, 90.0 / max(1, args.steps + args.warmup)))
    gbs, t_run, sample, n = oracle_sample_rate(case, per_step, threads)
    # the timed steps: the same sample, K times, after W warm-ups
    from paged_kv_cache_plan_gb300 import workloads as W
    import torch
    lens = torch.clamp(case.seq_lens, max=n).to(torch.int32)
    c = W.DecodeCase(case.name, case.q, case.k_pages, case.v_pages, case.page_table, lens,
                     case.heads, case.kv_heads, case.head_dim, case.head_dim_v, case.page_size,
                     case.k_row_pitch, case.v_row_pitch, case.scale, case.dtype, case.mla,
                     0, 0, {}, case.q_len)
    P = oracle.problem(**W.oracle_problem_kwargs(c))
    for _ in range(args.warmup):
        oracle.decode(P, c.q, c.k_pages, c.v_pages, c.page_table, c.seq_lens, threads=threads)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.decode(P, c.q, c.k_pages, c.v_pages, c.page_table, c.seq_lens, threads=threads)
    dt = time.perf_counter() - t0
    op_b = (int(lens.sum()) * (case.k_row_pitch * 2 if case.mla else
                               case.kv_heads * (case.head_dim + case.head_dim_v) * 2))
    value = op_b * args.steps / dt / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt / args.steps * 1e3, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": case.name, "sample_tokens_per_request": n},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def prefill_arm(args, world, rank, local):
    """The second workload: dense causal prefill at head_dim 64, named
    prefill_d64_b<B>_h<Hq>kv<Hkv>_L<L>. Times prefill_d64_run with CUDA events
    after an L2 flush, and reports algorithmic TFLOP/s (causal: 4 x 64 x
    L (L + 1) / 2 flops per request and head) against the measured bf16
    tensor peak."""
    import re
    import torch
    import numpy as np
    from paged_kv_cache_plan_gb300 import build as _build
    _build.build()
    from paged_kv_cache_plan_gb300 import prefill_d64
    from paged_kv_cache_plan_gb300 import workloads as W
    m = re.fullmatch(r"prefill_d64_b(\d+)_h(\d+)kv(\d+)_L(\d+)", args.workload)
    if not m:
        raise SystemExit(f"unknown workload {args.workload}")
    B, H, Hkv, L = (int(x) for x in m.groups())
    torch.cuda.set_device(local)
    case = W.prefill_case(batch=B, heads=H, kv_heads=Hkv, seq_len=L, seed=1006 + L)
    q, k, v = case.q.cuda(), case.k_pages.cuda(), case.v_pages.cuda()
    out = torch.empty((B, L, H, 64), dtype=torch.float32, device="cuda")
    lse = torch.empty((B, L, H), dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
    evict = torch.ones(FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()

    def step():
        prefill_d64(q, k, v, out=out, lse=lse, status=status)

    for _ in range(args.warmup):
        flush.fill_(1.0)
        evict.sum()
        step()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        for a, b in evs:
            flush.fill_(1.0)
            evict.sum()
            a.record(stream)
            step()
            b.record(stream)
        torch.cuda.synchronize()
    barrier(world)
    assert int(status.item()) == 0, "a pipeline wait ran out"
    ms = max_over_ranks(float(np.mean([a.elapsed_time(b) for a, b in evs])), world)
    flops = 4.0 * 64 * L * (L + 1) / 2 * B * H
    tflops = flops / (ms * 1e-3) / 1e12
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peak, src = float(json.load(f)["bf16_tflops"]), "measured (MEASURED_PEAKS.json bf16_tflops)"
    except Exception:
        peak, src = 1900.0, "fallback"
    line = {
        "metric": "dense causal prefill TFLOP/s at head_dim 64 (second workload)",
        "value": round(tflops * world, 2), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": case.name, "batch": B, "heads": H, "kv_heads": Hkv,
                   "seq_len": L, "head_dim": 64, "causal": True,
                   "l2": "flushed before every step (512 MB write, then 512 MB read, outside the events)"},
        "roofline": {"bound": "tensor", "achieved": round(tflops, 2), "peak": peak,
                     "unit": "TFLOP/s", "frac": round(tflops / peak, 4), "traffic": None,
                     "kernel": "prefill_d64", "peak_source": src},
        # two launches per step once the prompt has query tiles past 1,024 tokens
        "gpu_launches": args.steps * (2 if L > 1024 else 1), "clocks": clk.summary(),
        "cpu_baseline": None,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="gqa_long_64k")
    ap.add_argument("--variant", default="auto")
    ap.add_argument("--splits", type=int, default=-1, help="-1 = the workload's own choice")
    ap.add_argument("--cpu-budget", type=float, default=6.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-prefix", action="store_true",
                    help="plan shared-prefix workloads as independent requests")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)

    world, rank, local = dist_init()
    if args.impl == "reference":
        reference_arm(args, world, rank)
        barrier(world)
        return

    if args.workload.startswith("prefill_d64_"):
        prefill_arm(args, world, rank, local)
        barrier(world)
        return

    import torch
    import numpy as np
    from paged_kv_cache_plan_gb300 import build as _build
    _build.build()
    from paged_kv_cache_plan_gb300 import (decode_run, decode_run_timed, plan_for_case)
    from paged_kv_cache_plan_gb300 import _lib

    torch.cuda.set_device(local)
    case = workload(args.workload)
    dev = case.to("cuda")
    kw = {"variant": args.variant}
    if args.splits >= 0:
        kw["splits"] = args.splits
    groups = [g for g in case.meta.get("prefix_group", []) if g >= 0]
    shared_prefix = (not args.no_prefix and case.q_len == 1
                     and any(groups.count(g) > 1 for g in set(groups)))
    plan = plan_for_case(case, shared_prefix=shared_prefix, **kw)
    tok = () if case.q_len == 1 else (case.q_len,)
    out = torch.empty((case.batch, *tok, case.heads, case.head_dim_v), dtype=torch.float32,
                      device="cuda")
    lse = torch.empty((case.batch, *tok, case.heads), dtype=torch.float32, device="cuda")
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
    evict = torch.ones(FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()

    def flush_l2():
        # Write a buffer larger than L2, then read another one: the read pushes
        # the written (dirty) lines back to HBM before the events start, so the
        # timed op neither hits in L2 nor pays for the flush's write-back.
        flush.fill_(1.0)
        evict.sum()
    bytes_op = case.kv_bytes_unique()

    def step():
        decode_run(plan, dev.q, dev.k_pages, dev.v_pages, dev.page_table, out, lse)

    for _ in range(args.warmup):
        flush_l2()
        step()
    torch.cuda.synchronize()
    assert plan.last_device_status() == 0

    # ---- timed region: K ops, each after an L2 flush outside its events
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        t_wall = time.perf_counter()
        for a, b in evs:
            flush_l2()
            a.record(stream)
            step()
            b.record(stream)
        torch.cuda.synchronize()
        t_wall = time.perf_counter() - t_wall
    barrier(world)
    ms = [a.elapsed_time(b) for a, b in evs]
    ms_op = float(np.mean(ms))
    ms_op_max = max_over_ranks(ms_op, world)
    value = bytes_op * world / (ms_op_max * 1e-3) / 1e9
    status = plan.last_device_status()
    assert status == 0, f"device status {status}"

    # ---- per-stage events (ev_mid between the stages), for the roofline
    n_prof = min(args.steps, 1000)
    pev = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(3)) for _ in range(n_prof)]
    for trio in pev:          # torch creates the CUDA event on its first record()
        for e in trio:
            e.record(stream)
    torch.cuda.synchronize()
    for e0, e1, e2 in pev:
        flush_l2()
        decode_run_timed(plan, dev.q, dev.k_pages, dev.v_pages, dev.page_table, out, lse,
                         e0, e1, e2)
    torch.cuda.synchronize()
    s1 = float(np.mean([e0.elapsed_time(e1) for e0, e1, _ in pev]))
    s2 = float(np.mean([e1.elapsed_time(e2) for _, e1, e2 in pev]))

    # ---- end to end through the C ABI from pinned host buffers
    q_h = case.q.pin_memory()
    pt_h = case.page_table.pin_memory()
    out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    lse_h = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
    q_d, pt_d = torch.empty_like(dev.q), torch.empty_like(dev.page_table)
    n_e2e = min(args.steps, 1000)
    eev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(n_e2e)]
    for a, b in eev:
        flush_l2()
        a.record(stream)
        q_d.copy_(q_h, non_blocking=True)
        pt_d.copy_(pt_h, non_blocking=True)
        decode_run(plan, q_d, dev.k_pages, dev.v_pages, pt_d, out, lse)
        out_h.copy_(out, non_blocking=True)
        lse_h.copy_(lse, non_blocking=True)
        b.record(stream)
    torch.cuda.synchronize()
    ms_e2e = max_over_ranks(float(np.mean([a.elapsed_time(b) for a, b in eev])), world)
    h2d = q_h.numel() * q_h.element_size() + pt_h.numel() * pt_h.element_size()
    d2h = out_h.numel() * 4 + lse_h.numel() * 4

    hbm, peak_src = peaks()
    achieved = bytes_op / (s1 * 1e-3) / 1e9
    vname = {v: k for k, v in _lib.VARIANTS.items()}[plan.info["variant"]]
    if plan.info["num_prefix_items"] > 0:
        vname = "mla_tc"   # the shared-prefix items dominate
    kernel_src = os.path.join(ROOT, "paged_kv_cache_plan_gb300", "csrc",
                              {"mla_tc": "stage1_mla_tc.cu", "mla_mma": "stage1_mla.cu",
                               "gqa_fma": "stage1_gqa_fma.cu"}.get(vname, "stage1_gqa_mma.cu"))
    traffic = recorded_traffic(kernel_src, case.name)
    clocks = clk.summary()

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        threads = os.cpu_count() or 1
        gbs, t_run, sample, _ = oracle_sample_rate(case, args.cpu_budget, threads)
        cpu = {"value": round(gbs, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
               "sample": sample}

    info = plan.info
    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_op_max, 5),
            "us_per_op": round(ms_op_max * 1e3, 2), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None,
            "dtype": case.dtype, "data": "synthetic",
            "config": {"workload": case.name, "batch": case.batch, "heads": case.heads,
                       "kv_heads": case.kv_heads, "head_dim": case.head_dim,
                       "head_dim_v": case.head_dim_v, "page_size": case.page_size,
                       "query_tokens": case.q_len,
                       "seq_lens": (case.seq_lens.tolist() if case.batch <= 16 else
                                    f"{case.batch} x {int(case.seq_lens[0])}"),
                       "kv_bytes_per_op": bytes_op,
                       "l2": "flushed before every step (512 MB write, then 512 MB read, outside the events)",
                       "variant": {v: k for k, v in _lib.VARIANTS.items()}[info["variant"]],
                       "splits_max": info["max_splits"], "chunk": info["chunk"],
                       "work_items": info["num_items"], "ctas_per_sm": info["ctas_per_sm"],
                       "shared_prefix_items": info["num_prefix_items"],
                       "stage2_tiles": info["stage2_tiles"],
                       "grid_order": ["auto", "split_major", "request_major"][info["grid_order"]],
                       "parallelism": "replicas" if world > 1 else "single GPU"},
            "frac_of_hbm_peak": round(value / hbm, 4),
            "stage_ms": {"stage1": round(s1, 5), "stage2": round(s2, 5)},
            "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": hbm,
                         "unit": "GB/s", "frac": round(achieved / hbm, 4),
                         "traffic": traffic, "kernel": "stage1",
                         "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)"
                         if peak_src == "measured" else "fallback 6.8 TB/s"},
            "e2e": {"value": round(bytes_op / (ms_e2e * 1e-3) / 1e9, 2), "unit": "GB/s",
                    "us_per_op": round(ms_e2e * 1e3, 2), "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h},
            "gpu_launches": ((info["num_prefix_items"] > 0) + (info["num_items"] > 0) + 1) * args.steps,
            "clocks": clocks,
            "cpu_baseline": cpu,
            "wall_s_timed_region": round(t_wall, 3),
        }
        print(json.dumps(line), flush=True)
    barrier(world)


if __name__ == "__main__":
    main()
