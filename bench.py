"""Benchmark: paged-KV split-KV decode attention on one GB300.

One step = one decode op (stage 1 + merge) over the workload's batch, timed
with CUDA events on the launching stream after an L2 flush (a 512 MB write,
then a 512 MB read that pushes the dirty lines out) that sits outside the
events. The default workload is the largest single-GPU configuration: MLA
decode with 128 heads over 128 requests of 16,384 distinct tokens each (one
576-wide latent row per token, page size 1, 2.42 GB of KV per op);
--workload picks another. Inputs are seeded N(0, 1) values drawn on the
device with the workloads module's shapes and page structure.

Prints one JSON line (rank 0). value = algorithmic KV bytes of one op /
device time per op (GB/s); ms_per_step is that device time. e2e repeats the
op through the C ABI from pinned host buffers (q and page table in, out and
lse back) with the copies inside the events; the KV cache stays resident in
HBM like model weights. roofline = the stage-1 kernel's algorithmic bytes /
its own event-timed duration against the measured HBM copy bandwidth.
cpu_baseline = the fp64 oracle on this host's cores, on a bounded sample.
per_config = every long-context GQA and MLA configuration, timed the same
way (fewer steps each), with its stage-1 fraction of the HBM peak.

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


def workload(name: str, device: str = "cpu", context=None):
    """A named workload; a trailing "_q<n>" asks for n query tokens per request
    (multi-token decode, causal among them) on the same cache. device !=
    "cpu" draws the values on that device (same shapes, distributions and
    page structure; other draws). context: cut every request to its first
    `context` tokens (the bounded CPU samples of the oracle legs)."""
    from paged_kv_cache_plan_gb300 import workloads as W
    q_len = 1
    base, sep, tail = name.rpartition("_q")
    if sep and tail.isdigit():
        name, q_len = base, int(tail)
    kw = {"q_len": q_len, "device": device}
    if name.startswith("gqa_long_"):
        L = int(name.split("_")[-1].rstrip("k")) * 1024
        return W.gqa_long(L if context is None else min(L, context), seed=1002 + L, **kw)
    if name == "gqa_tiny":
        return W.gqa_tiny(**kw)
    if name.startswith("mla16_b"):
        B = int(name[len("mla16_b"):])
        if context is None:
            return W.mla16(B, **kw)
        c = min(W.MLA16_CONTEXT, context)
        p = min(W.MLA16_PREFIX, max(0, c - (W.MLA16_CONTEXT - W.MLA16_PREFIX)))
        groups = (B + 7) // 8
        return W.mla16(B, context=c, prefix=p, pool_rows=groups * p + B * (c - p), **kw)
    if name.startswith("mla_h"):
        h, b = name[len("mla_h"):].split("_b")
        if context is None:
            return W.mla_many(int(h), int(b), **kw)
        return W.mla_many(int(h), int(b), context=min(W.MLA_MANY_CONTEXT, context), **kw)
    if name.startswith("gqa_varlen_"):
        if context is None:
            return W.gqa_varlen(name[len("gqa_varlen_"):], **kw)
        lens = [min(L, context) for L in W.VARLEN_LENS]
        return W.gqa_varlen(name[len("gqa_varlen_"):], lens=lens, pool_pages=None, **kw)
    raise SystemExit(f"unknown workload {name}")


def full_context(name: str) -> int:
    """Longest context of a named workload."""
    from paged_kv_cache_plan_gb300 import workloads as W
    name = name.rpartition("_q")[0] if name.rpartition("_q")[2].isdigit() else name
    if name.startswith("gqa_long_"):
        return int(name.split("_")[-1].rstrip("k")) * 1024
    if name.startswith("mla16_b"):
        return W.MLA16_CONTEXT
    if name.startswith("mla_h"):
        return W.MLA_MANY_CONTEXT
    if name.startswith("gqa_varlen_"):
        return max(W.VARLEN_LENS)
    return 512


# The per-configuration record that rides on the default line: every
# long-context and MLA configuration of the target, each timed like the
# headline (L2 flushed outside the events, clocks sampled).
PER_CONFIG = ("gqa_long_64k", "gqa_long_32k", "gqa_long_16k", "gqa_long_8k", "gqa_long_2k",
              "gqa_varlen_bf16", "gqa_varlen_fp16", "mla16_b1", "mla16_b8", "mla16_b24",
              "mla16_b48", "mla_h64_b64", "mla_h64_b128", "mla_h128_b64", "mla_h128_b128")


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def source_sha(paths) -> str:
    """First 16 hex digits of the SHA-256 of the kernel's source files, in order."""
    h = hashlib.sha256()
    for p in ([paths] if isinstance(paths, str) else paths):
        h.update(open(p, "rb").read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel_src, workload_name: str):
    """DRAM bytes per stage-1 launch from the committed ncu summary, if it was
    taken on the current kernel source (a file or a list of files); else None."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    try:
        with open(path) as f:
            rec = json.load(f)
        sha = source_sha(kernel_src)
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


def oracle_sample_rate(name: str, budget_s: float, threads: int):
    """Oracle GB/s (the op's KV bytes per second) on the workload cut to the
    first n tokens of each request (drawn on the CPU), n sized to the time
    budget. Returns (GB/s, seconds per run, sample description, n, case)."""
    import oracle
    from paged_kv_cache_plan_gb300 import workloads as W

    def op_bytes(c):
        if c.mla:
            return int(c.seq_lens.sum()) * c.k_row_pitch * 2
        return int(c.seq_lens.sum()) * c.kv_heads * (c.head_dim + c.head_dim_v) * 2

    def run(c):
        P = oracle.problem(**W.oracle_problem_kwargs(c))
        t0 = time.perf_counter()
        oracle.decode(P, c.q, c.k_pages, c.v_pages, c.page_table, c.seq_lens, threads=threads)
        return time.perf_counter() - t0

    full = workload(name, context=1)   # shapes only
    maxL = full_context(name)
    n = min(maxL, 256)
    c = workload(name, context=n)
    dt = run(c)
    while dt < budget_s / 4 and n < maxL:
        n = min(maxL, n * 4)
        c = workload(name, context=n)
        dt = run(c)
    reps, total, t_end = 0, 0.0, time.perf_counter() + budget_s
    while True:
        total += run(c)
        reps += 1
        if time.perf_counter() >= t_end:
            break
    gbs = op_bytes(c) * reps / total / 1e9
    sample = (f"{name} at an {n}-token context (of {maxL}), all "
              f"{full.batch * full.q_len * full.heads} (request, token, head) rows, {reps} runs, "
              f"fp64 oracle on {threads} threads")
    return gbs, total / reps, sample, n, c


def reference_arm(args, world, rank):
    """The oracle as the reference arm: each step a bounded sample."""
    if rank != 0:
        return
    import oracle
    from paged_kv_cache_plan_gb300 import workloads as W
    oracle.build()
    threads = os.cpu_count() or 1
    per_step = max(0.02, min(1.0, 90.0 / max(1, args.steps + args.warmup)))
    gbs, t_run, sample, n, c = oracle_sample_rate(args.workload, per_step, threads)
    # the timed steps: the same sample, K times, after W warm-ups
    P = oracle.problem(**W.oracle_problem_kwargs(c))
    for _ in range(args.warmup):
        oracle.decode(P, c.q, c.k_pages, c.v_pages, c.page_table, c.seq_lens, threads=threads)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.decode(P, c.q, c.k_pages, c.v_pages, c.page_table, c.seq_lens, threads=threads)
    dt = time.perf_counter() - t0
    op_b = (int(c.seq_lens.sum()) * (c.k_row_pitch * 2 if c.mla else
                                     c.kv_heads * (c.head_dim + c.head_dim_v) * 2))
    value = op_b * args.steps / dt / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt / args.steps * 1e3, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": workload(args.workload, context=1).name.rsplit("_L", 1)[0],
                   "sample_tokens_per_request": n},
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


# a kernel's own source files (the GQA consumers share their block streaming)
KERNEL_SRC = {"mla_tc": ("stage1_mla_tc.cu",), "mla_mma": ("stage1_mla.cu",),
              "gqa_fma": ("stage1_gqa_fma.cu", "stage1_gqa.cuh"),
              "gqa_mma": ("stage1_gqa_mma.cu", "stage1_gqa.cuh")}


class Timer:
    """Times decode ops on one workload: each op after an L2 flush (a buffer
    larger than L2 written, then another one read, so the written lines are
    back in HBM before the events start) that sits outside the events."""

    def __init__(self):
        import torch
        self.torch = torch
        self.flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
        self.evict = torch.ones(FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")

    def flush_l2(self):
        self.flush.fill_(1.0)
        self.evict.sum()

    def ops(self, fn, steps: int, warmup: int, clock_index=None):
        """Mean event time (ms) of `fn` over `steps` flushed ops, the wall time
        of the timed loop and the clock summary (if clock_index is given)."""
        torch = self.torch
        stream = torch.cuda.current_stream()
        for _ in range(warmup):
            self.flush_l2()
            fn()
        torch.cuda.synchronize()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(steps)]
        sampler = ClockSampler(clock_index) if clock_index is not None else None
        if sampler:
            sampler.__enter__()
        t_wall = time.perf_counter()
        for a, b in evs:
            self.flush_l2()
            a.record(stream)
            fn()
            b.record(stream)
        torch.cuda.synchronize()
        t_wall = time.perf_counter() - t_wall
        clocks = None
        if sampler:
            sampler.__exit__(None, None, None)
            clocks = sampler.summary()
        import numpy as np
        return float(np.mean([a.elapsed_time(b) for a, b in evs])), t_wall, clocks

    def stages(self, plan, dev, out, lse, steps: int):
        """Mean stage-1 and merge times (ms): an event between the stages."""
        torch = self.torch
        import numpy as np
        from paged_kv_cache_plan_gb300 import decode_run_timed
        stream = torch.cuda.current_stream()
        pev = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(3)) for _ in range(steps)]
        for trio in pev:          # torch creates the CUDA event on its first record()
            for e in trio:
                e.record(stream)
        torch.cuda.synchronize()
        for e0, e1, e2 in pev:
            self.flush_l2()
            decode_run_timed(plan, dev.q, dev.k_pages, dev.v_pages, dev.page_table, out, lse,
                             e0, e1, e2)
        torch.cuda.synchronize()
        return (float(np.mean([e0.elapsed_time(e1) for e0, e1, _ in pev])),
                float(np.mean([e1.elapsed_time(e2) for _, e1, e2 in pev])))


def plan_workload(case, args):
    """Plan a workload as the benchmark runs it: batches whose requests share
    prefixes in groups get a shared-prefix plan unless --no-prefix."""
    from paged_kv_cache_plan_gb300 import plan_for_case
    kw = {"variant": args.variant}
    if args.splits >= 0:
        kw["splits"] = args.splits
    groups = [g for g in case.meta.get("prefix_group", []) if g >= 0]
    shared_prefix = (not args.no_prefix and case.q_len == 1
                     and any(groups.count(g) > 1 for g in set(groups)))
    return plan_for_case(case, shared_prefix=shared_prefix, **kw)


def stage1_kernel_name(plan):
    from paged_kv_cache_plan_gb300 import _lib
    vname = {v: k for k, v in _lib.VARIANTS.items()}[plan.info["variant"]]
    return "mla_tc" if plan.info["num_prefix_items"] > 0 else vname


def measure(name, args, timer, clock_index, steps, warmup):
    """One workload drawn on the device, planned and timed: (record, case,
    plan, out, lse)."""
    import torch
    from paged_kv_cache_plan_gb300 import decode_run
    case = workload(name, device="cuda")
    plan = plan_workload(case, args)
    tok = () if case.q_len == 1 else (case.q_len,)
    out = torch.empty((case.batch, *tok, case.heads, case.head_dim_v), dtype=torch.float32,
                      device="cuda")
    lse = torch.empty((case.batch, *tok, case.heads), dtype=torch.float32, device="cuda")

    def step():
        decode_run(plan, case.q, case.k_pages, case.v_pages, case.page_table, out, lse)

    ms, t_wall, clocks = timer.ops(step, steps, warmup, clock_index)
    status = plan.last_device_status()
    assert status == 0, f"{name}: device status {status}"
    s1, s2 = timer.stages(plan, case, out, lse, min(steps, 1000))
    hbm, _ = peaks()
    kv = case.kv_bytes_unique()
    kern = stage1_kernel_name(plan)
    traffic = recorded_traffic(
        [os.path.join(ROOT, "paged_kv_cache_plan_gb300", "csrc", f) for f in KERNEL_SRC[kern]],
        case.name)
    info = plan.info
    rec = {
        "workload": case.name, "us_per_op": round(ms * 1e3, 2),
        "gbs": round(kv / (ms * 1e-3) / 1e9, 2), "frac_of_hbm_peak": round(kv / (ms * 1e-3) / 1e9 / hbm, 4),
        "stage1_us": round(s1 * 1e3, 2), "stage2_us": round(s2 * 1e3, 2),
        "stage1_frac": round(kv / (s1 * 1e-3) / 1e9 / hbm, 4),
        "traffic": traffic, "kv_bytes_per_op": kv, "kernel": kern,
        "splits_max": info["max_splits"], "work_items": info["num_items"],
        "shared_prefix_items": info["num_prefix_items"], "steps": steps,
        "clocks": clocks, "wall_s_timed_region": round(t_wall, 3),
    }
    return rec, case, plan, out, lse, ms, s1, s2, t_wall, clocks


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="mla_h128_b128")
    ap.add_argument("--variant", default="auto")
    ap.add_argument("--splits", type=int, default=-1, help="-1 = the workload's own choice")
    ap.add_argument("--cpu-budget", type=float, default=6.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-prefix", action="store_true",
                    help="plan shared-prefix workloads as independent requests")
    ap.add_argument("--per-config-steps", type=int, default=40,
                    help="timed ops per configuration of the per-config record (0 = skip it)")
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
    from paged_kv_cache_plan_gb300 import decode_run
    from paged_kv_cache_plan_gb300 import _lib

    torch.cuda.set_device(local)
    timer = Timer()

    # ---- timed region: K ops of the headline workload, each after an L2 flush
    barrier(world)
    torch.cuda.synchronize()
    rec, case, plan, out, lse, ms_op, s1, s2, t_wall, clocks = measure(
        args.workload, args, timer, local, args.steps, args.warmup)
    barrier(world)
    ms_op_max = max_over_ranks(ms_op, world)
    bytes_op = case.kv_bytes_unique()
    value = bytes_op * world / (ms_op_max * 1e-3) / 1e9
    stream = torch.cuda.current_stream()

    # ---- end to end through the C ABI from pinned host buffers
    q_h = case.q.cpu().pin_memory()
    pt_h = case.page_table.cpu().pin_memory()
    out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    lse_h = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
    q_d, pt_d = torch.empty_like(case.q), torch.empty_like(case.page_table)

    def e2e_step():
        q_d.copy_(q_h, non_blocking=True)
        pt_d.copy_(pt_h, non_blocking=True)
        decode_run(plan, q_d, case.k_pages, case.v_pages, pt_d, out, lse)
        out_h.copy_(out, non_blocking=True)
        lse_h.copy_(lse, non_blocking=True)

    ms_e2e, _, _ = timer.ops(e2e_step, min(args.steps, 1000), 3)
    ms_e2e = max_over_ranks(ms_e2e, world)
    h2d = q_h.numel() * q_h.element_size() + pt_h.numel() * pt_h.element_size()
    d2h = out_h.numel() * 4 + lse_h.numel() * 4

    hbm, peak_src = peaks()
    achieved = bytes_op / (s1 * 1e-3) / 1e9
    traffic = rec["traffic"]
    info = plan.info
    launches_per_op = (info["num_prefix_items"] > 0) + (info["num_items"] > 0) + 1
    head_cfg = {"workload": case.name, "batch": case.batch, "heads": case.heads,
                "kv_heads": case.kv_heads, "head_dim": case.head_dim,
                "head_dim_v": case.head_dim_v, "page_size": case.page_size,
                "query_tokens": case.q_len,
                "seq_lens": (case.seq_lens.tolist() if case.batch <= 16 else
                             f"{case.batch} x {int(case.seq_lens[0])}"),
                "kv_bytes_per_op": bytes_op,
                "l2": "flushed before every step (512 MB write, then 512 MB read, outside the events)",
                "inputs": "seeded N(0,1) values drawn on the device, seeded CPU page scatter",
                "variant": {v: k for k, v in _lib.VARIANTS.items()}[info["variant"]],
                "splits_max": info["max_splits"], "chunk": info["chunk"],
                "work_items": info["num_items"], "ctas_per_sm": info["ctas_per_sm"],
                "shared_prefix_items": info["num_prefix_items"],
                "stage2_tiles": info["stage2_tiles"],
                "grid_order": ["auto", "split_major", "request_major"][info["grid_order"]],
                "parallelism": "replicas" if world > 1 else "single GPU"}
    dtype = case.dtype
    del out, lse, plan, case, q_d, pt_d
    torch.cuda.empty_cache()

    # ---- every target configuration, timed the same way (rank 0, N = 1 only)
    per_config = None
    if rank == 0 and world == 1 and args.per_config_steps > 0:
        per_config = {}
        for name in PER_CONFIG:
            if name == args.workload:
                per_config[name] = {k: v for k, v in rec.items()}
                continue
            r = measure(name, args, timer, local, args.per_config_steps, 3)[0]
            per_config[name] = r
            torch.cuda.empty_cache()

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        threads = os.cpu_count() or 1
        gbs, t_run, sample, _, _ = oracle_sample_rate(args.workload, args.cpu_budget, threads)
        cpu = {"value": round(gbs, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
               "sample": sample}

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_op_max, 5),
            "us_per_op": round(ms_op_max * 1e3, 2), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None,
            "dtype": dtype,
            "data": "synthetic",
            "config": head_cfg,
            "frac_of_hbm_peak": round(value / world / hbm, 4),
            "stage_ms": {"stage1": round(s1, 5), "stage2": round(s2, 5)},
            "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": hbm,
                         "unit": "GB/s", "frac": round(achieved / hbm, 4),
                         "traffic": traffic, "kernel": "stage1 (" + rec["kernel"] + ")",
                         "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)"
                         if peak_src == "measured" else "fallback 6.8 TB/s"},
            "e2e": {"value": round(bytes_op / (ms_e2e * 1e-3) / 1e9, 2), "unit": "GB/s",
                    "us_per_op": round(ms_e2e * 1e3, 2), "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h},
            "gpu_launches": launches_per_op * args.steps,
            "clocks": clocks,
            "cpu_baseline": cpu,
            "wall_s_timed_region": round(t_wall, 3),
            "per_config": per_config,
        }
        print(json.dumps(line), flush=True)
    barrier(world)


if __name__ == "__main__":
    main()
