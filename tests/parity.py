"""Shared helpers of the GPU parity tests: run the CUDA path through the C ABI
on a seeded case, run the oracle on the same host tensors, compare.

Tolerances: max |out - oracle| <= 2e-3 and max |lse - oracle| <= 1e-4
(fp32 accumulation from bf16/fp16 inputs against the fp64 oracle). Because
softmax over long contexts is nearly flat, |out| shrinks like 1/sqrt(L), so
the relative L2 error of out is also held below 1e-2.
"""
from __future__ import annotations

import math
import os

import numpy as np
import torch

import oracle
from paged_kv_cache_plan_gb300 import plan_for_case, run_case
from paged_kv_cache_plan_gb300 import workloads as W

OUT_ATOL = 2e-3
LSE_ATOL = 1e-4
REL_L2 = 1e-2

THREADS = max(1, (os.cpu_count() or 1))


def oracle_full(case):
    P = oracle.problem(**W.oracle_problem_kwargs(case))
    return oracle.decode(P, case.q, case.k_pages, case.v_pages, case.page_table,
                         case.seq_lens, threads=THREADS)


def oracle_pairs(case, pairs):
    """The oracle on the listed (b, v) rows, spread over the host's threads
    (each chunk of rows is one call into the C oracle, which drops the GIL)."""
    from concurrent.futures import ThreadPoolExecutor
    P = oracle.problem(**W.oracle_problem_kwargs(case))
    pairs = list(pairs)
    n = max(1, min(THREADS, len(pairs)))
    chunks = [pairs[i::n] for i in range(n)]

    def run(ch):
        return oracle.decode(P, case.q, case.k_pages, case.v_pages, case.page_table,
                             case.seq_lens, pairs=ch)

    with ThreadPoolExecutor(n) as ex:
        res = list(ex.map(run, chunks))
    out = np.zeros((len(pairs), case.head_dim_v))
    lse = np.zeros((len(pairs),))
    for i, (o, l) in enumerate(res):
        out[i::n] = o
        lse[i::n] = l
    return out, lse


def run_gpu(case, dev_case=None, poison=True, **plan_kw):
    """Plan + run through the C ABI; out/lse start NaN-filled so that a head
    the kernels skip cannot pass. Returns (out, lse, plan) on the host, as
    [B, q_len * Hq, Dv] / [B, q_len * Hq] (the oracle's (token, head) rows)."""
    dev = dev_case if dev_case is not None else case.to("cuda")
    plan = plan_for_case(case, **plan_kw)
    tok = () if case.q_len == 1 else (case.q_len,)
    out = torch.full((case.batch, *tok, case.heads, case.head_dim_v),
                     float("nan") if poison else 0.0, dtype=torch.float32, device="cuda")
    lse = torch.full((case.batch, *tok, case.heads), float("nan") if poison else 0.0,
                     dtype=torch.float32, device="cuda")
    run_case(plan, dev, out, lse)
    torch.cuda.synchronize()
    status = plan.last_device_status()
    assert status == 0, f"device status {status}"
    vh = case.q_len * case.heads
    out = out.reshape(case.batch, vh, case.head_dim_v)
    lse = lse.reshape(case.batch, vh)
    return out.cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64), plan


def compare(out, lse, ref_out, ref_lse, what=""):
    assert out.shape == ref_out.shape and lse.shape == ref_lse.shape
    empty = np.isneginf(ref_lse)
    assert np.array_equal(np.isneginf(lse), empty), f"{what}: empty-head mismatch"
    assert np.all(out[empty] == 0), f"{what}: empty heads must give 0"
    assert np.all(np.isfinite(out)), f"{what}: non-finite output"
    e_out = np.abs(out - ref_out).max() if out.size else 0.0
    fin = ~empty
    e_lse = np.abs(lse[fin] - ref_lse[fin]).max() if fin.any() else 0.0
    num = np.linalg.norm((out - ref_out)[fin])
    den = np.linalg.norm(ref_out[fin])
    rel = num / den if den > 0 else num
    assert e_out <= OUT_ATOL, f"{what}: max|out err| {e_out:.3g} > {OUT_ATOL}"
    assert e_lse <= LSE_ATOL, f"{what}: max|lse err| {e_lse:.3g} > {LSE_ATOL}"
    assert rel <= REL_L2, f"{what}: relative L2 {rel:.3g} > {REL_L2}"
    return dict(max_out=float(e_out), max_lse=float(e_lse), rel_l2=float(rel))


def check_case(case, ref=None, **plan_kw):
    out, lse, plan = run_gpu(case, **plan_kw)
    ref_out, ref_lse = ref if ref is not None else oracle_full(case)
    return compare(out, lse, ref_out, ref_lse, case.name), plan


def sample_pairs(case, n, seed=0):
    rng = np.random.default_rng(seed)
    B, H = case.batch, case.q_len * case.heads
    pairs = {(0, 0), (B - 1, H - 1)}
    while len(pairs) < min(n, B * H):
        pairs.add((int(rng.integers(B)), int(rng.integers(H))))
    return sorted(pairs)


def edge_pairs(case, extra=8, seed=0):
    """Rows of a full-size case the oracle checks one by one: every (query
    token, head) row of the first and the last request, the first and last
    row of every request, and `extra` random rows. A fault confined to one
    head block, one request of a group or a late split shows up in one of
    them."""
    B, H = case.batch, case.q_len * case.heads
    pairs = {(b, h) for b in (0, B - 1) for h in range(H)}
    pairs |= {(b, h) for b in range(B) for h in (0, H - 1)}
    pairs |= set(sample_pairs(case, extra, seed))
    return sorted(pairs)


def check_sampled(case, n=8, dev_case=None, pairs=None, **plan_kw):
    """Full-size run on the GPU, the oracle on n sampled (b, h) heads (or on
    the given pairs)."""
    out, lse, plan = run_gpu(case, dev_case=dev_case, **plan_kw)
    assert np.all(np.isfinite(out)) and np.all(np.isfinite(lse))
    if pairs is None:
        pairs = sample_pairs(case, n)
    ref_o, ref_l = oracle_pairs(case, pairs)
    got_o = np.stack([out[b, h] for b, h in pairs])
    got_l = np.array([lse[b, h] for b, h in pairs])
    return compare(got_o, got_l, ref_o, ref_l, case.name), plan


def lse_closed_form_check(lse, L):
    """q = 0 sanity: lse = ln L."""
    return np.abs(lse - math.log(L)).max()
