"""Bit-exactness and robustness of the CUDA path.

Bit-exact (north of any tolerance): relabelling physical pages, split-major
versus request-major grid order (a pure relabelling, as the aiter pull 4758
page requires of its split-major grid: bit-identical output), merge tiling.
Within tolerance: any split count. Also: the debug page-id checks report an
out-of-pool id through the status word (never a fault), graph capture, and
plans that differ only in batch or lengths stay distinct."""
import numpy as np
import pytest
import torch

import parity as Pt
from paged_kv_cache_plan_gb300 import _lib, plan_for_case, run_case
from paged_kv_cache_plan_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _cases():
    return {
        "gqa_fma": (W.gqa_case(batch=3, heads=16, kv_heads=2, head_dim=256, page_size=16,
                               seq_lens=[3000, 17, 900], pool_pages=400, seed=91), "gqa_fma"),
        "gqa_mma": (W.gqa_case(batch=3, heads=16, kv_heads=2, head_dim=256, page_size=16,
                               seq_lens=[3000, 17, 900], pool_pages=400, seed=91), "gqa_mma"),
        "mla": (W.mla_case(batch=4, heads=16, seq_len=2000, prefix_len=1500, group=2,
                           pool_rows=8000, seed=92), "mla_mma"),
        "mla_tc": (W.mla_case(batch=3, heads=64, seq_len=1700, prefix_len=1200, group=2,
                              pool_rows=6000, seed=93), "mla_tc"),
    }


CASES = _cases()


@pytest.mark.parametrize("name", sorted(CASES))
def test_page_relabelling_bit_exact(cuda_ok, name):
    case, variant = CASES[name]
    o1, l1, _ = Pt.run_gpu(case, variant=variant, splits=5)
    for seed in (1, 2):
        o2, l2, _ = Pt.run_gpu(W.permute_pages(case, seed), variant=variant, splits=5)
        assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


@pytest.mark.parametrize("name", sorted(CASES))
def test_grid_order_bit_exact(cuda_ok, name):
    case, variant = CASES[name]
    o1, l1, p1 = Pt.run_gpu(case, variant=variant, grid_order="split_major")
    o2, l2, p2 = Pt.run_gpu(case, variant=variant, grid_order="request_major")
    assert p1.info["grid_order"] == 1 and p2.info["grid_order"] == 2
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


@pytest.mark.parametrize("name", sorted(CASES))
def test_stage2_tiling_bit_exact(cuda_ok, name):
    case, variant = CASES[name]
    ref = None
    for tiles in (1, 2, 4, 8):
        o, l, p = Pt.run_gpu(case, variant=variant, stage2_tiles=tiles, splits=9)
        assert p.info["stage2_tiles"] == tiles
        if ref is None:
            ref = (o, l)
        else:
            assert np.array_equal(ref[0], o) and np.array_equal(ref[1], l)


@pytest.mark.parametrize("name", sorted(CASES))
def test_split_count_invariance(cuda_ok, name):
    case, variant = CASES[name]
    ref = Pt.oracle_full(case)
    for splits in (1, 2, 4, 7, 256):
        Pt.check_case(case, ref=ref, variant=variant, splits=splits)


def test_variants_agree_within_tolerance(cuda_ok):
    case, _ = CASES["gqa_fma"]
    o1, l1, _ = Pt.run_gpu(case, variant="gqa_fma")
    o2, l2, _ = Pt.run_gpu(case, variant="gqa_mma")
    assert np.abs(o1 - o2).max() <= 2 * Pt.OUT_ATOL and np.abs(l1 - l2).max() <= 2 * Pt.LSE_ATOL


def test_page_id_checks_report_status(cuda_ok):
    # checks on: an id outside the pool is replaced by page 0 inside the
    # kernel and reported through the status word; nothing faults
    case = W.gqa_case(batch=2, heads=8, kv_heads=2, head_dim=128, page_size=16,
                      seq_lens=[100, 50], pool_pages=20, seed=93)
    bad = case.page_table.clone()
    bad[1, 2] = 10_000
    dev = case.to("cuda")
    dev.page_table = bad.cuda()
    for variant in ("gqa_fma", "gqa_mma"):
        plan = plan_for_case(case, variant=variant, checks=True)
        run_case(plan, dev)
        assert plan.last_device_status() == _lib.PKVD_EDEVICE_CHECK
        # the status word is cleared by the read, and a clean run stays clean
        run_case(plan, case.to("cuda"))
        assert plan.last_device_status() == 0
    mla = W.mla_case(batch=2, heads=16, seq_len=300, pool_rows=700, seed=94)
    mdev = mla.to("cuda")
    mbad = mla.page_table.clone()
    mbad[0, 299] = -5
    mdev.page_table = mbad.cuda()
    plan = plan_for_case(mla, checks=True)
    run_case(plan, mdev)
    assert plan.last_device_status() == _lib.PKVD_EDEVICE_CHECK


def test_cuda_graph_replay_matches_eager(cuda_ok):
    case, variant = CASES["gqa_mma"]
    dev = case.to("cuda")
    plan = plan_for_case(case, variant=variant)
    out_e, lse_e = run_case(plan, dev)
    torch.cuda.synchronize()
    out = torch.full_like(out_e, float("nan"))
    lse = torch.full_like(lse_e, float("nan"))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        run_case(plan, dev, out, lse, stream=s)   # warm-up outside capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    out.fill_(float("nan"))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        run_case(plan, dev, out, lse)
    for _ in range(3):
        out.fill_(float("nan"))
        g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, out_e) and torch.equal(lse, lse_e)


def test_plans_differing_only_in_batch(cuda_ok):
    # Specs that differ only in batch (then only in lengths) must each give
    # their own correct result, in either order.
    c4 = W.gqa_case(batch=4, heads=8, kv_heads=2, head_dim=128, page_size=16,
                    seq_lens=[2048] * 4, seed=95)
    c6 = W.gqa_case(batch=6, heads=8, kv_heads=2, head_dim=128, page_size=16,
                    seq_lens=[256, 512, 768, 1024, 1536, 2048], seed=96)
    r4, r6 = Pt.oracle_full(c4), Pt.oracle_full(c6)
    for order in ((c4, r4), (c6, r6), (c4, r4)):
        Pt.check_case(order[0], ref=order[1])


def test_repeated_runs_identical(cuda_ok):
    case, variant = CASES["mla"]
    dev = case.to("cuda")
    plan = plan_for_case(case, variant=variant)
    o1, l1 = run_case(plan, dev)
    o1, l1 = o1.clone(), l1.clone()
    for _ in range(3):
        o2, l2 = run_case(plan, dev)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
