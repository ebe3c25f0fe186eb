"""GPU parity of shared-prefix plans (decode_plan_prefix): requests in a
group share their first prefix_len tokens, which one tensor-core work item
reads once for up to 64 / heads members; the private tokens run per request;
the merge combines both kinds of partials. Checked against the oracle (which
knows nothing of the grouping) and against the plain plan."""
import numpy as np
import pytest
import torch

import parity as Pt
from paged_kv_cache_plan_gb300 import _lib, plan_for_case, run_case
from paged_kv_cache_plan_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _check_prefix(case, ref=None):
    out, lse, plan = Pt.run_gpu(case, shared_prefix=True)
    assert plan.info["num_prefix_items"] > 0
    ref_o, ref_l = ref if ref is not None else Pt.oracle_full(case)
    res = Pt.compare(out, lse, ref_o, ref_l, case.name + " shared prefix")
    o2, l2, _ = Pt.run_gpu(case)   # the plain plan, same tolerance
    Pt.compare(out, lse, o2, l2, case.name + " prefix vs plain")
    return res


@pytest.mark.parametrize("batch,group,heads", [(6, 3, 16), (5, 5, 16), (4, 2, 32), (8, 8, 16)])
def test_groups(cuda_ok, batch, group, heads):
    case = W.mla_case(batch=batch, heads=heads, seq_len=1500, prefix_len=1100, group=group,
                      seed=111)
    _check_prefix(case)


def test_ungrouped_request_and_whole_sequence_prefix(cuda_ok):
    case = W.mla_case(batch=5, heads=16, seq_len=1300, prefix_len=1300, group=2, seed=112)
    case.meta["prefix_group"][4] = -1    # shares nothing (its rows are its group's anyway)
    case.meta["prefix_len"][4] = 0
    _check_prefix(case)


def test_fp16(cuda_ok):
    case = W.mla_case(batch=4, heads=16, seq_len=2000, prefix_len=1500, group=4,
                      dtype="fp16", seed=113)
    _check_prefix(case)


@pytest.mark.parametrize("prefix", [1, 64, 500, 1023])
@pytest.mark.parametrize("heads", [16, 64])
def test_short_prefixes_with_private_tails(cuda_ok, prefix, heads):
    # too short to batch on the tensor-memory kernel: every member reads the
    # prefix itself (the tensor-memory kernel only over requests of 1,024
    # tokens or more), at the standard tolerances
    case = W.mla_case(batch=5, heads=heads, seq_len=prefix + 700, prefix_len=prefix, group=3,
                      seed=114 + prefix)
    out, lse, plan = Pt.run_gpu(case, shared_prefix=True)
    assert plan.info["num_prefix_items"] == 0
    assert plan.info["variant"] == (4 if prefix + 700 >= 1024 else 3)
    ref_o, ref_l = Pt.oracle_full(case)
    Pt.compare(out, lse, ref_o, ref_l, case.name + " short shared prefix")


def test_long_prefix_short_tails(cuda_ok):
    # 64 heads: the prefix items on the tensor-memory kernel, 1- to 40-token
    # private tails on the mma.sync kernel
    case = W.mla_case(batch=4, heads=64, seq_len=2100, prefix_len=2060, group=4, seed=118)
    case.seq_lens[:] = torch.tensor([2061, 2070, 2100, 2060], dtype=torch.int32)
    res = _check_prefix(case)


def test_prefix_page_relabelling_bit_exact(cuda_ok):
    case = W.mla_case(batch=6, heads=16, seq_len=2500, prefix_len=1800, group=3,
                      pool_rows=9000, seed=119)
    o1, l1, p1 = Pt.run_gpu(case, shared_prefix=True)
    assert p1.info["num_prefix_items"] > 0
    for seed in (1, 2):
        o2, l2, _ = Pt.run_gpu(W.permute_pages(case, seed), shared_prefix=True)
        assert np.array_equal(o1, o2) and np.array_equal(l1, l2), f"relabelling {seed}"


def test_prefix_promise_checked(cuda_ok):
    # with checks on, a member whose prefix page differs from the first
    # member's is reported (PKVD_EDEVICE_CHECK); the same plan without the
    # difference reports nothing
    case = W.mla_case(batch=4, heads=16, seq_len=1500, prefix_len=1200, group=4,
                      pool_rows=7000, seed=120)
    dev = case.to("cuda")
    plan = plan_for_case(case, shared_prefix=True, checks=True)
    assert plan.info["num_prefix_items"] > 0
    out = torch.empty((4, 16, 512), device="cuda")
    lse = torch.empty((4, 16), device="cuda")
    run_case(plan, dev, out, lse)
    assert plan.last_device_status() == _lib.PKVD_OK
    bad = case.page_table.clone()
    bad[2, 700] = int(case.page_table[2, 1300])   # still inside the pool
    dev.page_table = bad.cuda()
    run_case(plan, dev, out, lse)
    assert plan.last_device_status() == _lib.PKVD_EDEVICE_CHECK


@pytest.mark.parametrize("batch", [8, 48])
def test_mla16_shared_prefix_full_size(cuda_ok, batch):
    # every head of the first and last request, the first and last head of
    # every request (each member of every group), a few random rows
    case = W.mla16(batch)
    res, plan = Pt.check_sampled(case, pairs=Pt.edge_pairs(case), shared_prefix=True)
    assert plan.info["num_prefix_items"] > 0
