"""GPU parity of shared-prefix plans (decode_plan_prefix): requests in a
group share their first prefix_len tokens, which one tensor-core work item
reads once for up to 64 / heads members; the private tokens run per request;
the merge combines both kinds of partials. Checked against the oracle (which
knows nothing of the grouping) and against the plain plan."""
import numpy as np
import pytest

import parity as Pt
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


@pytest.mark.parametrize("batch", [8, 48])
def test_mla16_shared_prefix_full_size(cuda_ok, batch):
    case = W.mla16(batch)
    res, plan = Pt.check_sampled(case, n=8, shared_prefix=True)
    assert plan.info["num_prefix_items"] > 0
