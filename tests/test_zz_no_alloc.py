"""decode_run_static, the entry point that allocates no device memory.

Callers that cannot call cudaMalloc (a host application that owns all device
memory through its own pool, or code where allocating is forbidden) use
decode_run_static instead of decode_plan_ex + decode_run: it keeps all of its
scratch in one static device array inside the library. This file checks,
through the C ABI, that two calls in a row give the same results as the
planned entry point, and that a problem too large for the array is refused
before anything runs. It is named so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

import parity as Pt
from paged_kv_cache_plan_gb300 import _lib, plan_for_case, run_case
from paged_kv_cache_plan_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _run_static(desc, case, dev, out, lse):
    seq = (ctypes.c_int32 * case.batch)(*case.seq_lens.tolist())
    ptr = lambda t: ctypes.c_void_p(t.data_ptr())
    return _lib.lib().decode_run_static(
        ctypes.byref(desc), ctypes.cast(seq, ctypes.c_void_p), ptr(dev.q), ptr(dev.k_pages),
        ptr(dev.v_pages), ptr(dev.page_table), ptr(out), ptr(lse),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


CASES = {
    "gqa": lambda: W.gqa_case(batch=3, heads=16, kv_heads=2, head_dim=256, page_size=16,
                              seq_lens=[5000, 17, 900], pool_pages=500, seed=301),
    "mla": lambda: W.mla_case(batch=2, heads=16, seq_len=3000, prefix_len=2000, group=2,
                              pool_rows=9000, seed=302),
    # several query tokens per request
    "gqa_q3": lambda: W.gqa_case(batch=2, heads=8, kv_heads=2, head_dim=128, page_size=16,
                                 seq_lens=[700, 33], pool_pages=60, seed=303, q_len=3),
    "mla_q4": lambda: W.mla_case(batch=2, heads=16, seq_len=2000, prefix_len=0,
                                 pool_rows=5000, seed=304, q_len=4),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_static_scratch_matches_planned_entry_point(cuda_ok, name):
    case = CASES[name]()
    dev = case.to("cuda")
    plan = plan_for_case(case)
    ref_out, ref_lse = run_case(plan, dev)
    torch.cuda.synchronize()
    vh = case.q_len * case.heads   # (query token, head) rows per request
    ref_out = ref_out.reshape(case.batch, vh, case.head_dim_v).cpu().double().numpy()
    ref_lse = ref_lse.reshape(case.batch, vh).cpu().double().numpy()
    for call in range(2):
        out = torch.full((case.batch, vh, case.head_dim_v), float("nan"), device="cuda")
        lse = torch.full((case.batch, vh), float("nan"), device="cuda")
        _lib.check(_run_static(plan.desc, case, dev, out, lse), "decode_run_static")
        torch.cuda.synchronize()
        o = out.cpu().double().numpy()
        l = lse.cpu().double().numpy()
        assert np.all(np.isfinite(o)) and np.all(np.isfinite(l)), f"call {call}"
        assert np.abs(o - ref_out).max() <= Pt.OUT_ATOL, f"call {call}"
        assert np.abs(l - ref_lse).max() <= Pt.LSE_ATOL, f"call {call}"


def test_static_scratch_rejects_too_large(cuda_ok):
    # 128 heads x 256 splits x 512 columns of fp32 partials is 64 MiB > 16 MiB
    case = W.mla_case(batch=1, heads=128, seq_len=4096, pool_rows=4096, seed=303)
    dev = case.to("cuda")
    desc = plan_for_case(case, splits=256).desc
    out = torch.full((1, 128, 512), float("nan"), device="cuda")
    lse = torch.full((1, 128), float("nan"), device="cuda")
    assert _run_static(desc, case, dev, out, lse) == _lib.PKVD_ENOMEM
    torch.cuda.synchronize()
    assert torch.isnan(out).all() and torch.isnan(lse).all()
