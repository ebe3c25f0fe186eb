"""decode_run_static, the entry point that allocates no device memory.

Callers that cannot call cudaMalloc (a host application that owns all device
memory through its own pool, or code where allocating is forbidden) use
decode_run_static instead of decode_plan_ex + decode_run: it keeps all of its
scratch in one static device array inside the library. This file checks,
through the C ABI, that two calls in a row give bit-for-bit the results of the
planned entry point (same planner, same kernels, same inputs) and the oracle's
within the usual tolerance, that the second call changes the device's free
memory by nothing, that its status query reports a page id outside the pool,
and that a problem too large for the array, or a stream being captured, is
refused before anything runs. It is named so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

import parity as Pt
from paged_kv_cache_plan_gb300 import _lib, plan_for_case, run_case
from paged_kv_cache_plan_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _run_static(desc, case, dev, out, lse, stream=None):
    seq = (ctypes.c_int32 * case.batch)(*case.seq_lens.tolist())
    ptr = lambda t: ctypes.c_void_p(t.data_ptr())
    s = stream if stream is not None else torch.cuda.current_stream()
    return _lib.lib().decode_run_static(
        ctypes.byref(desc), ctypes.cast(seq, ctypes.c_void_p), ptr(dev.q), ptr(dev.k_pages),
        ptr(dev.v_pages), ptr(dev.page_table), ptr(out), ptr(lse),
        ctypes.c_void_p(s.cuda_stream))


def _static_status():
    return _lib.lib().decode_run_static_status(
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


CASES = {
    "gqa": lambda: W.gqa_case(batch=3, heads=16, kv_heads=2, head_dim=256, page_size=16,
                              seq_lens=[5000, 17, 900], pool_pages=500, seed=301),
    "mla": lambda: W.mla_case(batch=2, heads=16, seq_len=3000, prefix_len=2000, group=2,
                              pool_rows=9000, seed=302),
    "mla_tc": lambda: W.mla_case(batch=2, heads=64, seq_len=2100, pool_rows=4300, seed=305),
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
    ref_out = ref_out.reshape(case.batch, vh, case.head_dim_v).cpu().numpy()
    ref_lse = ref_lse.reshape(case.batch, vh).cpu().numpy()
    orc_out, orc_lse = Pt.oracle_full(case)
    for call in range(2):
        out = torch.full((case.batch, vh, case.head_dim_v), float("nan"), device="cuda")
        lse = torch.full((case.batch, vh), float("nan"), device="cuda")
        torch.cuda.synchronize()
        free0, _ = torch.cuda.mem_get_info()
        _lib.check(_run_static(plan.desc, case, dev, out, lse), "decode_run_static")
        assert _static_status() == _lib.PKVD_OK      # synchronises the stream
        free1, _ = torch.cuda.mem_get_info()
        if call == 1:   # the first call may load the kernels' code; later ones take nothing
            assert free1 == free0, f"free device memory moved by {free0 - free1} bytes"
        o, l = out.cpu().numpy(), lse.cpu().numpy()
        # same planner, kernels and inputs as the planned entry point: same bits
        assert np.array_equal(o, ref_out), f"call {call}: out differs from decode_run"
        assert np.array_equal(l, ref_lse), f"call {call}: lse differs from decode_run"
        Pt.compare(o.astype(np.float64), l.astype(np.float64), orc_out, orc_lse,
                   f"{name} static call {call}")


def test_static_status_reports_bad_page(cuda_ok):
    # checks on: a page id outside the pool is replaced by page 0 on the device
    # (nothing faults) and the status query returns PKVD_EDEVICE_CHECK; the
    # next clean call reports PKVD_OK again
    case = W.gqa_case(batch=2, heads=8, kv_heads=2, head_dim=128, page_size=16,
                      seq_lens=[100, 50], pool_pages=20, seed=306)
    dev = case.to("cuda")
    desc = plan_for_case(case, checks=True).desc
    out = torch.empty((2, 8, 128), device="cuda")
    lse = torch.empty((2, 8), device="cuda")
    good = dev.page_table
    bad = case.page_table.clone()
    bad[1, 2] = 10_000
    dev.page_table = bad.cuda()
    _lib.check(_run_static(desc, case, dev, out, lse), "decode_run_static")
    assert _static_status() == _lib.PKVD_EDEVICE_CHECK
    dev.page_table = good
    _lib.check(_run_static(desc, case, dev, out, lse), "decode_run_static")
    assert _static_status() == _lib.PKVD_OK


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


def test_static_scratch_refuses_capture(cuda_ok):
    # the work list is copied from host memory the call frees on return, so a
    # stream under capture is refused before anything is queued
    case = CASES["gqa_q3"]()
    dev = case.to("cuda")
    desc = plan_for_case(case).desc
    out = torch.full((2, 24, 128), float("nan"), device="cuda")
    lse = torch.full((2, 24), float("nan"), device="cuda")
    x = torch.zeros(4, device="cuda")
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        g.capture_begin()
        rc = _run_static(desc, case, dev, out, lse, stream=side)
        x.add_(1.0)   # keeps the captured graph non-empty
        g.capture_end()
    torch.cuda.current_stream().wait_stream(side)
    assert rc == _lib.PKVD_EUNSUPPORTED
    g.replay()
    torch.cuda.synchronize()
    assert torch.isnan(out).all() and float(x[0]) == 1.0
