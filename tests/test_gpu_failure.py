"""Failure detection on the GPU without a fault: a pipeline wait that nothing
completes gives up after its limit and reports PKVD_ETIMEOUT, and the CUDA
context stays usable for a decode right after it."""
import pytest

import parity as Pt
from paged_kv_cache_plan_gb300 import _lib, selftest_wait_timeout
from paged_kv_cache_plan_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("limit_us", [1000, 20000])
def test_bounded_wait_runs_out(cuda_ok, limit_us):
    status, waited = selftest_wait_timeout(limit_us)
    assert status == _lib.PKVD_ETIMEOUT
    # it waited at least its limit and not much more (one check every 32 tries)
    assert limit_us <= waited < limit_us + 200000


def test_context_usable_after_timeout(cuda_ok):
    selftest_wait_timeout(1000)
    Pt.check_case(W.gqa_tiny(), variant="gqa_mma")


def test_selftest_arguments(cuda_ok):
    import ctypes
    L = _lib.lib()
    assert L.decode_selftest_wait_timeout(None, 1000, None) == _lib.PKVD_EINVAL
    import torch
    st = torch.zeros(2, dtype=torch.int32, device="cuda")
    assert L.decode_selftest_wait_timeout(ctypes.c_void_p(st.data_ptr()), 0, None) == _lib.PKVD_EINVAL
    assert L.decode_selftest_wait_timeout(ctypes.c_void_p(st.data_ptr()), 10**8, None) == _lib.PKVD_EINVAL
