"""ctypes binding of the C ABI in include/pkvd.h (argument marshalling only).

The names match the C entry points: decode_plan, decode_plan_ex,
decode_plan_prefix, decode_run, decode_run_timed, decode_run_static,
decode_run_static_status, decode_cp_ranges, decode_plan_cp, decode_plan_cp_compute,
decode_merge_ranks, decode_plan_destroy, decode_workspace_bytes, decode_plan_query,
decode_last_device_status, decode_plan_compute, decode_plan_prefix_compute,
decode_status_string, decode_selftest_wait_timeout, prefill_d64_run. Every
step of the computation runs in libpkvd.so's
CUDA kernels; if the library is missing this module raises instead of
falling back to anything else.
"""
from __future__ import annotations

import ctypes
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libpkvd.so")

PKVD_OK, PKVD_EINVAL, PKVD_EUNSUPPORTED, PKVD_ECUDA = 0, -1, -2, -3
PKVD_ENOMEM, PKVD_EDEVICE_CHECK, PKVD_ETIMEOUT = -4, -5, -6
PKVD_BF16, PKVD_FP16 = 0, 1
PKVD_FAMILY_GQA, PKVD_FAMILY_MLA = 0, 1
VARIANTS = {"auto": 0, "gqa_fma": 1, "gqa_mma": 2, "mla_mma": 3, "mla_tc": 4}
GRID_ORDERS = {"auto": 0, "split_major": 1, "request_major": 2}


class PlanDesc(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "batch", "heads", "kv_heads", "head_dim", "head_dim_v", "page_size", "dtype",
        "splits", "grid_order", "stage2_tiles", "variant", "checks", "num_sms",
        "ctas_per_sm", "min_chunk", "q_len")] + [
        (n, ctypes.c_int64) for n in ("max_pages_per_seq", "num_pool_pages",
                                      "k_row_pitch", "v_row_pitch")] + [
        ("scale", ctypes.c_float), ("reserved2", ctypes.c_int32)]


class PrefillDesc(ctypes.Structure):
    """pkvd_prefill_desc (include/pkvd.h)."""
    _fields_ = [("batch", ctypes.c_int32), ("heads", ctypes.c_int32),
                ("kv_heads", ctypes.c_int32), ("seq_len", ctypes.c_int32),
                ("dtype", ctypes.c_int32), ("scale", ctypes.c_float),
                ("reserved", ctypes.c_int32 * 2)]


class PlanInfo(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "family", "variant", "grid_order", "stage2_tiles", "stage2_threads", "num_sms",
        "ctas_per_sm", "heads_per_unit", "units_per_request", "num_items",
        "num_partial_rows", "max_splits")] + [
        ("chunk", ctypes.c_int64), ("workspace_bytes", ctypes.c_int64)] + [
        (n, ctypes.c_int32) for n in ("block_tokens", "pipeline_stages",
                                      "stage1_smem_bytes", "stage1_threads", "kv_tiles",
                                      "num_prefix_items")]

    def as_dict(self) -> dict:
        return {n: getattr(self, n) for n, _ in self._fields_}


class WorkItem(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "request", "unit", "split", "partial_row", "tok_begin", "tok_end",
        "grouped", "query_pos")]


# Every function the header declares, with (restype, argtypes).
_vp, _i32, _i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
_pp = ctypes.POINTER(ctypes.c_void_p)
SIGNATURES = {
    "decode_plan": (ctypes.c_int, [_pp, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                   ctypes.c_int, _vp, ctypes.c_int]),
    "decode_plan_ex": (ctypes.c_int, [_pp, ctypes.POINTER(PlanDesc), _vp]),
    "decode_run": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp]),
    "decode_run_timed": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp]),
    "decode_plan_destroy": (ctypes.c_int, [_vp]),
    "decode_workspace_bytes": (ctypes.c_size_t, [_vp]),
    "decode_plan_query": (ctypes.c_int, [_vp, ctypes.POINTER(PlanInfo)]),
    "decode_last_device_status": (ctypes.c_int, [_vp, _vp]),
    "decode_plan_compute": (ctypes.c_int, [ctypes.POINTER(PlanDesc), _vp,
                                           ctypes.POINTER(PlanInfo), _vp, _i64]),
    "decode_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "decode_plan_prefix": (ctypes.c_int, [_pp, ctypes.POINTER(PlanDesc), _vp, _vp, _vp]),
    "decode_plan_prefix_compute": (ctypes.c_int, [ctypes.POINTER(PlanDesc), _vp, _vp, _vp,
                                                  ctypes.POINTER(PlanInfo), _vp, _i64]),
    "decode_run_static": (ctypes.c_int, [ctypes.POINTER(PlanDesc), _vp, _vp, _vp, _vp, _vp,
                                         _vp, _vp, _vp]),
    "decode_run_static_status": (ctypes.c_int, [_vp]),
    "decode_cp_ranges": (ctypes.c_int, [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                        _vp, _vp, _vp]),
    "decode_plan_cp": (ctypes.c_int, [_pp, ctypes.POINTER(PlanDesc), _vp, ctypes.c_int,
                                      ctypes.c_int]),
    "decode_plan_cp_compute": (ctypes.c_int, [ctypes.POINTER(PlanDesc), _vp, ctypes.c_int,
                                              ctypes.c_int, ctypes.POINTER(PlanInfo), _vp, _i64]),
    "decode_merge_ranks": (ctypes.c_int, [ctypes.c_int, _i64, ctypes.c_int, _vp, _vp, _vp, _vp,
                                          _vp]),
    "decode_selftest_wait_timeout": (ctypes.c_int, [_vp, _i64, _vp]),
    "prefill_d64_run": (ctypes.c_int, [ctypes.POINTER(PrefillDesc), _vp, _vp, _vp, _vp, _vp, _vp,
                                       _vp]),
}

_lock = threading.Lock()
_lib = None


def lib() -> ctypes.CDLL:
    """Load libpkvd.so (built by paged_kv_cache_plan_gb300.build)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is missing: build it with "
                    "`python -m paged_kv_cache_plan_gb300.build` (there is no fallback path)")
            import torch  # noqa: F401  (loads the same CUDA runtime first)
            L = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _lib = L
    return _lib


def status_string(code: int) -> str:
    return lib().decode_status_string(int(code)).decode()


class PkvdError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {status_string(code)} ({code})")
        self.code = code


def check(code: int, what: str) -> None:
    if code != PKVD_OK:
        raise PkvdError(code, what)
