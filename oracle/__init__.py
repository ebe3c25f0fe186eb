"""Plain fp64 CPU oracle for paged-KV split-KV decode attention.

TEST INFRASTRUCTURE ONLY. The tests, the package's smoke check and the
benchmark's CPU-baseline leg are the only callers. The CUDA library never
imports, links or runs anything here, and this module imports nothing from
the CUDA side: the two meet only in the tests, on inputs made by the seeded
workload generator.

The arithmetic lives in ``oracle.c`` (see its header for the definition it
writes out and the passages it follows). This module compiles it with gcc
(no FMA contraction, so x86 and Arm give the same bits) and wraps its entry
points for numpy / torch CPU arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")

BF16, FP16 = 0, 1

# Planted mistakes for the test-of-tests (mirror of the MUT_* codes in oracle.c).
MUTATIONS = {
    "no_scale": 1,
    "head_map_mod": 2,
    "slot_off_by_one": 3,
    "lse_log2": 4,
    "v_from_k": 5,
    "no_max_shift": 6,
    "divide_by_L": 7,
    "pages_reversed": 8,
    "merge_no_norm": 9,
    "drop_last_key": 10,
    "no_causal": 11,
}


class Problem(ctypes.Structure):
    _fields_ = [
        ("batch", ctypes.c_int32),
        ("heads", ctypes.c_int32),
        ("kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("head_dim_v", ctypes.c_int32),
        ("page_size", ctypes.c_int32),
        ("dtype", ctypes.c_int32),
        ("mutation", ctypes.c_int32),
        ("max_pages", ctypes.c_int64),
        ("k_row_pitch", ctypes.c_int64),
        ("v_row_pitch", ctypes.c_int64),
        ("scale", ctypes.c_double),
        ("q_len", ctypes.c_int32),
    ]


_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into _build/liboracle.so (skipped when up to date)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", "-o", tmp, _SRC, "-lm", "-lpthread"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            path = build()
            L = ctypes.CDLL(path)
            P = ctypes.POINTER(Problem)
            vp = ctypes.c_void_p
            i32, i64 = ctypes.c_int32, ctypes.c_int64
            L.orc_decode.argtypes = [P, vp, vp, vp, vp, vp, vp, vp]
            L.orc_decode_pairs.argtypes = [P, vp, vp, vp, vp, vp, vp, i64, vp, vp]
            L.orc_decode_threads.argtypes = [P, vp, vp, vp, vp, vp, i32, vp, vp]
            L.orc_partial.argtypes = [P, vp, vp, vp, vp, vp, i32, i32, i64, i64, vp, vp]
            L.orc_merge.argtypes = [i32, i32, vp, vp, i32, vp, vp]
            L.orc_to_double.argtypes = [vp, i64, i32, vp]
            for f in ("orc_decode", "orc_decode_pairs", "orc_decode_threads",
                      "orc_partial", "orc_merge"):
                getattr(L, f).restype = ctypes.c_int
            L.orc_to_double.restype = None
            _lib = L
    return _lib


def _ptr(a):
    """Data pointer of a contiguous CPU torch tensor or numpy array."""
    if a is None:
        return None
    if hasattr(a, "data_ptr"):
        if a.device.type != "cpu" or not a.is_contiguous():
            raise ValueError("oracle inputs must be contiguous CPU tensors")
        return ctypes.c_void_p(a.data_ptr())
    if not a.flags["C_CONTIGUOUS"]:
        raise ValueError("oracle inputs must be C-contiguous")
    return ctypes.c_void_p(a.ctypes.data)


def _i32(a):
    if hasattr(a, "data_ptr"):
        import torch
        return a.to(torch.int32).contiguous()
    return np.ascontiguousarray(a, dtype=np.int32)


def problem(*, batch, heads, kv_heads, head_dim, head_dim_v, page_size, dtype,
            max_pages, k_row_pitch, v_row_pitch, scale, mutation=0, q_len=1) -> Problem:
    return Problem(int(batch), int(heads), int(kv_heads), int(head_dim),
                   int(head_dim_v), int(page_size),
                   FP16 if dtype in ("fp16", FP16) else BF16, int(mutation),
                   int(max_pages), int(k_row_pitch), int(v_row_pitch),
                   float(scale), int(q_len))


def _check(rc, what):
    if rc != 0:
        raise RuntimeError(f"oracle {what} failed with code {rc}")


def decode(P: Problem, q, k_pages, v_pages, page_table, seq_lens, *,
           pairs=None, threads: int = 0):
    """fp64 out and lse. With ``pairs`` ([n, 2] of (b, v), v = token * Hq +
    head) only those are computed and the results come back as out [n, Dv],
    lse [n]; otherwise out [B, q_len * Hq, Dv], lse [B, q_len * Hq] (q_len =
    1: [B, Hq, ...]). ``threads`` > 0 spreads the full decode over that many
    host threads (same arithmetic per head)."""
    L = lib()
    pt, sl = _i32(page_table), _i32(seq_lens)
    if pairs is not None:
        pr = np.ascontiguousarray(np.asarray(pairs, dtype=np.int32).reshape(-1, 2))
        n = pr.shape[0]
        out = np.zeros((n, P.head_dim_v), dtype=np.float64)
        lse = np.zeros((n,), dtype=np.float64)
        _check(L.orc_decode_pairs(ctypes.byref(P), _ptr(q), _ptr(k_pages),
                                  _ptr(v_pages), _ptr(pt), _ptr(sl), _ptr(pr),
                                  n, _ptr(out), _ptr(lse)), "decode_pairs")
        return out, lse
    vh = max(P.q_len, 1) * P.heads
    out = np.zeros((P.batch, vh, P.head_dim_v), dtype=np.float64)
    lse = np.zeros((P.batch, vh), dtype=np.float64)
    if threads and threads > 0:
        _check(L.orc_decode_threads(ctypes.byref(P), _ptr(q), _ptr(k_pages),
                                    _ptr(v_pages), _ptr(pt), _ptr(sl),
                                    int(threads), _ptr(out), _ptr(lse)),
               "decode_threads")
    else:
        _check(L.orc_decode(ctypes.byref(P), _ptr(q), _ptr(k_pages),
                            _ptr(v_pages), _ptr(pt), _ptr(sl), _ptr(out),
                            _ptr(lse)), "decode")
    return out, lse


def partial(P: Problem, q, k_pages, v_pages, page_table, seq_lens, b, h, t0, t1):
    """Normalised partial output and lse of (b, v) over the tokens of
    [t0, t1) that query token v // Hq may see."""
    L = lib()
    pt, sl = _i32(page_table), _i32(seq_lens)
    o = np.zeros((P.head_dim_v,), dtype=np.float64)
    lse = np.zeros((1,), dtype=np.float64)
    _check(L.orc_partial(ctypes.byref(P), _ptr(q), _ptr(k_pages), _ptr(v_pages),
                         _ptr(pt), _ptr(sl), int(b), int(h), int(t0), int(t1),
                         _ptr(o), _ptr(lse)), "partial")
    return o, float(lse[0])


def merge(o_parts, lse_parts, mutation: int = 0):
    """Merge normalised partials [S, Dv] with their lse [S]."""
    L = lib()
    o_parts = np.ascontiguousarray(o_parts, dtype=np.float64)
    lse_parts = np.ascontiguousarray(lse_parts, dtype=np.float64)
    S, dv = o_parts.shape
    out = np.zeros((dv,), dtype=np.float64)
    lse = np.zeros((1,), dtype=np.float64)
    _check(L.orc_merge(int(S), int(dv), _ptr(o_parts), _ptr(lse_parts),
                       int(mutation), _ptr(out), _ptr(lse)), "merge")
    return out, float(lse[0])


def to_double(bits_u16, dtype) -> np.ndarray:
    """Exact widening of stored 16-bit elements (uint16 bit patterns)."""
    L = lib()
    src = np.ascontiguousarray(bits_u16, dtype=np.uint16)
    dst = np.zeros(src.shape, dtype=np.float64)
    L.orc_to_double(_ptr(src), int(src.size),
                    FP16 if dtype in ("fp16", FP16) else BF16, _ptr(dst))
    return dst
