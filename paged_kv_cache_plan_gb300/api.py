"""Python surface of the C ABI: plan once, run many times.

    plan = decode_plan(batch, heads, kv_heads, head_dim, page_size, seq_lens, splits)
    decode_run(plan, q, k_pages, v_pages, page_table, out, lse)

Several query tokens per request (make_desc(..., q_len=n), n > 1): q, out and
lse carry a token axis, [B, n, Hq, ...], and token j sees the cache up to its
own position L - n + j. prefill_d64(q, k, v) runs the dense causal prefill at
head_dim 64. decode_plan_prefix plans MLA requests that share a prefix.

Tensors are torch CUDA tensors (PyTorch provides device memory and streams
only). Shapes, dtypes and alignment are checked here; the arithmetic runs in
the library's kernels.
"""
from __future__ import annotations

import ctypes
import math
from typing import Optional, Sequence

import torch

from . import _lib
from ._lib import PlanDesc, PlanInfo, WorkItem, check

_DTYPES = {torch.bfloat16: _lib.PKVD_BF16, torch.float16: _lib.PKVD_FP16,
           "bf16": _lib.PKVD_BF16, "fp16": _lib.PKVD_FP16}


def _seq_array(seq_lens) -> ctypes.Array:
    vals = [int(x) for x in (seq_lens.tolist() if hasattr(seq_lens, "tolist") else seq_lens)]
    return (ctypes.c_int32 * max(1, len(vals)))(*vals)


def make_desc(batch: int, heads: int, kv_heads: int, head_dim: int, page_size: int, *,
              head_dim_v: int = 0, dtype="bf16", splits: int = 0, grid_order: str = "auto",
              stage2_tiles: int = 0, variant: str = "auto", checks: bool = False,
              num_sms: int = 0, ctas_per_sm: int = 0, min_chunk: int = 0,
              max_pages_per_seq: int = 0, num_pool_pages: int = 0, k_row_pitch: int = 0,
              v_row_pitch: int = 0, scale: float = 0.0, q_len: int = 0) -> PlanDesc:
    d = PlanDesc()
    d.batch, d.heads, d.kv_heads, d.head_dim = batch, heads, kv_heads, head_dim
    d.head_dim_v, d.page_size, d.dtype = head_dim_v, page_size, _DTYPES[dtype]
    d.splits, d.grid_order = splits, _lib.GRID_ORDERS[grid_order]
    d.stage2_tiles, d.variant, d.checks = stage2_tiles, _lib.VARIANTS[variant], int(bool(checks))
    d.num_sms, d.ctas_per_sm, d.min_chunk = num_sms, ctas_per_sm, min_chunk
    d.max_pages_per_seq, d.num_pool_pages = max_pages_per_seq, num_pool_pages
    d.k_row_pitch, d.v_row_pitch, d.scale = k_row_pitch, v_row_pitch, scale
    d.q_len = q_len
    return d


class Plan:
    """Owns a pkvd_plan* (freed on close / garbage collection)."""

    def __init__(self, handle: ctypes.c_void_p, desc: PlanDesc):
        self._h = handle
        self.desc = desc
        info = PlanInfo()
        check(_lib.lib().decode_plan_query(self._h, ctypes.byref(info)), "decode_plan_query")
        self.info = info.as_dict()

    @property
    def handle(self) -> ctypes.c_void_p:
        if self._h is None:
            raise ValueError("plan was destroyed")
        return self._h

    def workspace_bytes(self) -> int:
        return int(_lib.lib().decode_workspace_bytes(self.handle))

    def last_device_status(self, stream: Optional[torch.cuda.Stream] = None) -> int:
        s = (stream or torch.cuda.current_stream()).cuda_stream
        return int(_lib.lib().decode_last_device_status(self.handle, ctypes.c_void_p(s)))

    def close(self) -> None:
        if self._h is not None:
            check(_lib.lib().decode_plan_destroy(self._h), "decode_plan_destroy")
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def decode_plan_ex(desc: PlanDesc, seq_lens: Sequence[int]) -> Plan:
    h = ctypes.c_void_p()
    check(_lib.lib().decode_plan_ex(ctypes.byref(h), ctypes.byref(desc),
                                    ctypes.cast(_seq_array(seq_lens), ctypes.c_void_p)),
          "decode_plan_ex")
    return Plan(h, desc)


def decode_plan(batch: int, heads: int, kv_heads: int, head_dim: int, page_size: int,
                seq_lens: Sequence[int], splits: int = 0, **kw) -> Plan:
    """Plan a decode op. Keyword arguments are the optional pkvd_plan_desc
    fields (dtype, head_dim_v, grid_order, stage2_tiles, variant, checks, ...)."""
    return decode_plan_ex(make_desc(batch, heads, kv_heads, head_dim, page_size,
                                    splits=splits, **kw), seq_lens)


def decode_plan_compute(desc: PlanDesc, seq_lens: Sequence[int], with_items: bool = True):
    """The split planner alone, on the host (no CUDA): (info dict, work items)."""
    L = _lib.lib()
    info = PlanInfo()
    seq = _seq_array(seq_lens)
    check(L.decode_plan_compute(ctypes.byref(desc), ctypes.cast(seq, ctypes.c_void_p),
                                ctypes.byref(info), None, 0), "decode_plan_compute")
    items = []
    if with_items and info.num_items > 0:
        arr = (WorkItem * info.num_items)()
        check(L.decode_plan_compute(ctypes.byref(desc), ctypes.cast(seq, ctypes.c_void_p),
                                    ctypes.byref(info), ctypes.cast(arr, ctypes.c_void_p),
                                    info.num_items), "decode_plan_compute")
        items = [(w.request, w.unit, w.split, w.partial_row, w.tok_begin, w.tok_end)
                 for w in arr]
    return info.as_dict(), items


def _i32_array(vals) -> ctypes.Array:
    vals = [int(x) for x in (vals.tolist() if hasattr(vals, "tolist") else vals)]
    return (ctypes.c_int32 * max(1, len(vals)))(*vals)


def decode_plan_prefix(desc: PlanDesc, seq_lens: Sequence[int], prefix_group: Sequence[int],
                       prefix_len: Sequence[int]) -> Plan:
    """Shared-prefix plan (MLA): consecutive requests with one prefix_group id
    >= 0 share their first prefix_len tokens (same pages)."""
    h = ctypes.c_void_p()
    arrs = [_seq_array(seq_lens), _i32_array(prefix_group), _i32_array(prefix_len)]
    check(_lib.lib().decode_plan_prefix(ctypes.byref(h), ctypes.byref(desc),
                                        *[ctypes.cast(x, ctypes.c_void_p) for x in arrs]),
          "decode_plan_prefix")
    return Plan(h, desc)


def decode_plan_prefix_compute(desc: PlanDesc, seq_lens: Sequence[int],
                               prefix_group: Sequence[int], prefix_len: Sequence[int]):
    """Host-only shared-prefix planning: (info dict, grouped prefix items,
    per-request items); items as (request, unit, split, partial_row,
    tok_begin, tok_end, grouped)."""
    L = _lib.lib()
    info = PlanInfo()
    arrs = [_seq_array(seq_lens), _i32_array(prefix_group), _i32_array(prefix_len)]
    ptrs = [ctypes.cast(x, ctypes.c_void_p) for x in arrs]
    check(L.decode_plan_prefix_compute(ctypes.byref(desc), *ptrs, ctypes.byref(info), None, 0),
          "decode_plan_prefix_compute")
    n = info.num_prefix_items + info.num_items
    arr = (WorkItem * max(1, n))()
    check(L.decode_plan_prefix_compute(ctypes.byref(desc), *ptrs, ctypes.byref(info),
                                       ctypes.cast(arr, ctypes.c_void_p), n),
          "decode_plan_prefix_compute")
    rows = [(w.request, w.unit, w.split, w.partial_row, w.tok_begin, w.tok_end, w.grouped)
            for w in arr[:n]]
    return info.as_dict(), rows[:info.num_prefix_items], rows[info.num_prefix_items:]


def cp_ranges(world: int, rank: int, seq_lens: Sequence[int], page_size: int):
    """Token range of every request on context-parallel rank `rank` of
    `world` (decode_cp_ranges): (begin list, length list)."""
    n = len(seq_lens)
    begin = (ctypes.c_int32 * max(1, n))()
    length = (ctypes.c_int32 * max(1, n))()
    check(_lib.lib().decode_cp_ranges(int(world), int(rank), n, int(page_size),
                                      ctypes.cast(_seq_array(seq_lens), ctypes.c_void_p),
                                      ctypes.cast(begin, ctypes.c_void_p),
                                      ctypes.cast(length, ctypes.c_void_p)), "decode_cp_ranges")
    return list(begin[:n]), list(length[:n])


def decode_plan_cp(desc: PlanDesc, seq_lens: Sequence[int], world: int, rank: int) -> Plan:
    """Plan of rank `rank`'s token ranges of a context-parallel decode."""
    h = ctypes.c_void_p()
    check(_lib.lib().decode_plan_cp(ctypes.byref(h), ctypes.byref(desc),
                                    ctypes.cast(_seq_array(seq_lens), ctypes.c_void_p),
                                    int(world), int(rank)), "decode_plan_cp")
    return Plan(h, desc)


def decode_plan_cp_compute(desc: PlanDesc, seq_lens: Sequence[int], world: int, rank: int):
    """Host-only planning of a rank's plan: (info dict, items as (request,
    unit, split, partial_row, tok_begin, tok_end))."""
    L = _lib.lib()
    info = PlanInfo()
    seq = _seq_array(seq_lens)
    check(L.decode_plan_cp_compute(ctypes.byref(desc), ctypes.cast(seq, ctypes.c_void_p),
                                   int(world), int(rank), ctypes.byref(info), None, 0),
          "decode_plan_cp_compute")
    items = []
    if info.num_items > 0:
        arr = (WorkItem * info.num_items)()
        check(L.decode_plan_cp_compute(ctypes.byref(desc), ctypes.cast(seq, ctypes.c_void_p),
                                       int(world), int(rank), ctypes.byref(info),
                                       ctypes.cast(arr, ctypes.c_void_p), info.num_items),
              "decode_plan_cp_compute")
        items = [(w.request, w.unit, w.split, w.partial_row, w.tok_begin, w.tok_end)
                 for w in arr]
    return info.as_dict(), items


def decode_merge_ranks(o_parts: torch.Tensor, lse_parts: torch.Tensor, out: torch.Tensor,
                       lse: torch.Tensor, stream=None) -> None:
    """Merge the ranks' rows (decode_merge_ranks): o_parts [R, ..., Dv] and
    lse_parts [R, ...] fp32 CUDA tensors, out [..., Dv] and lse [...]."""
    R = o_parts.shape[0]
    dv = o_parts.shape[-1]
    rows = lse_parts[0].numel()
    for name, t in (("o_parts", o_parts), ("lse_parts", lse_parts), ("out", out), ("lse", lse)):
        if t.device.type != "cuda" or t.dtype != torch.float32 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous fp32 CUDA tensor")
    if (lse_parts.shape[0] != R or o_parts.numel() != R * rows * dv or out.numel() != rows * dv
            or lse.numel() != rows):
        raise ValueError("o_parts [R, rows, Dv], lse_parts [R, rows], out [rows, Dv], lse [rows]")
    s = (stream or torch.cuda.current_stream()).cuda_stream
    check(_lib.lib().decode_merge_ranks(int(R), int(rows), int(dv), _ptr(o_parts), _ptr(lse_parts),
                                        _ptr(out), _ptr(lse), ctypes.c_void_p(s)),
          "decode_merge_ranks")


def gather_ranks(o_r: torch.Tensor, lse_r: torch.Tensor, group=None):
    """All-gather every rank's rows (torch.distributed, the process group's
    backend: NCCL on GPUs, gloo on the CPU): returns o_parts [R, *o_r.shape],
    lse_parts [R, *lse_r.shape] in rank order."""
    import torch.distributed as dist
    R = dist.get_world_size(group)
    # concatenated along the first dimension (the form every backend takes)
    o_parts = torch.empty((R * o_r.shape[0], *o_r.shape[1:]), dtype=o_r.dtype, device=o_r.device)
    l_parts = torch.empty((R * lse_r.shape[0], *lse_r.shape[1:]), dtype=lse_r.dtype,
                          device=lse_r.device)
    dist.all_gather_into_tensor(o_parts, o_r.contiguous(), group=group)
    dist.all_gather_into_tensor(l_parts, lse_r.contiguous(), group=group)
    return o_parts.view(R, *o_r.shape), l_parts.view(R, *lse_r.shape)


def cp_decode(plan: Plan, q, k_pages, v_pages, page_table, out, lse, group=None,
              stream=None) -> None:
    """Context-parallel decode step on this rank: its range (decode_run of a
    decode_plan_cp plan), the all-gather of every rank's rows, the merge
    (decode_merge_ranks) into out / lse, identical on every rank."""
    o_r = torch.empty_like(out)
    l_r = torch.empty_like(lse)
    decode_run(plan, q, k_pages, v_pages, page_table, o_r, l_r, stream)
    o_parts, l_parts = gather_ranks(o_r, l_r, group)
    decode_merge_ranks(o_parts, l_parts, out, lse, stream)


def _ptr(t: Optional[torch.Tensor]) -> Optional[ctypes.c_void_p]:
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _check_tensors(plan: Plan, q, k_pages, v_pages, page_table, out, lse) -> None:
    d = plan.desc
    dt = {_lib.PKVD_BF16: torch.bfloat16, _lib.PKVD_FP16: torch.float16}[d.dtype]
    dv = d.head_dim_v or (512 if d.head_dim == 576 else d.head_dim)
    for name, t, dtype in (("q", q, dt), ("k_pages", k_pages, dt), ("v_pages", v_pages, dt),
                           ("page_table", page_table, torch.int32), ("out", out, torch.float32),
                           ("lse", lse, torch.float32)):
        if not isinstance(t, torch.Tensor):
            raise TypeError(f"{name} must be a torch tensor")
        if t.device.type != "cuda":
            raise ValueError(f"{name} must be a CUDA tensor")
        if t.dtype != dtype:
            raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    # one query token: [B, Hq, ...]; q_len > 1: [B, q_len, Hq, ...]
    tok = () if d.q_len <= 1 else (d.q_len,)
    for name, t, want in (("q", q, (d.batch, *tok, d.heads, d.head_dim)),
                          ("out", out, (d.batch, *tok, d.heads, dv)),
                          ("lse", lse, (d.batch, *tok, d.heads))):
        if tuple(t.shape) != want:
            raise ValueError(f"{name} shape {tuple(t.shape)} != {want}")
    if page_table.dim() != 2 or page_table.shape[0] != d.batch:
        raise ValueError("page_table must be [batch, max_pages_per_seq]")


def decode_run(plan: Plan, q: torch.Tensor, k_pages: torch.Tensor, v_pages: torch.Tensor,
               page_table: torch.Tensor, out: torch.Tensor, lse: torch.Tensor,
               stream: Optional[torch.cuda.Stream] = None) -> None:
    """Enqueue stage 1 and the merge on ``stream`` (default: current stream)."""
    _check_tensors(plan, q, k_pages, v_pages, page_table, out, lse)
    if plan.desc.max_pages_per_seq and page_table.shape[1] != plan.desc.max_pages_per_seq:
        raise ValueError("page_table row length differs from the plan's max_pages_per_seq")
    s = (stream or torch.cuda.current_stream()).cuda_stream
    check(_lib.lib().decode_run(plan.handle, _ptr(q), _ptr(k_pages), _ptr(v_pages),
                                _ptr(page_table), _ptr(out), _ptr(lse), ctypes.c_void_p(s)),
          "decode_run")


def decode_run_timed(plan: Plan, q, k_pages, v_pages, page_table, out, lse, ev_begin=None,
                     ev_mid=None, ev_end=None, stream: Optional[torch.cuda.Stream] = None) -> None:
    """decode_run that records torch.cuda.Events around and between the stages."""
    _check_tensors(plan, q, k_pages, v_pages, page_table, out, lse)
    s = (stream or torch.cuda.current_stream()).cuda_stream
    for e in (ev_begin, ev_mid, ev_end):
        if e is not None and not e.cuda_event:
            e.record(stream or torch.cuda.current_stream())   # create the CUDA event
    ev = [ctypes.c_void_p(e.cuda_event) if e is not None else None
          for e in (ev_begin, ev_mid, ev_end)]
    check(_lib.lib().decode_run_timed(plan.handle, _ptr(q), _ptr(k_pages), _ptr(v_pages),
                                      _ptr(page_table), _ptr(out), _ptr(lse),
                                      ctypes.c_void_p(s), *ev), "decode_run_timed")


def selftest_wait_timeout(limit_us: int = 2000, stream=None):
    """Run the bounded-wait self-test (decode_selftest_wait_timeout): a wait
    that nothing completes must give up after limit_us. Returns (status,
    microseconds waited)."""
    st = torch.zeros(2, dtype=torch.int32, device="cuda")
    s = (stream or torch.cuda.current_stream()).cuda_stream
    check(_lib.lib().decode_selftest_wait_timeout(_ptr(st), int(limit_us), ctypes.c_void_p(s)),
          "decode_selftest_wait_timeout")
    torch.cuda.synchronize()
    v = st.cpu().tolist()
    return int(v[0]), int(v[1])


def prefill_d64(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, *, scale: float = 0.0,
                out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                status: Optional[torch.Tensor] = None, stream=None):
    """Dense causal prefill attention at head_dim 64 (prefill_d64_run):
    q [B, L, Hq, 64], k / v [B, Hkv, L, 64] (bf16 or fp16, contiguous, on the
    GPU). Returns (out [B, L, Hq, 64] fp32, lse [B, L, Hq] fp32, status), with
    status a device int32 that is nonzero if a pipeline wait ran out.
    Asynchronous on ``stream``."""
    if q.dim() != 4 or k.dim() != 4 or v.shape != k.shape:
        raise ValueError("q must be [B, L, Hq, 64] and k, v [B, Hkv, L, 64]")
    B, L, H, D = q.shape
    Hkv = k.shape[1]
    if D != 64 or tuple(k.shape) != (B, Hkv, L, 64):
        raise ValueError(f"shapes q {tuple(q.shape)}, k {tuple(k.shape)} do not match")
    for name, t in (("q", q), ("k", k), ("v", v)):
        if t.device.type != "cuda" or not t.is_contiguous() or t.dtype != q.dtype:
            raise ValueError(f"{name} must be a contiguous CUDA tensor of q's dtype")
    if q.dtype not in (torch.bfloat16, torch.float16):
        raise TypeError("bf16 or fp16 inputs")
    dev = q.device
    if out is None:
        out = torch.empty((B, L, H, 64), dtype=torch.float32, device=dev)
    if lse is None:
        lse = torch.empty((B, L, H), dtype=torch.float32, device=dev)
    if status is None:
        status = torch.zeros(1, dtype=torch.int32, device=dev)
    if tuple(out.shape) != (B, L, H, 64) or tuple(lse.shape) != (B, L, H):
        raise ValueError("out must be [B, L, Hq, 64] and lse [B, L, Hq]")
    d = _lib.PrefillDesc()
    d.batch, d.heads, d.kv_heads, d.seq_len = B, H, Hkv, L
    d.dtype = _lib.PKVD_FP16 if q.dtype == torch.float16 else _lib.PKVD_BF16
    d.scale = scale
    s = (stream or torch.cuda.current_stream()).cuda_stream
    check(_lib.lib().prefill_d64_run(ctypes.byref(d), _ptr(q), _ptr(k), _ptr(v), _ptr(out),
                                     _ptr(lse), _ptr(status), ctypes.c_void_p(s)),
          "prefill_d64_run")
    return out, lse, status


def plan_for_case(case, *, shared_prefix: bool = False, **kw) -> Plan:
    """Plan matching a workloads.DecodeCase (splits from the case unless
    given). shared_prefix: use the case's prefix groups (decode_plan_prefix)."""
    kw.setdefault("splits", 0 if shared_prefix else case.splits)
    if case.q_len != 1:
        kw.setdefault("q_len", case.q_len)
    desc = make_desc(case.batch, case.heads, case.kv_heads, case.head_dim, case.page_size,
                     head_dim_v=case.head_dim_v, dtype=case.dtype,
                     max_pages_per_seq=case.max_pages, num_pool_pages=case.pool_pages,
                     k_row_pitch=case.k_row_pitch, v_row_pitch=case.v_row_pitch,
                     scale=case.scale, **kw)
    if shared_prefix:
        return decode_plan_prefix(desc, case.seq_lens.tolist(), case.meta["prefix_group"],
                                  case.meta["prefix_len"])
    return decode_plan_ex(desc, case.seq_lens.tolist())


def run_case(plan: Plan, case_dev, out: Optional[torch.Tensor] = None,
             lse: Optional[torch.Tensor] = None, stream=None):
    """Run a plan on a DecodeCase whose tensors are on the GPU; returns (out, lse)."""
    dev = case_dev.q.device
    tok = () if case_dev.q_len == 1 else (case_dev.q_len,)
    if out is None:
        out = torch.empty((case_dev.batch, *tok, case_dev.heads, case_dev.head_dim_v),
                          dtype=torch.float32, device=dev)
    if lse is None:
        lse = torch.empty((case_dev.batch, *tok, case_dev.heads), dtype=torch.float32,
                          device=dev)
    decode_run(plan, case_dev.q, case_dev.k_pages, case_dev.v_pages, case_dev.page_table,
               out, lse, stream)
    return out, lse


LN2 = math.log(2.0)
