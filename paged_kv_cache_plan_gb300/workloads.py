"""Seeded synthetic decode workloads.

This module only draws inputs: values, page tables and sequence lengths. It
holds none of the attention arithmetic, so both the CUDA path and the CPU
oracle can take its tensors without sharing any of the method.

Recipe (the same for every workload):
  * q, K and V values are i.i.d. N(0, 1) in fp32 from a seeded CPU
    ``torch.Generator``, rounded to bf16 or fp16 (round to nearest even);
  * physical pages come from a seeded ``torch.randperm`` of the pool, handed
    out to the requests in order, so the page table is a random scatter;
  * page-table entries past a request's last page are 0 (a valid page: no
    kernel may read them, and a wrong read still stays in bounds);
  * MLA rows are one 576-wide latent row per token (512 no-rope + 64 rope);
    V is the first 512 elements of the same row, page size 1.

Layouts (all contiguous):
  q          [B, Hq, D]; with q_len > 1 query tokens per request
             [B, q_len, Hq, D] (the request's last q_len positions)
  k_pages    [P, Hkv, ps, k_row_pitch]      (MLA: [P, 1, 1, 576])
  v_pages    [P, Hkv, ps, v_row_pitch]      (MLA: the same tensor as k_pages)
  page_table [B, max_pages] int32
  seq_lens   [B] int32
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import List, Optional, Sequence

import torch

_DT = {"bf16": torch.bfloat16, "fp16": torch.float16}


@dataclass
class DecodeCase:
    name: str
    q: torch.Tensor
    k_pages: torch.Tensor
    v_pages: torch.Tensor
    page_table: torch.Tensor
    seq_lens: torch.Tensor
    heads: int
    kv_heads: int
    head_dim: int
    head_dim_v: int
    page_size: int
    k_row_pitch: int
    v_row_pitch: int
    scale: float
    dtype: str
    mla: bool = False
    splits: int = 0
    unique_rows: int = 0          # distinct KV rows the batch reads (per KV head)
    meta: dict = field(default_factory=dict)
    q_len: int = 1                # query tokens per request (last positions)

    @property
    def batch(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def pool_pages(self) -> int:
        return int(self.k_pages.shape[0])

    @property
    def max_pages(self) -> int:
        return int(self.page_table.shape[1])

    def kv_bytes_unique(self) -> int:
        """Compulsory KV bytes of one decode op: every distinct K and V row
        read once (MLA: one 1,152-byte latent row per distinct token)."""
        el = 2
        if self.mla:
            return self.unique_rows * self.k_row_pitch * el
        return self.unique_rows * self.kv_heads * (self.head_dim + self.head_dim_v) * el

    def kv_bytes_logical(self) -> int:
        """KV bytes summed over requests, shared prefixes counted per request."""
        el = 2
        toks = int(self.seq_lens.to(torch.int64).sum())
        if self.mla:
            return toks * self.k_row_pitch * el
        return toks * self.kv_heads * (self.head_dim + self.head_dim_v) * el

    def to(self, device) -> "DecodeCase":
        """Copy of the case with every tensor on ``device`` (aliasing kept)."""
        k = self.k_pages.to(device)
        v = k if self.v_pages.data_ptr() == self.k_pages.data_ptr() else self.v_pages.to(device)
        return DecodeCase(self.name, self.q.to(device), k, v, self.page_table.to(device),
                          self.seq_lens.to(device), self.heads, self.kv_heads,
                          self.head_dim, self.head_dim_v, self.page_size,
                          self.k_row_pitch, self.v_row_pitch, self.scale, self.dtype,
                          self.mla, self.splits, self.unique_rows, dict(self.meta), self.q_len)


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator()
    g.manual_seed(int(seed))
    return g


def _randn(shape, g: torch.Generator, dtype: str, chunk_rows: int = 1 << 16) -> torch.Tensor:
    """N(0,1) fp32 rounded to ``dtype``, on g's device; drawn in row chunks to
    bound memory."""
    shape = tuple(int(s) for s in shape)
    out = torch.empty(shape, dtype=_DT[dtype], device=g.device)
    flat = out.view(shape[0], -1)
    for r0 in range(0, shape[0], chunk_rows):
        r1 = min(shape[0], r0 + chunk_rows)
        flat[r0:r1] = torch.randn((r1 - r0, flat.shape[1]), generator=g,
                                  dtype=torch.float32, device=g.device).to(_DT[dtype])
    return out


def _value_gen(seed: int, g: torch.Generator, device: str) -> torch.Generator:
    """Generator of the values: the structure generator itself on the CPU;
    on another device a generator there, seeded from the same seed (same
    distribution and structure, other draws: for timing only)."""
    if str(device) == "cpu":
        return g
    gd = torch.Generator(device=device)
    gd.manual_seed(int(seed) + 0x5EED)
    return gd


def gqa_case(*, batch: int = 1, heads: int, kv_heads: int, head_dim: int,
             page_size: int, seq_lens: Sequence[int], pool_pages: Optional[int] = None,
             dtype: str = "bf16", seed: int = 0, splits: int = 0,
             scale: Optional[float] = None, name: str = "gqa",
             q_len: int = 1, device: str = "cpu") -> DecodeCase:
    """GQA decode: Hq query heads over Hkv KV heads (consecutive groups),
    HND pages [P, Hkv, ps, D], a seeded random page scatter; q_len query
    tokens per request. device != "cpu" draws the values there (timing only)."""
    lens = [int(x) for x in seq_lens]
    assert len(lens) == batch
    g = _gen(seed)
    npages = [(L + page_size - 1) // page_size for L in lens]
    need = sum(npages)
    P = need if pool_pages is None else int(pool_pages)
    assert P >= need, "pool too small for the requested contexts"
    gv = _value_gen(seed, g, device)
    q = _randn((batch, heads, head_dim) if q_len == 1 else (batch, q_len, heads, head_dim),
               gv, dtype)
    k = _randn((max(P, 1), kv_heads, page_size, head_dim), gv, dtype)
    v = _randn((max(P, 1), kv_heads, page_size, head_dim), gv, dtype)
    perm = torch.randperm(max(P, 1), generator=g).to(torch.int32)
    maxp = max(1, max(npages) if npages else 1)
    pt = torch.zeros((batch, maxp), dtype=torch.int32)
    nxt = 0
    for b, n in enumerate(npages):
        pt[b, :n] = perm[nxt:nxt + n]
        nxt += n
    return DecodeCase(name, q, k, v, pt.to(q.device),
                      torch.tensor(lens, dtype=torch.int32, device=q.device), heads,
                      kv_heads, head_dim, head_dim, page_size, head_dim, head_dim,
                      float(scale if scale is not None else 1.0 / math.sqrt(head_dim)),
                      dtype, False, splits, unique_rows=sum(lens), q_len=q_len)


def mla_case(*, batch: int, heads: int, seq_len: int, prefix_len: int = 0,
             group: int = 8, pool_rows: Optional[int] = None, dtype: str = "bf16",
             seed: int = 0, splits: int = 0, scale: Optional[float] = None,
             name: str = "mla", q_len: int = 1, device: str = "cpu") -> DecodeCase:
    """MLA decode: one 576-wide latent row (512 + 64) per token shared by all
    heads, page size 1. Requests in consecutive groups of ``group`` share the
    physical rows of their first ``prefix_len`` tokens; the rest are private.
    Rows are scattered over the pool by a seeded permutation; only the rows a
    request reads are drawn (the rest of the pool stays zero). device !=
    "cpu" draws the values there (timing only)."""
    D, DV = 576, 512
    g = _gen(seed)
    ngroups = (batch + group - 1) // group if prefix_len > 0 else 0
    unique = ngroups * prefix_len + batch * (seq_len - prefix_len)
    R = unique if pool_rows is None else int(pool_rows)
    assert R >= unique, "pool too small"
    gv = _value_gen(seed, g, device)
    q = _randn((batch, heads, D) if q_len == 1 else (batch, q_len, heads, D), gv, dtype)
    perm = torch.randperm(R, generator=g).to(torch.int64)
    pt = torch.empty((batch, seq_len), dtype=torch.int64)
    nxt = 0
    for gi in range(ngroups):
        rows = perm[nxt:nxt + prefix_len]
        nxt += prefix_len
        for b in range(gi * group, min(batch, (gi + 1) * group)):
            pt[b, :prefix_len] = rows
    for b in range(batch):
        n = seq_len - prefix_len
        pt[b, prefix_len:] = perm[nxt:nxt + n]
        nxt += n
    used = perm[:nxt].to(q.device)
    pool = torch.zeros((R, 1, 1, D), dtype=_DT[dtype], device=q.device)
    vals = _randn((nxt, D), gv, dtype)
    pool.view(R, D).index_copy_(0, used, vals)
    del vals
    # shared-prefix description for decode_plan_prefix: consecutive groups
    meta = {"prefix_group": [b // group if prefix_len > 0 else -1 for b in range(batch)],
            "prefix_len": [prefix_len if prefix_len > 0 else 0] * batch}
    return DecodeCase(name, q, pool, pool, pt.to(torch.int32).to(q.device),
                      torch.full((batch,), seq_len, dtype=torch.int32, device=q.device),
                      heads, 1, D, DV,
                      1, D, D, float(scale if scale is not None else 1.0 / math.sqrt(D)),
                      dtype, True, splits, unique_rows=unique, meta=meta, q_len=q_len)


# ---------------------------------------------------------------------------
# The named workloads. Seeds are 1000 + workload number (+ a sub-sweep term).

GQA_LONG_CONTEXTS = (2048, 8192, 16384, 32768, 65536)
MLA16_BATCHES = (1, 8, 24, 48)
MLA16_CONTEXT, MLA16_PREFIX, MLA16_POOL_ROWS = 68_000, 63_240, 2_000_000
MLA_MANY = ((64, 64), (64, 128), (128, 64), (128, 128))  # (heads, batch)
MLA_MANY_CONTEXT = 16_384
VARLEN_LENS = (256, 512, 768, 1024, 1536, 2048, 8192, 32768, 65536, 131072)
VARLEN_POOL_PAGES = 300_000 // 16  # a pool sized for 300K tokens


def _qsuffix(q_len: int) -> str:
    return "" if q_len == 1 else f"_q{q_len}"


def gqa_tiny(seed: int = 1001, q_len: int = 1, device: str = "cpu") -> DecodeCase:
    """Batch 1, 4 query heads on 1 KV head, d 128, 512 tokens, page 16,
    32 pages shuffled in a pool of 32, 4 KV splits."""
    return gqa_case(batch=1, heads=4, kv_heads=1, head_dim=128, page_size=16,
                    seq_lens=[512], pool_pages=32, seed=seed, splits=4,
                    name="gqa_tiny_b1_h4kv1_d128_L512" + _qsuffix(q_len), q_len=q_len,
                    device=device)


def gqa_long(context: int, seed: Optional[int] = None, q_len: int = 1,
             device: str = "cpu") -> DecodeCase:
    """Batch 1, 16 query heads over 2 KV heads (group 8), d 256, page 16,
    pool = context/16 pages in random order."""
    return gqa_case(batch=1, heads=16, kv_heads=2, head_dim=256, page_size=16,
                    seq_lens=[context], seed=1002 + context if seed is None else seed,
                    name=f"gqa_long_b1_h16kv2_d256_L{context}" + _qsuffix(q_len), q_len=q_len,
                    device=device)


def mla16(batch: int, seed: Optional[int] = None, context: int = MLA16_CONTEXT,
          prefix: int = MLA16_PREFIX, pool_rows: int = MLA16_POOL_ROWS,
          splits: Optional[int] = None, q_len: int = 1, device: str = "cpu") -> DecodeCase:
    """16 heads on one 576-wide latent row, page 1, 68,000-token contexts whose
    first 63,240 tokens are shared by groups of 8, a 2,000,000-row pool
    (over 2 GiB, so 64-bit offsets). The split count is the planner's own
    choice unless `splits` forces one (the aiter page's kernel used
    256 // batch, `splits=max(1, 256 // batch)` reproduces that)."""
    return mla_case(batch=batch, heads=16, seq_len=context, prefix_len=prefix,
                    group=8, pool_rows=pool_rows,
                    seed=1003 + batch if seed is None else seed,
                    splits=0 if splits is None else splits,
                    name=f"mla16_b{batch}_L{context}_prefix{prefix}" + _qsuffix(q_len),
                    q_len=q_len, device=device)


def mla_many(heads: int, batch: int, seed: Optional[int] = None,
             context: int = MLA_MANY_CONTEXT, q_len: int = 1,
             device: str = "cpu") -> DecodeCase:
    """nhead 64/128 on the 576-wide latent row, page 1, 16,384 distinct
    tokens per request."""
    return mla_case(batch=batch, heads=heads, seq_len=context, prefix_len=0,
                    seed=1004 + heads + batch if seed is None else seed,
                    name=f"mla_h{heads}_b{batch}_L{context}" + _qsuffix(q_len), q_len=q_len,
                    device=device)


def gqa_varlen(dtype: str = "bf16", seed: Optional[int] = None,
               lens: Sequence[int] = VARLEN_LENS,
               pool_pages: Optional[int] = VARLEN_POOL_PAGES, q_len: int = 1,
               device: str = "cpu") -> DecodeCase:
    """Batch 10, 32 query heads over 8 KV heads, d 128, page 16, the varlen
    context mix, pages scattered over a 300K-token pool."""
    return gqa_case(batch=len(lens), heads=32, kv_heads=8, head_dim=128,
                    page_size=16, seq_lens=list(lens), pool_pages=pool_pages,
                    dtype=dtype, seed=(1005 if dtype == "bf16" else 1105) if seed is None else seed,
                    name=f"gqa_varlen_{dtype}_b{len(lens)}_h32kv8_d128" + _qsuffix(q_len),
                    q_len=q_len, device=device)


def prefill_case(*, batch: int, heads: int, kv_heads: int, seq_len: int, dtype: str = "bf16",
                 seed: int = 0, name: Optional[str] = None) -> DecodeCase:
    """Dense causal prefill at head_dim 64, as a case of the decode problem
    with every token a query: q [B, L, Hq, 64] (q_len = L), K and V
    [B, Hkv, L, 64] = one page of L tokens per request (page b of request b)."""
    g = _gen(seed)
    L = int(seq_len)
    q = _randn((batch, L, heads, 64), g, dtype)
    k = _randn((batch, kv_heads, L, 64), g, dtype)
    v = _randn((batch, kv_heads, L, 64), g, dtype)
    pt = torch.arange(batch, dtype=torch.int32).view(batch, 1)
    return DecodeCase(name or f"prefill_d64_b{batch}_h{heads}kv{kv_heads}_L{L}", q, k, v, pt,
                      torch.full((batch,), L, dtype=torch.int32), heads, kv_heads, 64, 64, L,
                      64, 64, 0.125, dtype, False, 0, unique_rows=batch * L, q_len=L)


def permute_pages(case: DecodeCase, seed: int) -> DecodeCase:
    """The same logical problem with every physical page relabelled: pages move
    to new pool slots and the page table follows them."""
    g = _gen(seed)
    P = case.pool_pages
    perm = torch.randperm(P, generator=g)          # new slot of old page p = perm[p]
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(P)
    k = case.k_pages[inv].contiguous()             # new[perm[p]] = old[p]
    v = k if case.v_pages.data_ptr() == case.k_pages.data_ptr() else case.v_pages[inv].contiguous()
    pt = perm.to(torch.int32)[case.page_table.to(torch.int64)]
    return DecodeCase(case.name + f"_perm{seed}", case.q, k, v, pt.to(torch.int32),
                      case.seq_lens, case.heads, case.kv_heads, case.head_dim,
                      case.head_dim_v, case.page_size, case.k_row_pitch, case.v_row_pitch,
                      case.scale, case.dtype, case.mla, case.splits, case.unique_rows,
                      dict(case.meta), case.q_len)


def oracle_problem_kwargs(case: DecodeCase) -> dict:
    """Shape fields in the form the oracle's ``problem()`` takes."""
    return dict(batch=case.batch, heads=case.heads, kv_heads=case.kv_heads,
                head_dim=case.head_dim, head_dim_v=case.head_dim_v,
                page_size=case.page_size, dtype=case.dtype, max_pages=case.max_pages,
                k_row_pitch=case.k_row_pitch, v_row_pitch=case.v_row_pitch,
                scale=case.scale, q_len=case.q_len)
