"""GPU parity of the dense causal prefill at head_dim 64 (prefill_d64_run)
against the fp64 oracle, which computes it as the decode problem with every
token a query on one page per request."""
import numpy as np
import pytest
import torch

import parity as Pt
from paged_kv_cache_plan_gb300 import prefill_d64
from paged_kv_cache_plan_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _run(case):
    q, k, v = case.q.cuda(), case.k_pages.cuda(), case.v_pages.cuda()
    out = torch.full((case.batch, case.q_len, case.heads, 64), float("nan"), device="cuda")
    lse = torch.full((case.batch, case.q_len, case.heads), float("nan"), device="cuda")
    out, lse, status = prefill_d64(q, k, v, out=out, lse=lse)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    vh = case.q_len * case.heads
    return (out.reshape(case.batch, vh, 64).cpu().double().numpy(),
            lse.reshape(case.batch, vh).cpu().double().numpy())


@pytest.mark.parametrize("seq_len", [1, 37, 128, 129, 300, 1000])
@pytest.mark.parametrize("heads,kv_heads", [(4, 2), (8, 1)])
def test_small(cuda_ok, seq_len, heads, kv_heads):
    case = W.prefill_case(batch=2, heads=heads, kv_heads=kv_heads, seq_len=seq_len,
                          seed=seq_len + heads)
    out, lse = _run(case)
    ref_o, ref_l = Pt.oracle_full(case)
    Pt.compare(out, lse, ref_o, ref_l, case.name)


def test_one_part_rows(cuda_ok):
    # query tiles from 1,024 tokens on use a one-part P; full oracle at 1,500
    case = W.prefill_case(batch=1, heads=2, kv_heads=1, seq_len=1500, seed=9)
    out, lse = _run(case)
    Pt.compare(out, lse, *Pt.oracle_full(case), case.name)


@pytest.mark.parametrize("seq_len", [1100, 1408, 2300])
def test_late_tile_counts(cuda_ok, seq_len):
    # late query tiles (one-part P) in odd and even counts: 1,100 tokens
    # leave one late tile, 1,408 three, 2,300 ten with a partial last tile
    case = W.prefill_case(batch=1, heads=2, kv_heads=2, seq_len=seq_len, seed=seq_len)
    out, lse = _run(case)
    Pt.compare(out, lse, *Pt.oracle_full(case), case.name)


def test_fp16(cuda_ok):
    case = W.prefill_case(batch=1, heads=4, kv_heads=4, seq_len=513, dtype="fp16", seed=5)
    out, lse = _run(case)
    Pt.compare(out, lse, *Pt.oracle_full(case), case.name)


def test_long_sampled(cuda_ok):
    # 4,096 tokens, 16 heads: the oracle on sampled (token, head) rows,
    # including the first and last rows of query tiles
    case = W.prefill_case(batch=1, heads=16, kv_heads=4, seq_len=4096, seed=7)
    out, lse = _run(case)
    rows = [(0, t * 16 + h) for t, h in [(0, 0), (127, 3), (128, 5), (1000, 15), (2047, 8),
                                         (2048, 1), (4095, 0), (4095, 15)]]
    ref_o, ref_l = Pt.oracle_pairs(case, rows)
    got_o = np.stack([out[b, v] for b, v in rows])
    got_l = np.array([lse[b, v] for b, v in rows])
    Pt.compare(got_o, got_l, ref_o, ref_l, case.name)
