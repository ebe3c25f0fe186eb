"""GPU parity of the tensor-memory MLA kernel (tcgen05, 64-head blocks).

It rounds P to one 16-bit value before the P.V product. The planner takes
it (AUTO) and accepts it (forced) only when every non-empty request has at
least 1,024 tokens, where the rounding errors average out far below the
output tolerance; shorter requests are refused for it and run on the
mma.sync kernel with its two-part P. Every test here holds the standard
tolerances.
"""
import math

import numpy as np
import pytest
import torch

import parity as Pt
from paged_kv_cache_plan_gb300 import _lib
from paged_kv_cache_plan_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("heads,batch,seq_len", [(64, 2, 2048), (128, 2, 1500), (64, 3, 1089)])
def test_long_contexts(cuda_ok, heads, batch, seq_len):
    case = W.mla_case(batch=batch, heads=heads, seq_len=seq_len,
                      pool_rows=batch * seq_len + 300, seed=101)
    res, plan = Pt.check_case(case, variant="mla_tc")
    assert plan.info["variant"] == 4 and plan.info["heads_per_unit"] == 64
    Pt.check_case(case, variant="mla_tc", splits=3)


@pytest.mark.parametrize("heads,q_len,batch,seq_len", [
    (16, 1, 1, 3000),    # 16 of 64 rows used
    (32, 1, 2, 1500),
    (48, 1, 2, 1100),
    (16, 3, 2, 1200),    # 48 (token, head) rows
    (32, 3, 1, 2000),    # 96 rows: one full unit and one half-used unit
    (80, 1, 1, 1024),    # 80 rows: the second unit holds 16
])
def test_padded_units(cuda_ok, heads, q_len, batch, seq_len):
    # a request whose (query token, head) rows are not a multiple of 64: the
    # last unit's unused rows carry zero queries and write nothing
    case = W.mla_case(batch=batch, heads=heads, seq_len=seq_len, q_len=q_len,
                      pool_rows=batch * seq_len + 200, seed=108)
    res, plan = Pt.check_case(case, variant="mla_tc")
    assert plan.info["variant"] == 4
    assert plan.info["units_per_request"] == -(-q_len * heads // 64)
    Pt.check_case(case, variant="mla_tc", splits=5)


def test_auto_picks_tensor_memory_kernel(cuda_ok):
    case = W.mla_case(batch=1, heads=128, seq_len=1024, pool_rows=1100, seed=102)
    res, plan = Pt.check_case(case)
    assert plan.info["variant"] == 4


def test_fp16(cuda_ok):
    case = W.mla_case(batch=2, heads=64, seq_len=1300, pool_rows=2700, dtype="fp16", seed=103)
    Pt.check_case(case, variant="mla_tc")


@pytest.mark.parametrize("seq_len", [1, 2, 63, 64, 65, 129, 700, 1023])
def test_short_lengths_refused_then_auto_within_tolerance(cuda_ok, seq_len):
    case = W.mla_case(batch=2, heads=64, seq_len=seq_len, pool_rows=2 * seq_len + 40, seed=104)
    with pytest.raises(_lib.PkvdError) as e:
        Pt.run_gpu(case, variant="mla_tc")
    assert e.value.code == _lib.PKVD_EUNSUPPORTED
    res, plan = Pt.check_case(case)   # AUTO: the mma.sync kernel, standard tolerances
    assert plan.info["variant"] == 3


def test_split_shorter_than_a_block(cuda_ok):
    # a forced split count that leaves the last split a handful of tokens
    case = W.mla_case(batch=2, heads=64, seq_len=1100, pool_rows=2300, seed=107)
    Pt.check_case(case, variant="mla_tc", splits=16)


def test_empty_request(cuda_ok):
    case = W.mla_case(batch=3, heads=64, seq_len=1200, pool_rows=3700, seed=105)
    case.seq_lens[1] = 0
    out, lse, _ = Pt.run_gpu(case, variant="mla_tc")
    assert np.all(out[1] == 0) and np.all(np.isneginf(lse[1]))
    ref_o, ref_l = Pt.oracle_full(case)
    Pt.compare(out, lse, ref_o, ref_l, "empty request")


def test_growing_scores_rescale(cuda_ok):
    # Scores that climb along the sequence, so that the running maximum is
    # raised again and again by more than the lazy-rescale margin: every
    # head's query is 24 u for a unit vector u on the 64 rope dims, and key t
    # carries (96 t / L) u there. V (the first 512 dims) stays N(0, 1/16).
    case = W.mla_case(batch=1, heads=64, seq_len=2048, pool_rows=2100, seed=106)
    g = torch.Generator().manual_seed(7)
    u = torch.zeros(576)
    u[512:] = torch.randn(64, generator=g)
    u = u / u.norm()
    case.q[:] = (u * 24.0).to(case.q.dtype)
    rows = case.page_table[0, :2048].to(torch.int64)
    ramp = torch.arange(2048, dtype=torch.float32) / 2047.0 * 96.0
    kv = case.k_pages.view(-1, 576)
    kv[rows] = (kv[rows].float() * 0.25 + ramp[:, None] * u[None, :]).to(kv.dtype)
    s = (case.q[0, 0].double() @ kv[rows].double().T) * case.scale / math.log(2.0)
    assert float(s.max() - s[:64].max()) > 3 * 8.0   # several lazy rescales happen
    Pt.check_case(case, variant="mla_tc")
