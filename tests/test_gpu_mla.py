"""GPU parity of the MLA path (576-wide latent rows, V = the first 512)."""
import pytest
import torch

import parity as Pt
from paged_kv_cache_plan_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_small_shared_prefix(cuda_ok, dtype):
    case = W.mla_case(batch=5, heads=16, seq_len=1000, prefix_len=600, group=2,
                      pool_rows=20000, dtype=dtype, seed=81)
    Pt.check_case(case)
    Pt.check_case(case, splits=7)


@pytest.mark.parametrize("seq_len", [1, 2, 63, 64, 65, 129, 3000])
def test_lengths(cuda_ok, seq_len):
    case = W.mla_case(batch=2, heads=16, seq_len=seq_len, pool_rows=2 * seq_len + 50, seed=82)
    Pt.check_case(case)


def test_several_head_blocks(cuda_ok):
    case = W.mla_case(batch=3, heads=48, seq_len=700, pool_rows=3000, seed=83)
    Pt.check_case(case)


def test_mla16_batch1_full_size(cuda_ok):
    # 68,000-token context, 2,000,000-row pool (over 2 GiB: 64-bit offsets),
    # 256 splits; every head checked against the oracle
    case = W.mla16(1)
    Pt.check_case(case)


@pytest.mark.parametrize("batch", [8, 48])
def test_mla16_shared_prefix_full_size(cuda_ok, batch):
    # every head of the first and last request, the first and last head of
    # every request (each member of every prefix group), a few random rows
    case = W.mla16(batch)
    Pt.check_sampled(case, pairs=Pt.edge_pairs(case))


@pytest.mark.parametrize("heads,batch", [(64, 64), (64, 128), (128, 64), (128, 128)])
def test_mla_many_heads_full_size(cuda_ok, heads, batch):
    # 128 heads: both 64-head items of the first and last request in full
    case = W.mla_many(heads, batch)
    res, plan = Pt.check_sampled(case, pairs=Pt.edge_pairs(case))
    assert plan.info["variant"] == 4
