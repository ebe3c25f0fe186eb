"""GPU parity of the GQA path against the fp64 oracle (through the C ABI)."""
import pytest
import torch

import parity as Pt
from paged_kv_cache_plan_gb300 import workloads as W

pytestmark = pytest.mark.gpu

VARIANTS = ["gqa_fma", "gqa_mma"]


@pytest.fixture(scope="module")
def tiny():
    c = W.gqa_tiny()
    return c, Pt.oracle_full(c)


@pytest.mark.parametrize("variant", VARIANTS)
def test_tiny_forced_four_splits(cuda_ok, tiny, variant):
    case, ref = tiny
    err, plan = Pt.check_case(case, ref=ref, variant=variant)
    assert plan.info["max_splits"] == 4 and plan.info["num_items"] == 4


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("splits", [0, 1, 2, 7, 32, 512])
def test_tiny_split_counts(cuda_ok, tiny, variant, splits):
    case, ref = tiny
    Pt.check_case(case, ref=ref, variant=variant, splits=splits)


@pytest.mark.parametrize("context", W.GQA_LONG_CONTEXTS)
@pytest.mark.parametrize("variant", VARIANTS)
def test_long_context(cuda_ok, context, variant):
    case = W.gqa_long(context)
    Pt.check_case(case, variant=variant)


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("variant", VARIANTS)
def test_varlen_batch(cuda_ok, dtype, variant):
    case = W.gqa_varlen(dtype)
    Pt.check_case(case, variant=variant)


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("group,head_dim", [(1, 128), (2, 256), (4, 128), (8, 128), (16, 256)])
@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_groups_dims_dtypes(cuda_ok, variant, group, head_dim, dtype):
    if variant == "gqa_fma" and group > 8:
        pytest.skip("the FMA path covers groups up to 8")
    lens = [1, 15, 16, 17, 333, 1000, 4096 + 5]
    case = W.gqa_case(batch=len(lens), heads=2 * group, kv_heads=2, head_dim=head_dim,
                      page_size=16, seq_lens=lens, pool_pages=400, dtype=dtype,
                      seed=31 + group + head_dim)
    Pt.check_case(case, variant=variant)


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("page_size", [1, 7, 16, 32])
def test_page_sizes(cuda_ok, variant, page_size):
    lens = [3, 100, 777]
    npages = sum(-(-L // page_size) for L in lens)
    case = W.gqa_case(batch=3, heads=8, kv_heads=2, head_dim=128, page_size=page_size,
                      seq_lens=lens, pool_pages=npages + 11, seed=40 + page_size)
    Pt.check_case(case, variant=variant)


@pytest.mark.parametrize("variant", VARIANTS)
def test_empty_and_single_token_requests(cuda_ok, variant):
    case = W.gqa_case(batch=4, heads=8, kv_heads=2, head_dim=256, page_size=16,
                      seq_lens=[0, 1, 0, 2], pool_pages=8, seed=51)
    Pt.check_case(case, variant=variant)
    case = W.gqa_case(batch=2, heads=8, kv_heads=2, head_dim=256, page_size=16,
                      seq_lens=[0, 0], pool_pages=2, seed=52)
    Pt.check_case(case, variant=variant)


@pytest.mark.parametrize("variant", VARIANTS)
def test_tails_ending_mid_warp(cuda_ok, variant):
    # 16,384-key spans plus tails that end inside a four-key pass and inside
    # a 16-token block, at d 256 and d 128
    for d in (256, 128):
        lens = [16384, 16384 + 1, 16384 + 6, 16384 + 15]
        case = W.gqa_case(batch=4, heads=16, kv_heads=2, head_dim=d, page_size=16,
                          seq_lens=lens, seed=60 + d)
        Pt.check_case(case, variant=variant)


def test_q_zero_closed_form(cuda_ok):
    case = W.gqa_case(batch=2, heads=8, kv_heads=2, head_dim=128, page_size=16,
                      seq_lens=[1000, 37], seed=71)
    case.q.zero_()
    for variant in VARIANTS:
        out, lse, _ = Pt.run_gpu(case, variant=variant)
        import math
        assert abs(lse[0] - math.log(1000)).max() < 1e-5
        assert abs(lse[1] - math.log(37)).max() < 1e-5
