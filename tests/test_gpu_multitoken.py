"""GPU parity of multi-token decode (q_len query tokens per request, causal
among them) against the fp64 oracle, through the C ABI: the GQA mma kernel,
both MLA kernels, splits that cut through the causal tail, rows with no
visible token in a split, and page relabelling."""
import numpy as np
import pytest

import parity as Pt
from paged_kv_cache_plan_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _gqa(q_len, heads, kv_heads, head_dim, lens, dtype="bf16", seed=0, page_size=16):
    return W.gqa_case(batch=len(lens), heads=heads, kv_heads=kv_heads, head_dim=head_dim,
                      page_size=page_size, seq_lens=lens, dtype=dtype, seed=seed,
                      q_len=q_len, name=f"gqa_q{q_len}_h{heads}kv{kv_heads}_d{head_dim}")


@pytest.mark.parametrize("q_len,heads,kv_heads,head_dim", [
    (2, 8, 2, 128), (3, 16, 4, 128), (4, 8, 2, 128), (2, 16, 2, 256), (4, 4, 4, 256),
    (3, 15, 3, 128)])
@pytest.mark.parametrize("splits", [0, 3, 64])
def test_gqa(cuda_ok, q_len, heads, kv_heads, head_dim, splits):
    # lengths: the queries alone, a few pages, a split boundary just before
    # the tail, a long context
    lens = [q_len, 17, 33, 1000, 4099]
    case = _gqa(q_len, heads, kv_heads, head_dim, lens, seed=100 + q_len)
    Pt.check_case(case, variant="gqa_mma", splits=splits)


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_gqa_dtypes_page_sizes(cuda_ok, dtype):
    for ps in (1, 16, 32):
        case = _gqa(3, 8, 2, 128, [5, 64, 300], dtype=dtype, seed=7, page_size=ps)
        Pt.check_case(case, splits=0)


def test_gqa_tail_split_of_one_token(cuda_ok):
    # chunk 16 with L = 16k + 1: the last split holds only the newest token,
    # so every query token but the last sees nothing there
    case = _gqa(4, 8, 2, 128, [16 * 9 + 1, 16 * 3 + 1], seed=11)
    err, plan = Pt.check_case(case, splits=0, min_chunk=16)
    assert plan.info["chunk"] == 16


@pytest.mark.parametrize("q_len,heads", [(2, 16), (3, 16), (2, 32), (4, 16)])
def test_mla_mma(cuda_ok, q_len, heads):
    case = W.mla_case(batch=3, heads=heads, seq_len=700, prefix_len=0, seed=20 + q_len,
                      q_len=q_len)
    for splits in (0, 7, 256):
        Pt.check_case(case, variant="mla_mma", splits=splits)


@pytest.mark.parametrize("q_len,heads", [(4, 16), (2, 64), (2, 32)])
def test_mla_tensor_memory(cuda_ok, q_len, heads):
    # 1027 tokens: two splits (the causal tail inside the second), and one
    # split per token (the last splits hold tokens some query rows do not
    # see: rows with no visible token in an item)
    case = W.mla_case(batch=2, heads=heads, seq_len=1027, prefix_len=0, seed=30 + q_len,
                      q_len=q_len)
    for splits in (2, 1027):
        err, plan = Pt.check_case(case, variant="mla_tc", splits=splits)
        assert plan.info["variant"] == 4
    case = W.mla_case(batch=2, heads=heads, seq_len=5000, prefix_len=0, seed=40 + q_len,
                      q_len=q_len)
    err, plan = Pt.check_case(case)
    assert plan.info["variant"] == 4


def test_relabelling_bit_exact(cuda_ok):
    for case in (_gqa(3, 8, 2, 128, [40, 300], seed=5),
                 W.mla_case(batch=2, heads=16, seq_len=300, prefix_len=0, seed=6, q_len=2)):
        o1, l1, _ = Pt.run_gpu(case)
        o2, l2, _ = Pt.run_gpu(W.permute_pages(case, 3))
        assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_one_token_plan_unchanged(cuda_ok):
    # q_len 1 through the new fields gives the same bits as the plain plan
    case = _gqa(1, 8, 2, 128, [33, 1000], seed=9)
    o1, l1, _ = Pt.run_gpu(case)
    o2, l2, _ = Pt.run_gpu(case, q_len=1)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
