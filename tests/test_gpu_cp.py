"""Context-parallel decode on one GPU: every rank's plan (decode_plan_cp) is
run in turn on the same GPU, the ranks' rows are stacked in rank order (what
the all-gather would deliver) and merged by decode_merge_ranks; the result
must match the oracle at the standard tolerances and the unsharded plan.
The exchange itself is covered on the CPU (tests/test_cp_cpu.py, gloo)."""
import numpy as np
import pytest
import torch

import parity as Pt
from paged_kv_cache_plan_gb300 import (cp_ranges, decode_merge_ranks, decode_plan_cp, make_desc,
                                       run_case)
from paged_kv_cache_plan_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _desc(case, **kw):
    return make_desc(case.batch, case.heads, case.kv_heads, case.head_dim, case.page_size,
                     head_dim_v=case.head_dim_v, dtype=case.dtype,
                     max_pages_per_seq=case.max_pages, num_pool_pages=case.pool_pages,
                     k_row_pitch=case.k_row_pitch, v_row_pitch=case.v_row_pitch,
                     scale=case.scale, **kw)


def _cp_run(case, dev, world, **kw):
    seq = case.seq_lens.tolist()
    B, H, dv = case.batch, case.heads, case.head_dim_v
    o_parts = torch.full((world, B, H, dv), float("nan"), device="cuda")
    l_parts = torch.full((world, B, H), float("nan"), device="cuda")
    variants = []
    for r in range(world):
        plan = decode_plan_cp(_desc(case, **kw), seq, world, r)
        variants.append(plan.info["variant"])
        run_case(plan, dev, o_parts[r], l_parts[r])
        assert plan.last_device_status() == 0
    out = torch.full((B, H, dv), float("nan"), device="cuda")
    lse = torch.full((B, H), float("nan"), device="cuda")
    decode_merge_ranks(o_parts, l_parts, out, lse)
    torch.cuda.synchronize()
    return out.cpu().double().numpy(), lse.cpu().double().numpy(), variants


CASES = {
    "gqa_d256": lambda: W.gqa_case(batch=3, heads=16, kv_heads=2, head_dim=256, page_size=16,
                                   seq_lens=[5000, 17, 900], pool_pages=500, seed=501),
    "gqa_d128_fp16": lambda: W.gqa_case(batch=4, heads=32, kv_heads=8, head_dim=128,
                                        page_size=16, seq_lens=[3000, 1, 64, 2048],
                                        pool_pages=400, dtype="fp16", seed=502),
    "mla16": lambda: W.mla_case(batch=3, heads=16, seq_len=2600, pool_rows=8000, seed=503),
    "mla64_long": lambda: W.mla_case(batch=2, heads=64, seq_len=5000, pool_rows=10100, seed=504),
}


@pytest.mark.parametrize("world", [2, 3, 4])
@pytest.mark.parametrize("name", sorted(CASES))
def test_sharded_then_merged_matches_oracle(cuda_ok, name, world):
    case = CASES[name]()
    dev = case.to("cuda")
    out, lse, variants = _cp_run(case, dev, world)
    ref_o, ref_l = Pt.oracle_full(case)
    Pt.compare(out, lse, ref_o, ref_l, f"{name} over {world} ranks")
    # and the unsharded plan, same tolerances
    o1, l1, _ = Pt.run_gpu(case)
    Pt.compare(out, lse, o1, l1, f"{name} over {world} ranks vs one plan")


def test_empty_ranges_and_forced_splits(cuda_ok):
    # requests shorter than a page per rank leave the later ranks empty
    case = W.gqa_case(batch=3, heads=8, kv_heads=2, head_dim=128, page_size=16,
                      seq_lens=[40, 5, 0], pool_pages=10, seed=505)
    dev = case.to("cuda")
    begin, length = cp_ranges(4, 3, case.seq_lens.tolist(), 16)
    assert length == [0, 0, 0]
    out, lse, _ = _cp_run(case, dev, 4, splits=3)
    ref_o, ref_l = Pt.oracle_full(case)
    Pt.compare(out, lse, ref_o, ref_l, "short requests over 4 ranks")


def test_merge_is_rank_order_deterministic(cuda_ok):
    case = CASES["mla16"]()
    dev = case.to("cuda")
    a = _cp_run(case, dev, 3)
    b = _cp_run(case, dev, 3)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
