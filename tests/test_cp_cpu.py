"""Context-parallel decode, host side (no GPU): the ranks' token ranges, the
ranks' plans, and the exchange-then-merge protocol over a world_size-2 gloo
process group, with the oracle standing in for each rank's GPU decode.

A request's tokens are cut into `world` page-aligned ranges; each rank
decodes its range into a normalised output and a log-sum-exp, the ranks
all-gather those rows and merge them by log-sum-exp (the aiter pull 4758
page's split merge, Technical Details 3, with the ranges as splits). The
merged rows must equal the whole-context decode.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from paged_kv_cache_plan_gb300 import (_lib, cp_ranges, decode_plan_cp_compute, gather_ranks,
                                       make_desc)
from paged_kv_cache_plan_gb300 import workloads as W


@pytest.mark.parametrize("page_size", [1, 16])
@pytest.mark.parametrize("world", [1, 2, 3, 5, 8])
def test_ranges_cover_every_token_once(world, page_size):
    rng = np.random.default_rng(world * 31 + page_size)
    seq = [0, 1, 15, 16, 17, 1000] + [int(x) for x in rng.integers(0, 70000, 6)]
    got = {b: [] for b in range(len(seq))}
    for r in range(world):
        begin, length = cp_ranges(world, r, seq, page_size)
        for b, (t0, n) in enumerate(zip(begin, length)):
            assert n >= 0 and t0 % page_size == 0 or n == 0
            if n:
                got[b].append((t0, t0 + n))
    for b, L in enumerate(seq):
        spans = sorted(got[b])
        covered = sum(t1 - t0 for t0, t1 in spans)
        assert covered == L
        for (a0, a1), (b0, b1) in zip(spans, spans[1:]):
            assert a1 == b0            # contiguous, disjoint, in rank order
        if spans:
            assert spans[0][0] == 0 and spans[-1][1] == L


def test_rank_plans_walk_their_ranges():
    seq = [70000, 3000, 17, 0]
    for heads, kv, d, ps in ((16, 2, 256, 16), (128, 1, 576, 1)):
        for world in (2, 3):
            for r in range(world):
                begin, length = cp_ranges(world, r, seq, ps)
                desc = make_desc(len(seq), heads, kv, d, ps, num_sms=152, ctas_per_sm=1)
                info, items = decode_plan_cp_compute(desc, seq, world, r)
                for b in range(len(seq)):
                    spans = sorted((t0, t1) for (rb, u, _, _, t0, t1) in items
                                   if rb == b and u == 0)
                    if length[b] == 0:
                        assert not spans
                        continue
                    assert spans[0][0] == begin[b] and spans[-1][1] == begin[b] + length[b]
                    for x, y in zip(spans, spans[1:]):
                        assert x[1] == y[0]


@pytest.mark.parametrize("kw,code", [
    (dict(world=0, rank=0), _lib.PKVD_EINVAL),
    (dict(world=2, rank=2), _lib.PKVD_EINVAL),
    (dict(world=2, rank=-1), _lib.PKVD_EINVAL),
    (dict(world=2, rank=0, q_len=2), _lib.PKVD_EUNSUPPORTED),
])
def test_rank_plan_errors(kw, code):
    desc = make_desc(1, 8, 2, 128, 16, num_sms=152, ctas_per_sm=1, q_len=kw.get("q_len", 0))
    with pytest.raises(_lib.PkvdError) as e:
        decode_plan_cp_compute(desc, [100], kw["world"], kw["rank"])
    assert e.value.code == code


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _case():
    return W.gqa_case(batch=3, heads=8, kv_heads=2, head_dim=128, page_size=16,
                      seq_lens=[700, 33, 5], pool_pages=60, seed=401)


def _rank_main(rank, world, port, out_path):
    import oracle
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        case = _case()
        P = oracle.problem(**W.oracle_problem_kwargs(case))
        begin, length = cp_ranges(world, rank, case.seq_lens.tolist(), case.page_size)
        B, H, dv = case.batch, case.heads, case.head_dim_v
        o_r = torch.zeros((B, H, dv), dtype=torch.float64)
        l_r = torch.full((B, H), float("-inf"), dtype=torch.float64)
        for b in range(B):
            for h in range(H):
                o, l = oracle.partial(P, case.q, case.k_pages, case.v_pages, case.page_table,
                                      case.seq_lens, b, h, begin[b], begin[b] + length[b])
                o_r[b, h] = torch.from_numpy(o)
                l_r[b, h] = l
        o_parts, l_parts = gather_ranks(o_r, l_r)
        out = np.zeros((B, H, dv))
        lse = np.zeros((B, H))
        for b in range(B):
            for h in range(H):
                out[b, h], lse[b, h] = oracle.merge(o_parts[:, b, h].numpy(),
                                                    l_parts[:, b, h].numpy())
        np.savez(out_path + f".{rank}.npz", out=out, lse=lse)
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2])
def test_gloo_exchange_then_merge_equals_whole_context(tmp_path, world):
    import oracle
    oracle.build()
    port = _free_port()
    out_path = str(tmp_path / "cp")
    mp.start_processes(_rank_main, args=(world, port, out_path), nprocs=world, join=True,
                       start_method="spawn")
    case = _case()
    ref_o, ref_l = oracle.decode(oracle.problem(**W.oracle_problem_kwargs(case)), case.q,
                                 case.k_pages, case.v_pages, case.page_table, case.seq_lens)
    for r in range(world):
        got = np.load(out_path + f".{r}.npz")
        assert np.abs(got["out"] - ref_o).max() < 1e-12
        fin = np.isfinite(ref_l)
        assert np.array_equal(np.isfinite(got["lse"]), fin)
        assert np.abs(got["lse"][fin] - ref_l[fin]).max() < 1e-12
