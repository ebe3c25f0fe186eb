"""CPU checks of bench.py's workload names (no GPU needed): the named
workloads and the query-token suffix build the cases they describe."""
import bench


def test_query_token_suffix():
    c = bench.workload("gqa_tiny_q3")
    assert c.q_len == 3 and tuple(c.q.shape) == (1, 3, 4, 128)
    assert c.name.endswith("_q3")
    c1 = bench.workload("gqa_tiny")
    assert c1.q_len == 1 and tuple(c1.q.shape) == (1, 4, 128)
    # the cache is the same one: only the queries differ
    assert c.k_pages.shape == c1.k_pages.shape


def test_long_gqa_names():
    c = bench.workload("gqa_long_2k")
    assert int(c.seq_lens[0]) == 2048 and c.heads == 16 and c.kv_heads == 2
    assert c.kv_bytes_unique() == 2 * 2048 * 512 * 2


def test_per_config_names_resolve():
    # every configuration of the per-config record names a workload; cut to a
    # short context here so that the CPU draws stay small
    for name in bench.PER_CONFIG:
        c = bench.workload(name, context=64)
        assert int(c.seq_lens.max()) <= 64 and c.batch >= 1
        assert bench.full_context(name) >= 2048
    assert bench.full_context("mla_h128_b128") == 16384
    assert bench.full_context("mla16_b8") == 68000


def test_headline_is_the_largest_single_gpu_config():
    # the default line times the configuration with the most KV bytes per op
    import argparse
    # (distinct KV rows: a shared prefix counts once per group of 8)
    from paged_kv_cache_plan_gb300 import workloads as W
    sizes = {}
    for name in bench.PER_CONFIG:
        c = bench.workload(name, context=1)
        per_token = (c.k_row_pitch * 2 if c.mla
                     else c.kv_heads * (c.head_dim + c.head_dim_v) * 2)
        if name.startswith("mla16_b"):
            rows = (-(-c.batch // 8) * W.MLA16_PREFIX
                    + c.batch * (W.MLA16_CONTEXT - W.MLA16_PREFIX))
        elif name.startswith("gqa_varlen_"):
            rows = sum(W.VARLEN_LENS)
        else:
            rows = bench.full_context(name) * c.batch
        sizes[name] = (rows * per_token, c.heads)   # ties: more heads is more work
    assert max(sizes, key=sizes.get) == "mla_h128_b128"


def test_reference_arm_line(capsys):
    import json
    import sys
    argv = sys.argv
    sys.argv = ["bench.py", "--impl", "reference", "--workload", "gqa_tiny", "--steps", "3",
                "--warmup", "3"]
    try:
        bench.main()
    finally:
        sys.argv = argv
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0 and line["unit"] == "GB/s"
    assert line["cpu_baseline"]["kind"] == "oracle" and line["e2e"]["h2d_bytes_per_step"] == 0
