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
