"""CPU tests of the C-ABI library: it loads, exports every declared entry
point, and its host planner (decode_plan_compute, no CUDA call) lays out the
splits, grid order and merge tiling as documented. No kernel runs here."""
import os
import re

import pytest

from paged_kv_cache_plan_gb300 import _lib, decode_plan_compute, make_desc

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from paged_kv_cache_plan_gb300 import build
    build.build()
    return _lib.lib()


def _header_functions():
    src = open(os.path.join(ROOT, "include", "pkvd.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:int|size_t|const char \*)\s*(\w+)\s*\(", src, re.M)))


def test_exports_every_declared_symbol(L):
    names = _header_functions()
    assert len(names) >= 10
    for n in names:
        assert hasattr(L, n), f"libpkvd.so does not export {n}"
    assert set(names) == set(_lib.SIGNATURES)


def test_status_strings(L):
    for code in (0, -1, -2, -3, -4, -5, -6):
        assert _lib.status_string(code) not in ("", "unknown status")
    assert _lib.status_string(123) == "unknown status"


def _plan(*args, seq, **kw):
    kw.setdefault("num_sms", 152)
    kw.setdefault("ctas_per_sm", 1)
    return decode_plan_compute(make_desc(*args, **kw), seq)


def _check_cover(info, items, seq, units):
    # every (request, unit) token range is covered exactly once, in split order
    by = {}
    for (b, u, s, row, t0, t1) in items:
        by.setdefault((b, u), []).append((s, t0, t1, row))
    for b, L in enumerate(seq):
        for u in range(units):
            got = sorted(by.get((b, u), []))
            if L == 0:
                assert not got
                continue
            assert [g[0] for g in got] == list(range(len(got)))
            assert got[0][1] == 0 and got[-1][2] == L
            for a, c in zip(got, got[1:]):
                assert a[2] == c[1] and a[1] < a[2]
    rows = sorted({(b, s, row) for (b, u, s, row, t0, t1) in items})
    assert len({r for (_, _, r) in rows}) == info["num_partial_rows"]


def test_auto_split_fills_one_wave(L):
    for seq, sms, occ in (([65536], 152, 1), ([65536], 152, 2), ([2048], 152, 2),
                          ([256, 512, 768, 1024, 1536, 2048, 8192, 32768, 65536, 131072], 152, 2)):
        kv = 2 if len(seq) == 1 else 8
        heads = 16 if kv == 2 else 32
        d = 256 if kv == 2 else 128
        info, items = _plan(len(seq), heads, kv, d, 16, seq=seq, num_sms=sms, ctas_per_sm=occ)
        assert info["num_items"] <= sms * occ
        assert info["chunk"] % 16 == 0
        _check_cover(info, items, seq, kv)
        # a smaller chunk would need more than one wave
        C = info["chunk"] - 16
        if C >= 32:
            assert sum(-(-L // C) for L in seq) * kv > sms * occ


def test_forced_splits(L):
    info, items = _plan(1, 4, 1, 128, 16, seq=[512], splits=4)
    assert info["num_items"] == 4 and info["chunk"] == 128
    assert [(t0, t1) for (*_, t0, t1) in items] == [(0, 128), (128, 256), (256, 384), (384, 512)]
    # more splits than tokens: one token each
    info, items = _plan(1, 4, 1, 128, 16, seq=[10], splits=64)
    assert info["num_items"] == 10 and info["max_splits"] == 10
    # MLA policy 256 / batch at 68,000 tokens
    for B in (1, 8, 24, 48):
        info, items = _plan(B, 16, 1, 576, 1, seq=[68000] * B, splits=max(1, 256 // B))
        assert info["max_splits"] == 256 // B
        _check_cover(info, items, [68000] * B, 1)


def test_grid_orders_same_items(L):
    seq = [100, 0, 37, 300]
    a_info, a = _plan(4, 8, 2, 128, 16, seq=seq, grid_order="split_major", splits=3)
    b_info, b = _plan(4, 8, 2, 128, 16, seq=seq, grid_order="request_major", splits=3)
    assert a_info["grid_order"] == 1 and b_info["grid_order"] == 2
    assert sorted(a) == sorted(b) and a != b
    # split-major: split index never decreases along the grid
    assert [it[2] for it in a] == sorted(it[2] for it in a)
    auto1, _ = _plan(1, 8, 2, 128, 16, seq=[100])
    auto4, _ = _plan(4, 8, 2, 128, 16, seq=seq)
    assert auto1["grid_order"] == 2 and auto4["grid_order"] == 1


def test_stage2_tiling_gate(L):
    # batch 1, 16 heads on 152 SMs: idle machine -> 8 slices of 512
    info, _ = _plan(1, 16, 1, 576, 1, seq=[68000])
    assert info["stage2_tiles"] == 8
    # many heads: the grid already fills the machine -> untiled
    info, _ = _plan(64, 128, 1, 576, 1, seq=[16384] * 64)
    assert info["stage2_tiles"] == 1
    # d 128 cannot be cut into 8 slices of at least 32
    info, _ = _plan(1, 4, 1, 128, 16, seq=[512])
    assert info["stage2_tiles"] == 4
    info, _ = _plan(1, 4, 1, 128, 16, seq=[512], stage2_tiles=2)
    assert info["stage2_tiles"] == 2


def test_variant_resolution(L):
    assert _plan(1, 16, 2, 256, 16, seq=[10])[0]["variant"] == 2      # MMA by default
    assert _plan(1, 32, 2, 128, 16, seq=[10])[0]["variant"] == 2      # MMA, group 16
    assert _plan(1, 16, 2, 256, 16, seq=[10], variant="gqa_fma")[0]["variant"] == 1
    assert _plan(1, 128, 1, 576, 1, seq=[10])[0]["variant"] == 3
    info = _plan(2, 128, 1, 576, 1, seq=[10, 20])[0]
    assert info["units_per_request"] == 8 and info["heads_per_unit"] == 16
    # tensor-memory MLA kernel: 64-head blocks, only for long contexts by default
    info = _plan(2, 128, 1, 576, 1, seq=[1024, 4096])[0]
    assert info["variant"] == 4 and info["heads_per_unit"] == 64 and info["units_per_request"] == 2
    assert info["block_tokens"] == 64 and info["stage1_threads"] == 448
    assert _plan(2, 128, 1, 576, 1, seq=[1023, 4096])[0]["variant"] == 3
    # row counts that are not a multiple of 64 take it too (padded last unit)
    info = _plan(1, 48, 1, 576, 1, seq=[4096])[0]
    assert info["variant"] == 4 and info["units_per_request"] == 1
    assert _plan(1, 16, 1, 576, 1, seq=[1023])[0]["variant"] == 3
    assert _plan(1, 64, 1, 576, 1, seq=[1024], variant="mla_tc")[0]["variant"] == 4
    # its one-part P is refused below 1,024 tokens (empty requests do not count)
    for seq in ([100], [1023, 4096], [4096, 1]):
        with pytest.raises(_lib.PkvdError) as e:
            _plan(len(seq), 64, 1, 576, 1, seq=seq, variant="mla_tc")
        assert e.value.code == _lib.PKVD_EUNSUPPORTED
    assert _plan(2, 64, 1, 576, 1, seq=[0, 2048], variant="mla_tc")[0]["variant"] == 4


@pytest.mark.parametrize("heads,q_len,units", [(16, 1, 1), (48, 1, 1), (16, 5, 2), (32, 3, 2),
                                               (80, 1, 2), (128, 1, 2)])
def test_tensor_memory_units_are_padded(L, heads, q_len, units):
    # the last 64-row unit of a request may be partly used
    info, items = _plan(2, heads, 1, 576, 1, seq=[2048, 1500], variant="mla_tc", q_len=q_len)
    assert info["variant"] == 4 and info["heads_per_unit"] == 64
    assert info["units_per_request"] == units
    _check_cover(info, items, [2048, 1500], units)


def test_tensor_memory_split_choice(L):
    # one resident block per SM: the split count minimises waves x (tokens + fill)
    info, items = _plan(64, 64, 1, 576, 1, seq=[16384] * 64, variant="mla_tc")
    waves = -(-info["num_items"] // 152)
    assert info["chunk"] % 64 == 0
    assert waves * (info["chunk"] + 128) <= 2 * (16384 + 128)   # better than one split per request
    _check_cover(info, items, [16384] * 64, 1)


@pytest.mark.parametrize("kw,code", [
    (dict(args=(1, 6, 4, 128, 16)), _lib.PKVD_EUNSUPPORTED),        # heads % kv_heads
    (dict(args=(1, 4, 1, 96, 16)), _lib.PKVD_EUNSUPPORTED),         # head_dim
    (dict(args=(1, 8, 2, 576, 1)), _lib.PKVD_EUNSUPPORTED),         # MLA with kv_heads 2
    (dict(args=(1, 24, 1, 576, 1)), _lib.PKVD_EUNSUPPORTED),        # MLA heads % 16
    (dict(args=(1, 4, 1, 128, 0)), _lib.PKVD_EINVAL),               # page size
    (dict(args=(0, 4, 1, 128, 16)), _lib.PKVD_EINVAL),              # batch
    (dict(args=(1, 4, 1, 128, 16), checks=True), _lib.PKVD_EINVAL), # checks need the pool size
    (dict(args=(1, 4, 1, 128, 16), stage2_tiles=3), _lib.PKVD_EINVAL),
    (dict(args=(1, 4, 1, 128, 16), k_row_pitch=100), _lib.PKVD_EINVAL),   # pitch < D
    (dict(args=(1, 4, 1, 128, 16), k_row_pitch=132), _lib.PKVD_EINVAL),   # 264 B not 16-B aligned
    (dict(args=(1, 4, 1, 128, 16), max_pages_per_seq=3), _lib.PKVD_EINVAL),
    (dict(args=(1, 32, 1, 128, 16), variant="gqa_fma"), _lib.PKVD_EUNSUPPORTED),   # group 32
    (dict(args=(1, 4, 1, 128, 16), variant="mla_mma"), _lib.PKVD_EUNSUPPORTED),
    (dict(args=(1, 16, 1, 576, 1), variant="mla_tc"), _lib.PKVD_EUNSUPPORTED),    # 100 tokens
    (dict(args=(1, 8, 2, 128, 16), variant="mla_tc"), _lib.PKVD_EUNSUPPORTED),
])
def test_argument_errors(L, kw, code):
    args = kw.pop("args")
    with pytest.raises(_lib.PkvdError) as e:
        _plan(*args, seq=[100] * args[0] if args[0] > 0 else [], **kw)
    assert e.value.code == code


def test_negative_length_rejected(L):
    with pytest.raises(_lib.PkvdError) as e:
        _plan(2, 4, 1, 128, 16, seq=[5, -1])
    assert e.value.code == _lib.PKVD_EINVAL


def test_plan_identity_includes_batch_and_lengths(L):
    # Two specs that differ only in batch (or only in lengths) must lay out
    # different work: the plan is a value of every shape field.
    a, ia = _plan(4, 8, 2, 128, 16, seq=[2048] * 4)
    b, ib = _plan(6, 8, 2, 128, 16, seq=[256, 512, 768, 1024, 1536, 2048])
    assert ia != ib and a["num_partial_rows"] != b["num_partial_rows"]
    c, ic = _plan(4, 8, 2, 128, 16, seq=[2048, 2048, 2048, 2047])
    assert ic != ia


def test_empty_batch_entries(L):
    info, items = _plan(3, 4, 1, 128, 16, seq=[0, 0, 0])
    assert info["num_items"] == 0 and info["num_partial_rows"] == 0
    info, items = _plan(3, 4, 1, 128, 16, seq=[0, 33, 0])
    assert all(it[0] == 1 for it in items)


def _prefix_plan(B, heads, seq, groups, plen, **kw):
    from paged_kv_cache_plan_gb300 import decode_plan_prefix_compute
    kw.setdefault("num_sms", 152)
    kw.setdefault("ctas_per_sm", 2)
    return decode_plan_prefix_compute(make_desc(B, heads, 1, 576, 1, **kw), seq, groups, plen)


def _check_prefix_cover(seq, groups, plen, info, pre, rest):
    """Every token of every request is covered exactly once, by grouped
    prefix items (members b0 .. b0 + unit - 1) or by its own items; returns
    the prefix splits of each request."""
    B = len(seq)
    assert info["num_prefix_items"] == len(pre) and info["num_items"] == len(rest)
    assert all(g == 1 and 1 <= u <= 4 for (_, u, _, _, _, _, g) in pre)
    assert all(g == 0 for (*_, g) in rest)
    cover = {b: [] for b in range(B)}
    prefix_splits = {b: set() for b in range(B)}
    for (b0, unit, s, _, t0, t1, _) in pre:
        for b in range(b0, b0 + unit):
            assert groups[b] == groups[b0] and t1 <= plen[b]
            cover[b].append((t0, t1))
            prefix_splits[b].add(s)
    for (b, u, s, row, t0, t1, _) in rest:
        if u == 0:   # every head block of a request walks the same tokens
            cover[b].append((t0, t1))
    for b in range(B):
        got = sorted(cover[b])
        if seq[b] == 0:
            assert not got
            continue
        assert got[0][0] == 0 and got[-1][1] == seq[b]
        for x, y in zip(got, got[1:]):
            assert x[1] == y[0]
        assert prefix_splits[b] == set(range(len(prefix_splits[b])))
    # partial rows: each request's prefix splits, then its private splits
    nrows = sum(len(prefix_splits[b]) for b in range(B)) + len(rest)
    assert info["num_partial_rows"] == nrows - len(rest) + len([r for r in rest if r[1] == 0])
    assert len({row for (_, u, _, row, _, _, _) in rest if u == 0}) == \
        len([r for r in rest if r[1] == 0])
    return prefix_splits


def test_shared_prefix_plan_covers_every_token_once(L):
    seq = [3000, 3000, 3000, 1500, 2000, 2100, 1100, 900, 900]
    groups = [0, 0, 0, 1, 1, -1, 2, 3, 3]
    plen = [1700, 1700, 1700, 1200, 1200, 0, 1100, 500, 500]
    info, pre, rest = _prefix_plan(len(seq), 16, seq, groups, plen)
    splits = _check_prefix_cover(seq, groups, plen, info, pre, rest)
    assert info["num_prefix_items"] > 0
    # group 3's 500-token prefix is too short to group: read per request
    assert not splits[7] and not splits[8]
    assert all(splits[b] for b in range(7) if b != 5)
    # no prefix split but a prefix's last is shorter than 1,024 tokens
    for (b0, _, _, _, t0, t1, _) in pre:
        assert t1 - t0 >= 1024 or t1 == plen[b0]


def test_random_shared_prefix_plans_cover_every_token_once(L):
    # seeded mixes of groups (runs of 1 to 8 consecutive requests), ungrouped
    # requests and empty ones, short and long prefixes
    import random
    rng = random.Random(31)
    for _ in range(150):
        heads = rng.choice((16, 32, 64))
        seq, groups, plen = [], [], []
        g = 0
        while len(seq) < rng.randint(1, 14):
            if rng.random() < 0.3:
                seq.append(rng.choice((0, 1, rng.randint(2, 30000))))
                groups.append(-1)
                plen.append(0)
                continue
            n, p = rng.randint(1, 8), rng.choice((1, rng.randint(2, 1023),
                                                  rng.randint(1024, 60000)))
            for _ in range(n):
                seq.append(p + rng.choice((0, 1, rng.randint(2, 5000))))
                groups.append(g)
                plen.append(p)
            g += 1
        info, pre, rest = _prefix_plan(len(seq), heads, seq, groups, plen,
                                       ctas_per_sm=rng.choice((1, 2)))
        _check_prefix_cover(seq, groups, plen, info, pre, rest)
        for (b0, unit, *_rest) in pre:
            assert unit <= 64 // heads and plen[b0] >= 1024


@pytest.mark.parametrize("prefix", [1, 64, 500, 1023])
def test_short_shared_prefix_is_not_grouped(L, prefix):
    # the grouped items run on the tensor-memory kernel, whose one-part P is
    # kept to long items: a short prefix is read by each request itself
    seq = [prefix + 300, prefix + 300, prefix + 7, prefix]
    groups, plen = [0] * 4, [prefix] * 4
    for heads in (16, 64):
        info, pre, rest = _prefix_plan(4, heads, seq, groups, plen)
        assert info["num_prefix_items"] == 0 and not pre
        assert info["variant"] == 3   # mma.sync with its two-part P
        _check_prefix_cover(seq, groups, plen, info, pre, rest)


def test_shared_prefix_private_variant(L):
    # long prefixes, short private tails: the grouped prefix items go to the
    # tensor-memory kernel and the tails to the mma.sync kernel
    info, pre, rest = _prefix_plan(2, 64, [5000, 5000], [0, 0], [4990, 4990])
    assert info["num_prefix_items"] > 0 and info["variant"] == 3
    info, pre, rest = _prefix_plan(2, 64, [9000, 9000], [0, 0], [4000, 4000])
    assert info["num_prefix_items"] > 0 and info["variant"] == 4
    with pytest.raises(_lib.PkvdError) as e:   # a forced tensor-memory tail that is too short
        _prefix_plan(2, 64, [5000, 5000], [0, 0], [4990, 4990], variant="mla_tc")
    assert e.value.code == _lib.PKVD_EUNSUPPORTED


def test_shared_prefix_units_of_four_requests(L):
    info, pre, rest = _prefix_plan(8, 16, [68000] * 8, [0] * 8, [63240] * 8)
    units = {(b0, u) for (b0, u, *_) in pre}
    assert units == {(0, 4), (4, 4)}
    info, pre, _ = _prefix_plan(2, 32, [5000] * 2, [0] * 2, [4000] * 2)
    assert {(b0, u) for (b0, u, *_) in pre} == {(0, 2)}


@pytest.mark.parametrize("heads,groups,plen,seq,code", [
    (16, [0, 1, 0], [10] * 3, [20] * 3, _lib.PKVD_EINVAL),        # members not consecutive
    (16, [0, 0], [10, 11], [20, 20], _lib.PKVD_EINVAL),           # prefix lengths differ
    (16, [0, 0], [21, 21], [20, 20], _lib.PKVD_EINVAL),           # longer than the request
    (16, [0, 0], [0, 0], [20, 20], _lib.PKVD_EINVAL),             # empty prefix in a group
    (128, [0, 0], [10, 10], [20, 20], _lib.PKVD_EUNSUPPORTED),    # 128 heads exceed 64 rows
    (48, [0, 0], [10, 10], [20, 20], _lib.PKVD_EUNSUPPORTED),     # 48 does not divide 64
])
def test_shared_prefix_errors(L, heads, groups, plen, seq, code):
    with pytest.raises(_lib.PkvdError) as e:
        _prefix_plan(len(seq), heads, seq, groups, plen)
    assert e.value.code == code


def test_shared_prefix_needs_mla(L):
    from paged_kv_cache_plan_gb300 import decode_plan_prefix_compute
    with pytest.raises(_lib.PkvdError) as e:
        decode_plan_prefix_compute(make_desc(2, 8, 2, 128, 16, num_sms=152, ctas_per_sm=1),
                                   [32, 32], [0, 0], [16, 16])
    assert e.value.code == _lib.PKVD_EUNSUPPORTED


def _merge_threads(max_splits, dv_slice):
    # one thread per float4 column (blocks of 32..128) for at most 8 splits,
    # else the 256-thread split-parallel merge
    if max_splits <= 8:
        return min(128, max(32, -(-(dv_slice // 4) // 32) * 32))
    return 256


@pytest.mark.parametrize("shape", [
    (1, 16, 2, 256, 16, [65536], {}),                 # many splits
    (1, 4, 1, 128, 16, [512], {"splits": 4}),         # few splits, sliced Dv
    (64, 128, 1, 576, 1, [16384] * 64, {}),           # few splits, untiled 512
    (10, 32, 8, 128, 16, [256, 512, 8192, 65536] + [1024] * 6, {}),
])
def test_merge_block_shape(L, shape):
    B, H, Hkv, D, ps, seq, kw = shape
    info, _ = _plan(B, H, Hkv, D, ps, seq=seq, **kw)
    dv = 512 if D == 576 else D
    assert info["stage2_threads"] == _merge_threads(info["max_splits"], dv // info["stage2_tiles"])


def test_merge_block_shape_follows_prefix_splits(L):
    # the prefix splits raise the per-request split count after the private
    # tokens were planned; the merge shape must follow the final count
    for B, seq, plen in ((8, [68000] * 8, [63240] * 8), (2, [3000, 3000], [2900, 2900])):
        info, _, _ = _prefix_plan(B, 16, seq, [0] * B, plen)
        assert info["stage2_threads"] == _merge_threads(info["max_splits"],
                                                        512 // info["stage2_tiles"])


# ---------------------------------------------------------------- several query tokens

@pytest.mark.parametrize("args,seq,kw,code", [
    ((2, 8, 2, 128, 16), [100, 2], dict(q_len=3), _lib.PKVD_EINVAL),     # L < q_len
    ((1, 8, 2, 128, 16), [100], dict(q_len=-1), _lib.PKVD_EINVAL),
    ((1, 8, 2, 128, 16), [100], dict(q_len=9), _lib.PKVD_EUNSUPPORTED),  # over 8 tokens
    ((1, 16, 2, 128, 16), [100], dict(q_len=3), _lib.PKVD_EUNSUPPORTED), # 3 x group 8 > 16
    ((1, 8, 2, 128, 16), [100], dict(q_len=2, variant="gqa_fma"), _lib.PKVD_EUNSUPPORTED),
    ((1, 16, 1, 576, 1), [1000], dict(q_len=2, variant="mla_tc"), _lib.PKVD_EUNSUPPORTED),
])
def test_query_token_errors(L, args, seq, kw, code):
    with pytest.raises(_lib.PkvdError) as e:
        _plan(*args, seq=seq, **kw)
    assert e.value.code == code


def test_query_tokens_layout(L):
    # GQA: an item covers q_len x group (token, head) rows of one KV head
    info, items = _plan(2, 8, 2, 128, 16, seq=[300, 0], q_len=2)
    assert info["heads_per_unit"] == 8 and info["units_per_request"] == 2
    assert all(it[6] == 300 - 2 for it in _items_full(L, (2, 8, 2, 128, 16), [300, 0], q_len=2))
    # MLA: 16 heads x 4 tokens fill a 64-row tensor-memory item on long contexts
    info, _ = _plan(3, 16, 1, 576, 1, seq=[4096] * 3, q_len=4)
    assert info["variant"] == 4 and info["heads_per_unit"] == 64
    assert info["units_per_request"] == 1
    # 16 heads x 2 tokens: 32 rows, one zero-padded 64-row unit
    info, _ = _plan(3, 16, 1, 576, 1, seq=[4096] * 3, q_len=2)
    assert info["variant"] == 4 and info["units_per_request"] == 1
    # short contexts: the mma.sync kernel's 16-row units
    info, _ = _plan(3, 16, 1, 576, 1, seq=[900] * 3, q_len=2)
    assert info["variant"] == 3 and info["units_per_request"] == 2
    # the merge runs over batch x q_len x heads rows: 1 x 4 x 16 = 64 rows tile 2 ways
    info, _ = _plan(1, 16, 1, 576, 1, seq=[68000], q_len=4)
    assert info["stage2_tiles"] == 2
    # no shared-prefix plans with several query tokens
    from paged_kv_cache_plan_gb300 import decode_plan_prefix_compute
    with pytest.raises(_lib.PkvdError) as e:
        decode_plan_prefix_compute(make_desc(2, 16, 1, 576, 1, num_sms=152, ctas_per_sm=2,
                                             q_len=2), [3000, 3000], [0, 0], [2000, 2000])
    assert e.value.code == _lib.PKVD_EUNSUPPORTED


def _items_full(L, args, seq, **kw):
    # every field of the work items, query_pos included
    import ctypes
    desc = make_desc(*args, num_sms=152, ctas_per_sm=1, **kw)
    info = _lib.PlanInfo()
    arr = (_lib.WorkItem * 4096)()
    s = (ctypes.c_int32 * len(seq))(*seq)
    rc = L.decode_plan_compute(ctypes.byref(desc), ctypes.cast(s, ctypes.c_void_p),
                               ctypes.byref(info), ctypes.cast(arr, ctypes.c_void_p), 4096)
    assert rc == 0
    return [(w.request, w.unit, w.split, w.partial_row, w.tok_begin, w.tok_end, w.query_pos)
            for w in arr[:info.num_items]]


def test_prefill_and_selftest_argument_errors(L):
    # argument checks happen before any CUDA call, so they run here too
    import ctypes
    d = _lib.PrefillDesc()
    d.batch, d.heads, d.kv_heads, d.seq_len, d.dtype = 1, 4, 2, 128, _lib.PKVD_BF16
    buf = (ctypes.c_uint8 * 64)()
    p = ctypes.cast(buf, ctypes.c_void_p)
    aligned = ctypes.c_void_p((p.value + 15) // 16 * 16)
    ptrs = [aligned] * 6
    assert L.prefill_d64_run(None, *ptrs, None) == _lib.PKVD_EINVAL
    assert L.prefill_d64_run(ctypes.byref(d), None, *ptrs[1:], None) == _lib.PKVD_EINVAL
    for field, bad in (("seq_len", 0), ("batch", 0), ("dtype", 7)):
        e = _lib.PrefillDesc.from_buffer_copy(d)
        setattr(e, field, bad)
        assert L.prefill_d64_run(ctypes.byref(e), *ptrs, None) == _lib.PKVD_EINVAL
    e = _lib.PrefillDesc.from_buffer_copy(d)
    e.kv_heads = 3
    assert L.prefill_d64_run(ctypes.byref(e), *ptrs, None) == _lib.PKVD_EUNSUPPORTED
    misaligned = ctypes.c_void_p(aligned.value + 4)
    assert L.prefill_d64_run(ctypes.byref(d), misaligned, *ptrs[1:], None) == _lib.PKVD_EINVAL
    assert L.decode_selftest_wait_timeout(None, 1000, None) == _lib.PKVD_EINVAL
    assert L.decode_selftest_wait_timeout(aligned, 0, None) == _lib.PKVD_EINVAL


def test_query_token_plans_cover_every_token_once(L):
    for args, seq, q in (((3, 8, 2, 128, 16), [300, 5, 4099], 3),
                         ((2, 16, 1, 576, 1), [2000, 70], 4)):
        info, items = _plan(*args, seq=seq, q_len=q)
        _check_cover(info, items, seq, info["units_per_request"])


def _random_case(rng):
    # one seeded planner case inside the documented domain: GQA (head_dim 128
    # or 256, q_len * group <= 16) or MLA shape, a length mix with empty and
    # one-token requests (every non-empty request holds its q_len queries),
    # auto or forced splits, any grid order
    batch = rng.randint(1, 12)
    if rng.random() < 0.5:
        kv = rng.choice((1, 2, 4, 8))
        group = rng.choice((1, 2, 4, 8, 16))
        args = (batch, kv * group, kv, rng.choice((128, 256)), rng.choice((1, 16, 64)))
        q_len = rng.randint(1, min(4, 16 // group))
    else:
        args = (batch, rng.choice((16, 32, 48, 64, 128)), 1, 576, rng.choice((1, 64)))
        q_len = rng.randint(1, 4)
    seq = [rng.choice((0, q_len, rng.randint(2, 300), rng.randint(300, 20000),
                       rng.randint(20000, 140000))) for _ in range(batch)]
    seq = [L and max(L, q_len) for L in seq]
    kw = dict(q_len=q_len, grid_order=rng.choice(("auto", "split_major", "request_major")),
              ctas_per_sm=rng.choice((1, 2)))
    if rng.random() < 0.4:
        kw["splits"] = rng.randint(1, 300)
    return args, seq, kw


def test_random_plans_cover_every_token_once(L):
    import random
    rng = random.Random(20261202)
    checked = 0
    for _ in range(300):
        args, seq, kw = _random_case(rng)
        if not any(seq):
            continue
        info, items = _plan(*args, seq=seq, **kw)
        assert info["num_items"] == len(items)
        _check_cover(info, items, seq, info["units_per_request"])
        # the split count of a request never exceeds what was asked or its tokens
        per = {}
        for (b, u, s, *_rest) in items:
            per[(b, u)] = max(per.get((b, u), 0), s + 1)
        assert max(per.values()) == info["max_splits"]
        for (b, u), n in per.items():
            assert n <= seq[b]
            if "splits" in kw:
                assert n <= kw["splits"]
        checked += 1
    assert checked > 250


def test_random_refusals_follow_the_documented_domain(L):
    import random
    rng = random.Random(7)
    for _ in range(100):
        args, seq, kw = _random_case(rng)
        q = kw["q_len"] = rng.randint(2, 8)
        # argument checks (lengths) come before the shape checks
        if any(0 < L < q for L in seq):
            code = _lib.PKVD_EINVAL             # a request shorter than its queries
        elif args[3] != 576 and q * (args[1] // args[2]) > 16:
            code = _lib.PKVD_EUNSUPPORTED       # more query rows than one 16-row tile
        else:
            _plan(*args, seq=seq, **kw)
            continue
        with pytest.raises(_lib.PkvdError) as e:
            _plan(*args, seq=seq, **kw)
        assert e.value.code == code, (args, seq, kw)
