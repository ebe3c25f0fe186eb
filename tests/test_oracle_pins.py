"""Pins for the fp64 oracle: checks against things other than itself.

Each pin is a plain function of a mutation code (0 = the oracle as written).
The test-of-tests at the bottom plants each known mistake in the oracle (on
the CPU) and requires that at least one pin fails, the way the TensorFold
pull 1932 page ("Tests run") requires its score check to fail when the
folds run in the wrong order or a block is skipped.

What pins what:
  * decoders        -- every bf16 / fp16 bit pattern against torch / numpy
  * q = 0           -- output is the plain mean of the V rows, lse = ln L
  * one key         -- output is that V row, lse = scale * q.k
  * two keys        -- closed-form softmax of scores {c, c + 1}, also at c = 1024
  * library check   -- torch fp64 softmax(q K^T scale) V and logsumexp on the
                       rows gathered by tensor indexing of the [P, Hkv, ps, D]
                       layout, for GQA and for the MLA-shaped aliased rows
  * head groups     -- KV head kv serves query heads kv*g .. kv*g+g-1
  * relabelling     -- permuting physical pages changes nothing (bit-exact)
  * split + merge   -- any split of the tokens, merged, equals the one-shot
                       result (aiter pull 4758, Technical Details 3)
  * several query tokens -- token j of q_len equals a one-token decode of the
                       request cut to its first L - q_len + j + 1 tokens
                       (bit-exact), and torch fp64 with an explicit causal
                       mask on the gathered rows
"""
import math

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_plan_gb300 import workloads as W


def _P(case, mutation=0):
    return oracle.problem(**W.oracle_problem_kwargs(case), mutation=mutation)


def _decode(case, mutation=0, **kw):
    return oracle.decode(_P(case, mutation), case.q, case.k_pages, case.v_pages,
                         case.page_table, case.seq_lens, **kw)


def _rows(case, b, kv):
    """K and V rows of request b, KV head kv, in logical order, gathered by
    tensor indexing of the [P, Hkv, ps, pitch] layout (fp64)."""
    L = int(case.seq_lens[b])
    ks, vs = [], []
    for t in range(L):
        page = int(case.page_table[b, t // case.page_size])
        slot = t % case.page_size
        ks.append(case.k_pages[page, kv, slot, :case.head_dim].double())
        vs.append(case.v_pages[page, kv, slot, :case.head_dim_v].double())
    if not ks:
        return (torch.zeros(0, case.head_dim, dtype=torch.float64),
                torch.zeros(0, case.head_dim_v, dtype=torch.float64))
    return torch.stack(ks), torch.stack(vs)


def _small_gqa(seed=7, lens=(13, 7, 1), heads=4, kv_heads=2, d=8, ps=4, dtype="bf16",
               extra_pages=5):
    need = sum((L + ps - 1) // ps for L in lens)
    return W.gqa_case(batch=len(lens), heads=heads, kv_heads=kv_heads, head_dim=d,
                      page_size=ps, seq_lens=list(lens), pool_pages=need + extra_pages,
                      dtype=dtype, seed=seed)


def _small_mla(seed=11, batch=3, heads=4, seq_len=9, prefix=5):
    # MLA-shaped rows at a small width: one shared latent row, V aliases the
    # first head_dim_v elements of it, page size 1.
    c = W.mla_case(batch=batch, heads=heads, seq_len=seq_len, prefix_len=prefix,
                   group=2, pool_rows=64, seed=seed)
    # narrow the 576-wide row to 24 (16 + 8) so the pins stay tiny
    D, DV = 24, 16
    pool = c.k_pages[..., :D].contiguous()
    q = c.q[..., :D].contiguous()
    return W.DecodeCase("mla_small", q, pool, pool, c.page_table, c.seq_lens, heads, 1,
                        D, DV, 1, D, D, 1.0 / math.sqrt(D), "bf16", True, 0,
                        c.unique_rows)


# ----------------------------------------------------------------------------
# pins (each raises AssertionError when the oracle is wrong)

def pin_decoders(mutation=0):
    bits = np.arange(1 << 16, dtype=np.uint16)
    got_b = oracle.to_double(bits, "bf16")
    ref_b = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double().numpy()
    got_h = oracle.to_double(bits, "fp16")
    ref_h = bits.view(np.float16).astype(np.float64)
    for got, ref in ((got_b, ref_b), (got_h, ref_h)):
        nan = np.isnan(ref)
        assert np.array_equal(np.isnan(got), nan)
        assert np.array_equal(got[~nan], ref[~nan])


def pin_q_zero_mean(mutation=0):
    # Every V row of request b, KV head kv, token t holds a value that names
    # (t, kv, d) exactly in bf16; pool rows no request reads hold 1000.
    case = _small_gqa(seed=3, lens=(13, 7, 1, 16))
    case.q.zero_()
    case.v_pages.fill_(1000.0)
    for b in range(case.batch):
        L = int(case.seq_lens[b])
        for t in range(L):
            page = int(case.page_table[b, t // case.page_size])
            for kv in range(case.kv_heads):
                vals = torch.tensor([(t % 16) + 0.5 * kv + 0.25 * d + 8 * b
                                     for d in range(case.head_dim_v)])
                case.v_pages[page, kv, t % case.page_size] = vals.to(torch.bfloat16)
    out, lse = _decode(case, mutation)
    g = case.heads // case.kv_heads
    for b in range(case.batch):
        L = int(case.seq_lens[b])
        for h in range(case.heads):
            kv = h // g
            exp = [sum((t % 16) + 0.5 * kv + 0.25 * d + 8 * b for t in range(L)) / L
                   for d in range(case.head_dim_v)]
            np.testing.assert_allclose(out[b, h], exp, rtol=0, atol=1e-12)
            assert abs(lse[b, h] - math.log(L)) < 1e-12


def pin_single_key(mutation=0):
    case = _small_gqa(seed=5, lens=(1, 1), d=16)
    out, lse = _decode(case, mutation)
    g = case.heads // case.kv_heads
    for b in range(case.batch):
        for h in range(case.heads):
            k, v = _rows(case, b, h // g)
            qd = case.q[b, h].double()
            np.testing.assert_array_equal(out[b, h], v[0].numpy())
            exp_lse = case.scale * float(qd @ k[0])
            assert abs(lse[b, h] - exp_lse) < 1e-12


def pin_two_keys(mutation=0):
    # q = (a, 1, 0, 0), keys (c, 0, 0, 0) and (c, 1, 0, 0), scale 1: the
    # scores are a*c and a*c + 1 (all exact in bf16). a*c = 1024 overflows
    # exp() unless the maximum is taken out first.
    for a, c in ((0.0, 0.0), (2.0, 3.0), (32.0, 32.0)):
        case = W.gqa_case(batch=1, heads=1, kv_heads=1, head_dim=4, page_size=1,
                          seq_lens=[2], pool_pages=3, seed=1, scale=1.0)
        case.q.zero_()
        case.q[0, 0, 0] = a
        case.q[0, 0, 1] = 1.0
        pages = [int(case.page_table[0, t]) for t in range(2)]
        case.k_pages.zero_()
        case.k_pages[pages[0], 0, 0, 0] = c
        case.k_pages[pages[1], 0, 0, 0] = c
        case.k_pages[pages[1], 0, 0, 1] = 1.0
        v0 = case.v_pages[pages[0], 0, 0].double().numpy()
        v1 = case.v_pages[pages[1], 0, 0].double().numpy()
        out, lse = _decode(case, mutation)
        e = math.e
        np.testing.assert_allclose(out[0, 0], (v0 + e * v1) / (1 + e), rtol=0, atol=1e-12)
        assert abs(lse[0, 0] - (a * c + math.log(1 + e))) < 1e-12


def _torch_ref(case):
    g = case.heads // case.kv_heads
    out = np.zeros((case.batch, case.heads, case.head_dim_v))
    lse = np.zeros((case.batch, case.heads))
    for b in range(case.batch):
        for h in range(case.heads):
            k, v = _rows(case, b, h // g)
            if k.shape[0] == 0:
                lse[b, h] = -math.inf
                continue
            s = (k @ case.q[b, h].double()) * case.scale
            out[b, h] = (torch.softmax(s, dim=0) @ v).numpy()
            lse[b, h] = float(torch.logsumexp(s, dim=0))
    return out, lse


def pin_library_crosscheck(mutation=0):
    cases = [_small_gqa(seed=21, lens=(13, 7, 1, 0, 33), heads=8, kv_heads=2, d=16, ps=4),
             _small_gqa(seed=22, lens=(5, 17), heads=6, kv_heads=3, d=8, ps=3, dtype="fp16"),
             _small_mla()]
    for case in cases:
        out, lse = _decode(case, mutation)
        ref_o, ref_l = _torch_ref(case)
        np.testing.assert_allclose(out, ref_o, rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse, ref_l, rtol=0, atol=1e-12)


def pin_head_groups(mutation=0):
    case = _small_gqa(seed=9, lens=(6,), heads=6, kv_heads=3, d=8, ps=2, extra_pages=0)
    case.q.zero_()
    for kv in range(case.kv_heads):
        case.v_pages[:, kv] = float(kv + 1)
    out, _ = _decode(case, mutation)
    for h in range(case.heads):
        assert np.all(out[0, h] == float(h // 2 + 1))


def pin_relabelling(mutation=0):
    case = _small_gqa(seed=13, lens=(29, 3, 16), d=8, ps=4, extra_pages=9)
    o1, l1 = _decode(case, mutation)
    for s in (1, 2):
        o2, l2 = _decode(W.permute_pages(case, s), mutation)
        assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def pin_split_merge(mutation=0):
    case = _small_gqa(seed=17, lens=(37, 5), heads=4, kv_heads=1, d=8, ps=4)
    out, lse = _decode(case, mutation)
    P = _P(case, mutation)
    for b in range(case.batch):
        L = int(case.seq_lens[b])
        for cuts in ([L], [1, L], [4, 8, L], [L - 1, L] if L > 1 else [L],
                     list(range(1, L + 1)), [3, 3, 3, L, L]):
            cuts = sorted(min(c, L) for c in cuts)
            for h in range(case.heads):
                parts, lses, t0 = [], [], 0
                for t1 in cuts:
                    o, l = oracle.partial(P, case.q, case.k_pages, case.v_pages,
                                          case.page_table, case.seq_lens, b, h, t0, t1)
                    parts.append(o)
                    lses.append(l)
                    t0 = t1
                mo, ml = oracle.merge(np.stack(parts), np.array(lses), mutation)
                np.testing.assert_allclose(mo, out[b, h], rtol=0, atol=1e-12)
                assert abs(ml - lse[b, h]) < 1e-12


def pin_merge_closed_form(mutation=0):
    # two partials with lse 0 and ln 3 weigh 1/4 and 3/4; an empty split
    # (lse -inf) carries no weight; all-empty gives 0 and -inf.
    o = np.array([[1.0, 2.0], [5.0, -2.0], [np.nan, np.nan]])
    l = np.array([0.0, math.log(3.0), -math.inf])
    out, lse = oracle.merge(o[:2], l[:2], mutation)
    np.testing.assert_allclose(out, [4.0, -1.0], rtol=0, atol=1e-14)
    assert abs(lse - math.log(4.0)) < 1e-14
    out, lse = oracle.merge(np.zeros((2, 2)), np.array([-math.inf, -math.inf]), mutation)
    assert np.all(out == 0) and lse == -math.inf


def pin_empty_request(mutation=0):
    case = _small_gqa(seed=19, lens=(0, 4), d=8, ps=4)
    out, lse = _decode(case, mutation)
    assert np.all(out[0] == 0) and np.all(lse[0] == -math.inf)
    assert np.all(np.isfinite(lse[1]))


def pin_pairs_and_threads(mutation=0):
    case = _small_gqa(seed=23, lens=(13, 7, 1), heads=4, kv_heads=2, d=8, ps=4)
    out, lse = _decode(case, mutation)
    pairs = [(2, 3), (0, 0), (1, 2)]
    po, pl = _decode(case, mutation, pairs=pairs)
    for i, (b, h) in enumerate(pairs):
        assert np.array_equal(po[i], out[b, h]) and pl[i] == lse[b, h]
    to, tl = _decode(case, mutation, threads=3)
    assert np.array_equal(to, out) and np.array_equal(tl, lse)


def _truncated(case, j):
    """One-token problem of query token j: the requests cut to L - q_len + j + 1
    tokens (same pages), q = token j's rows."""
    lens = (case.seq_lens - case.q_len + j + 1).clamp(min=0).to(torch.int32)
    return W.DecodeCase(case.name + f"_tok{j}", case.q[:, j].contiguous(), case.k_pages,
                        case.v_pages, case.page_table, lens, case.heads, case.kv_heads,
                        case.head_dim, case.head_dim_v, case.page_size, case.k_row_pitch,
                        case.v_row_pitch, case.scale, case.dtype, case.mla, case.splits,
                        case.unique_rows, dict(case.meta), 1)


def _multi_token_cases():
    gqa = W.gqa_case(batch=3, heads=4, kv_heads=2, head_dim=8, page_size=4,
                     seq_lens=[13, 3, 9], pool_pages=12, seed=31, q_len=3)
    mla = W.mla_case(batch=2, heads=4, seq_len=7, prefix_len=4, group=2, pool_rows=40,
                     seed=33, q_len=4)
    D, DV = 24, 16   # narrowed rows, as in _small_mla
    pool = mla.k_pages[..., :D].contiguous()
    mla = W.DecodeCase("mla_small_q4", mla.q[..., :D].contiguous(), pool, pool,
                       mla.page_table, mla.seq_lens, 4, 1, D, DV, 1, D, D,
                       1.0 / math.sqrt(D), "bf16", True, 0, mla.unique_rows, {}, 4)
    return [gqa, mla]


def pin_multi_token_truncation(mutation=0):
    for case in _multi_token_cases():
        out, lse = _decode(case, mutation)
        H = case.heads
        assert out.shape == (case.batch, case.q_len * H, case.head_dim_v)
        for j in range(case.q_len):
            to, tl = _decode(_truncated(case, j), mutation)
            assert np.array_equal(out[:, j * H:(j + 1) * H], to)
            assert np.array_equal(lse[:, j * H:(j + 1) * H], tl)


def pin_multi_token_library(mutation=0):
    for case in _multi_token_cases():
        out, lse = _decode(case, mutation)
        g = case.heads // case.kv_heads
        for b in range(case.batch):
            L = int(case.seq_lens[b])
            for j in range(case.q_len):
                for h in range(case.heads):
                    k, v = _rows(case, b, h // g)
                    s = (k @ case.q[b, j, h].double()) * case.scale
                    s[L - case.q_len + j + 1:] = -math.inf     # causal within the tokens
                    vh = j * case.heads + h
                    np.testing.assert_allclose(out[b, vh], (torch.softmax(s, 0) @ v).numpy(),
                                               rtol=0, atol=1e-12)
                    assert abs(lse[b, vh] - float(torch.logsumexp(s, 0))) < 1e-12


def pin_multi_token_split_merge(mutation=0):
    # split partials of a query token's row, merged, equal its one-shot
    # result; a split past the token's own position is empty (lse -inf)
    case = _multi_token_cases()[0]
    out, lse = _decode(case, mutation)
    P = _P(case, mutation)
    H = case.heads
    for b in range(case.batch):
        L = int(case.seq_lens[b])
        for j in range(case.q_len):
            vh = j * H + (b % H)
            cuts = sorted({max(1, L // 3), max(1, L - 2), L})
            parts, lses, t0 = [], [], 0
            for t1 in cuts:
                o, l = oracle.partial(P, case.q, case.k_pages, case.v_pages, case.page_table,
                                      case.seq_lens, b, vh, t0, t1)
                if t0 > L - case.q_len + j:   # nothing here is visible to token j
                    assert l == -math.inf and np.all(o == 0)
                parts.append(o)
                lses.append(l)
                t0 = t1
            mo, ml = oracle.merge(np.stack(parts), np.array(lses), mutation)
            np.testing.assert_allclose(mo, out[b, vh], rtol=0, atol=1e-12)
            assert abs(ml - lse[b, vh]) < 1e-12


def pin_prefill_as_decode(mutation=0):
    # dense causal prefill = every token a query on one page per request:
    # torch fp64 softmax with the upper triangle masked, per (request, head)
    case = W.prefill_case(batch=2, heads=4, kv_heads=2, seq_len=23, seed=41)
    out, lse = _decode(case, mutation)
    q, k, v = case.q.double(), case.k_pages.double(), case.v_pages.double()
    B, L, H, D = q.shape
    g = H // case.kv_heads
    mask = torch.triu(torch.ones(L, L, dtype=torch.bool), 1)
    for b in range(B):
        for h in range(H):
            s = ((q[b, :, h] @ k[b, h // g].T) * case.scale).masked_fill(mask, -math.inf)
            got_o = out[b].reshape(L, H, D)[:, h]
            got_l = lse[b].reshape(L, H)[:, h]
            np.testing.assert_allclose(got_o, (torch.softmax(s, -1) @ v[b, h // g]).numpy(),
                                       rtol=0, atol=1e-12)
            np.testing.assert_allclose(got_l, torch.logsumexp(s, -1).numpy(), rtol=0, atol=1e-12)


PINS = [pin_decoders, pin_q_zero_mean, pin_single_key, pin_two_keys,
        pin_library_crosscheck, pin_head_groups, pin_relabelling, pin_split_merge,
        pin_merge_closed_form, pin_empty_request, pin_pairs_and_threads,
        pin_multi_token_truncation, pin_multi_token_library, pin_multi_token_split_merge,
        pin_prefill_as_decode]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin):
    pin(0)


@pytest.mark.parametrize("name", sorted(oracle.MUTATIONS))
def test_planted_mistake_is_caught(name):
    code = oracle.MUTATIONS[name]
    caught = []
    for pin in PINS:
        try:
            pin(code)
        except (AssertionError, FloatingPointError, RuntimeError):
            caught.append(pin.__name__)
    assert caught, f"no pin catches the planted mistake {name}"
