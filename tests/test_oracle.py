"""Pins for the CPU oracle (no GPU).

Each test checks the oracle against something other than itself: a library
routine (torch's fp64 scaled_dot_product_attention, torch's e4m3 decoder),
closed forms, hand-counted values from tests/golden/, invariances the
problem statement fixes (page permutation, HND vs NHD, chunking, GQA vs
repeated kv heads), and brute force on tiny inputs.  A last group plants
mistakes in a copy of oracle.c and checks that the pins catch them.
"""
import json
import math
import os
import re
import subprocess
import tempfile

import numpy as np
import pytest
import torch

import oracle
import workload

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- helpers

def _kv_index(inp, b, t):
    """(page, slot) of logical token t of request b, by torch indexing."""
    P = inp.page_size
    return int(inp.block_tables[b, t // P]), t % P


def _gather_torch(inp, pool, b):
    """[kv_len, Hkv, D] float64 of request b, via torch advanced indexing."""
    kv = int(inp.seq_lens[b])
    P = inp.page_size
    t = torch.arange(kv)
    pages = inp.block_tables[b].long()[t // P]
    slots = t % P
    if inp.layout == "HND":
        x = pool[pages, :, slots, :]          # [kv, Hkv, D]
    else:
        x = pool[pages, slots, :, :]
    return x.to(torch.float64)


def _sdpa_reference(inp):
    """Output [T, H, D] float64 from torch's scaled_dot_product_attention.

    Masks are built with torch.ones().tril/triu (not from the oracle's
    formula); sinks enter as one extra key with K = 0, V = 0 and an additive
    logit equal to the sink.
    """
    T, H, D = inp.q.shape
    Hkv = inp.num_kv_heads
    G = H // Hkv
    out = torch.zeros((T, H, D), dtype=torch.float64)
    for b in range(inp.batch):
        q0, q1 = int(inp.cum_q[b]), int(inp.cum_q[b + 1])
        ql, kl = q1 - q0, int(inp.seq_lens[b])
        if ql == 0:
            continue
        K = _gather_torch(inp, inp.k_pool, b).repeat_interleave(G, dim=1)  # [kl, H, D]
        V = _gather_torch(inp, inp.v_pool, b).repeat_interleave(G, dim=1)
        Q = inp.q[q0:q1].to(torch.float64)                                  # [ql, H, D]
        allowed = torch.ones((ql, kl), dtype=torch.bool).tril(diagonal=kl - ql)
        if inp.window_left >= 0:
            allowed &= torch.ones((ql, kl), dtype=torch.bool).triu(diagonal=kl - ql - inp.window_left)
        add = torch.zeros((ql, kl), dtype=torch.float64).masked_fill(~allowed, float("-inf"))
        if inp.sinks is not None:
            K = torch.cat([K, torch.zeros((1, H, D), dtype=torch.float64)], 0)
            V = torch.cat([V, torch.zeros((1, H, D), dtype=torch.float64)], 0)
            add = add.unsqueeze(0).repeat(H, 1, 1)
            sink_col = inp.sinks.to(torch.float64).view(H, 1, 1).expand(H, ql, 1)
            add = torch.cat([add, sink_col], dim=2)
        o = torch.nn.functional.scaled_dot_product_attention(
            Q.transpose(0, 1), K.transpose(0, 1), V.transpose(0, 1), attn_mask=add, scale=inp.bmm1_scale
        )
        out[q0:q1] = o.transpose(0, 1) * inp.bmm2_scale
    return out


def _oracle_full(inp):
    out, st, _ = oracle.attention(inp)
    assert (st == 0).all()
    return out.reshape(inp.q.shape[0], inp.q.shape[1], inp.head_dim)


def _small(seed=0, **kw):
    args = dict(q_lens=[7, 1, 12, 5], kv_lens=[7, 9, 30, 5], num_heads=4, num_kv_heads=2,
                head_dim=16, page_size=4, seed=seed)
    args.update(kw)
    return workload.build(**args)


# ---------------------------------------------------------------- decoders

def test_e4m3_decoder_matches_torch_all_codes():
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float32).tolist()
    for c in range(256):
        v = oracle.e4m3_value(c)
        if math.isnan(ref[c]):
            assert math.isnan(v), c
        else:
            assert v == ref[c], (c, v, ref[c])


def test_bf16_decoder_matches_torch():
    g = torch.Generator().manual_seed(3)
    bits = torch.randint(0, 1 << 16, (4096,), generator=g, dtype=torch.int32)
    bits[:4] = torch.tensor([0, 0x8000, 0x3F80, 0xC2F7])
    ref = bits.to(torch.int16).view(torch.bfloat16).to(torch.float64).tolist()
    for b, r in zip(bits.tolist(), ref):
        v = oracle.bf16_value(b)
        assert (math.isnan(v) and math.isnan(r)) or v == r


# ---------------------------------------------------------------- library cross-check

@pytest.mark.parametrize("layout", ["HND", "NHD"])
@pytest.mark.parametrize("window", [-1, 0, 3, 11])
@pytest.mark.parametrize("sinks", [False, True])
def test_matches_torch_sdpa_fp64(layout, window, sinks):
    inp = _small(seed=11, layout=layout, window_left=window, with_sinks=sinks, bmm2_scale=0.75)
    ref = _sdpa_reference(inp)
    got = torch.from_numpy(_oracle_full(inp))
    assert torch.allclose(got, ref, rtol=0, atol=1e-12), (got - ref).abs().max()


def test_matches_torch_sdpa_fp8_kv():
    inp = _small(seed=5, kv_dtype="fp8_e4m3", with_sinks=True, window_left=6)
    ref = _sdpa_reference(inp)
    got = torch.from_numpy(_oracle_full(inp))
    assert torch.allclose(got, ref, rtol=0, atol=1e-12)


def test_matches_torch_sdpa_gqa8_d64():
    inp = workload.build([33, 17], [40, 17], 16, 2, 64, 16, "NHD", seed=9, with_sinks=True)
    ref = _sdpa_reference(inp)
    got = torch.from_numpy(_oracle_full(inp))
    assert torch.allclose(got, ref, rtol=0, atol=1e-12)


# ---------------------------------------------------------------- closed forms

def test_single_key_gives_bmm2_times_v():
    inp = workload.build([1], [1], 2, 1, 16, 4, seed=2, bmm2_scale=1.7)
    out = _oracle_full(inp)
    page = int(inp.block_tables[0, 0])
    v = inp.v_pool[page, 0, 0].to(torch.float64).numpy()
    for h in range(2):
        np.testing.assert_allclose(out[0, h], 1.7 * v, rtol=0, atol=1e-14)


def test_identical_v_rows_give_that_row():
    inp = _small(seed=4, bmm2_scale=0.5, with_sinks=False, window_left=5)
    row = torch.randn(16, generator=torch.Generator().manual_seed(1)).to(torch.bfloat16)
    inp.v_pool[:] = row
    out = _oracle_full(inp)
    np.testing.assert_allclose(out, np.broadcast_to(0.5 * row.double().numpy(), out.shape), rtol=0, atol=1e-13)


def test_zero_query_gives_mean_of_visible_values():
    # q = 0: every visible key has the same weight.  Request 0 has 3 cached
    # tokens and 2 queries: rows see keys 0..3 and 0..4.
    inp = workload.build([2], [5], 1, 1, 8, 2, seed=6)
    inp.q.zero_()
    out = _oracle_full(inp)
    V = _gather_torch(inp, inp.v_pool, 0)[:, 0]  # [5, 8]
    np.testing.assert_allclose(out[0, 0], V[:4].mean(0).numpy(), rtol=0, atol=1e-14)
    np.testing.assert_allclose(out[1, 0], V[:5].mean(0).numpy(), rtol=0, atol=1e-14)


def _visible_counts(inp, sink_value):
    """n per row from out0 = n / (n + e^sink) with q = 0 and V[..., 0] = 1."""
    o0 = _oracle_full(inp)[:, 0, 0]
    if sink_value is None:
        return o0
    e = math.exp(sink_value)
    return o0 * e / (1.0 - o0)


@pytest.mark.parametrize("window", [-1, 2, 0])
def test_visible_counts_match_hand_count(window):
    gold = json.load(open(os.path.join(GOLDEN, "tiny_visible_counts.json")))
    inp = workload.config(1)
    inp.window_left = window
    inp.q.zero_()
    inp.v_pool[..., 0] = 1.0
    inp.sinks = torch.full((inp.num_heads,), 0.25)
    n = _visible_counts(inp, 0.25)
    want = gold["visible_per_row"][f"window_{window}"]
    np.testing.assert_allclose(n, want, rtol=1e-12)
    assert round(sum(n)) == gold["visible_pairs_per_head"][f"window_{window}"]


def test_tiny_config_page_usage():
    gold = json.load(open(os.path.join(GOLDEN, "tiny_visible_counts.json")))
    inp = workload.config(1)
    used = [(k + inp.page_size - 1) // inp.page_size for k in inp.kv_lens]
    assert used == gold["pages_used"]
    assert inp.k_pool.shape[0] == 8
    ids = [int(inp.block_tables[b, c]) for b in range(2) for c in range(used[b])]
    assert len(set(ids)) == 4 and all(0 <= i < 8 for i in ids)


# ---------------------------------------------------------------- identities

def test_sinks_minus_inf_equals_no_sinks():
    a = _small(seed=8, with_sinks=True)
    a.sinks = torch.full_like(a.sinks, float("-inf"))
    b = _small(seed=8, with_sinks=False)
    np.testing.assert_array_equal(_oracle_full(a), _oracle_full(b))


def test_window_minus_one_equals_any_large_window():
    a = _small(seed=10, window_left=-1)
    ref = _oracle_full(a)
    for w in (29, 30, 1000):
        a.window_left = w
        np.testing.assert_array_equal(_oracle_full(a), ref)


def test_page_permutation_invariance():
    inp = _small(seed=12, with_sinks=True, window_left=7)
    ref = _oracle_full(inp)
    N = inp.k_pool.shape[0]
    perm = torch.randperm(N, generator=torch.Generator().manual_seed(99))
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(N)
    # new pool page perm[i] holds old page i
    k2 = torch.empty_like(inp.k_pool)
    v2 = torch.empty_like(inp.v_pool)
    k2[perm] = inp.k_pool
    v2[perm] = inp.v_pool
    inp.k_pool, inp.v_pool = k2, v2
    inp.block_tables = perm[inp.block_tables.long()].to(torch.int32)
    np.testing.assert_array_equal(_oracle_full(inp), ref)


def test_hnd_nhd_and_strided_views_agree():
    a = _small(seed=13, layout="HND", with_sinks=True)
    ref = _oracle_full(a)
    # NHD copy of the same pool
    b = _small(seed=13, layout="HND", with_sinks=True)
    b.layout = "NHD"
    b.k_pool = a.k_pool.permute(0, 2, 1, 3).contiguous()
    b.v_pool = a.v_pool.permute(0, 2, 1, 3).contiguous()
    np.testing.assert_array_equal(_oracle_full(b), ref)
    # HND-shaped view of token-major storage (TokenSpeed _get_kv_cache_permuted)
    c = _small(seed=13, layout="HND", with_sinks=True)
    c.k_pool = b.k_pool.permute(0, 2, 1, 3)
    c.v_pool = b.v_pool.permute(0, 2, 1, 3)
    assert not c.k_pool.is_contiguous()
    np.testing.assert_array_equal(_oracle_full(c), ref)


def test_chunk_rows_equal_tail_of_full_prefill():
    full = workload.build([20], [20], 4, 2, 16, 4, seed=14, with_sinks=True, window_left=9)
    ref = _oracle_full(full)
    chunk = workload.build([6], [20], 4, 2, 16, 4, seed=14, with_sinks=True, window_left=9)
    chunk.k_pool, chunk.v_pool, chunk.block_tables = full.k_pool, full.v_pool, full.block_tables
    chunk.sinks = full.sinks
    chunk.q = full.q[14:].clone()
    np.testing.assert_allclose(_oracle_full(chunk), ref[14:], rtol=0, atol=1e-12)


def test_gqa_equals_mha_with_repeated_kv_heads():
    g = _small(seed=15, with_sinks=True)
    ref = _oracle_full(g)
    m = _small(seed=15, with_sinks=True)
    m.k_pool = g.k_pool.repeat_interleave(2, dim=1).contiguous()
    m.v_pool = g.v_pool.repeat_interleave(2, dim=1).contiguous()
    np.testing.assert_array_equal(_oracle_full(m), ref)


def test_poison_outside_visible_range_changes_nothing():
    inp = _small(seed=16, window_left=4, with_sinks=True, table_pad="garbage", pool_factor=2.0)
    ref = _oracle_full(inp)
    # NaN every page slot that no request uses at a visible position
    P = inp.page_size
    used = set()
    for b in range(inp.batch):
        for t in range(int(inp.seq_lens[b])):
            used.add(_kv_index(inp, b, t))
    for pg in range(inp.k_pool.shape[0]):
        for sl in range(P):
            if (pg, sl) not in used:
                inp.k_pool[pg, :, sl] = float("nan")
                inp.v_pool[pg, :, sl] = float("nan")
    np.testing.assert_array_equal(_oracle_full(inp), ref)


# ---------------------------------------------------------------- gather

@pytest.mark.parametrize("layout", ["HND", "NHD"])
@pytest.mark.parametrize("dtype", ["bf16", "fp8_e4m3"])
def test_gather_matches_torch_indexing(layout, dtype):
    inp = _small(seed=17, layout=layout, kv_dtype=dtype, table_pad="garbage")
    for which, pool in (("k", inp.k_pool), ("v", inp.v_pool)):
        got, ok = oracle.gather(inp, which)
        assert ok
        for b in range(inp.batch):
            c0, kl = int(inp.cum_kv[b]), int(inp.seq_lens[b])
            t = torch.arange(kl)
            pages = inp.block_tables[b].long()[t // inp.page_size]
            slots = t % inp.page_size
            ref = pool[pages, :, slots] if layout == "HND" else pool[pages, slots]
            assert torch.equal(got[c0:c0 + kl].view(torch.uint8), ref.contiguous().view(torch.uint8))


def test_gather_flags_out_of_pool_ids():
    inp = _small(seed=18)
    inp.block_tables[0, 0] = inp.k_pool.shape[0] + 5
    _, ok = oracle.gather(inp, "k")
    assert not ok


# ---------------------------------------------------------------- ragged page table

def test_ragged_lengths_hand_cases():
    """kv length = (pages - 1) * P + last_page_len, 0 without pages, -1 if malformed."""
    ip = torch.tensor([0, 3, 4, 4, 6, 6, 7], dtype=torch.int32)
    last = torch.tensor([1, 4, 9, 0, 2, 5], dtype=torch.int32)
    assert oracle.ragged_lengths(ip, last, 4).tolist() == [9, 4, 0, -1, 0, -1]
    assert oracle.ragged_lengths(torch.tensor([0, 2, 1], dtype=torch.int32), torch.tensor([1, 1], dtype=torch.int32),
                                 4).tolist() == [5, -1]


@pytest.mark.parametrize("layout", ["HND", "NHD"])
@pytest.mark.parametrize("dtype", ["bf16", "fp8_e4m3"])
def test_gather_ragged_matches_torch_indexing(layout, dtype):
    """Token t of request b from page indices[indptr[b] + t // P], slot t % P,
    written out with torch advanced indexing."""
    inp = _small(seed=19, layout=layout, kv_dtype=dtype, table_pad="garbage")
    idx, ip, last = workload.ragged_page_table(inp)
    P = inp.page_size
    for which, pool in (("k", inp.k_pool), ("v", inp.v_pool)):
        got, ok = oracle.gather_ragged(inp, idx, ip, last, which)
        assert ok
        for b in range(inp.batch):
            n = int(ip[b + 1] - ip[b])
            kl = (n - 1) * P + int(last[b]) if n > 0 else 0
            c0 = int(inp.cum_kv[b])
            t = torch.arange(kl)
            pages = idx.long()[int(ip[b]) + t // P]
            ref = pool[pages, :, t % P] if layout == "HND" else pool[pages, t % P]
            assert torch.equal(got[c0:c0 + kl].view(torch.uint8), ref.contiguous().view(torch.uint8))


def test_ragged_table_describes_the_same_attention():
    """The ragged form of a batch's pages gives exactly the block-table form's output."""
    inp = _small(seed=20, window_left=5, with_sinks=True)
    idx, ip, last = workload.ragged_page_table(inp)
    a, st_a, _ = oracle.attention(inp)
    r, st_r, _ = oracle.attention_ragged(inp, idx, ip, last)
    assert (st_a == 0).all() and (st_r == 0).all()
    np.testing.assert_array_equal(a, r)


def test_gather_ragged_flags_bad_tables():
    inp = _small(seed=21)
    idx, ip, last = workload.ragged_page_table(inp)
    bad_last = last.clone()
    bad_last[0] = inp.page_size + 1
    assert not oracle.gather_ragged(inp, idx, ip, bad_last, "k")[1]
    bad_idx = idx.clone()
    bad_idx[0] = inp.k_pool.shape[0] + 3
    assert not oracle.gather_ragged(inp, bad_idx, ip, last, "k")[1]


# ---------------------------------------------------------------- work list

def _brute_items(inp, rows_per_tile, nqt, bn):
    """Every item by enumerating all visible (row, key) pairs."""
    items = []
    per = rows_per_tile * nqt
    for b in range(inp.batch):
        ql = int(inp.cum_q[b + 1] - inp.cum_q[b])
        kl = int(inp.seq_lens[b])
        if ql == 0:
            continue
        for it in range((ql + per - 1) // per):
            for hk in range(inp.num_kv_heads):
                tiles, qtiles = set(), set()
                for i in range(it * per, min(ql, (it + 1) * per)):
                    pos = kl - ql + i
                    for j in range(kl):
                        vis = j <= pos and (inp.window_left < 0 or j >= pos - inp.window_left)
                        if vis:
                            tiles.add(j // bn)
                            qtiles.add((i - it * per) // rows_per_tile)
                # the item computes every tile between its first and last
                span = max(tiles) - min(tiles) + 1
                items.append((b, hk, it, span * len(qtiles)))
    return items


@pytest.mark.parametrize("window", [-1, 0, 5, 40])
def test_worklist_costs_match_brute_force(window):
    inp = workload.build([1, 37, 64, 65, 3], [1, 100, 64, 200, 130], 8, 2, 16, 8, window_left=window, seed=19)
    for rpt, nqt, bn, cap in ((16, 2, 32, 1023), (8, 1, 16, 1023), (16, 2, 32, 3)):
        got = oracle.worklist(inp, rpt, nqt, bn, cap)
        brute = _brute_items(inp, rpt, nqt, bn)
        assert sorted(map(tuple, got.tolist())) == sorted(brute)
        # longest first (capped), ties in enumeration order
        keys = [(-min(c, cap), brute.index((b, h, i, c))) for b, h, i, c in got.tolist()]
        assert keys == sorted(keys)


def test_worklist_skips_invalid_requests():
    inp = workload.build([4, 4], [8, 8], 2, 1, 16, 4, seed=20)
    inp.seq_lens[1] = 2  # q_len 4 > kv_len 2
    got = oracle.worklist(inp, 8, 2, 16, 1023)
    assert set(got[:, 0].tolist()) == {0}


# ---------------------------------------------------------------- the K/V write before the attention

def _e4m3_codes_torch(x: torch.Tensor) -> torch.Tensor:
    """torch's binary32 -> e4m3 cast (round to nearest even), as raw codes."""
    return x.to(torch.float8_e4m3fn).view(torch.uint8)


def test_e4m3_encoder_round_trips_every_finite_code():
    for c in range(256):
        if c & 0x7F == 0x7F:  # the two NaN codes
            continue
        assert oracle.e4m3_encode(oracle.e4m3_value(c)) == c, hex(c)


def test_e4m3_encoder_breaks_ties_to_the_even_code():
    for c in range(0x7E):
        lo, hi = oracle.e4m3_value(c), oracle.e4m3_value(c + 1)
        mid = np.float32((lo + hi) / 2)  # exact: e4m3 values carry at most 4 significant bits
        assert float(mid) == (lo + hi) / 2
        even = c if c % 2 == 0 else c + 1
        assert oracle.e4m3_encode(float(mid)) == even, hex(c)
        assert oracle.e4m3_encode(-float(mid)) == 0x80 | even, hex(c)
        below = np.nextafter(mid, np.float32(-1.0))
        above = np.nextafter(mid, np.float32(1e9))
        assert oracle.e4m3_encode(float(below)) == c and oracle.e4m3_encode(float(above)) == c + 1, hex(c)


def test_e4m3_encoder_matches_torch_cast_in_range():
    g = torch.Generator().manual_seed(77)
    uniform = (torch.rand(20000, generator=g, dtype=torch.float64) * 2 - 1) * 448
    sign = torch.where(torch.rand(20000, generator=g) < 0.5, -1.0, 1.0).double()
    spread = torch.exp(torch.rand(20000, generator=g, dtype=torch.float64) * 25 - 19).clamp(max=448) * sign
    x = torch.cat([uniform, spread]).float()
    got = torch.tensor([oracle.e4m3_encode(v) for v in x.tolist()], dtype=torch.uint8)
    assert torch.equal(got, _e4m3_codes_torch(x))


def test_e4m3_encoder_saturates_at_448():
    for v in [448.0, 449.0, 463.0, 464.0, 465.0, 1.0e4, 3.0e38]:
        assert oracle.e4m3_encode(v) == 0x7E and oracle.e4m3_encode(-v) == 0xFE, v
    assert oracle.e4m3_encode(float("nan")) == 0x7F


def _append_case(layout, fp8, T=40, N=12, P=8, H=3, D=16, seed=5):
    g = torch.Generator().manual_seed(seed)
    shape = (N, H, P, D) if layout == "HND" else (N, P, H, D)
    if fp8:
        kp = torch.randint(0, 0x7E, shape, generator=g, dtype=torch.uint8).view(torch.float8_e4m3fn)
        vp = torch.randint(0x80, 0xFE, shape, generator=g, dtype=torch.uint8).view(torch.float8_e4m3fn)
    else:
        kp = torch.randn(shape, generator=g).to(torch.bfloat16)
        vp = torch.randn(shape, generator=g).to(torch.bfloat16)
    k_new = (torch.randn((T, H, D), generator=g) * 3).to(torch.bfloat16)
    v_new = (torch.randn((T, H, D), generator=g) * 2).to(torch.bfloat16)
    loc = torch.randperm(N * P, generator=g)[:T].to(torch.int32)
    return kp, vp, k_new, v_new, loc


def _written_by_indexing(pool, new, loc, layout, scale):
    """The pool after the write, by torch indexing (and torch's cast, after clamping to +-448)."""
    P = pool.shape[2] if layout == "HND" else pool.shape[1]
    fp8 = pool.dtype == torch.float8_e4m3fn
    out = pool.clone()
    view = out.view(torch.uint8) if fp8 else out
    for n, s in enumerate(loc.tolist()):
        if s < 0 or s >= pool.shape[0] * P:
            continue
        page, slot = s // P, s % P
        rows = new[n]
        if fp8:
            rows = _e4m3_codes_torch((rows.float() / torch.tensor(scale, dtype=torch.float32)).clamp(-448, 448))
        if layout == "HND":
            view[page, :, slot, :] = rows
        else:
            view[page, slot, :, :] = rows
    return out


def _same_bits(a, b):
    return torch.equal(a.view(torch.uint8), b.view(torch.uint8))


@pytest.mark.parametrize("layout", ["HND", "NHD"])
@pytest.mark.parametrize("fp8,scales", [(False, (1.0, 1.0)), (True, (0.02, 0.03)), (True, (0.013, 0.004))])
def test_append_matches_torch_indexing(layout, fp8, scales):
    # (0.013, 0.004): quotients up to ~900, so the saturation is exercised
    kp, vp, k_new, v_new, loc = _append_case(layout, fp8)
    want_k = _written_by_indexing(kp, k_new, loc, layout, scales[0])
    want_v = _written_by_indexing(vp, v_new, loc, layout, scales[1])
    assert oracle.append_kv(k_new, v_new, kp, vp, loc, scales[0], scales[1], layout) == 0
    assert _same_bits(kp, want_k) and _same_bits(vp, want_v)


def test_append_skips_slots_outside_the_pool():
    kp, vp, k_new, v_new, loc = _append_case("HND", False, T=10)
    loc[3] = -1
    loc[7] = kp.shape[0] * kp.shape[2]
    want_k = _written_by_indexing(kp, k_new, loc, "HND", 1.0)
    assert oracle.append_kv(k_new, v_new, kp, vp, loc, 1.0, 1.0, "HND") == 2
    assert _same_bits(kp, want_k)


@pytest.mark.parametrize("layout", ["HND", "NHD"])
def test_append_then_gather_returns_the_new_tokens(layout):
    # the new tokens of each request are its last q_len keys: positions prefix .. kv_len - 1
    inp = workload.build([5, 17, 1], [9, 40, 33], 4, 2, 16, 8, layout, seed=31)
    g = torch.Generator().manual_seed(32)
    T, H, D, P = inp.q.shape[0], inp.num_kv_heads, inp.head_dim, inp.page_size
    k_new = torch.randn((T, H, D), generator=g).to(torch.bfloat16)
    v_new = torch.randn((T, H, D), generator=g).to(torch.bfloat16)
    loc = []
    for b in range(inp.batch):
        q_len = int(inp.cum_q[b + 1] - inp.cum_q[b])
        kv = int(inp.seq_lens[b])
        for t in range(kv - q_len, kv):
            page, slot = _kv_index(inp, b, t)
            loc.append(page * P + slot)
    assert oracle.append_kv(k_new, v_new, inp.k_pool, inp.v_pool, torch.tensor(loc, dtype=torch.int32),
                            1.0, 1.0, layout) == 0
    for which, new in (("k", k_new), ("v", v_new)):
        rows, ok = oracle.gather(inp, which)
        assert ok
        for b in range(inp.batch):
            q0, q1 = int(inp.cum_q[b]), int(inp.cum_q[b + 1])
            kv0, kv = int(inp.cum_kv[b]), int(inp.seq_lens[b])
            assert torch.equal(rows[kv0 + kv - (q1 - q0):kv0 + kv], new[q0:q1])


# ---------------------------------------------------------------- planted mistakes

_MUTANTS = {
    # a dropped sink term
    "drop_sink": ("den += exp((double)sinks[h] - m);", "den += 0.0;"),
    # window one key too wide
    "window_off_by_one": ("pos - window_left > 0 ? pos - window_left : 0", "pos - window_left - 1 > 0 ? pos - window_left - 1 : 0"),
    # causal alignment to the start instead of the end
    "start_aligned": ("int64_t pos = kv_len - q_len + i;", "int64_t pos = i;"),
    # wrong GQA head mapping
    "head_map": ("int hk = h / G;", "int hk = h % Hkv;"),
    # transposed page slot
    "slot": ("return pool_offset(p, layout, page, head, t % P, d);", "return pool_offset(p, layout, page, head, (P - 1) - t % P, d);"),
    # layout confusion
    "layout": ("if (layout == OR_HND)\n        return page", "if (layout != OR_HND)\n        return page"),
    # bmm2 applied before normalisation twice
    "bmm2": ("o[d] = bmm2_scale * acc[d] / den;", "o[d] = acc[d] / den;"),
    # e4m3 bias
    "e4m3_bias": ("v = ldexp(1.0 + (double)m / 8.0, e - 7);", "v = ldexp(1.0 + (double)m / 8.0, e - 8);"),
    # e4m3 encoding: ties to the odd code
    "e4m3_ties_odd": ("((lo & 1) ? hi : lo)", "((lo & 1) ? lo : hi)"),
    # e4m3 encoding: NaN instead of saturation above 448
    "e4m3_overflow_nan": ("        return sign | 0x7E;", "        return sign | 0x7F;"),
    # the write: scale not applied
    "append_unscaled": ("float q = x / scale;", "float q = x;"),
    # the write: slot within the page mirrored
    "append_slot": ("int64_t page = loc / P, slot = loc % P;", "int64_t page = loc / P, slot = (P - 1) - loc % P;"),
    # ragged table: the last page counted as full
    "ragged_last_full": ("(int32_t)((pages - 1) * P + last)", "(int32_t)(pages * P)"),
    # ragged table: a request's pages taken from the next request's slice
    "ragged_slice": ("int32_t page = indices[indptr[b] + t / P];", "int32_t page = indices[indptr[b + 1] - 1 - t / P];"),
}


def _build_mutant(name, tmpdir):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "oracle.c")).read()
    old, new = _MUTANTS[name]
    assert old in src, name
    path = os.path.join(tmpdir, f"{name}.c")
    open(path, "w").write(src.replace(old, new))
    so = os.path.join(tmpdir, f"lib{name}.so")
    subprocess.run(["gcc", "-O1", "-fopenmp", "-shared", "-fPIC", "-std=c11", "-o", so, path, "-lm"], check=True)
    return so


def _pins_pass(lib_path):
    """Run a handful of pins against the library at lib_path; True if all hold."""
    import ctypes

    saved = oracle._lib
    try:
        oracle._lib = None
        lib = ctypes.CDLL(lib_path)
        lib.oracle_attention.restype = ctypes.c_int
        lib.oracle_gather.restype = ctypes.c_int
        lib.oracle_worklist.restype = ctypes.c_int
        lib.oracle_e4m3_value.restype = ctypes.c_double
        lib.oracle_e4m3_value.argtypes = [ctypes.c_uint8]
        lib.oracle_bf16_value.restype = ctypes.c_double
        lib.oracle_bf16_value.argtypes = [ctypes.c_uint16]
        lib.oracle_e4m3_encode.restype = ctypes.c_uint8
        lib.oracle_e4m3_encode.argtypes = [ctypes.c_float]
        lib.oracle_append_kv.restype = ctypes.c_int64
        lib.oracle_gather_ragged.restype = ctypes.c_int
        lib.oracle_ragged_lengths.restype = None
        oracle._lib = lib
        checks = [
            lambda: test_matches_torch_sdpa_fp64("HND", 3, True),
            lambda: test_matches_torch_sdpa_fp64("NHD", -1, False),
            lambda: test_matches_torch_sdpa_fp8_kv(),
            lambda: test_matches_torch_sdpa_gqa8_d64(),
            lambda: test_e4m3_decoder_matches_torch_all_codes(),
            lambda: test_e4m3_encoder_breaks_ties_to_the_even_code(),
            lambda: test_e4m3_encoder_saturates_at_448(),
            lambda: test_append_matches_torch_indexing("NHD", True, (0.013, 0.004)),
            lambda: test_append_then_gather_returns_the_new_tokens("HND"),
            lambda: test_ragged_lengths_hand_cases(),
            lambda: test_gather_ragged_matches_torch_indexing("NHD", "bf16"),
        ]
        for c in checks:
            try:
                c()
            except AssertionError:
                return False
        return True
    finally:
        oracle._lib = saved


def test_pins_accept_the_unmodified_oracle():
    assert _pins_pass(oracle.build())


@pytest.mark.parametrize("name", sorted(_MUTANTS))
def test_pins_catch_planted_mistake(name):
    with tempfile.TemporaryDirectory() as d:
        assert not _pins_pass(_build_mutant(name, d)), f"mutant {name} survived the pins"
