"""Pins for the fp64 oracle: each test checks it against something other than
itself -- a hand-worked example, a closed form, brute force with an explicit
K+1 score column, a library attention routine, or a layout invariant -- so
that a dropped term, a wrong sign or index, or a transposed operand in the
oracle fails at least one of them.

Sources: GPT-OSS 20B model files (README "Attention sinks"; src/attention.linnet,
SinkAttention.decode_rows and the grouping of sink_attention by kv head);
Mistral 7B Instruct v0.3 model files (README "Entries", decode_paged;
src/attention.linnet, GroupedQueryAttention.decode_paged).
"""
import json
import math
import os

import numpy as np
import pytest
import scipy.special
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bf16_from(values) -> np.ndarray:
    """uint16 bit patterns of float values that are exactly representable in bf16."""
    t = torch.tensor(values, dtype=torch.float32)
    b = t.to(torch.bfloat16)
    assert torch.equal(b.float(), t), "fixture value not exact in bf16"
    return b.view(torch.int16).numpy().view(np.uint16)


def rand_bf16(gen, *shape, std=1.0):
    t = (torch.randn(*shape, generator=gen, dtype=torch.float32) * std).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def as_float(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _eval(expr: str) -> float:
    return float(eval(expr, {"__builtins__": {}}, {"e": math.e, "log": math.log, "exp": math.exp}))


# ---------------------------------------------------------------------------
# Worked examples (tests/golden)


def test_golden_sink_softmax_worked():
    g = json.load(open(os.path.join(GOLDEN, "sink_softmax_worked.json")))
    n = g["position"]
    q = bf16_from(g["q"]).reshape(1, 1, g["head_dim"])
    k = bf16_from(g["k"]).reshape(1, 1, n + 1, g["head_dim"])
    v = bf16_from(g["v"]).reshape(1, 1, n + 1, g["head_dim"])
    pos = np.array([n], dtype=np.int32)
    sinks = np.array([g["sink"]], dtype=np.float32)
    for case in g["cases"]:
        out, lse, lse_real = oracle.decode_rows(q, k, v, pos, sinks, window=case["window"],
                                                scale=g["scale"])
        want = np.array([_eval(x) for x in case["out"]])
        np.testing.assert_allclose(out[0, 0], want, rtol=1e-14, atol=1e-15)
        assert lse[0, 0] == pytest.approx(_eval(case["lse"]), rel=1e-14)
        assert lse_real[0, 0] == pytest.approx(_eval(case["lse_real"]), rel=1e-14)


def test_golden_page_slots_worked():
    g = json.load(open(os.path.join(GOLDEN, "page_slots_worked.json")))
    table = np.array(g["table"], dtype=np.int32)
    for case in g["cases"]:
        got = oracle.page_slots(table, np.array(case["positions"], dtype=np.int32),
                                g["page_size"], g["num_pages"])
        want = [int(_eval(x)) for x in case["slots"]]
        assert got.tolist() == want


def test_page_slots_rejects_out_of_range():
    table = np.array([[3, 9]], dtype=np.int32)
    with pytest.raises(ValueError):   # listed page 9 is outside an 8-page pool
        oracle.page_slots(table, np.array([64], dtype=np.int32), 64, 8)
    with pytest.raises(ValueError):   # position beyond the table's two pages
        oracle.page_slots(table, np.array([128], dtype=np.int32), 64, 16)


# ---------------------------------------------------------------------------
# Brute force: an explicit K+1 score column, softmaxed and then dropped.


def brute_force_k_plus_one(q, k, v, n, window, scale, sink):
    """One head: concatenate the sink as an extra score, softmax over the
    K+1 entries with scipy, drop the sink's probability, weight V.  The mask
    is evaluated position by position from its definition."""
    qf, kf, vf = as_float(q), as_float(k), as_float(v)
    scores, kept = [], []
    for s in range(n + 1):
        seen = s <= n and (window <= 0 or s > n - window)
        if seen:
            scores.append(scale * float(np.dot(qf, kf[s])))
            kept.append(s)
    column = np.array(scores + [sink if sink is not None else -np.inf])
    p = scipy.special.softmax(column)
    return p[:-1] @ vf[kept]


@pytest.mark.parametrize("hq,hkv,d,n,window,with_sink", [
    (1, 1, 4, 0, 0, True),
    (2, 1, 4, 5, 0, True),
    (4, 2, 8, 19, 0, False),
    (6, 2, 4, 17, 5, True),
    (3, 3, 8, 9, 1, True),
    (4, 1, 6, 12, 13, True),
    (8, 2, 8, 20, 3, False),
])
def test_oracle_equals_k_plus_one_column(hq, hkv, d, n, window, with_sink):
    gen = torch.Generator().manual_seed(hq * 1000 + n * 10 + window)
    rows = 3
    q = rand_bf16(gen, rows, hq, d)
    k = rand_bf16(gen, rows, hkv, n + 1, d)
    v = rand_bf16(gen, rows, hkv, n + 1, d)
    positions = np.array([n, max(n - 3, 0), n // 2], dtype=np.int32)
    sinks = (torch.randn(hq, generator=gen) * 2).numpy().astype(np.float32) if with_sink else None
    scale = 0.375   # exact in fp32, the type of the scale argument
    out, _, _ = oracle.decode_rows(q, k, v, positions, sinks, window=window, scale=scale)
    group = hq // hkv
    for b in range(rows):
        for h in range(hq):
            want = brute_force_k_plus_one(q[b, h], k[b, h // group], v[b, h // group],
                                          int(positions[b]), window, scale,
                                          None if sinks is None else float(sinks[h]))
            np.testing.assert_allclose(out[b, h], want, rtol=1e-12, atol=1e-14)


# ---------------------------------------------------------------------------
# Library routine: without a sink the op is plain scaled dot-product attention
# with each kv head copied out to its query heads (the ungrouped form the
# grouped one must equal).


@pytest.mark.parametrize("hq,hkv,d,window", [(14, 2, 16, 0), (8, 8, 8, 0), (8, 2, 32, 7),
                                             (32, 8, 8, 0)])
def test_no_sink_equals_sdpa_with_replicated_kv(hq, hkv, d, window):
    gen = torch.Generator().manual_seed(7 + hq + d + window)
    rows, length = 4, 40
    q = rand_bf16(gen, rows, hq, d)
    k = rand_bf16(gen, rows, hkv, length, d)
    v = rand_bf16(gen, rows, hkv, length, d)
    positions = np.array([39, 0, 17, 25], dtype=np.int32)
    scale = float(np.float32(1.0 / math.sqrt(d)))   # the scale argument is fp32
    out, lse, lse_real = oracle.decode_rows(q, k, v, positions, None, window=window, scale=scale)
    group = hq // hkv
    qt = torch.from_numpy(as_float(q))
    kt = torch.from_numpy(as_float(k)).repeat_interleave(group, dim=1)
    vt = torch.from_numpy(as_float(v)).repeat_interleave(group, dim=1)
    for b in range(rows):
        n = int(positions[b])
        s = torch.arange(length)
        mask = s <= n
        if window > 0:
            mask &= s > n - window
        ref = torch.nn.functional.scaled_dot_product_attention(
            qt[b][:, None, :], kt[b], vt[b], attn_mask=mask[None, None, :], scale=scale)
        np.testing.assert_allclose(out[b], ref[:, 0, :].numpy(), rtol=1e-12, atol=1e-13)
        logits = (qt[b][:, None, :] @ kt[b].transpose(-1, -2))[:, 0, :] * scale
        ref_lse = torch.logsumexp(logits.masked_fill(~mask, -math.inf), dim=-1)
        np.testing.assert_allclose(lse_real[b], ref_lse.numpy(), rtol=1e-13)
        np.testing.assert_allclose(lse[b], ref_lse.numpy(), rtol=1e-13)


def test_sink_minus_infinity_is_no_sink():
    gen = torch.Generator().manual_seed(3)
    q = rand_bf16(gen, 2, 4, 8)
    k = rand_bf16(gen, 2, 2, 10, 8)
    v = rand_bf16(gen, 2, 2, 10, 8)
    pos = np.array([9, 4], dtype=np.int32)
    a = oracle.decode_rows(q, k, v, pos, None)[0]
    b = oracle.decode_rows(q, k, v, pos, np.full(4, -np.inf, dtype=np.float32))[0]
    np.testing.assert_array_equal(a, b)


# ---------------------------------------------------------------------------
# Closed forms.


def test_huge_sink_drives_output_to_zero():
    gen = torch.Generator().manual_seed(4)
    q = rand_bf16(gen, 2, 4, 16)
    k = rand_bf16(gen, 2, 2, 30, 16)
    v = rand_bf16(gen, 2, 2, 30, 16)
    pos = np.array([29, 3], dtype=np.int32)
    out, lse, _ = oracle.decode_rows(q, k, v, pos, np.full(4, 1e4, dtype=np.float32))
    assert np.all(np.isfinite(out))
    assert np.max(np.abs(out)) <= 1e-30
    np.testing.assert_allclose(lse, 1e4, rtol=1e-15)


def test_real_key_mass_is_logistic_of_sink_minus_lse():
    """With every value row equal to 1, out is the total probability on real
    keys, which must be 1 / (1 + exp(sink - lse_real)) (< 1 with a sink)."""
    gen = torch.Generator().manual_seed(5)
    hq, hkv, d, length = 8, 2, 16, 50
    q = rand_bf16(gen, 3, hq, d)
    k = rand_bf16(gen, 3, hkv, length, d)
    v = bf16_from(np.ones((3, hkv, length, d)))
    pos = np.array([49, 10, 0], dtype=np.int32)
    sinks = (torch.randn(hq, generator=gen) * 3).numpy().astype(np.float32)
    scale = 1.0 / math.sqrt(d)
    out, _, lse_real = oracle.decode_rows(q, k, v, pos, sinks, scale=scale)
    # lse_real from a library log-sum-exp over the scores of a library matmul
    qt = torch.from_numpy(as_float(q))
    kt = torch.from_numpy(as_float(k)).repeat_interleave(hq // hkv, dim=1)
    for b in range(3):
        n = int(pos[b])
        logits = (qt[b][:, None, :] @ kt[b, :, : n + 1].transpose(-1, -2))[:, 0, :] * scale
        ref_lse = torch.logsumexp(logits, dim=-1).numpy()
        np.testing.assert_allclose(lse_real[b], ref_lse, rtol=1e-13)
        mass = 1.0 / (1.0 + np.exp(sinks.astype(np.float64) - ref_lse))
        for h in range(hq):
            np.testing.assert_allclose(out[b, h], mass[h], rtol=1e-13)
        assert np.all(mass < 1.0)


def test_single_key_closed_form():
    """n = 0: one key, out = v0 / (1 + exp(sink - s0))."""
    gen = torch.Generator().manual_seed(6)
    d = 8
    q = rand_bf16(gen, 1, 2, d)
    k = rand_bf16(gen, 1, 1, 1, d)
    v = rand_bf16(gen, 1, 1, 1, d)
    sinks = np.array([0.5, -1.25], dtype=np.float32)
    scale = 0.25
    out, _, _ = oracle.decode_rows(q, k, v, np.array([0], dtype=np.int32), sinks, scale=scale)
    for h in range(2):
        s0 = scale * float(as_float(q[0, h]) @ as_float(k[0, 0, 0]))
        want = as_float(v[0, 0, 0]) / (1.0 + math.exp(float(sinks[h]) - s0))
        np.testing.assert_allclose(out[0, h], want, rtol=1e-14)


def test_equal_keys_closed_form():
    """All attended keys equal: every score is s, so out = mean(V over A) *
    |A| e^s / (|A| e^s + e^sink)."""
    gen = torch.Generator().manual_seed(8)
    d, length, n, window = 8, 40, 37, 11
    q = rand_bf16(gen, 1, 1, d)
    key = rand_bf16(gen, d)
    k = np.broadcast_to(key, (1, 1, length, d)).copy()
    v = rand_bf16(gen, 1, 1, length, d)
    sink = np.array([0.75], dtype=np.float32)
    scale = 0.5
    out, _, _ = oracle.decode_rows(q, k, v, np.array([n], dtype=np.int32), sink, window=window,
                                   scale=scale)
    s = scale * float(as_float(q[0, 0]) @ as_float(key))
    attended = as_float(v[0, 0, n - window + 1: n + 1])
    count = attended.shape[0]
    assert count == window
    want = attended.mean(axis=0) * count * math.exp(s) / (count * math.exp(s) + math.exp(0.75))
    np.testing.assert_allclose(out[0, 0], want, rtol=1e-13)


def test_window_one_keeps_only_the_new_token():
    gen = torch.Generator().manual_seed(9)
    d = 16
    q = rand_bf16(gen, 1, 1, d)
    k = rand_bf16(gen, 1, 1, 20, d)
    v = rand_bf16(gen, 1, 1, 20, d)
    sink = np.array([-0.25], dtype=np.float32)
    out, _, _ = oracle.decode_rows(q, k, v, np.array([19], dtype=np.int32), sink, window=1,
                                   scale=0.125)
    s = 0.125 * float(as_float(q[0, 0]) @ as_float(k[0, 0, 19]))
    want = as_float(v[0, 0, 19]) / (1.0 + math.exp(-0.25 - s))
    np.testing.assert_allclose(out[0, 0], want, rtol=1e-14)


@pytest.mark.parametrize("n", [0, 63, 64, 126, 127])
def test_window_at_least_context_is_full(n):
    gen = torch.Generator().manual_seed(10 + n)
    q = rand_bf16(gen, 1, 8, 16)
    k = rand_bf16(gen, 1, 1, 128, 16)
    v = rand_bf16(gen, 1, 1, 128, 16)
    sinks = torch.randn(8, generator=gen).numpy().astype(np.float32)
    pos = np.array([n], dtype=np.int32)
    full = oracle.decode_rows(q, k, v, pos, sinks, window=0)[0]
    for w in (n + 1, 128, 10_000):
        np.testing.assert_array_equal(oracle.decode_rows(q, k, v, pos, sinks, window=w)[0], full)
    if n > 0:
        narrower = oracle.decode_rows(q, k, v, pos, sinks, window=n)[0]
        assert not np.array_equal(narrower, full)


def test_inactive_row_is_zero():
    gen = torch.Generator().manual_seed(11)
    q = rand_bf16(gen, 2, 2, 8)
    k = rand_bf16(gen, 2, 1, 4, 8)
    v = rand_bf16(gen, 2, 1, 4, 8)
    out, lse, _ = oracle.decode_rows(q, k, v, np.array([-1, 3], dtype=np.int32), None)
    assert np.all(out[0] == 0.0) and np.all(np.isneginf(lse[0]))
    assert np.any(out[1] != 0.0)


# ---------------------------------------------------------------------------
# Layout invariants for the paged form.


def _contiguous_case(seed, rows, hq, hkv, d, length):
    gen = torch.Generator().manual_seed(seed)
    q = rand_bf16(gen, rows, hq, d)
    k = rand_bf16(gen, rows, hkv, length, d)
    v = rand_bf16(gen, rows, hkv, length, d)
    sinks = torch.randn(hq, generator=gen).numpy().astype(np.float32)
    return q, k, v, sinks


def _identity_page_major_pool(cache, page):
    """[R, Hkv, L, D] -> page-major pool where row b owns pages b*L/P ...
    (a pure reshape/transpose: no slot arithmetic)."""
    rows, hkv, length, d = cache.shape
    per_row = length // page
    tiles = cache.reshape(rows, hkv, per_row, page, d).transpose(0, 2, 1, 3, 4)
    return np.ascontiguousarray(tiles).reshape(-1), per_row


@pytest.mark.parametrize("window", [0, 50])
def test_paged_identity_table_equals_contiguous(window):
    rows, hq, hkv, d, page = 3, 8, 2, 16, 64
    length = 3 * page
    q, k, v, sinks = _contiguous_case(12, rows, hq, hkv, d, length)
    positions = np.array([191, 64, 5], dtype=np.int32)
    k_pool, per_row = _identity_page_major_pool(k, page)
    v_pool, _ = _identity_page_major_pool(v, page)
    table = np.arange(rows * per_row, dtype=np.int32).reshape(rows, per_row)
    want = oracle.decode_rows(q, k, v, positions, sinks, window=window)
    got = oracle.decode_paged(q, k_pool, v_pool, table, positions, kv_heads=hkv, page_size=page,
                              num_pages=rows * per_row, sinks=sinks, window=window)
    for a, b in zip(got, want):
        np.testing.assert_array_equal(a, b)


def test_paged_result_invariant_under_page_permutation_and_layout():
    """Relabelling the pool's pages by a permutation (moving the page tiles
    and rewriting the table) and switching to the head-major layout must not
    change any output."""
    rows, hq, hkv, d, page = 4, 6, 3, 8, 64
    length = 4 * page
    q, k, v, sinks = _contiguous_case(13, rows, hq, hkv, d, length)
    positions = np.array([255, 130, 63, 0], dtype=np.int32)
    k_pool, per_row = _identity_page_major_pool(k, page)
    v_pool, _ = _identity_page_major_pool(v, page)
    num_pages = rows * per_row
    table = np.arange(num_pages, dtype=np.int32).reshape(rows, per_row)
    base = oracle.decode_paged(q, k_pool, v_pool, table, positions, kv_heads=hkv,
                               page_size=page, num_pages=num_pages, sinks=sinks)

    perm = np.random.default_rng(0).permutation(num_pages)
    tile = hkv * page * d

    def relabel(pool):
        out = np.empty_like(pool)
        for old in range(num_pages):
            out[perm[old] * tile:(perm[old] + 1) * tile] = pool[old * tile:(old + 1) * tile]
        return out

    table_p = perm[table].astype(np.int32)
    k_p, v_p = relabel(k_pool), relabel(v_pool)
    got = oracle.decode_paged(q, k_p, v_p, table_p, positions, kv_heads=hkv, page_size=page,
                              num_pages=num_pages, sinks=sinks)
    for a, b in zip(got, base):
        np.testing.assert_array_equal(a, b)

    def head_major(pool):
        return np.ascontiguousarray(
            pool.reshape(num_pages, hkv, page, d).transpose(1, 0, 2, 3)).reshape(-1)

    got = oracle.decode_paged(q, head_major(k_p), head_major(v_p), table_p, positions,
                              kv_heads=hkv, page_size=page, num_pages=num_pages, sinks=sinks,
                              layout=oracle.HEAD_MAJOR)
    for a, b in zip(got, base):
        np.testing.assert_array_equal(a, b)


# ---------------------------------------------------------------------------
# Append (write_tokens at page_slots).


@pytest.mark.parametrize("layout", [oracle.PAGE_MAJOR, oracle.HEAD_MAJOR])
def test_append_token_by_token_rebuilds_the_cache(layout):
    """Appending positions 0..L-1 one call at a time into a pool whose pages
    are handed out in a shuffled order rebuilds exactly the contiguous cache
    (read back through the same shuffled order by reshaping, not by slot
    arithmetic)."""
    rows, hkv, d, page, pages_per_row = 2, 3, 8, 64, 3
    length = page * pages_per_row
    gen = torch.Generator().manual_seed(14)
    cache = rand_bf16(gen, rows, hkv, length, d)
    num_pages = rows * pages_per_row + 2
    order = np.random.default_rng(1).permutation(num_pages).astype(np.int32)
    table = order[: rows * pages_per_row].reshape(rows, pages_per_row)
    pool = np.zeros(num_pages * hkv * page * d, dtype=np.uint16)
    for n in range(length):
        positions = np.array([n, n], dtype=np.int32)
        slots = oracle.page_slots(table, positions, page, num_pages)
        oracle.write_tokens(pool, cache[:, :, n, :], slots, kv_heads=hkv, head_dim=d,
                            page_size=page, num_pages=num_pages, layout=layout)
    if layout == oracle.PAGE_MAJOR:
        tiles = pool.reshape(num_pages, hkv, page, d)
    else:
        tiles = pool.reshape(hkv, num_pages, page, d).transpose(1, 0, 2, 3)
    for b in range(rows):
        rebuilt = np.concatenate([tiles[p] for p in table[b]], axis=1)   # [Hkv, L, D]
        np.testing.assert_array_equal(rebuilt, cache[b])
    untouched = sorted(set(range(num_pages)) - set(table.reshape(-1).tolist()))
    for p in untouched:
        assert not tiles[p].any()


def test_append_skips_inactive_rows():
    pool = np.zeros(2 * 1 * 64 * 4, dtype=np.uint16)
    table = np.array([[0], [1]], dtype=np.int32)
    slots = oracle.page_slots(table, np.array([-1, 5], dtype=np.int32), 64, 2)
    assert slots[0] == -1
    kv = np.full((2, 1, 4), 0x3F80, dtype=np.uint16)
    oracle.write_tokens(pool, kv, slots, kv_heads=1, head_dim=4, page_size=64, num_pages=2)
    tiles = pool.reshape(2, 64, 4)
    assert not tiles[0].any()
    assert (tiles[1, 5] == 0x3F80).all() and tiles[1].sum() == 4 * 0x3F80


# ---------------------------------------------------------------------------
# Paged prefill: packed prompt tokens, each a decode step of its own row.


def _prefill_setup(seed, rows, hq, hkv, d, pages_per_row, page=64):
    """A pool built by pure reshape from contiguous per-row caches (row b owns
    pages b*k .. b*k+k-1, identity table)."""
    length = pages_per_row * page
    q_dummy, k, v, sinks = _contiguous_case(seed, rows, hq, hkv, d, length)
    k_pool, per_row = _identity_page_major_pool(k, page)
    v_pool, _ = _identity_page_major_pool(v, page)
    table = np.arange(rows * per_row, dtype=np.int32).reshape(rows, per_row)
    return k, v, sinks, k_pool, v_pool, table


def test_prefill_one_token_per_row_is_decode():
    rows, hq, hkv, d = 3, 8, 2, 16
    k, v, sinks, k_pool, v_pool, table = _prefill_setup(20, rows, hq, hkv, d, 3)
    gen = torch.Generator().manual_seed(21)
    q = rand_bf16(gen, rows, hq, d)
    positions = np.array([191, 70, 0], dtype=np.int32)
    geo = dict(kv_heads=hkv, page_size=64, num_pages=table.size, sinks=sinks, window=40)
    want = oracle.decode_paged(q, k_pool, v_pool, table, positions, **geo)
    got = oracle.prefill_paged(q, k_pool, v_pool, table, np.arange(rows, dtype=np.int32),
                               positions, **geo)
    for a, b in zip(got, want):
        np.testing.assert_array_equal(a, b)
    # tokens may name rows in any order; each follows its own row's pages
    perm = np.array([2, 0, 1], dtype=np.int32)
    got = oracle.prefill_paged(q[perm], k_pool, v_pool, table, perm, positions[perm], **geo)
    np.testing.assert_array_equal(got[0], want[0][perm])


@pytest.mark.parametrize("hq,hkv", [(8, 2), (4, 4)])
def test_prefill_whole_prompt_equals_causal_sdpa(hq, hkv):
    """A prompt of L tokens at positions 0..L-1 of one row, no sink and no
    window: plain causal attention, checked against the library routine
    with KV replicated per head."""
    d, L = 16, 150
    k, v, _, k_pool, v_pool, table = _prefill_setup(22, 1, hq, hkv, d, 3)
    gen = torch.Generator().manual_seed(23)
    q = rand_bf16(gen, L, hq, d)
    positions = np.arange(L, dtype=np.int32)
    scale = 0.25
    out, _, _ = oracle.prefill_paged(q, k_pool, v_pool, table, np.zeros(L, dtype=np.int32),
                                     positions, kv_heads=hkv, num_pages=table.size, scale=scale)
    qt = torch.from_numpy(as_float(q)).permute(1, 0, 2)                  # [Hq, L, D]
    kt = torch.from_numpy(as_float(k[0, :, :L])).repeat_interleave(hq // hkv, dim=0)
    vt = torch.from_numpy(as_float(v[0, :, :L])).repeat_interleave(hq // hkv, dim=0)
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, is_causal=True,
                                                           scale=scale)
    np.testing.assert_allclose(out, ref.permute(1, 0, 2).numpy(), rtol=1e-12, atol=1e-13)


def test_prefill_with_sink_and_window_equals_k_plus_one_column():
    rows, hq, hkv, d = 2, 6, 2, 8
    k, v, sinks, k_pool, v_pool, table = _prefill_setup(24, rows, hq, hkv, d, 2)
    gen = torch.Generator().manual_seed(25)
    tokens = 12
    q = rand_bf16(gen, tokens, hq, d)
    token_rows = np.array([0] * 6 + [1] * 6, dtype=np.int32)
    positions = np.array([60, 61, 62, 63, 64, 65, 0, 1, 2, 100, 101, 127], dtype=np.int32)
    window, scale = 5, 0.375
    out, _, _ = oracle.prefill_paged(q, k_pool, v_pool, table, token_rows, positions,
                                     kv_heads=hkv, num_pages=table.size, sinks=sinks,
                                     window=window, scale=scale)
    for p in range(tokens):
        r = token_rows[p]
        for h in range(hq):
            want = brute_force_k_plus_one(q[p, h], k[r, h // (hq // hkv)], v[r, h // (hq // hkv)],
                                          int(positions[p]), window, scale, float(sinks[h]))
            np.testing.assert_allclose(out[p, h], want, rtol=1e-12, atol=1e-14)


def test_prefill_in_chunks_equals_one_pass():
    """Writing a prompt's K/V and attending in two chunks gives the second
    chunk the same result as one pass over the whole prompt."""
    hq, hkv, d, L, cut = 4, 2, 8, 100, 37
    gen = torch.Generator().manual_seed(26)
    q = rand_bf16(gen, L, hq, d)
    kv_k = rand_bf16(gen, L, hkv, d)
    kv_v = rand_bf16(gen, L, hkv, d)
    num_pages = 4
    order = np.array([3, 0, 2, 1], dtype=np.int32)
    table = order[None, :2].copy()
    geo = dict(kv_heads=hkv, head_dim=d, page_size=64, num_pages=num_pages)

    def run(chunks):
        kp = np.zeros(num_pages * hkv * 64 * d, dtype=np.uint16)
        vp = np.zeros_like(kp)
        outs = []
        for lo, hi in chunks:
            pos = np.arange(lo, hi, dtype=np.int32)
            rows = np.zeros(hi - lo, dtype=np.int32)
            slots = np.array([table[0, s // 64] * 64 + s % 64 for s in pos], dtype=np.int64)
            oracle.write_tokens(kp, kv_k[lo:hi], slots, **geo)
            oracle.write_tokens(vp, kv_v[lo:hi], slots, **geo)
            outs.append(oracle.prefill_paged(q[lo:hi], kp, vp, table, rows, pos, kv_heads=hkv,
                                             num_pages=num_pages)[0])
        return np.concatenate(outs)

    np.testing.assert_array_equal(run([(0, cut), (cut, L)]), run([(0, L)]))


def test_prefill_rejects_rows_outside_the_table():
    k, v, sinks, k_pool, v_pool, table = _prefill_setup(27, 2, 4, 2, 8, 1)
    q = np.zeros((1, 4, 8), dtype=np.uint16)
    with pytest.raises(ValueError):
        oracle.prefill_paged(q, k_pool, v_pool, table, np.array([2], dtype=np.int32),
                             np.array([3], dtype=np.int32), kv_heads=2, num_pages=table.size)


# ---------------------------------------------------------------------------
# Rotary embedding (rope_rows) at the pages' precision.


def _bf16_of(values: np.ndarray) -> np.ndarray:
    """Library rounding (torch) of float64 values to bf16 bit patterns."""
    t = torch.from_numpy(np.asarray(values, dtype=np.float64)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def test_rope_table_against_numpy_float32():
    """The tables: f32 inverse frequencies and angles as the pages compute
    them, cos/sin cast to bf16.  numpy float32 exp/log may differ from libm by
    an ulp, which moves a bf16 table value by at most one ulp, rarely."""
    d, theta = 128, 1e6
    i = np.arange(d // 2, dtype=np.float32)
    inv = np.exp(-(i * np.float32(2.0) / np.float32(d)) * np.log(np.float32(theta)))
    diffs, total = 0, 0
    for pos in (0, 1, 7, 63, 64, 1000, 4095, 32767):
        ang = (np.float32(pos) * inv).astype(np.float32)
        want_c = _bf16_of(np.cos(ang.astype(np.float64)))
        want_s = _bf16_of(np.sin(ang.astype(np.float64)))
        got_c, got_s = oracle.rope_table(d, theta, pos)
        for g, w in ((got_c, want_c), (got_s, want_s)):
            gf, wf = as_float(g), as_float(w)
            assert np.all(np.abs(gf - wf) <= 2.0 ** -7 * np.maximum(np.abs(wf), 2.0 ** -20))
            diffs += int(np.sum(g != w))
            total += g.size
    assert diffs <= total // 50
    c0, s0 = oracle.rope_table(d, theta, 0)
    assert np.all(as_float(c0) == 1.0) and np.all(as_float(s0) == 0.0)


def test_rope_is_complex_rotation_of_half_pairs():
    """Pairing dimension i with i + D/2 and rotating by the table angle is the
    complex product (x_i + j x_{i+D/2}) (cos_i + j sin_i), rounded to bf16."""
    gen = torch.Generator().manual_seed(30)
    n, heads, d, theta = 5, 3, 64, 1e6
    x = rand_bf16(gen, n, heads, d)
    pos = np.array([0, 1, 100, 4096, 30000], dtype=np.int32)
    out = oracle.rope(x, pos, theta)
    np.testing.assert_array_equal(out[0], x[0])          # position 0 is the identity
    for r in range(n):
        c, s = oracle.rope_table(d, theta, int(pos[r]))
        rot = as_float(c) + 1j * as_float(s)
        for h in range(heads):
            z = (as_float(x[r, h, : d // 2]) + 1j * as_float(x[r, h, d // 2:])) * rot
            np.testing.assert_array_equal(out[r, h, : d // 2], _bf16_of(z.real))
            np.testing.assert_array_equal(out[r, h, d // 2:], _bf16_of(z.imag))


def test_rope_inactive_rows_unchanged_and_rounding_matches_library():
    gen = torch.Generator().manual_seed(31)
    x = rand_bf16(gen, 2, 2, 16)
    out = oracle.rope(x, np.array([-1, 3], dtype=np.int32), 1e6)
    np.testing.assert_array_equal(out[0], x[0])
    # the oracle's RNE conversion equals torch's on awkward values (ties, tiny, huge)
    vals = np.array([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -1.5 - 2.0 ** -9, 3.0e38, 1e-40,
                     65504.5, 0.0, 2.0 ** -133])
    z = np.zeros((1, 1, 2 * len(vals)), dtype=np.uint16)
    assert _bf16_of(vals).dtype == np.uint16
    # a rotation by angle 0 returns the bf16 of the inputs; feed exact bf16 inputs and
    # check the values round-trip
    exact = _bf16_of(vals)
    z[0, 0, : len(vals)] = exact
    z[0, 0, len(vals):] = exact
    np.testing.assert_array_equal(oracle.rope(z, np.array([0], dtype=np.int32), 1e6), z)
