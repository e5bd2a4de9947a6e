"""GPU parity of the paired-SM prefill kernel (PGD_KERNEL_PREFILL_PAIR: head_dim
128, clusters of two CTAs sharing each tcgen05 product): against the oracle
on the prefill cases of the one-SM kernels -- group sizes, runs, windows,
sinks, both pool layouts, step_paged, padding blocks, bad entries, poisoned
slots, rescaling scores, the full Mistral-shaped prefill on sampled tokens --
and every output of the full Mistral-shaped prefill close to the one-SM
tcgen05 kernel's."""
import numpy as np
import pytest
import torch

import paged_gqa_decode_gb300 as pgd
from pgd_inputs import PREFILL_WORKLOADS, PrefillWorkload, make_prefill_batch
from tests.parity import compare
from tests.test_gpu_prefill import DEV, prefill_check

pytestmark = pytest.mark.gpu

PAIR = pgd.KERNEL_PREFILL_PAIR


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    yield
    torch.cuda.synchronize()


@pytest.mark.parametrize("hq,hkv,window,sinks", [(32, 8, 0, False), (16, 4, 65, True),
                                                 (8, 8, 0, True), (4, 2, 30, True),
                                                 (12, 4, 0, True), (10, 2, 1, True)])
@pytest.mark.parametrize("fused", [False, True])
def test_pair_small(hq, hkv, window, sinks, fused):
    """Group sizes 1-5 (blocks of 128 / G tokens per tile, 25 tokens and 125
    rows at G = 5), chunks starting on and off page boundaries, windows of 1,
    30 and 65 positions."""
    wl = PrefillWorkload("pair", rows=4, q_heads=hq, kv_heads=hkv, head_dim=128, prefix_lo=0,
                         prefix_hi=300, chunk=0, window=window, sinks=sinks)
    b = make_prefill_batch(wl, 41 + hq + window, DEV, prefix=[0, 63, 64, 200],
                           chunks=[1, 64, 100, 130])
    prefill_check(b, kernel=PAIR, fused=fused, what=f"pair {hq}/{hkv} w={window} fused={fused}")


@pytest.mark.parametrize("layout", [pgd.PAGE_MAJOR, pgd.HEAD_MAJOR])
def test_pair_long_prefix_both_layouts(layout):
    wl = PrefillWorkload("pair_long", rows=3, q_heads=16, kv_heads=4, head_dim=128, prefix_lo=0,
                         prefix_hi=3000, chunk=0, window=0, sinks=True)
    b = make_prefill_batch(wl, 43, DEV, prefix=[2000, 37, 1500], chunks=[70, 150, 9])
    prefill_check(b, layout=layout, kernel=PAIR, what=f"pair long layout={layout}")


def test_pair_interleaved_token_order():
    wl = PrefillWorkload("pair_mixed", rows=3, q_heads=8, kv_heads=2, head_dim=128, prefix_lo=0,
                         prefix_hi=300, chunk=0, window=100, sinks=True)
    b = make_prefill_batch(wl, 13, DEV, prefix=[0, 120, 250], chunks=[40, 40, 40])
    perm = np.random.default_rng(0).permutation(len(b.rows_np))
    t = torch.as_tensor(perm, device=DEV)
    b.rows_np, b.positions_np = b.rows_np[perm], b.positions_np[perm]
    b.rows, b.positions = b.rows[t].contiguous(), b.positions[t].contiguous()
    b.q, b.k_new, b.v_new = b.q[t].contiguous(), b.k_new[t].contiguous(), b.v_new[t].contiguous()
    prefill_check(b, kernel=PAIR, what="pair interleaved")


@pytest.mark.parametrize("fused", [False, True])
def test_pair_step_paged(fused):
    wl = PrefillWorkload("pair_step", rows=5, q_heads=32, kv_heads=8, head_dim=128, prefix_lo=0,
                         prefix_hi=2000, chunk=0, window=0, sinks=False)
    b = make_prefill_batch(wl, 14, DEV, prefix=[0, 900, 1500, 64, 1999],
                           chunks=[150, 70, 1, 1, 1])
    prefill_check(b, kernel=PAIR, fused=fused, what=f"pair step_paged fused={fused}")


@pytest.mark.parametrize("fused", [False, True])
def test_pair_full_size_sampled(fused):
    wl = PREFILL_WORKLOADS["mistral_prefill"]
    b = make_prefill_batch(wl, 2000, DEV)
    rng = np.random.default_rng(3)
    tokens = len(b.rows_np)
    idx = np.unique(np.concatenate([rng.choice(tokens, size=190, replace=False),
                                    [0, tokens - 1]]))
    prefill_check(b, sample=idx, kernel=PAIR, fused=fused, what="pair mistral_prefill")


@pytest.mark.parametrize("window", [0, 128])
def test_pair_close_to_the_one_sm_kernel_everywhere(window):
    """Every output of the full Mistral-shaped prefill against the one-SM
    tcgen05 kernel's (itself checked against the oracle), within the
    tolerance.  They are not bit-identical: the paired kernel takes its lazy
    running-max decisions per two pages."""
    wl = PREFILL_WORKLOADS["mistral_prefill"].replace(window=window)
    b = make_prefill_batch(wl, 2100 + window, DEV)
    kw = dict(num_kv_heads=wl.kv_heads)
    want = pgd.paged_prefill_attention(b.q, b.k_pool, b.v_pool, b.table, b.rows, b.positions,
                                       b.sinks, window, wl.scale, kernel=pgd.KERNEL_PREFILL_UMMA,
                                       **kw)
    got = pgd.paged_prefill_attention(b.q, b.k_pool, b.v_pool, b.table, b.rows, b.positions,
                                      b.sinks, window, wl.scale, kernel=PAIR, **kw)
    assert pgd.get_device_error() == pgd.OK
    compare(got, want.float().cpu().numpy().astype(np.float64), f"pair vs one-SM w={window}")


def test_pair_step_equals_the_three_calls():
    wl = PrefillWorkload("pair_fused", rows=4, q_heads=32, kv_heads=8, head_dim=128, prefix_lo=0,
                         prefix_hi=900, chunk=0, window=30, sinks=True)
    a = make_prefill_batch(wl, 59, DEV, prefix=[0, 700, 65, 300], chunks=[90, 140, 33, 64])
    b = make_prefill_batch(wl, 59, DEV, prefix=[0, 700, 65, 300], chunks=[90, 140, 33, 64])
    for x in (a, b):
        x.positions[7] = -1
    kw = dict(num_kv_heads=wl.kv_heads, layout=pgd.HEAD_MAJOR, kernel=PAIR)
    slots = pgd.page_slots(a.table, a.positions, a.rows, num_pages=a.num_pages)
    pgd.kv_write_slots(a.k_new, a.v_new, slots, a.k_pool, a.v_pool, layout=pgd.HEAD_MAJOR)
    want = pgd.paged_prefill_attention(a.q, a.k_pool, a.v_pool, a.table, a.rows, a.positions,
                                       a.sinks, wl.window, wl.scale, **kw)
    assert pgd.get_device_error() == pgd.OK
    got = pgd.paged_prefill_step(b.q, b.k_new, b.v_new, b.k_pool, b.v_pool, b.table, b.rows,
                                 b.positions, b.sinks, wl.window, wl.scale, **kw)
    assert pgd.get_device_error() == pgd.OK
    assert torch.equal(b.k_pool, a.k_pool) and torch.equal(b.v_pool, a.v_pool)
    assert torch.equal(got, want)
    assert torch.all(got[7] == 0)


def test_pair_bad_rows_and_pages_are_zero_and_reported():
    wl = PrefillWorkload("pair_bad", rows=2, q_heads=8, kv_heads=2, head_dim=128, prefix_lo=0,
                         prefix_hi=100, chunk=0)
    b = make_prefill_batch(wl, 15, DEV, prefix=[0, 50], chunks=[10, 10])
    rows = b.rows.clone()
    rows[3] = 7
    out = pgd.paged_prefill_attention(b.q, b.k_pool, b.v_pool, b.table, rows, b.positions,
                                      num_kv_heads=2, kernel=PAIR)
    assert pgd.get_device_error() == pgd.EDEVICE_BOUNDS
    assert torch.all(out[3] == 0) and torch.any(out[4] != 0)
    table = b.table.clone()
    table[1, 0] = 10 ** 6
    out = pgd.paged_prefill_attention(b.q, b.k_pool, b.v_pool, table, b.rows, b.positions,
                                      num_kv_heads=2, kernel=PAIR)
    assert pgd.get_device_error() == pgd.EDEVICE_BOUNDS
    assert torch.all(out[10:] == 0) and torch.any(out[:10] != 0)


def test_pair_poisoned_slots_outside_attention_are_never_read():
    wl = PrefillWorkload("pair_poison", rows=3, q_heads=16, kv_heads=4, head_dim=128, prefix_lo=0,
                         prefix_hi=600, chunk=0, window=90, sinks=True)
    b = make_prefill_batch(wl, 17, DEV, prefix=[10, 300, 523], chunks=[70, 33, 40])
    keep = np.zeros(b.num_pages * 64, dtype=bool)
    for r, n in zip(b.rows_np, b.positions_np):
        for s in range(max(0, int(n) - wl.window + 1), int(n) + 1):
            keep[b.table_np[r, s // 64] * 64 + s % 64] = True
    nan_slots = torch.from_numpy(~keep).to(DEV)
    for pool in (b.k_pool, b.v_pool):
        view = pool.view(b.num_pages, wl.kv_heads, 64, wl.head_dim)
        view.masked_fill_(nan_slots.view(b.num_pages, 1, 64, 1).expand_as(view), float("nan"))
    prefill_check(b, kernel=PAIR, what="pair poison")


def test_pair_large_logits():
    wl = PrefillWorkload("pair_large", rows=2, q_heads=32, kv_heads=8, head_dim=128, prefix_lo=0,
                         prefix_hi=2000, chunk=0, window=0, sinks=True)
    b = make_prefill_batch(wl, 18, DEV, prefix=[1900, 700], chunks=[96, 64])
    b.q = (b.q.float() * 6.0).to(torch.bfloat16)
    b.v_pool.mul_(0.5)
    b.v_new = b.v_new * 0.5
    prefill_check(b, kernel=PAIR, what="pair large logits")


@pytest.mark.parametrize("hq,hkv", [(16, 4), (8, 8)])
def test_pair_padding_tokens_fill_whole_blocks(hq, hkv):
    wl = PrefillWorkload("pair_pad", rows=3, q_heads=hq, kv_heads=hkv, head_dim=128, prefix_lo=0,
                         prefix_hi=900, chunk=0, window=0, sinks=True)
    b = make_prefill_batch(wl, 19 + hq, DEV, prefix=[300, 0, 777], chunks=[200, 190, 300])
    block = 128 // (hq // hkv)
    pad = np.zeros(len(b.rows_np), dtype=bool)
    pad[block:3 * block] = True
    pad[-(block + 5):] = True
    b.positions_np = np.where(pad, -1, b.positions_np).astype(np.int32)
    b.positions = torch.from_numpy(b.positions_np).to(DEV)
    prefill_check(b, kernel=PAIR, what=f"pair padding {hq}/{hkv}")
    out = pgd.paged_prefill_attention(b.q, b.k_pool, b.v_pool, b.table, b.rows, b.positions,
                                      b.sinks, 0, wl.scale, num_kv_heads=hkv, kernel=PAIR)
    assert pgd.get_device_error() == pgd.OK
    padded = torch.from_numpy(pad).to(DEV)
    assert torch.all(out[padded] == 0) and torch.all(out[~padded].abs().sum((1, 2)) > 0)


def test_pair_scores_far_below_zero():
    wl = PrefillWorkload("pair_negative", rows=2, q_heads=16, kv_heads=4, head_dim=128,
                         prefix_lo=0, prefix_hi=500, chunk=0, window=0, sinks=False)
    b = make_prefill_batch(wl, 155, DEV, prefix=[300, 0], chunks=[70, 90])
    b.q.fill_(-64.0)
    b.k_pool.fill_(2.0)
    b.k_new.fill_(2.0)
    prefill_check(b, sinks=None, kernel=PAIR, what="pair negative scores")


def test_pair_scores_rise_every_page():
    wl = PrefillWorkload("pair_rising", rows=2, q_heads=16, kv_heads=4, head_dim=128,
                         prefix_lo=0, prefix_hi=1500, chunk=0, window=0, sinks=True)
    b = make_prefill_batch(wl, 159, DEV, prefix=[1400, 200], chunks=[40, 64])
    step = 6.0
    b.q.fill_(0.25)
    view = b.k_pool.view(b.num_pages, wl.kv_heads, 64, 128)
    for r in range(2):
        n_pages = (int(b.positions_np[b.rows_np == r].max()) // 64) + 1
        for j in range(n_pages):
            view[int(b.table_np[r, j])] = step * j
    pages = torch.as_tensor(b.positions_np // 64, device=DEV, dtype=torch.float32)
    b.k_new = (pages.view(-1, 1, 1) * step).expand_as(b.k_new).to(torch.bfloat16).contiguous()
    prefill_check(b, kernel=PAIR, what="pair rising scores")


def test_pair_kernel_count_and_head_dim_64_refused():
    w = PREFILL_WORKLOADS["mistral_prefill"]
    dims = pgd.make_dims(rows=4096, num_q_heads=w.q_heads, num_kv_heads=w.kv_heads,
                         head_dim=w.head_dim, num_pages=10000, max_pages_per_row=140)
    assert pgd.prefill_step_kernel_count(dims, 8, kernel=PAIR) == 2
    assert pgd.attention_kernel_count(dims, 8, kernel=PAIR) == 2
    assert pgd.attention_kernel_count(dims, 8, window=128, kernel=PAIR) == 1
    d64 = pgd.make_dims(rows=64, num_q_heads=64, num_kv_heads=8, head_dim=64, num_pages=100,
                        max_pages_per_row=10)
    with pytest.raises(pgd.PgdError):
        pgd.attention_kernel_count(d64, 8, kernel=PAIR)


@pytest.mark.parametrize("rows,prefix,kernel", [(1, 0, PAIR), (2, None, pgd.KERNEL_PREFILL_UMMA),
                                                (8, None, pgd.KERNEL_PREFILL_UMMA)])
def test_auto_takes_the_pair_kernel_for_few_short_items(rows, prefix, kernel):
    """AUTO runs the paired kernel when blocks x kv heads are at most half
    the SM count and too short to cut into key parts (one 512-token
    Mistral-shaped chunk from position 0: 64 items of at most 8 pages), the
    one-SM kernel when they are more (two chunks: 128 items; eight: 512):
    its outputs equal that kernel's."""
    wl = PREFILL_WORKLOADS["mistral_prefill"].replace(rows=rows)
    b = make_prefill_batch(wl, 2200 + rows, DEV, prefix=None if prefix is None else [prefix] * rows)
    kw = dict(num_kv_heads=wl.kv_heads)
    args = (b.q, b.k_pool, b.v_pool, b.table, b.rows, b.positions, b.sinks, 0, wl.scale)
    auto = pgd.paged_prefill_attention(*args, **kw)
    want = pgd.paged_prefill_attention(*args, kernel=kernel, **kw)
    assert pgd.get_device_error() == pgd.OK
    assert torch.equal(auto, want)
