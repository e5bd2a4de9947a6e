"""GPU parity of the tcgen05 prefill cut into key parts (AUTO, calls whose
work items are at most half the SMs): each item's pages are split over
several work units that write partials, and a combine launch merges them with
the sink.  Against the oracle on small cases (group sizes, windows, sinks,
both call forms), items with several runs and parts without pages, bad rows
and pages, inactive tokens, poisoned slots and a huge sink; every output of
one long Mistral-shaped and one gpt-oss-shaped chunk close to the one-SM
kernel's without parts; the launch counts."""
import math

import numpy as np
import pytest
import torch

import paged_gqa_decode_gb300 as pgd
from pgd_inputs import PREFILL_WORKLOADS, PrefillWorkload, make_prefill_batch
from tests.parity import compare
from tests.test_gpu_prefill import DEV, prefill_check

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    yield
    torch.cuda.synchronize()


def sm_count() -> int:
    return torch.cuda.get_device_properties(0).multi_processor_count


def expected_parts(tokens, hq, hkv, max_pages, window) -> int:
    """The key-part count AUTO takes (the rule pgd.h states): at most half as
    many items as SMs, min(8, SMs / items, L / 8) parts, L the table width
    or, with a window, the pages a block's keys can span; 1 below 2."""
    block = 2 * (128 // (hq // hkv))
    items = math.ceil(tokens / block) * hkv
    if items * 2 > sm_count():
        return 1
    pages = max_pages
    if window > 0:
        pages = min(pages, (window + block - 2) // 64 + 2)
    parts = min(8, sm_count() // items, pages // 8)
    return parts if parts >= 2 else 1


def assert_parts(b, window):
    """The call is cut into key parts: one launch more than without."""
    wl = b.wl
    tokens = len(b.rows_np)
    parts = expected_parts(tokens, wl.q_heads, wl.kv_heads, b.table.shape[1], window)
    assert parts > 1, "the case does not exercise key parts"
    dims = pgd.make_dims(rows=tokens, num_q_heads=wl.q_heads, num_kv_heads=wl.kv_heads,
                         head_dim=wl.head_dim, num_pages=b.num_pages,
                         max_pages_per_row=b.table.shape[1])
    table_rows = b.table.shape[0]
    direct = pgd.attention_kernel_count(dims, table_rows, window=window,
                                        kernel=pgd.KERNEL_PREFILL_UMMA)
    assert pgd.attention_kernel_count(dims, table_rows, window=window) == direct + 1
    assert pgd.prefill_step_kernel_count(dims, table_rows, window=window) == 3
    return parts


@pytest.mark.parametrize("hq,hkv,d,window,sinks", [(32, 8, 128, 0, False),
                                                   (16, 4, 128, 1000, True),
                                                   (8, 8, 128, 0, True),
                                                   (10, 2, 128, 0, True),
                                                   (64, 8, 64, 0, True),
                                                   (14, 2, 64, 900, False),
                                                   (4, 2, 64, 0, True)])
@pytest.mark.parametrize("fused", [False, True])
def test_parts_small(hq, hkv, d, window, sinks, fused):
    """Group sizes 1-8 (7: blocks of 18 tokens a tile), chunks on and off
    page boundaries over prefixes of up to 1500 positions, full and windowed."""
    wl = PrefillWorkload("parts", rows=3, q_heads=hq, kv_heads=hkv, head_dim=d, prefix_lo=0,
                         prefix_hi=1600, chunk=0, window=window, sinks=sinks)
    b = make_prefill_batch(wl, 61 + hq + d + window, DEV, prefix=[0, 700, 1500],
                           chunks=[40, 130, 64])
    assert_parts(b, window)
    prefill_check(b, fused=fused, what=f"parts {hq}/{hkv} d{d} w={window} fused={fused}")


def test_parts_runs_and_parts_without_pages():
    """A block holding two rows' tokens (two runs): a one-page run, which
    falls in one part only (the other parts hold none of its pages), and a
    63-page run spread over all parts."""
    wl = PrefillWorkload("parts_runs", rows=2, q_heads=16, kv_heads=4, head_dim=128,
                         prefix_lo=0, prefix_hi=4000, chunk=0, window=0, sinks=True)
    b = make_prefill_batch(wl, 71, DEV, prefix=[0, 4000], chunks=[20, 10])
    assert assert_parts(b, 0) >= 4
    prefill_check(b, what="parts: runs and empty parts")


@pytest.mark.parametrize("d", [128, 64])
def test_parts_interleaved_tokens(d):
    wl = PrefillWorkload("parts_mixed", rows=3, q_heads=8, kv_heads=2, head_dim=d, prefix_lo=0,
                         prefix_hi=2000, chunk=0, window=0, sinks=True)
    b = make_prefill_batch(wl, 73, DEV, prefix=[0, 1200, 1900], chunks=[40, 40, 40])
    perm = np.random.default_rng(1).permutation(len(b.rows_np))
    t = torch.as_tensor(perm, device=DEV)
    b.rows_np, b.positions_np = b.rows_np[perm], b.positions_np[perm]
    b.rows, b.positions = b.rows[t].contiguous(), b.positions[t].contiguous()
    b.q, b.k_new, b.v_new = b.q[t].contiguous(), b.k_new[t].contiguous(), b.v_new[t].contiguous()
    assert_parts(b, 0)
    prefill_check(b, what=f"parts interleaved d{d}")


@pytest.mark.parametrize("name", ["mistral_prefill", "gptoss_prefill_sliding"])
def test_parts_one_long_chunk_close_to_one_sm_kernel(name):
    """One chunk (64 items at both shapes; the gpt-oss one without its window)
    over a prefix of 6000 positions: every output against the one-SM kernel
    without parts (itself checked against the oracle), and sampled tokens
    against the oracle."""
    window = 0
    wl = PREFILL_WORKLOADS[name].replace(rows=1, window=window)
    b = make_prefill_batch(wl, 75, DEV, prefix=[6000])
    parts = assert_parts(b, window)
    assert parts >= 2
    kw = dict(num_kv_heads=wl.kv_heads)
    args = (b.q, b.k_pool, b.v_pool, b.table, b.rows, b.positions, b.sinks, window, wl.scale)
    slots = pgd.page_slots(b.table, b.positions, b.rows, num_pages=b.num_pages)
    pgd.kv_write_slots(b.k_new, b.v_new, slots, b.k_pool, b.v_pool)
    want = pgd.paged_prefill_attention(*args, kernel=pgd.KERNEL_PREFILL_UMMA, **kw)
    got = pgd.paged_prefill_attention(*args, **kw)
    assert pgd.get_device_error() == pgd.OK
    compare(got, want.float().cpu().numpy().astype(np.float64), f"{name} parts vs one-SM")
    b2 = make_prefill_batch(wl, 75, DEV, prefix=[6000])
    rng = np.random.default_rng(5)
    idx = np.unique(np.concatenate([rng.choice(len(b2.rows_np), size=48, replace=False),
                                    [0, len(b2.rows_np) - 1]]))
    prefill_check(b2, sample=idx, what=f"{name} one chunk, parts")


def test_parts_bad_rows_pages_and_inactive_tokens():
    wl = PrefillWorkload("parts_bad", rows=2, q_heads=8, kv_heads=2, head_dim=128, prefix_lo=0,
                         prefix_hi=1500, chunk=0)
    b = make_prefill_batch(wl, 77, DEV, prefix=[0, 1400], chunks=[10, 12])
    assert_parts(b, 0)
    kw = dict(num_kv_heads=2)
    rows = b.rows.clone()
    rows[3] = 7
    out = pgd.paged_prefill_attention(b.q, b.k_pool, b.v_pool, b.table, rows, b.positions, **kw)
    assert pgd.get_device_error() == pgd.EDEVICE_BOUNDS
    assert torch.all(out[3] == 0) and torch.all(out[4:].abs().sum((1, 2)) > 0)
    table = b.table.clone()
    table[1, 3] = 10 ** 6
    out = pgd.paged_prefill_attention(b.q, b.k_pool, b.v_pool, table, b.rows, b.positions, **kw)
    assert pgd.get_device_error() == pgd.EDEVICE_BOUNDS
    assert torch.all(out[10:] == 0) and torch.all(out[:10].abs().sum((1, 2)) > 0)
    positions = b.positions.clone()
    positions[[2, 15]] = -1
    out = pgd.paged_prefill_attention(b.q, b.k_pool, b.v_pool, b.table, b.rows, positions, **kw)
    assert pgd.get_device_error() == pgd.OK
    assert torch.all(out[[2, 15]] == 0)
    live = torch.ones(len(b.rows_np), dtype=torch.bool, device=DEV)
    live[[2, 15]] = False
    assert torch.all(out[live].abs().sum((1, 2)) > 0)


def test_parts_poisoned_slots_outside_attention_are_never_read():
    wl = PrefillWorkload("parts_poison", rows=3, q_heads=16, kv_heads=4, head_dim=128,
                         prefix_lo=0, prefix_hi=2000, chunk=0, window=1100, sinks=True)
    b = make_prefill_batch(wl, 79, DEV, prefix=[10, 1300, 1923], chunks=[70, 33, 40])
    assert_parts(b, wl.window)
    keep = np.zeros(b.num_pages * 64, dtype=bool)
    for r, n in zip(b.rows_np, b.positions_np):
        for s in range(max(0, int(n) - wl.window + 1), int(n) + 1):
            keep[b.table_np[r, s // 64] * 64 + s % 64] = True
    nan_slots = torch.from_numpy(~keep).to(DEV)
    for pool in (b.k_pool, b.v_pool):
        view = pool.view(b.num_pages, wl.kv_heads, 64, wl.head_dim)
        view.masked_fill_(nan_slots.view(b.num_pages, 1, 64, 1).expand_as(view), float("nan"))
    prefill_check(b, what="parts poison")


def test_parts_huge_sink_gives_zero_without_nan():
    wl = PrefillWorkload("parts_sink", rows=2, q_heads=16, kv_heads=4, head_dim=64, prefix_lo=0,
                         prefix_hi=1500, chunk=0, window=0, sinks=True)
    b = make_prefill_batch(wl, 81, DEV, prefix=[0, 1400], chunks=[30, 50])
    assert_parts(b, 0)
    sinks = torch.full_like(b.sinks, 1e4)
    prefill_check(b, sinks=sinks, what="parts huge sink")
    out = pgd.paged_prefill_attention(b.q, b.k_pool, b.v_pool, b.table, b.rows, b.positions,
                                      sinks, 0, wl.scale, num_kv_heads=4)
    assert pgd.get_device_error() == pgd.OK
    assert torch.all(torch.isfinite(out.float())) and out.float().abs().max().item() < 1e-6


def test_parts_step_equals_the_three_calls():
    wl = PrefillWorkload("parts_fused", rows=3, q_heads=32, kv_heads=8, head_dim=128,
                         prefix_lo=0, prefix_hi=2000, chunk=0, window=0, sinks=True)
    prefix, chunks = [0, 1700, 650], [90, 70, 33]
    a = make_prefill_batch(wl, 83, DEV, prefix=prefix, chunks=chunks)
    b = make_prefill_batch(wl, 83, DEV, prefix=prefix, chunks=chunks)
    for x in (a, b):
        x.positions[7] = -1
    assert_parts(a, 0)
    kw = dict(num_kv_heads=wl.kv_heads, layout=pgd.HEAD_MAJOR)
    slots = pgd.page_slots(a.table, a.positions, a.rows, num_pages=a.num_pages)
    pgd.kv_write_slots(a.k_new, a.v_new, slots, a.k_pool, a.v_pool, layout=pgd.HEAD_MAJOR)
    want = pgd.paged_prefill_attention(a.q, a.k_pool, a.v_pool, a.table, a.rows, a.positions,
                                       a.sinks, 0, wl.scale, **kw)
    assert pgd.get_device_error() == pgd.OK
    got = pgd.paged_prefill_step(b.q, b.k_new, b.v_new, b.k_pool, b.v_pool, b.table, b.rows,
                                 b.positions, b.sinks, 0, wl.scale, **kw)
    assert pgd.get_device_error() == pgd.OK
    assert torch.equal(b.k_pool, a.k_pool) and torch.equal(b.v_pool, a.v_pool)
    assert torch.equal(got, want)
    assert torch.all(got[7] == 0)


def test_short_windows_and_short_tables_take_no_parts():
    """A 128-position window bounds every item to a few pages, and a table of
    under 16 pages leaves no part 8 pages long: no key parts then."""
    wl = PREFILL_WORKLOADS["gptoss_prefill_sliding"].replace(rows=1)
    dims = pgd.make_dims(rows=256, num_q_heads=wl.q_heads, num_kv_heads=wl.kv_heads,
                         head_dim=wl.head_dim, num_pages=2000, max_pages_per_row=140)
    one_sm = pgd.attention_kernel_count(dims, 1, window=128, kernel=pgd.KERNEL_PREFILL_UMMA)
    assert pgd.attention_kernel_count(dims, 1, window=128) == one_sm
    assert pgd.attention_kernel_count(dims, 1) == one_sm + 2  # block order, kernel, combine
    short = pgd.make_dims(rows=256, num_q_heads=wl.q_heads, num_kv_heads=wl.kv_heads,
                          head_dim=wl.head_dim, num_pages=2000, max_pages_per_row=15)
    assert pgd.attention_kernel_count(short, 1) == 2  # block order, kernel


@pytest.mark.parametrize("d,hq,hkv", [(128, 32, 8), (64, 64, 8), (64, 14, 2)])
def test_parts_write_only_their_outputs(d, hq, hkv):
    """The combine writes each token's rows and nothing past them: the call's
    output is the first P rows of a larger buffer whose last row holds a
    sentinel, which stays; every output close to the kernel without parts."""
    wl = PrefillWorkload("parts_guard", rows=2, q_heads=hq, kv_heads=hkv, head_dim=d,
                         prefix_lo=0, prefix_hi=2500, chunk=0, window=0, sinks=True)
    b = make_prefill_batch(wl, 87 + d + hq, DEV, prefix=[2400, 1100], chunks=[77, 50])
    assert_parts(b, 0)
    tokens = len(b.rows_np)
    buf = torch.full((tokens + 1, hq, d), 7.0, dtype=torch.bfloat16, device=DEV)
    out = buf[:tokens]
    kw = dict(num_kv_heads=hkv)
    args = (b.q, b.k_pool, b.v_pool, b.table, b.rows, b.positions, b.sinks, 0, wl.scale)
    pgd.paged_prefill_attention(*args, out=out, **kw)
    want = pgd.paged_prefill_attention(*args, kernel=pgd.KERNEL_PREFILL_UMMA, **kw)
    assert pgd.get_device_error() == pgd.OK
    assert torch.all(buf[tokens] == 7.0), "a write past the call's outputs"
    compare(out, want.float().cpu().numpy().astype(np.float64), f"parts guard d{d} {hq}/{hkv}")
