"""GPU parity for the prefill row: page_slots and kv_write_slots bit-exact
against the oracle, paged prefill attention (packed prompt chunks over their
rows' pages, with sinks and windows) and step_paged (prompts and decode steps
in one call) within the tolerance, on small cases and sampled tokens of the
full prefill workloads."""
import math

import numpy as np
import pytest
import torch

import oracle
import paged_gqa_decode_gb300 as pgd
from pgd_inputs import (PREFILL_WORKLOADS, WORKLOADS, PrefillWorkload, bf16_bits, draw_layout,
                        make_batch, make_prefill_batch)
from tests.oracle_side import snapshot_pages
from tests.parity import compare

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    yield
    torch.cuda.synchronize()


def pages_needed(n_last: np.ndarray) -> np.ndarray:
    return n_last // 64 + 1


def prefill_check(b, *, window=None, sinks="batch", layout=pgd.PAGE_MAJOR, sample=None, pps=0,
                  kernel=pgd.KERNEL_AUTO, what="", fused=False):
    """Oracle inputs are copied out before the CUDA path writes anything; the
    oracle then does its own slot computation, writes and prefill.  The CUDA
    path is page_slots + kv_write_slots + paged_prefill_attention, or with
    `fused` the one paged_prefill_step call (page_slots is then called only to
    check the slots)."""
    wl = b.wl
    window = wl.window if window is None else window
    sinks = b.sinks if isinstance(sinks, str) else sinks
    rows_used = sorted(set(b.rows_np.tolist()))
    last = np.array([b.positions_np[b.rows_np == r].max() for r in rows_used])
    k_host, v_host, ctable, num = snapshot_pages(
        b.k_pool, b.v_pool, b.table_np, rows_used, pages_needed(last), kv_heads=wl.kv_heads,
        head_dim=wl.head_dim, layout=layout)
    slots = pgd.page_slots(b.table, b.positions, b.rows, num_pages=b.num_pages)
    if fused:
        out = pgd.paged_prefill_step(b.q, b.k_new, b.v_new, b.k_pool, b.v_pool, b.table, b.rows,
                                     b.positions, sinks, window, wl.scale,
                                     num_kv_heads=wl.kv_heads, layout=layout,
                                     pages_per_split=pps, kernel=kernel)
    else:
        pgd.kv_write_slots(b.k_new, b.v_new, slots, b.k_pool, b.v_pool, layout=layout)
        out = pgd.paged_prefill_attention(b.q, b.k_pool, b.v_pool, b.table, b.rows, b.positions,
                                          sinks, window, wl.scale, num_kv_heads=wl.kv_heads,
                                          layout=layout, pages_per_split=pps, kernel=kernel)
    status = pgd.get_device_error()
    assert status == pgd.OK, pgd.status_string(status)
    # slots: bit-exact against the oracle's page_slots on the original table
    per_token_table = b.table_np[b.rows_np]
    want_slots = oracle.page_slots(per_token_table, b.positions_np, 64, b.num_pages)
    assert np.array_equal(slots.cpu().numpy().astype(np.int64), want_slots)
    # the oracle's own write and prefill on the compact pool
    crow = {r: i for i, r in enumerate(rows_used)}
    crows = np.array([crow[int(r)] for r in b.rows_np], dtype=np.int32)
    oslots = oracle.page_slots(ctable[crows], b.positions_np, 64, num)
    geo = dict(kv_heads=wl.kv_heads, head_dim=wl.head_dim, page_size=64, num_pages=num,
               layout=layout)
    oracle.write_tokens(k_host, bf16_bits(b.k_new), oslots, **geo)
    oracle.write_tokens(v_host, bf16_bits(b.v_new), oslots, **geo)
    idx = np.arange(len(b.rows_np)) if sample is None else np.asarray(sample)
    sinks_np = None if sinks is None else sinks.cpu().numpy()
    want, _, _ = oracle.prefill_paged(bf16_bits(b.q)[idx], k_host, v_host, ctable, crows[idx],
                                      b.positions_np[idx], kv_heads=wl.kv_heads, num_pages=num,
                                      layout=layout, sinks=sinks_np, window=window,
                                      scale=wl.scale)
    got = out.index_select(0, torch.as_tensor(idx, device=out.device))
    return compare(got, want, what or wl.name)


# ---------------------------------------------------------------------------


def test_page_slots_decode_mode_bit_exact():
    wl = WORKLOADS["gptoss_full"]
    lay = draw_layout(wl, 1002)
    table = torch.from_numpy(lay.table).to(DEV)
    pos = torch.from_numpy(lay.positions).to(DEV)
    got = pgd.page_slots(table, pos, num_pages=lay.num_pages).cpu().numpy()
    want = oracle.page_slots(lay.table, lay.positions, 64, lay.num_pages)
    assert np.array_equal(got.astype(np.int64), want)
    assert pgd.get_device_error() == pgd.OK


def test_page_slots_bad_entries_give_minus_one_and_an_error():
    table = torch.tensor([[3, 7], [5, 99]], dtype=torch.int32, device=DEV)
    pos = torch.tensor([70, 64, -1, 200], dtype=torch.int32, device=DEV)
    rows = torch.tensor([0, 1, 0, 0], dtype=torch.int32, device=DEV)
    got = pgd.page_slots(table, pos, rows, num_pages=8).cpu().tolist()
    assert got == [7 * 64 + 6, -1, -1, -1]
    assert pgd.get_device_error() == pgd.EDEVICE_BOUNDS


@pytest.mark.parametrize("layout", [pgd.PAGE_MAJOR, pgd.HEAD_MAJOR])
def test_write_slots_bit_exact(layout):
    wl = PREFILL_WORKLOADS["mistral_prefill"].replace(rows=3, chunk=70)
    b = make_prefill_batch(wl, 5, DEV, prefix=[0, 63, 130])
    k_host, v_host = bf16_bits(b.k_pool).copy(), bf16_bits(b.v_pool).copy()
    slots = pgd.page_slots(b.table, b.positions, b.rows, num_pages=b.num_pages)
    slots[5] = -1                                   # a padding token writes nothing
    pgd.kv_write_slots(b.k_new, b.v_new, slots, b.k_pool, b.v_pool, layout=layout)
    assert pgd.get_device_error() == pgd.OK
    s64 = slots.cpu().numpy().astype(np.int64)
    geo = dict(kv_heads=wl.kv_heads, head_dim=wl.head_dim, page_size=64,
               num_pages=b.num_pages, layout=layout)
    oracle.write_tokens(k_host, bf16_bits(b.k_new), s64, **geo)
    oracle.write_tokens(v_host, bf16_bits(b.v_new), s64, **geo)
    assert np.array_equal(bf16_bits(b.k_pool), k_host)
    assert np.array_equal(bf16_bits(b.v_pool), v_host)


SMALL = [
    # name, q, kv, d, window, sinks
    ("mistral", 32, 8, 128, 0, False),
    ("gptoss_sliding", 64, 8, 64, 128, True),
    ("gptoss_full", 64, 8, 64, 0, True),
    ("qwen", 14, 2, 64, 0, False),
    ("narrow_window", 16, 4, 128, 65, True),
    ("window_one", 8, 8, 64, 1, True),
]


@pytest.mark.parametrize("name,hq,hkv,d,window,sinks", SMALL)
@pytest.mark.parametrize("kernel,pps", [(pgd.KERNEL_TENSOR_CORE, 0), (pgd.KERNEL_TENSOR_CORE, 1),
                                        (pgd.KERNEL_PREFILL_TILED, 0),
                                        (pgd.KERNEL_PREFILL_UMMA, 0)])
@pytest.mark.parametrize("fused", [False, True])
def test_prefill_small(name, hq, hkv, d, window, sinks, kernel, pps, fused):
    wl = PrefillWorkload(name, rows=4, q_heads=hq, kv_heads=hkv, head_dim=d, prefix_lo=0,
                         prefix_hi=300, chunk=0, window=window, sinks=sinks)
    b = make_prefill_batch(wl, 11 + hq + d, DEV, prefix=[0, 63, 64, 200],
                           chunks=[1, 64, 100, 130])
    prefill_check(b, pps=pps, kernel=kernel, fused=fused,
                  what=f"prefill {name} k={kernel} pps={pps} fused={fused}")


TILED_KERNELS = [pgd.KERNEL_PREFILL_TILED, pgd.KERNEL_PREFILL_UMMA]


@pytest.mark.parametrize("kernel", TILED_KERNELS)
@pytest.mark.parametrize("hq,hkv,d", [(8, 8, 64), (4, 2, 128), (12, 4, 64), (10, 2, 64),
                                      (64, 8, 64)])
def test_prefill_tiled_groups_and_long_prefix(hq, hkv, d, kernel):
    """Group sizes 1, 2, 3, 5 and 8 in the token-block kernels (blocks of
    128 / G tokens on the tcgen05 kernel, so 25 tokens and 125 query rows for
    G = 5), chunks that start mid-page after long prefixes."""
    wl = PrefillWorkload("tiled", rows=3, q_heads=hq, kv_heads=hkv, head_dim=d, prefix_lo=0,
                         prefix_hi=3000, chunk=0, window=0, sinks=True)
    b = make_prefill_batch(wl, 16 + hq, DEV, prefix=[2000, 37, 1500], chunks=[70, 150, 9])
    prefill_check(b, kernel=kernel, what=f"kernel {kernel} {hq}/{hkv} d{d}")


@pytest.mark.parametrize("layout", [pgd.PAGE_MAJOR, pgd.HEAD_MAJOR])
def test_prefill_head_major_and_cuda_core(layout):
    wl = PrefillWorkload("hm", rows=3, q_heads=16, kv_heads=4, head_dim=64, prefix_lo=0,
                         prefix_hi=300, chunk=0, window=0, sinks=True)
    b = make_prefill_batch(wl, 12, DEV, prefix=[10, 0, 190], chunks=[80, 5, 70])
    prefill_check(b, layout=layout, kernel=pgd.KERNEL_CUDA_CORE if layout else pgd.KERNEL_AUTO)


@pytest.mark.parametrize("kernel", TILED_KERNELS)
@pytest.mark.parametrize("d", [64, 128])
def test_prefill_token_block_kernels_head_major(kernel, d):
    """The token-block kernels on the head-major pool: a (page, kv head) tile
    is still 64 contiguous rows, at another row of the pool."""
    wl = PrefillWorkload("hm_tiles", rows=3, q_heads=16, kv_heads=4, head_dim=d, prefix_lo=0,
                         prefix_hi=900, chunk=0, window=0, sinks=True)
    b = make_prefill_batch(wl, 23 + d, DEV, prefix=[700, 0, 130], chunks=[90, 140, 33])
    prefill_check(b, layout=pgd.HEAD_MAJOR, kernel=kernel, what=f"head-major k={kernel} d{d}")


@pytest.mark.parametrize("kernel", [pgd.KERNEL_AUTO] + TILED_KERNELS)
def test_prefill_interleaved_token_order(kernel):
    """Packed tokens need not be grouped by row or sorted by position."""
    wl = PrefillWorkload("mixed", rows=3, q_heads=8, kv_heads=2, head_dim=128, prefix_lo=0,
                         prefix_hi=300, chunk=0, window=100, sinks=True)
    b = make_prefill_batch(wl, 13, DEV, prefix=[0, 120, 250], chunks=[40, 40, 40])
    perm = np.random.default_rng(0).permutation(len(b.rows_np))
    t = torch.as_tensor(perm, device=DEV)
    b.rows_np, b.positions_np = b.rows_np[perm], b.positions_np[perm]
    b.rows, b.positions = b.rows[t].contiguous(), b.positions[t].contiguous()
    b.q, b.k_new, b.v_new = b.q[t].contiguous(), b.k_new[t].contiguous(), b.v_new[t].contiguous()
    prefill_check(b, kernel=kernel)


@pytest.mark.parametrize("kernel", [pgd.KERNEL_AUTO] + TILED_KERNELS)
@pytest.mark.parametrize("fused", [False, True])
def test_step_paged_prompts_and_steps_in_one_call(kernel, fused):
    """step_paged: two rows prefill a chunk, three other rows take a decode
    step; one write of every token and one attention call over all of them
    matches the oracle's prefill over the same concatenation (which for the
    step tokens is exactly decode_paged)."""
    wl = PrefillWorkload("step", rows=5, q_heads=32, kv_heads=8, head_dim=128, prefix_lo=0,
                         prefix_hi=2000, chunk=0, window=0, sinks=False)
    b = make_prefill_batch(wl, 14, DEV, prefix=[0, 900, 1500, 64, 1999],
                           chunks=[150, 70, 1, 1, 1])
    prefill_check(b, kernel=kernel, fused=fused, what=f"step_paged fused={fused}")


@pytest.mark.parametrize("kernel", [pgd.KERNEL_AUTO] + TILED_KERNELS)
@pytest.mark.parametrize("name,sample", [("mistral_prefill", 192), ("gptoss_prefill_sliding", 256)])
@pytest.mark.parametrize("fused", [False, True])
def test_prefill_full_size_sampled(name, sample, kernel, fused):
    wl = PREFILL_WORKLOADS[name]
    b = make_prefill_batch(wl, 2000 + list(PREFILL_WORKLOADS).index(name), DEV)
    rng = np.random.default_rng(3)
    tokens = len(b.rows_np)
    idx = np.unique(np.concatenate([rng.choice(tokens, size=sample - 2, replace=False),
                                    [0, tokens - 1]]))
    prefill_check(b, sample=idx, kernel=kernel, fused=fused)


@pytest.mark.parametrize("kernel", [pgd.KERNEL_AUTO, pgd.KERNEL_TENSOR_CORE] + TILED_KERNELS)
@pytest.mark.parametrize("layout,d,window", [(pgd.PAGE_MAJOR, 128, 0), (pgd.PAGE_MAJOR, 64, 100),
                                             (pgd.HEAD_MAJOR, 64, 0), (pgd.HEAD_MAJOR, 128, 30)])
def test_prefill_step_equals_the_three_calls(kernel, layout, d, window):
    """paged_prefill_step leaves the pools bit-identical to page_slots +
    kv_write_slots and gives bit-identical outputs to the attention call
    after them (the same attention kernels, the same block order), with
    inactive tokens among the packed ones."""
    wl = PrefillWorkload("fused", rows=4, q_heads=32, kv_heads=8, head_dim=d, prefix_lo=0,
                         prefix_hi=900, chunk=0, window=window, sinks=True)
    a = make_prefill_batch(wl, 31 + d + window, DEV, prefix=[0, 700, 65, 300],
                           chunks=[90, 140, 33, 64])
    b = make_prefill_batch(wl, 31 + d + window, DEV, prefix=[0, 700, 65, 300],
                           chunks=[90, 140, 33, 64])
    for x in (a, b):
        x.positions[7] = -1   # an inactive token: not written, zero output
    kw = dict(num_kv_heads=wl.kv_heads, layout=layout, kernel=kernel)
    slots = pgd.page_slots(a.table, a.positions, a.rows, num_pages=a.num_pages)
    pgd.kv_write_slots(a.k_new, a.v_new, slots, a.k_pool, a.v_pool, layout=layout)
    want = pgd.paged_prefill_attention(a.q, a.k_pool, a.v_pool, a.table, a.rows, a.positions,
                                       a.sinks, window, wl.scale, **kw)
    assert pgd.get_device_error() == pgd.OK
    got = pgd.paged_prefill_step(b.q, b.k_new, b.v_new, b.k_pool, b.v_pool, b.table, b.rows,
                                 b.positions, b.sinks, window, wl.scale, **kw)
    assert pgd.get_device_error() == pgd.OK
    assert torch.equal(b.k_pool, a.k_pool) and torch.equal(b.v_pool, a.v_pool)
    assert torch.equal(got, want)
    assert torch.all(got[7] == 0)


@pytest.mark.parametrize("kernel", [pgd.KERNEL_TENSOR_CORE] + TILED_KERNELS)
def test_prefill_step_bad_entries_are_not_written(kernel):
    """A token whose row, page index or page is out of range is reported, not
    written, and its output is zero; the other tokens are written and
    attend as in the three calls."""
    wl = PrefillWorkload("fused_bad", rows=2, q_heads=8, kv_heads=2, head_dim=64, prefix_lo=0,
                         prefix_hi=100, chunk=0)
    b = make_prefill_batch(wl, 15, DEV, prefix=[0, 50], chunks=[10, 10])
    rows, positions, table = b.rows.clone(), b.positions.clone(), b.table.clone()
    rows[3] = 7                                  # outside the table
    positions[4] = 64 * b.table.shape[1] + 1     # beyond its table row
    before_k, before_v = b.k_pool.clone(), b.v_pool.clone()
    out = pgd.paged_prefill_step(b.q, b.k_new, b.v_new, b.k_pool, b.v_pool, table, rows,
                                 positions, num_kv_heads=2, kernel=kernel)
    assert pgd.get_device_error() == pgd.EDEVICE_BOUNDS
    assert torch.all(out[3] == 0) and torch.all(out[4] == 0) and torch.any(out[5] != 0)
    # the 18 good tokens' rows were written, nothing else
    changed_k = (b.k_pool != before_k).view(-1, 64).any(dim=1).sum().item()
    assert changed_k == 18 * wl.kv_heads
    assert torch.equal((b.v_pool != before_v).view(-1, 64).any(dim=1),
                       (b.k_pool != before_k).view(-1, 64).any(dim=1))


def test_prefill_step_kernel_count():
    w = PREFILL_WORKLOADS["mistral_prefill"]
    dims = pgd.make_dims(rows=4096, num_q_heads=w.q_heads, num_kv_heads=w.kv_heads,
                         head_dim=w.head_dim, num_pages=10000, max_pages_per_row=140)
    # the write launch + the tcgen05 kernel (its counter and order prepared)
    assert pgd.prefill_step_kernel_count(dims, 8) == 2
    assert pgd.attention_kernel_count(dims, 8) == 2
    assert pgd.prefill_step_kernel_count(dims, 8, kernel=pgd.KERNEL_PREFILL_TILED) == 2
    assert pgd.prefill_step_kernel_count(dims, 8, window=128) == 2
    one = pgd.make_dims(rows=8, num_q_heads=w.q_heads, num_kv_heads=w.kv_heads,
                        head_dim=w.head_dim, num_pages=10000, max_pages_per_row=140)
    # one token per row: the per-token decode kernels (the window kernel here)
    assert pgd.prefill_step_kernel_count(one, 8, window=100) == 2
    zero = pgd.make_dims(rows=0, num_q_heads=w.q_heads, num_kv_heads=w.kv_heads,
                         head_dim=w.head_dim, num_pages=10000, max_pages_per_row=140)
    assert pgd.prefill_step_kernel_count(zero, 8) == 0


@pytest.mark.parametrize("kernel", [pgd.KERNEL_TENSOR_CORE] + TILED_KERNELS)
def test_prefill_bad_rows_and_pages_are_zero_and_reported(kernel):
    wl = PrefillWorkload("bad", rows=2, q_heads=8, kv_heads=2, head_dim=64, prefix_lo=0,
                         prefix_hi=100, chunk=0)
    b = make_prefill_batch(wl, 15, DEV, prefix=[0, 50], chunks=[10, 10])
    rows = b.rows.clone()
    rows[3] = 7
    out = pgd.paged_prefill_attention(b.q, b.k_pool, b.v_pool, b.table, rows, b.positions,
                                      num_kv_heads=2, kernel=kernel)
    assert pgd.get_device_error() == pgd.EDEVICE_BOUNDS
    assert torch.all(out[3] == 0) and torch.any(out[4] != 0)
    table = b.table.clone()
    table[1, 0] = 10 ** 6          # row 1's first page is outside the pool
    out = pgd.paged_prefill_attention(b.q, b.k_pool, b.v_pool, table, b.rows, b.positions,
                                      num_kv_heads=2, kernel=kernel)
    assert pgd.get_device_error() == pgd.EDEVICE_BOUNDS
    assert torch.all(out[10:] == 0) and torch.any(out[:10] != 0)


@pytest.mark.parametrize("kernel", [pgd.KERNEL_TENSOR_CORE] + TILED_KERNELS)
def test_prefill_poisoned_slots_outside_attention_are_never_read(kernel):
    """Every pool position that no token attends to holds NaN before the
    chunk is written (including the rest of each row's last page and, with the
    window, the positions below it on its first page): any read of one that
    reached a result would show."""
    wl = PrefillWorkload("poison", rows=3, q_heads=16, kv_heads=4, head_dim=128, prefix_lo=0,
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
    prefill_check(b, kernel=kernel, what=f"poison k={kernel}")


@pytest.mark.parametrize("kernel", TILED_KERNELS)
def test_prefill_large_logits(kernel):
    """Queries scaled by 6 give scores with a spread of tens of units in log2,
    so the running maximum is raised many times along a row (on the tcgen05
    kernel each raise by more than 2^8 rescales that row of O in TMEM).  The
    softmax is then nearly one-hot, so an output is close to a single V entry;
    V is halved (exactly) to keep outputs below 2.56, above which rounding to
    bf16 alone can exceed the 1e-2 absolute bound."""
    wl = PrefillWorkload("large", rows=2, q_heads=32, kv_heads=8, head_dim=128, prefix_lo=0,
                         prefix_hi=2000, chunk=0, window=0, sinks=True)
    b = make_prefill_batch(wl, 18, DEV, prefix=[1900, 700], chunks=[96, 64])
    b.q = (b.q.float() * 6.0).to(torch.bfloat16)
    b.v_pool.mul_(0.5)
    b.v_new = b.v_new * 0.5
    prefill_check(b, kernel=kernel, what=f"large logits k={kernel}")


@pytest.mark.parametrize("kernel", [pgd.KERNEL_TENSOR_CORE] + TILED_KERNELS)
@pytest.mark.parametrize("hq,hkv,d", [(16, 4, 128), (8, 8, 128), (64, 8, 64)])
def test_prefill_padding_tokens_fill_whole_blocks(hq, hkv, d, kernel):
    """Padding tokens (position < 0) give zero outputs and write nothing.
    Here they fill whole blocks of 128 / G consecutive tokens (and the tail),
    so the token-block kernels meet work items with no pages at all, which
    must still hand their slot back to the loaders."""
    wl = PrefillWorkload("pad", rows=3, q_heads=hq, kv_heads=hkv, head_dim=d, prefix_lo=0,
                         prefix_hi=900, chunk=0, window=0, sinks=True)
    b = make_prefill_batch(wl, 19 + hq, DEV, prefix=[300, 0, 777], chunks=[200, 190, 300])
    block = 128 // (hq // hkv)
    pad = np.zeros(len(b.rows_np), dtype=bool)
    pad[block:3 * block] = True                  # two whole blocks in the middle
    pad[-(block + 5):] = True                    # the last block and a ragged piece
    for r in range(3):                           # every row keeps an active token
        assert not pad[b.rows_np == r].all()
    b.positions_np = np.where(pad, -1, b.positions_np).astype(np.int32)
    b.positions = torch.from_numpy(b.positions_np).to(DEV)
    prefill_check(b, kernel=kernel, what=f"padding k={kernel} {hq}/{hkv}")
    out = pgd.paged_prefill_attention(b.q, b.k_pool, b.v_pool, b.table, b.rows, b.positions,
                                      b.sinks, 0, wl.scale, num_kv_heads=hkv, kernel=kernel)
    assert pgd.get_device_error() == pgd.OK
    padded = torch.from_numpy(pad).to(DEV)
    assert torch.all(out[padded] == 0) and torch.all(out[~padded].abs().sum((1, 2)) > 0)


@pytest.mark.parametrize("kernel", [pgd.KERNEL_TENSOR_CORE] + TILED_KERNELS)
@pytest.mark.parametrize("d,window", [(128, 0), (64, 100)])
def test_prefill_scores_far_below_zero(kernel, d, window):
    """q = -64 and every key 2 in every dimension: all scores equal, about
    -1450 (d 128) in score units, so the output is the mean of V over the
    attended keys.  A running maximum raised above the true one by anything
    (a stray value) would underflow every weight to zero."""
    wl = PrefillWorkload("negative", rows=2, q_heads=16, kv_heads=4, head_dim=d, prefix_lo=0,
                         prefix_hi=500, chunk=0, window=window, sinks=False)
    b = make_prefill_batch(wl, 27 + d, DEV, prefix=[300, 0], chunks=[70, 90])
    b.q.fill_(-64.0)
    b.k_pool.fill_(2.0)
    b.k_new.fill_(2.0)
    prefill_check(b, sinks=None, kernel=kernel, what=f"negative scores k={kernel} d{d}")


@pytest.mark.parametrize("kernel", [pgd.KERNEL_TENSOR_CORE] + TILED_KERNELS)
@pytest.mark.parametrize("d", [64, 128])
def test_prefill_scores_rise_every_page(kernel, d):
    """q = 1/4 and every key of logical page j equal to step * j in every
    dimension: a token's scores grow by about 23 log2 units from one page to
    the next, more than the lazy-rescale slack of 8, so on the tcgen05 kernel
    the reference maximum is raised (and O rescaled) on page after page.  The
    keys (multiples of 6 or 8 below 256) are exact in bf16."""
    wl = PrefillWorkload("rising", rows=2, q_heads=16, kv_heads=4, head_dim=d, prefix_lo=0,
                         prefix_hi=1500, chunk=0, window=0, sinks=True)
    b = make_prefill_batch(wl, 31 + d, DEV, prefix=[1400, 200], chunks=[40, 64])
    step = 8.0 if d == 64 else 6.0   # sqrt(d) * step / 4 * log2(e) ~ 23 per page
    b.q.fill_(0.25)
    view = b.k_pool.view(b.num_pages, wl.kv_heads, 64, d)
    for r in range(2):
        n_pages = (int(b.positions_np[b.rows_np == r].max()) // 64) + 1
        for j in range(n_pages):
            view[int(b.table_np[r, j])] = step * j
    pages = torch.as_tensor(b.positions_np // 64, device=DEV, dtype=torch.float32)
    b.k_new = (pages.view(-1, 1, 1) * step).expand_as(b.k_new).to(torch.bfloat16).contiguous()
    prefill_check(b, kernel=kernel, what=f"rising scores k={kernel} d{d}")
