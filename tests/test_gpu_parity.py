"""GPU parity: libpgd (through its C ABI) against the fp64 oracle on the same
seeded inputs.  Append indexing must be bit-exact; attention output must be
within max abs 1e-2 and max rel 2e-2 (bf16 output, fp32 accumulation).

Covers the five workloads at full size: qwen_small, qwen_serve and
gptoss_full on every row through append + decode; gptoss_sliding and
mistral_serve on every row through the call the benchmark times (the fused
decode step) and on sampled rows through append + decode.  And the edge
cases: contexts around page boundaries, window boundaries, group sizes 1..8 with padding, head_dim 64 and 128, sink of
-inf / huge / none, shared and reversed page lists, inactive rows, both pool
layouts, split sizes that force the combine kernel, poisoned (NaN) slots
outside every attended set, device-side bounds errors, and CUDA graphs."""
import math

import numpy as np
import pytest
import torch

import oracle
import paged_gqa_decode_gb300 as pgd
from pgd_inputs import WORKLOADS, Workload, bf16_bits, layout_from_contexts, make_batch
from tests.parity import compare, gpu_step, oracle_step, snapshot_rows

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    yield
    torch.cuda.synchronize()


def run_and_check(batch, *, window=None, sinks="batch", layout=pgd.PAGE_MAJOR, rows=None,
                  pages_per_split=0, kernel=pgd.KERNEL_AUTO, what=""):
    wl = batch.wl
    window = wl.window if window is None else window
    sinks = batch.sinks if isinstance(sinks, str) else sinks
    rows = np.arange(len(batch.layout.positions)) if rows is None else np.asarray(rows)
    host = snapshot_rows(batch, rows, layout)
    got = gpu_step(batch, window=window, sinks=sinks, scale=wl.scale, layout=layout,
                   pages_per_split=pages_per_split, kernel=kernel)
    want, _, _ = oracle_step(batch, host, window=window, sinks=sinks, scale=wl.scale,
                             layout=layout)
    idx = torch.as_tensor(rows, device=got.device)
    return compare(got.index_select(0, idx), want, what or wl.name)


# ---------------------------------------------------------------------------
# Append: bit-exact against the oracle's page_slots + write_tokens.


@pytest.mark.parametrize("layout", [pgd.PAGE_MAJOR, pgd.HEAD_MAJOR])
@pytest.mark.parametrize("hkv,d", [(2, 64), (8, 128), (3, 64), (1, 128)])
def test_append_bit_exact(layout, hkv, d):
    wl = Workload("append", rows=9, q_heads=hkv, kv_heads=hkv, head_dim=d, ctx_lo=1, ctx_hi=300)
    contexts = [1, 64, 65, 128, 129, 300, 0, 63, 200]   # a 0 context is an inactive row
    lay = layout_from_contexts(wl, contexts, seed=5, num_pages=40)
    batch = make_batch(wl, seed=21, device=DEV, layout=lay)
    k_host, v_host = bf16_bits(batch.k_pool).copy(), bf16_bits(batch.v_pool).copy()
    pgd.kv_append_paged(batch.k_new, batch.v_new, batch.table, batch.positions, batch.k_pool,
                        batch.v_pool, layout=layout)
    assert pgd.get_device_error() == pgd.OK
    slots = oracle.page_slots(lay.table, lay.positions, 64, lay.num_pages)
    geo = dict(kv_heads=hkv, head_dim=d, page_size=64, num_pages=lay.num_pages, layout=layout)
    oracle.write_tokens(k_host, bf16_bits(batch.k_new), slots, **geo)
    oracle.write_tokens(v_host, bf16_bits(batch.v_new), slots, **geo)
    assert np.array_equal(bf16_bits(batch.k_pool), k_host)
    assert np.array_equal(bf16_bits(batch.v_pool), v_host)


# ---------------------------------------------------------------------------
# The five workloads.


@pytest.mark.parametrize("name", ["qwen_small", "qwen_serve", "gptoss_full"])
def test_workload_every_row(name):
    wl = WORKLOADS[name]
    batch = make_batch(wl, seed=1000 + list(WORKLOADS).index(name), device=DEV)
    run_and_check(batch)


@pytest.mark.parametrize("name,sample", [("gptoss_sliding", 32), ("mistral_serve", 6)])
def test_workload_full_size_sampled_rows(name, sample):
    """Full-size pool and batch, the benchmark's launch configuration; the
    oracle checks a seeded sample of rows, always including the longest and
    the shortest."""
    wl = WORKLOADS[name]
    batch = make_batch(wl, seed=1000 + list(WORKLOADS).index(name), device=DEV)
    pos = batch.layout.positions
    rng = np.random.default_rng(7)
    rows = set(rng.choice(wl.rows, size=sample - 2, replace=False).tolist())
    rows |= {int(np.argmax(pos)), int(np.argmin(pos))}
    run_and_check(batch, rows=sorted(rows))
    del batch
    torch.cuda.empty_cache()


@pytest.mark.parametrize("name", ["gptoss_sliding", "mistral_serve"])
def test_workload_full_size_every_row_decode_step(name):
    """The call the benchmark times, at full size and in its launch
    configuration: paged_decode_step (the append inside the decode launch,
    split size chosen by the library, the workload's window and sinks),
    checked on every row against the oracle's write_tokens + paged_attention
    over a host copy of the pool taken before the step."""
    wl = WORKLOADS[name]
    batch = make_batch(wl, seed=1000 + list(WORKLOADS).index(name), device=DEV)
    rows = np.arange(wl.rows)
    host = snapshot_rows(batch, rows)
    got = pgd.paged_decode_step(batch.q, batch.k_new, batch.v_new, batch.k_pool, batch.v_pool,
                                batch.table, batch.positions, batch.sinks, wl.window, wl.scale,
                                num_kv_heads=wl.kv_heads)
    assert pgd.get_device_error() == pgd.OK
    want, _, _ = oracle_step(batch, host, window=wl.window, sinks=batch.sinks, scale=wl.scale)
    compare(got, want, f"{name}: decode step, every row")
    del batch, host
    torch.cuda.empty_cache()


# ---------------------------------------------------------------------------
# Edge cases.

EDGE_CONTEXTS = [1, 2, 63, 64, 65, 127, 128, 129, 191, 192, 193, 255, 256, 257, 700]


@pytest.mark.parametrize("hq,hkv,d", [(14, 2, 64), (64, 8, 64), (32, 8, 128), (8, 8, 64),
                                      (6, 3, 128), (12, 4, 64), (10, 2, 128), (16, 8, 128)])
@pytest.mark.parametrize("window", [0, 1, 63, 64, 65, 128, 129])
def test_edge_contexts_windows_groups(hq, hkv, d, window):
    wl = Workload("edge", rows=len(EDGE_CONTEXTS), q_heads=hq, kv_heads=hkv, head_dim=d,
                  ctx_lo=1, ctx_hi=700, sinks=True)
    lay = layout_from_contexts(wl, EDGE_CONTEXTS, seed=hq + d + window)
    batch = make_batch(wl, seed=31 + window, device=DEV, layout=lay)
    run_and_check(batch, window=window, what=f"edge hq={hq} hkv={hkv} d={d} w={window}")


@pytest.mark.parametrize("hq,hkv,d", [(14, 2, 64), (64, 8, 64), (32, 8, 128), (8, 8, 128),
                                      (6, 3, 64)])
@pytest.mark.parametrize("window", [0, 65])
def test_cuda_core_kernel(hq, hkv, d, window):
    """The CUDA-core variant of the split kernel (selectable through the
    decode options) against the oracle on the edge contexts."""
    wl = Workload("edge_cc", rows=len(EDGE_CONTEXTS), q_heads=hq, kv_heads=hkv, head_dim=d,
                  ctx_lo=1, ctx_hi=700, sinks=True)
    lay = layout_from_contexts(wl, EDGE_CONTEXTS, seed=hq + d + window + 1)
    batch = make_batch(wl, seed=37 + window, device=DEV, layout=lay)
    run_and_check(batch, window=window, kernel=pgd.KERNEL_CUDA_CORE, pages_per_split=2,
                  what=f"cuda-core hq={hq} d={d} w={window}")


@pytest.mark.parametrize("name", ["gptoss_full", "qwen_serve"])
def test_cuda_core_kernel_workloads(name):
    wl = WORKLOADS[name]
    batch = make_batch(wl, seed=1000 + list(WORKLOADS).index(name), device=DEV)
    run_and_check(batch, kernel=pgd.KERNEL_CUDA_CORE)


@pytest.mark.parametrize("kind", ["none", "minus_inf", "huge", "mixed"])
@pytest.mark.parametrize("d", [64, 128])
def test_sink_values(kind, d):
    wl = Workload("sinks", rows=6, q_heads=8, kv_heads=2, head_dim=d, ctx_lo=1, ctx_hi=400)
    lay = layout_from_contexts(wl, [1, 65, 130, 257, 400, 64], seed=3)
    batch = make_batch(wl, seed=41, device=DEV, layout=lay)
    sinks = {
        "none": None,
        "minus_inf": torch.full((8,), -math.inf, device=DEV),
        "huge": torch.full((8,), 1e4, device=DEV),
        "mixed": torch.tensor([1e4, -math.inf, 0.0, 3.0, -3.0, 30.0, -30.0, 1.5], device=DEV),
    }[kind]
    stats = run_and_check(batch, sinks=sinks, what=f"sink {kind}")
    if kind == "huge":
        assert stats["max_abs"] <= 1e-6


@pytest.mark.parametrize("pps", [1, 2, 3, 5, 8, 12, 64])
@pytest.mark.parametrize("window", [0, 100])
def test_split_sizes_force_the_combine(pps, window):
    """Rows of 1 to 24 pages cut into 1 to 24 splits (with the window, up to
    3), merged by the combine kernel; one split writes directly.  The split
    kernel is asked for by name: with a window of at most 128 positions AUTO
    takes the window kernel, which has no splits."""
    wl = Workload("splits", rows=5, q_heads=16, kv_heads=4, head_dim=64, ctx_lo=1, ctx_hi=1500,
                  sinks=True)
    lay = layout_from_contexts(wl, [1500, 1, 640, 641, 1000], seed=9)
    batch = make_batch(wl, seed=51, device=DEV, layout=lay)
    run_and_check(batch, window=window, pages_per_split=pps, kernel=pgd.KERNEL_TENSOR_CORE,
                  what=f"pps={pps}")


@pytest.mark.parametrize("hq,hkv,d", [(14, 2, 64), (64, 8, 64), (32, 8, 128), (6, 3, 128)])
@pytest.mark.parametrize("window", [1, 64, 65, 127, 128])
@pytest.mark.parametrize("pps", [0, 1])
def test_split_kernel_windows(hq, hkv, d, window, pps):
    """Windows of at most 128 positions through the split kernel (asked for by
    name), as AUTO sends them to the window kernel.  V is scaled by 1/4
    (exact in bf16): with a window of one position an output is a single V
    row, and above |out| = 2.56 rounding to bf16 alone can exceed the 1e-2
    absolute bound."""
    wl = Workload("edge_split", rows=len(EDGE_CONTEXTS), q_heads=hq, kv_heads=hkv, head_dim=d,
                  ctx_lo=1, ctx_hi=700, sinks=True)
    lay = layout_from_contexts(wl, EDGE_CONTEXTS, seed=hq + d + window + 3)
    batch = make_batch(wl, seed=33 + window, device=DEV, layout=lay)
    batch.v_pool.mul_(0.25)
    batch.v_new.mul_(0.25)
    run_and_check(batch, window=window, pages_per_split=pps, kernel=pgd.KERNEL_TENSOR_CORE,
                  what=f"split kernel hq={hq} d={d} w={window} pps={pps}")


def window_rounds(d: int, window: int, sms: int) -> tuple[int, int]:
    """(one-unit CTAs per SM, units per large CTA) of the window kernel:
    a unit (row, kv head) keeps the window's K and V in shared memory, the
    hardware reserves 1 KB per CTA out of 228 KB per SM, and a CTA holds at
    most 227 KB, 1024 threads (a warp per 32 window rows) and 15 units."""
    tiles = 1 if window <= 64 else 2
    unit_smem = 2 * tiles * 64 * d * 2
    per_sm = (228 * 1024) // (unit_smem + 1024)
    units = min((227 * 1024) // unit_smem, 1024 // (64 * tiles), 15)
    return per_sm, units


@pytest.mark.parametrize("d,window", [(64, 128), (64, 100), (64, 65), (64, 64), (64, 7),
                                      (128, 64), (128, 33)])
@pytest.mark.parametrize("fused", [False, True])
@pytest.mark.parametrize("beyond", [False, True])
def test_window_kernel_one_round_of_large_ctas(d, window, fused, beyond):
    """A batch whose (row, kv head) units take two rounds of one-unit CTAs
    but fit one round of CTAs holding as many units as shared memory allows:
    the window kernel launches the large CTAs (each unit on a barrier of its
    own, the last CTA partly empty).  With `beyond`, a batch just past one
    round of large CTAs, which goes back to one-unit CTAs over several
    rounds.  Every row against the oracle, with inactive rows, contexts
    shorter than the window and the append either fused into the decode
    launch or a call of its own.  V is scaled by 1/4 (exact in bf16): rows of
    one or two positions output about one V row, and above |out| = 2.56
    rounding to bf16 alone can exceed the 1e-2 absolute bound."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    per_sm, units = window_rounds(d, window, sms)
    if units <= per_sm:
        pytest.skip("large CTAs hold no more units per SM than one-unit CTAs")
    hkv = 8
    if beyond:
        rows = (sms * units) // hkv + 3      # past one round of large CTAs
        assert rows * hkv > sms * units
    else:
        rows = (sms * per_sm) // hkv + 9     # more than one round of one-unit CTAs
        assert sms * per_sm < rows * hkv <= sms * units and (rows * hkv) % units != 0
    wl = Workload("window_round", rows=rows, q_heads=64, kv_heads=hkv, head_dim=d, ctx_lo=1,
                  ctx_hi=300, window=window, sinks=True)
    base = [0, 1, 2, 7, 63, 64, 65, 100, 127, 128, 129, 191, 192, 193, 255, 300]
    contexts = [base[(7 * b) % len(base)] for b in range(rows)]
    lay = layout_from_contexts(wl, contexts, seed=d + window + rows)
    batch = make_batch(wl, seed=41 + window + d, device=DEV, layout=lay)
    batch.v_pool.mul_(0.25)
    batch.v_new.mul_(0.25)
    if not fused:
        run_and_check(batch, what=f"window kernel d={d} w={window} rows={rows}")
        return
    idx = np.arange(rows)
    host = snapshot_rows(batch, idx)
    got = pgd.paged_decode_step(batch.q, batch.k_new, batch.v_new, batch.k_pool, batch.v_pool,
                                batch.table, batch.positions, batch.sinks, window, wl.scale,
                                num_kv_heads=hkv)
    assert pgd.get_device_error() == pgd.OK
    want, _, _ = oracle_step(batch, host, window=window, sinks=batch.sinks, scale=wl.scale)
    compare(got, want, f"window kernel, decode step d={d} w={window} rows={rows}")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("pps", [0, 3])
def test_head_major_layout(d, pps):
    wl = Workload("headmajor", rows=7, q_heads=16, kv_heads=4, head_dim=d, ctx_lo=1, ctx_hi=900,
                  sinks=True)
    lay = layout_from_contexts(wl, [900, 1, 64, 65, 500, 129, 0], seed=11)
    batch = make_batch(wl, seed=61, device=DEV, layout=lay)
    run_and_check(batch, layout=pgd.HEAD_MAJOR, pages_per_split=pps)


@pytest.mark.parametrize("pps", [0, 1])
def test_shared_prefix_and_reversed_pages(pps):
    """Rows 0 and 1 share their first three pages (a shared prefix) and
    differ in the page holding the new token; row 2 lists its pages in
    reverse pool order; row 3 is inactive and lists page 0."""
    wl = Workload("shared", rows=4, q_heads=8, kv_heads=2, head_dim=64, ctx_lo=1, ctx_hi=256,
                  sinks=True)
    table = np.zeros((4, 4), dtype=np.int32)
    table[0] = [5, 2, 7, 1]
    table[1] = [5, 2, 7, 3]
    table[2] = [11, 10, 9, 8]
    contexts = [250, 230, 256, 0]
    lay = layout_from_contexts(wl, contexts, seed=0, num_pages=12, table=table)
    batch = make_batch(wl, seed=71, device=DEV, layout=lay)
    run_and_check(batch, pages_per_split=pps)


@pytest.mark.parametrize("pps,kernel", [(0, pgd.KERNEL_AUTO), (0, pgd.KERNEL_TENSOR_CORE),
                                        (2, pgd.KERNEL_TENSOR_CORE)])
def test_poisoned_slots_outside_attention_are_never_read(pps, kernel):
    """Every pool position no row attends to holds NaN: any read of it that
    reached the result would show (window kernel and split kernel)."""
    wl = Workload("poison", rows=6, q_heads=8, kv_heads=2, head_dim=128, ctx_lo=1, ctx_hi=600,
                  sinks=True)
    window = 70
    lay = layout_from_contexts(wl, [600, 1, 64, 65, 129, 300], seed=13)
    batch = make_batch(wl, seed=81, device=DEV, layout=lay)
    keep = np.zeros(lay.num_pages * 64, dtype=bool)
    for b, n in enumerate(lay.positions):
        for s in range(max(0, n - window + 1), n + 1):
            keep[lay.table[b, s // 64] * 64 + s % 64] = True
    nan_slots = torch.from_numpy(~keep).to(DEV)
    for pool in (batch.k_pool, batch.v_pool):
        view = pool.view(lay.num_pages, wl.kv_heads, 64, wl.head_dim)
        mask = nan_slots.view(lay.num_pages, 1, 64, 1).expand_as(view)
        view.masked_fill_(mask, float("nan"))
    run_and_check(batch, window=window, pages_per_split=pps, kernel=kernel)


@pytest.mark.parametrize("d", [64, 128])
def test_scores_far_below_zero(d):
    """q = -64 and every key 2 in every dimension: all scores equal and far
    below zero, so the output is the mean of V over the attended keys; a
    running maximum raised above the true one would zero every weight."""
    wl = Workload("negative", rows=4, q_heads=16, kv_heads=4, head_dim=d, ctx_lo=1, ctx_hi=900)
    lay = layout_from_contexts(wl, [900, 65, 1, 300], seed=29)
    batch = make_batch(wl, seed=111, device=DEV, layout=lay)
    batch.q.fill_(-64.0)
    batch.k_pool.fill_(2.0)
    batch.k_new.fill_(2.0)
    run_and_check(batch, sinks=None, what=f"negative scores d{d}")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("pps", [0, 2])
def test_scores_rise_every_page(d, pps):
    """Keys of logical page j equal to step * j, q = 1/4: scores grow by about
    23 log2 units per page, so the running maximum changes on every page and
    within a split every earlier page's weight is rescaled away."""
    wl = Workload("rising", rows=3, q_heads=16, kv_heads=4, head_dim=d, ctx_lo=1, ctx_hi=1500,
                  sinks=True)
    lay = layout_from_contexts(wl, [1500, 130, 64], seed=37)
    batch = make_batch(wl, seed=121, device=DEV, layout=lay)
    step = 8.0 if d == 64 else 6.0
    batch.q.fill_(0.25)
    view = batch.k_pool.view(lay.num_pages, wl.kv_heads, 64, d)
    for r, n in enumerate(lay.positions):
        for j in range(int(n) // 64 + 1):
            view[int(lay.table[r, j])] = step * j
    pages = torch.as_tensor(lay.positions // 64, device=DEV, dtype=torch.float32)
    batch.k_new = (pages.view(-1, 1, 1) * step).expand_as(batch.k_new).to(torch.bfloat16).contiguous()
    run_and_check(batch, pages_per_split=pps, what=f"rising scores d{d} pps{pps}")


@pytest.mark.parametrize("pps", [0, 1])   # one split (written directly); two (combined)
@pytest.mark.parametrize("window", [0, 64, 100])   # split kernel; window kernel (1 and 2 tiles)
def test_inactive_rows_are_zero_and_untouched(pps, window):
    wl = Workload("inactive", rows=4, q_heads=4, kv_heads=1, head_dim=64, ctx_lo=1, ctx_hi=128)
    lay = layout_from_contexts(wl, [0, 100, 0, 1], seed=17, num_pages=6)
    batch = make_batch(wl, seed=91, device=DEV, layout=lay)
    pgd.kv_append_paged(batch.k_new, batch.v_new, batch.table, batch.positions, batch.k_pool,
                        batch.v_pool)
    out = torch.full_like(batch.q, 7.0)          # every output must be written
    out = pgd.paged_decode_attention(batch.q, batch.k_pool, batch.v_pool, batch.table,
                                     batch.positions, None, window, wl.scale, out=out,
                                     num_kv_heads=wl.kv_heads, pages_per_split=pps)
    assert pgd.get_device_error() == pgd.OK
    assert torch.all(out[0] == 0) and torch.all(out[2] == 0)
    assert torch.any(out[1] != 0) and torch.all(out[3] != 7.0)


def test_zero_rows_is_a_no_op():
    q = torch.empty(0, 8, 64, dtype=torch.bfloat16, device=DEV)
    pool = torch.zeros(4 * 2 * 64 * 64, dtype=torch.bfloat16, device=DEV)
    table = torch.zeros(0, 3, dtype=torch.int32, device=DEV)
    pos = torch.zeros(0, dtype=torch.int32, device=DEV)
    out = pgd.paged_decode_attention(q, pool, pool, table, pos, num_kv_heads=2)
    assert out.shape == (0, 8, 64)


def test_kernel_count_follows_the_split_plan():
    """One kernel when every row fits one split (the split kernel writes the
    outputs), two when a row can span several (split + combine)."""
    def dims(wl, maxp, rows=None):
        return pgd.make_dims(rows=wl.rows if rows is None else rows, num_q_heads=wl.q_heads,
                             num_kv_heads=wl.kv_heads, head_dim=wl.head_dim, num_pages=100000,
                             max_pages_per_row=maxp)
    w = WORKLOADS
    assert pgd.attention_kernel_count(dims(w["qwen_serve"], 10)) == 1
    assert pgd.attention_kernel_count(dims(w["gptoss_full"], 64)) == 2       # 3 splits
    assert pgd.attention_kernel_count(dims(w["mistral_serve"], 512)) == 2    # 8 splits
    # windows of at most 128 positions: the window kernel alone (AUTO)
    assert pgd.attention_kernel_count(dims(w["gptoss_sliding"], 512), window=128) == 1
    assert pgd.attention_kernel_count(dims(w["gptoss_sliding"], 512), window=128,
                                      pages_per_split=1) == 1
    assert pgd.attention_kernel_count(dims(w["gptoss_sliding"], 512), window=128,
                                      pages_per_split=1,
                                      kernel=pgd.KERNEL_TENSOR_CORE) == 2    # 3 splits
    assert pgd.attention_kernel_count(dims(w["gptoss_sliding"], 512), window=129) == 1
    assert pgd.attention_kernel_count(dims(w["gptoss_sliding"], 512), window=129,
                                      pages_per_split=1) == 2
    assert pgd.attention_kernel_count(dims(w["qwen_serve"], 10), pages_per_split=10) == 1
    assert pgd.attention_kernel_count(dims(w["qwen_serve"], 10), pages_per_split=9) == 2
    assert pgd.attention_kernel_count(dims(w["qwen_serve"], 10),
                                      kernel=pgd.KERNEL_CUDA_CORE) == 1
    assert pgd.attention_kernel_count(dims(w["gptoss_full"], 64, rows=0)) == 0
    # prefill: tokens in runs take the tcgen05 kernel (after a pass that orders its
    # token blocks longest first, without a window); one token per row the split kernel
    assert pgd.attention_kernel_count(dims(w["mistral_serve"], 512, rows=4096), table_rows=8) == 2
    assert pgd.attention_kernel_count(dims(w["mistral_serve"], 512, rows=4096), table_rows=8,
                                      window=128) == 1
    assert pgd.attention_kernel_count(dims(w["mistral_serve"], 512, rows=4096), table_rows=8,
                                      kernel=pgd.KERNEL_PREFILL_TILED) == 1
    assert pgd.attention_kernel_count(dims(w["mistral_serve"], 512, rows=8), table_rows=8) == 2
    # one token per table row with a window: the per-token path, i.e. the window kernel
    assert pgd.attention_kernel_count(dims(w["gptoss_sliding"], 512, rows=8), table_rows=8,
                                      window=128) == 1


# ---------------------------------------------------------------------------
# Errors: caught on the host, or recorded on the device without a fault.


def test_device_bounds_errors_do_not_fault():
    wl = Workload("bounds", rows=3, q_heads=8, kv_heads=2, head_dim=64, ctx_lo=1, ctx_hi=200)
    lay = layout_from_contexts(wl, [200, 100, 50], seed=19, num_pages=10)
    batch = make_batch(wl, seed=101, device=DEV, layout=lay)
    bad_table = batch.table.clone()
    bad_table[1, 1] = 10 ** 6                      # row 1's last page: outside the pool
    out = pgd.paged_decode_attention(batch.q, batch.k_pool, batch.v_pool, bad_table,
                                     batch.positions, num_kv_heads=2)
    assert pgd.get_device_error() == pgd.EDEVICE_BOUNDS
    assert torch.all(out[1] == 0)
    bad_pos = batch.positions.clone()
    bad_pos[2] = 64 * batch.table.shape[1] + 5      # beyond the row's table
    for pps in (1, 0):        # split kernel, balanced kernel
        out = pgd.paged_decode_attention(batch.q, batch.k_pool, batch.v_pool, batch.table,
                                         bad_pos, num_kv_heads=2, pages_per_split=pps)
        assert pgd.get_device_error() == pgd.EDEVICE_BOUNDS
        assert torch.all(out[2] == 0) and torch.any(out[0] != 0)
    before = batch.k_pool.clone()
    pgd.kv_append_paged(batch.k_new, batch.v_new, bad_table, bad_pos, batch.k_pool, batch.v_pool)
    assert pgd.get_device_error() == pgd.EDEVICE_BOUNDS
    # rows 1 and 2 were skipped; row 0 was written
    changed = (batch.k_pool != before).view(-1, 64 * 64).any(dim=1).nonzero().flatten()
    assert changed.numel() == 2
    # the context is still healthy: a valid step matches the oracle
    batch2 = make_batch(wl, seed=102, device=DEV, layout=lay)
    run_and_check(batch2)


@pytest.mark.parametrize("pps", [1, 3, 5, 0])   # 10, 4 and 2 splits (combined); one split
def test_bad_table_entries_in_every_split(pps):
    """A bad table entry in the first split of one row and in a later split
    of another zeroes exactly those rows, whichever split holds it; a
    position beyond the table zeroes its row; the context stays usable."""
    wl = Workload("bounds_merge", rows=3, q_heads=16, kv_heads=2, head_dim=64, ctx_lo=1,
                  ctx_hi=600, sinks=True)
    lay = layout_from_contexts(wl, [600, 300, 100], seed=23)
    batch = make_batch(wl, seed=103, device=DEV, layout=lay)
    table = batch.table.clone()
    table[0, 7] = -1                  # row 0 (10 pages): a late split
    table[1, 1] = 10 ** 6             # row 1 (5 pages): the first split
    out = pgd.paged_decode_attention(batch.q, batch.k_pool, batch.v_pool, table,
                                     batch.positions, batch.sinks, 0, wl.scale,
                                     num_kv_heads=wl.kv_heads, pages_per_split=pps)
    assert pgd.get_device_error() == pgd.EDEVICE_BOUNDS
    assert torch.all(out[0] == 0) and torch.all(out[1] == 0) and torch.any(out[2] != 0)
    bad_pos = batch.positions.clone()
    bad_pos[0] = 64 * batch.table.shape[1] + 3
    out = pgd.paged_decode_attention(batch.q, batch.k_pool, batch.v_pool, batch.table, bad_pos,
                                     batch.sinks, 0, wl.scale, num_kv_heads=wl.kv_heads,
                                     pages_per_split=pps)
    assert pgd.get_device_error() == pgd.EDEVICE_BOUNDS
    assert torch.all(out[0] == 0) and torch.any(out[1] != 0) and torch.any(out[2] != 0)
    run_and_check(batch, pages_per_split=pps, what=f"after bounds errors, pps {pps}")


def test_window_kernel_reads_only_the_window_table_entries():
    """Window kernel: a bad table entry inside a row's window zeroes that row
    and is reported; a bad entry outside every window is never read."""
    wl = Workload("bounds_window", rows=3, q_heads=16, kv_heads=2, head_dim=64, ctx_lo=1,
                  ctx_hi=600, sinks=True)
    lay = layout_from_contexts(wl, [600, 300, 100], seed=23)
    batch = make_batch(wl, seed=104, device=DEV, layout=lay)
    host = snapshot_rows(batch, [1, 2])
    pgd.kv_append_paged(batch.k_new, batch.v_new, batch.table, batch.positions, batch.k_pool,
                        batch.v_pool)
    assert pgd.get_device_error() == pgd.OK
    table = batch.table.clone()
    table[1, 0] = 10 ** 6      # row 1 (n = 299): page 0 lies outside its window 200..299
    out = pgd.paged_decode_attention(batch.q, batch.k_pool, batch.v_pool, table,
                                     batch.positions, batch.sinks, 100, wl.scale,
                                     num_kv_heads=wl.kv_heads)
    assert pgd.get_device_error() == pgd.OK
    table[0, 9] = -1           # row 0 (n = 599): its window's last page
    out_bad = pgd.paged_decode_attention(batch.q, batch.k_pool, batch.v_pool, table,
                                         batch.positions, batch.sinks, 100, wl.scale,
                                         num_kv_heads=wl.kv_heads)
    assert pgd.get_device_error() == pgd.EDEVICE_BOUNDS
    assert torch.all(out_bad[0] == 0)
    assert torch.equal(out_bad[1:], out[1:])
    want, _, _ = oracle_step(batch, host, window=100, sinks=batch.sinks, scale=wl.scale)
    compare(out[1:], want, "window kernel, rows beside bad entries")
    # a position beyond its table row: that row is zero and reported
    bad_pos = batch.positions.clone()
    bad_pos[2] = 64 * batch.table.shape[1] + 5
    out_pos = pgd.paged_decode_attention(batch.q, batch.k_pool, batch.v_pool, batch.table,
                                         bad_pos, batch.sinks, 100, wl.scale,
                                         num_kv_heads=wl.kv_heads)
    assert pgd.get_device_error() == pgd.EDEVICE_BOUNDS
    assert torch.all(out_pos[2] == 0) and torch.equal(out_pos[:2], out[:2])


def test_window_kernel_large_ctas_bad_entries():
    """The window kernel's large CTAs (several units each): units whose row
    has a bad table entry inside its window or a position beyond its table
    leave early, zero their outputs and report; the other units of the same
    CTAs, which synchronise on barriers of their own, match the oracle."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    per_sm, units = window_rounds(64, 128, sms)
    if units <= per_sm:
        pytest.skip("large CTAs hold no more units per SM than one-unit CTAs")
    hkv = 8
    rows = (sms * per_sm) // hkv + 9
    wl = Workload("window_bad", rows=rows, q_heads=64, kv_heads=hkv, head_dim=64, ctx_lo=1,
                  ctx_hi=600, window=128, sinks=True)
    contexts = [[600, 300, 129, 64, 0, 1][b % 6] for b in range(rows)]
    lay = layout_from_contexts(wl, contexts, seed=29)
    batch = make_batch(wl, seed=105, device=DEV, layout=lay)
    batch.v_pool.mul_(0.25)
    batch.v_new.mul_(0.25)
    host = snapshot_rows(batch, np.arange(rows))
    pgd.kv_append_paged(batch.k_new, batch.v_new, batch.table, batch.positions, batch.k_pool,
                        batch.v_pool)
    assert pgd.get_device_error() == pgd.OK
    table = batch.table.clone()
    positions = batch.positions.clone()
    bad = [0, 7, 13, rows - 1]
    table[0, 9] = -1                               # row 0 (n = 599): its window's last page
    table[7, 4] = 10 ** 6                          # row 7 (n = 299): inside its window
    positions[13] = 64 * batch.table.shape[1] + 5  # beyond its table row
    table[rows - 1, 1] = 10 ** 6                   # last row (n = 599 or less), if in its window
    n_last = int(positions[rows - 1])
    if n_last < 0 or not (max(0, n_last - 127) // 64 <= 1 <= n_last // 64):
        bad.remove(rows - 1)
    out = pgd.paged_decode_attention(batch.q, batch.k_pool, batch.v_pool, table, positions,
                                     batch.sinks, 128, wl.scale, num_kv_heads=hkv)
    assert pgd.get_device_error() == pgd.EDEVICE_BOUNDS
    for b in bad:
        assert torch.all(out[b] == 0), f"row {b} not zeroed"
    want, _, _ = oracle_step(batch, host, window=128, sinks=batch.sinks, scale=wl.scale)
    good = np.array([b for b in range(rows) if b not in bad])
    compare(out.index_select(0, torch.as_tensor(good, device=out.device)), want[good],
            "window kernel large CTAs, rows beside bad ones")


def test_host_validation():
    q = torch.zeros(2, 8, 64, dtype=torch.bfloat16, device=DEV)
    pool = torch.zeros(4 * 2 * 64 * 64, dtype=torch.bfloat16, device=DEV)
    table = torch.zeros(2, 3, dtype=torch.int32, device=DEV)
    pos = torch.zeros(2, dtype=torch.int32, device=DEV)
    with pytest.raises(ValueError):
        pgd.paged_decode_attention(q.float(), pool, pool, table, pos, num_kv_heads=2)
    with pytest.raises(ValueError):
        pgd.paged_decode_attention(q.cpu(), pool, pool, table, pos, num_kv_heads=2)
    with pytest.raises(pgd.PgdError) as e:   # group of 16 has no kernel
        pgd.paged_decode_attention(torch.zeros(2, 32, 64, dtype=torch.bfloat16, device=DEV),
                                   pool, pool, table, pos, num_kv_heads=2)
    assert e.value.status == pgd.EUNSUPPORTED
    with pytest.raises(pgd.PgdError) as e:   # head_dim 96
        pgd.paged_decode_attention(torch.zeros(2, 8, 96, dtype=torch.bfloat16, device=DEV),
                                   torch.zeros(4 * 2 * 64 * 96, dtype=torch.bfloat16, device=DEV),
                                   torch.zeros(4 * 2 * 64 * 96, dtype=torch.bfloat16, device=DEV),
                                   table, pos, num_kv_heads=2)
    assert e.value.status == pgd.EUNSUPPORTED
    with pytest.raises(pgd.PgdError) as e:   # misaligned q
        raw = torch.zeros(2 * 8 * 64 + 1, dtype=torch.bfloat16, device=DEV)
        pgd.paged_decode_attention(raw[1:].view(2, 8, 64), pool, pool, table, pos,
                                   num_kv_heads=2)
    assert e.value.status == pgd.EINVAL
    with pytest.raises(pgd.PgdError) as e:   # workspace too small
        pgd.paged_decode_attention(q, pool, pool, table, pos, num_kv_heads=2,
                                   workspace=torch.zeros(16, dtype=torch.uint8, device=DEV),
                                   pages_per_split=1)
    assert e.value.status == pgd.EWORKSPACE


def test_cuda_graph_replay_matches_eager():
    wl = WORKLOADS["qwen_serve"]
    batch = make_batch(wl, seed=1001, device=DEV)
    want = gpu_step(batch, window=0, sinks=None, scale=wl.scale).clone()
    out = torch.empty_like(want)
    dims = pgd.make_dims(rows=wl.rows, num_q_heads=wl.q_heads, num_kv_heads=wl.kv_heads,
                         head_dim=wl.head_dim, num_pages=batch.layout.num_pages,
                         max_pages_per_row=batch.table.shape[1])
    ws = torch.empty(pgd.paged_decode_workspace_bytes(dims), dtype=torch.uint8, device=DEV)
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):   # warm up on the capture stream
        pgd.paged_decode_attention(batch.q, batch.k_pool, batch.v_pool, batch.table,
                                   batch.positions, None, 0, wl.scale, num_kv_heads=wl.kv_heads,
                                   out=out, workspace=ws)
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        pgd.kv_append_paged(batch.k_new, batch.v_new, batch.table, batch.positions,
                            batch.k_pool, batch.v_pool)
        pgd.paged_decode_attention(batch.q, batch.k_pool, batch.v_pool, batch.table,
                                   batch.positions, None, 0, wl.scale, num_kv_heads=wl.kv_heads,
                                   out=out, workspace=ws)
    out.zero_()
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, want)


def test_bounded_waits_time_out_into_an_error_and_the_context_survives():
    """A pipeline wait that nothing satisfies gives up after its limit and
    reports PGD_EDEVICE_TIMEOUT; no fault, and a normal step works after.
    The self-test also runs a decode split's give-up path after the timeout:
    a row's only split must leave zeros, and a split abandoned beside a valid
    one must make the combine's merge give zeros (no stale partial used)."""
    status, waits, abandoned = pgd.selftest_bounded_wait()
    assert status == pgd.EDEVICE_TIMEOUT
    assert waits == 0
    assert abandoned == 0
    wl = WORKLOADS["qwen_small"]
    batch = make_batch(wl, seed=1000, device=DEV)
    run_and_check(batch)
