"""paged_decode_step (append fused into the decode launch) against the two
calls it replaces: the pools must end bit-identical to kv_append_paged's and
the output bit-identical to paged_decode_attention's over those pools (the
latter is checked against the oracle elsewhere); one case is also checked
against the oracle directly.  Covers several splits per row, windows,
inactive rows, both pool layouts, the CUDA-core consumer, a bad table entry
and CUDA-graph capture."""
import numpy as np
import pytest
import torch

import paged_gqa_decode_gb300 as pgd
from pgd_inputs import WORKLOADS, Workload, layout_from_contexts, make_batch
from tests.parity import compare, oracle_step, snapshot_rows

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    yield


def both(batch, *, window, sinks, layout=pgd.PAGE_MAJOR, pps=0, kernel=pgd.KERNEL_AUTO):
    wl = batch.wl
    kw = dict(num_kv_heads=wl.kv_heads, layout=layout, pages_per_split=pps, kernel=kernel)
    k1, v1 = batch.k_pool.clone(), batch.v_pool.clone()
    pgd.kv_append_paged(batch.k_new, batch.v_new, batch.table, batch.positions, k1, v1,
                        layout=layout)
    want = pgd.paged_decode_attention(batch.q, k1, v1, batch.table, batch.positions, sinks,
                                      window, wl.scale, **kw)
    assert pgd.get_device_error() == pgd.OK
    k2, v2 = batch.k_pool.clone(), batch.v_pool.clone()
    got = pgd.paged_decode_step(batch.q, batch.k_new, batch.v_new, k2, v2, batch.table,
                                batch.positions, sinks, window, wl.scale, **kw)
    assert pgd.get_device_error() == pgd.OK
    assert torch.equal(k1, k2) and torch.equal(v1, v2), "pools differ from kv_append_paged's"
    assert torch.equal(got, want), "output differs from append + decode"
    return got


@pytest.mark.parametrize("name", ["qwen_small", "qwen_serve", "gptoss_full"])
def test_step_workloads(name):
    wl = WORKLOADS[name]
    batch = make_batch(wl, seed=1000 + list(WORKLOADS).index(name), device=DEV)
    both(batch, window=wl.window, sinks=batch.sinks)


@pytest.mark.parametrize("hq,hkv,d", [(14, 2, 64), (64, 8, 64), (32, 8, 128), (6, 3, 128)])
@pytest.mark.parametrize("window", [0, 1, 65, 128])
@pytest.mark.parametrize("pps", [0, 1, 3])
@pytest.mark.parametrize("layout", [pgd.PAGE_MAJOR, pgd.HEAD_MAJOR])
def test_step_edges(hq, hkv, d, window, pps, layout):
    """Contexts around page boundaries and an inactive row; with pps 1 or 3
    the split kernel is asked for by name and the new token's page is the
    last of several splits; with pps 0 (AUTO) windows go to the window
    kernel, which takes the new token from k_new / v_new."""
    wl = Workload("step", rows=8, q_heads=hq, kv_heads=hkv, head_dim=d, ctx_lo=1, ctx_hi=700,
                  sinks=True)
    lay = layout_from_contexts(wl, [1, 63, 64, 65, 0, 129, 256, 700], seed=hq + d + window)
    batch = make_batch(wl, seed=41 + pps, device=DEV, layout=lay)
    kernel = pgd.KERNEL_AUTO if pps == 0 else pgd.KERNEL_TENSOR_CORE
    both(batch, window=window, sinks=batch.sinks, layout=layout, pps=pps, kernel=kernel)


@pytest.mark.parametrize("d", [64, 128])
def test_step_cuda_core_and_oracle(d):
    wl = Workload("step_cc", rows=5, q_heads=16, kv_heads=4, head_dim=d, ctx_lo=1, ctx_hi=400,
                  sinks=True)
    lay = layout_from_contexts(wl, [400, 1, 130, 0, 64], seed=7)
    batch = make_batch(wl, seed=77, device=DEV, layout=lay)
    both(batch, window=0, sinks=batch.sinks, kernel=pgd.KERNEL_CUDA_CORE)
    # and straight against the oracle (pools snapshotted before the step)
    rows = np.arange(wl.rows)
    host = snapshot_rows(batch, rows, pgd.PAGE_MAJOR)
    got = pgd.paged_decode_step(batch.q, batch.k_new, batch.v_new, batch.k_pool, batch.v_pool,
                                batch.table, batch.positions, batch.sinks, 0, wl.scale,
                                num_kv_heads=wl.kv_heads)
    assert pgd.get_device_error() == pgd.OK
    want, _, _ = oracle_step(batch, host, window=0, sinks=batch.sinks, scale=wl.scale,
                             layout=pgd.PAGE_MAJOR)
    compare(got, want, "decode_step vs oracle")


def test_step_bad_last_page_is_reported_and_not_written():
    wl = Workload("step_bad", rows=3, q_heads=8, kv_heads=2, head_dim=64, ctx_lo=1, ctx_hi=200)
    lay = layout_from_contexts(wl, [200, 100, 50], seed=19, num_pages=10)
    batch = make_batch(wl, seed=101, device=DEV, layout=lay)
    table = batch.table.clone()
    table[1, 1] = 10 ** 6            # row 1's last page (positions 64..99) lies outside the pool
    k0 = batch.k_pool.clone()
    out = pgd.paged_decode_step(batch.q, batch.k_new, batch.v_new, batch.k_pool, batch.v_pool,
                                table, batch.positions, num_kv_heads=2)
    assert pgd.get_device_error() == pgd.EDEVICE_BOUNDS
    assert torch.all(out[1] == 0) and torch.any(out[0] != 0) and torch.any(out[2] != 0)
    # rows 0 and 2 appended: their slot pages' tiles for both kv heads
    changed = (batch.k_pool != k0).view(-1, 64 * 64).any(dim=1).nonzero().flatten()
    assert changed.numel() == 4


@pytest.mark.parametrize("pps", [0, 3])   # one split per row; 4 splits + the combine
def test_step_in_a_cuda_graph(pps):
    wl = WORKLOADS["qwen_serve"]
    batch = make_batch(wl, seed=1001, device=DEV)
    k0, v0 = batch.k_pool.clone(), batch.v_pool.clone()
    eager = both(batch, window=0, sinks=None, pps=pps)
    out = torch.empty_like(batch.q)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        pgd.paged_decode_step(batch.q, batch.k_new, batch.v_new, batch.k_pool, batch.v_pool,
                              batch.table, batch.positions, None, 0, wl.scale, out=out,
                              num_kv_heads=wl.kv_heads, pages_per_split=pps)
        torch.cuda.synchronize()
        batch.k_pool.copy_(k0)
        batch.v_pool.copy_(v0)
        with torch.cuda.graph(g, stream=side):
            pgd.paged_decode_step(batch.q, batch.k_new, batch.v_new, batch.k_pool, batch.v_pool,
                                  batch.table, batch.positions, None, 0, wl.scale, out=out,
                                  num_kv_heads=wl.kv_heads, pages_per_split=pps)
    torch.cuda.synchronize()
    batch.k_pool.copy_(k0)
    batch.v_pool.copy_(v0)
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert pgd.get_device_error() == pgd.OK
    assert torch.equal(out, eager)
