"""The seeded workload generator: deterministic, shaped like the five
workloads, and producing valid shuffled page tables."""
import numpy as np
import pytest
import torch

from pgd_inputs import WORKLOADS, draw_layout, layout_from_contexts, make_batch


@pytest.mark.parametrize("name", list(WORKLOADS))
def test_layouts_are_valid_and_seeded(name):
    wl = WORKLOADS[name]
    a, b = draw_layout(wl, 1000), draw_layout(wl, 1000)
    assert np.array_equal(a.table, b.table) and np.array_equal(a.positions, b.positions)
    assert not np.array_equal(draw_layout(wl, 1001).contexts, a.contexts)
    assert a.contexts.min() >= wl.ctx_lo and a.contexts.max() <= wl.ctx_hi
    assert np.array_equal(a.positions, a.contexts - 1)
    assert a.table.shape == (wl.rows, wl.max_pages_per_row)
    assert a.num_pages >= a.pages_used
    listed = []
    for r in range(wl.rows):
        k = -(-int(a.contexts[r]) // wl.page_size)
        listed.extend(a.table[r, :k].tolist())
        assert not a.table[r, k:].any()            # padding entries are page 0
    assert len(set(listed)) == len(listed)         # no page shared between rows
    assert min(listed) >= 0 and max(listed) < a.num_pages
    if wl.pool_pages is not None:
        assert a.num_pages == wl.pool_pages


def test_small_batch_shapes_and_determinism():
    wl = WORKLOADS["qwen_small"].replace(sinks=True)
    x, y = make_batch(wl, 3), make_batch(wl, 3)
    assert x.q.shape == (4, 14, 64) and x.k_new.shape == (4, 2, 64)
    assert x.k_pool.numel() == 32 * 2 * 64 * 64 and x.sinks.shape == (14,)
    assert x.q.dtype == torch.bfloat16 and x.sinks.dtype == torch.float32
    assert torch.equal(x.k_pool, y.k_pool) and torch.equal(x.q, y.q)
    assert abs(float(x.k_pool.float().std()) - 1.0) < 0.05


def test_explicit_contexts_and_inactive_rows():
    wl = WORKLOADS["qwen_small"]
    lay = layout_from_contexts(wl, [0, 1, 64, 65], seed=0, num_pages=8)
    assert lay.positions.tolist() == [-1, 0, 63, 64]
    assert lay.pages_used == 0 + 1 + 1 + 2
    with pytest.raises(ValueError):
        layout_from_contexts(wl, [640, 640], seed=0, num_pages=8)
