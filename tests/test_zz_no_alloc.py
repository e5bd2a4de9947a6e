"""The decode entry point for callers that cannot allocate device memory.

pgd_paged_decode_attention_static takes no workspace: its split partials go
to a static device array inside the library.  It serves callers such as
plugins whose host runtime owns every device allocation, or code on paths
where cudaMalloc/cudaFree (which can synchronise the device) are not
allowed.  These tests call it through the C ABI:

- twice on the same problem, with a call on other data of the same shape in
  between (which leaves its own partials at the same places of the shared
  array); both results must be identical to the workspace entry point's,
  pgd_paged_decode_attention, with the same options (the same kernels run),
  so a partial left over from another call cannot go unnoticed;
- against the fp64 oracle directly (pool copied to the host before the
  append), so its parity does not rest on the other entry point;
- with a problem needing more scratch than the array holds, which is refused
  before anything launches.

This file is collected last on purpose: it must pass on its own in a fresh
process and after every other test."""
import ctypes

import numpy as np
import pytest
import torch

import paged_gqa_decode_gb300 as pgd
from pgd_inputs import WORKLOADS, layout_from_contexts, make_batch
from tests.parity import compare, oracle_step, snapshot_rows

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
ESCRATCH_LIMIT = 7

CASES = [
    ("gptoss_full", None, 0),
    ("gptoss_sliding", [1, 64, 65, 129, 4000, 32768], 0),
    ("mistral_serve", [1024, 1, 700, 2049, 5000, 32768], 3),
]


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    so = pgd.load_library()
    vp = ctypes.c_void_p
    so.pgd_paged_decode_attention_static.argtypes = [
        ctypes.POINTER(pgd.Dims), vp, vp, vp, vp, vp, vp, ctypes.c_int32, ctypes.c_float, vp,
        ctypes.POINTER(pgd.DecodeOptions), vp]
    so.pgd_paged_decode_attention_static.restype = ctypes.c_int
    return so


def static_decode(so, batch, window, pages_per_split=0):
    wl = batch.wl
    dims = pgd.make_dims(rows=len(batch.layout.positions), num_q_heads=wl.q_heads,
                         num_kv_heads=wl.kv_heads, head_dim=wl.head_dim,
                         num_pages=batch.layout.num_pages, max_pages_per_row=batch.table.shape[1])
    opts = pgd.DecodeOptions(pages_per_split)
    out = torch.full_like(batch.q, float("nan"))
    sinks = None if batch.sinks is None else batch.sinks.data_ptr()
    rc = so.pgd_paged_decode_attention_static(
        ctypes.byref(dims), batch.q.data_ptr(), batch.k_pool.data_ptr(), batch.v_pool.data_ptr(),
        batch.table.data_ptr(), batch.positions.data_ptr(), sinks, window, wl.scale,
        out.data_ptr(), ctypes.byref(opts), torch.cuda.current_stream().cuda_stream)
    assert rc == pgd.OK, pgd.status_string(rc)
    assert pgd.get_device_error() == pgd.OK
    return out


def case_batch(name, contexts, seed):
    wl = WORKLOADS[name]
    lay = None
    if contexts is not None:
        wl = wl.replace(rows=len(contexts))
        lay = layout_from_contexts(wl, contexts, seed=3)
    return make_batch(wl, seed=seed, device=DEV, layout=lay)


def append(batch):
    pgd.kv_append_paged(batch.k_new, batch.v_new, batch.table, batch.positions, batch.k_pool,
                        batch.v_pool)
    assert pgd.get_device_error() == pgd.OK


@pytest.mark.parametrize("name,contexts,pps", CASES)
def test_static_scratch_equals_workspace_entry_across_calls(lib, name, contexts, pps):
    wl = WORKLOADS[name]
    batch = case_batch(name, contexts, seed=500)
    append(batch)
    want = pgd.paged_decode_attention(batch.q, batch.k_pool, batch.v_pool, batch.table,
                                      batch.positions, batch.sinks, wl.window, wl.scale,
                                      num_kv_heads=wl.kv_heads, pages_per_split=pps)
    assert pgd.get_device_error() == pgd.OK
    first = static_decode(lib, batch, wl.window, pps)
    # the same shapes on other data: its partials overwrite the first call's
    other = case_batch(name, contexts, seed=501)
    append(other)
    between = static_decode(lib, other, wl.window, pps)
    assert not torch.equal(between, want)
    second = static_decode(lib, batch, wl.window, pps)
    assert torch.equal(first, want), f"{name}: first static call differs from the workspace entry"
    assert torch.equal(second, want), f"{name}: static call after another problem differs"


@pytest.mark.parametrize("name,contexts,pps", CASES[1:])
def test_static_scratch_against_the_oracle(lib, name, contexts, pps):
    wl = WORKLOADS[name]
    batch = case_batch(name, contexts, seed=502)
    rows = np.arange(len(contexts))
    host = snapshot_rows(batch, rows)
    append(batch)
    got = static_decode(lib, batch, wl.window, pps)
    want, _, _ = oracle_step(batch, host, window=wl.window, sinks=batch.sinks, scale=wl.scale)
    compare(got, want, f"static scratch {name} vs oracle")


def test_static_scratch_refuses_problems_beyond_its_size(lib):
    wl = WORKLOADS["mistral_serve"]
    dims = pgd.make_dims(rows=4096, num_q_heads=64, num_kv_heads=8, head_dim=128,
                         num_pages=1024, max_pages_per_row=512)
    opts = pgd.DecodeOptions(1)
    need = pgd.paged_decode_workspace_bytes(dims, 1)
    assert need > 64 * 2 ** 20
    out = torch.zeros(4, dtype=torch.bfloat16, device=DEV)
    rc = lib.pgd_paged_decode_attention_static(
        ctypes.byref(dims), out.data_ptr(), out.data_ptr(), out.data_ptr(), out.data_ptr(),
        out.data_ptr(), None, 0, wl.scale, out.data_ptr(), ctypes.byref(opts),
        torch.cuda.current_stream().cuda_stream)
    assert rc == ESCRATCH_LIMIT
    assert pgd.status_string(rc) != "unknown status"
    assert torch.all(out == 0)
