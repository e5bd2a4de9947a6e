"""GPU parity for decode_rows over dense per-row caches [Batch, KvHeads,
MaxSeq, D] (the pages' decode_rows state): write_rows bit-exact, and decode
attention within the tolerance against the oracle's contiguous decode_rows."""
import numpy as np
import pytest
import torch

import oracle
import paged_gqa_decode_gb300 as pgd
from pgd_inputs import ROWS_WORKLOADS, Workload, bf16_bits, make_rows_batch
from tests.parity import compare

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    yield
    torch.cuda.synchronize()


def rows_check(b, *, window=None, sinks="batch", pps=0, kernel=pgd.KERNEL_AUTO, rows=None,
               step=False):
    wl = b.wl
    window = wl.window if window is None else window
    sinks = b.sinks if isinstance(sinks, str) else sinks
    idx = np.arange(len(b.positions_np)) if rows is None else np.asarray(rows)
    t = torch.as_tensor(idx, device=b.cache_k.device)
    k_host = bf16_bits(b.cache_k.index_select(0, t)).copy()
    v_host = bf16_bits(b.cache_v.index_select(0, t)).copy()
    if step:   # the append inside the decode launch
        out = pgd.decode_rows_step(b.q, b.k_new, b.v_new, b.cache_k, b.cache_v, b.positions,
                                   sinks, window, wl.scale, pages_per_split=pps, kernel=kernel)
    else:
        pgd.kv_append_rows(b.k_new, b.v_new, b.positions, b.cache_k, b.cache_v)
        out = pgd.decode_rows_attention(b.q, b.cache_k, b.cache_v, b.positions, sinks, window,
                                        wl.scale, pages_per_split=pps, kernel=kernel)
    assert pgd.get_device_error() == pgd.OK
    # the oracle's write_rows: row b's token goes to position n of row b
    kn, vn = bf16_bits(b.k_new)[idx], bf16_bits(b.v_new)[idx]
    for i, r in enumerate(idx):
        n = int(b.positions_np[r])
        if n >= 0:
            k_host[i, :, n, :] = kn[i]
            v_host[i, :, n, :] = vn[i]
    assert np.array_equal(bf16_bits(b.cache_k.index_select(0, t)), k_host)
    assert np.array_equal(bf16_bits(b.cache_v.index_select(0, t)), v_host)
    want, _, _ = oracle.decode_rows(bf16_bits(b.q)[idx], k_host, v_host, b.positions_np[idx],
                                    None if sinks is None else sinks.cpu().numpy(),
                                    window=window, scale=wl.scale)
    return compare(out.index_select(0, t), want, wl.name)


@pytest.mark.parametrize("step", [False, True])
@pytest.mark.parametrize("name", list(ROWS_WORKLOADS))
def test_rows_workloads(name, step):
    wl = ROWS_WORKLOADS[name]
    b = make_rows_batch(wl, 3000 + list(ROWS_WORKLOADS).index(name), DEV)
    rows_check(b, rows=None if name == "gptoss_rows_serve" else list(range(0, wl.rows, 8)),
               step=step)


@pytest.mark.parametrize("window", [0, 1, 64, 128])
@pytest.mark.parametrize("hq,hkv,d", [(64, 8, 64), (32, 8, 128), (14, 2, 64)])
@pytest.mark.parametrize("kernel,pps", [(pgd.KERNEL_AUTO, 0), (pgd.KERNEL_AUTO, 1),
                                        (pgd.KERNEL_CUDA_CORE, 2)])
@pytest.mark.parametrize("step", [False, True])
def test_rows_edges(window, hq, hkv, d, kernel, pps, step):
    wl = Workload("rows_edge", rows=7, q_heads=hq, kv_heads=hkv, head_dim=d, ctx_lo=1,
                  ctx_hi=320, sinks=True)
    b = make_rows_batch(wl, 7 + window + d, DEV, contexts=[1, 63, 64, 65, 129, 320, 0])
    rows_check(b, window=window, pps=pps, kernel=kernel, step=step)


def test_rows_fewer_rows_than_cache_rows():
    """A batch may use only the first rows of the caches."""
    wl = Workload("rows_part", rows=3, q_heads=8, kv_heads=2, head_dim=64, ctx_lo=1, ctx_hi=256)
    b = make_rows_batch(wl, 9, DEV, contexts=[100, 5, 256])
    extra = torch.zeros(2, 2, b.max_seq, 64, dtype=torch.bfloat16, device=DEV)
    b.cache_k = torch.cat([b.cache_k, extra]).contiguous()
    b.cache_v = torch.cat([b.cache_v, extra]).contiguous()
    rows_check(b)
    assert torch.all(b.cache_k[3:] == 0)
