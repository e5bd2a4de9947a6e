"""Randomised GPU parity: seeded random shapes (group sizes 1-8, head_dim 64
and 128), contexts (inactive rows, page boundaries, long rows), windows,
sinks, pool layouts, split sizes and kernel choices, for decode and for
packed prefill, each checked against the oracle like the hand-picked cases.
Every case is reproducible from its seed.

V is scaled by 1/4 (exact in bf16): with tiny windows an output is nearly a
single V row, and above |out| = 2.56 rounding to bf16 alone can exceed the
1e-2 absolute bound (a bf16 half-ulp at 4 is 1/64)."""
import numpy as np
import pytest

import paged_gqa_decode_gb300 as pgd
from pgd_inputs import PrefillWorkload, Workload, layout_from_contexts, make_batch, \
    make_prefill_batch
from tests.test_gpu_parity import run_and_check
from tests.test_gpu_prefill import prefill_check

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    yield


def heads(rng):
    hkv = int(rng.choice([1, 2, 3, 4, 8]))
    group = int(rng.integers(1, 9))
    return hkv * group, hkv


def context(rng, hi):
    kind = rng.integers(0, 4)
    if kind == 0:
        return 0                                   # inactive row
    if kind == 1:                                  # at or next to a page boundary
        return int(max(1, min(hi, 64 * rng.integers(1, hi // 64 + 1) + rng.integers(-1, 2))))
    return int(rng.integers(1, hi + 1))


@pytest.mark.parametrize("seed", range(64))
def test_random_decode(seed):
    rng = np.random.default_rng(7000 + seed)
    hq, hkv = heads(rng)
    d = int(rng.choice([64, 128]))
    rows = int(rng.integers(1, 13))
    hi = int(rng.choice([100, 700, 3000]))
    contexts = [context(rng, hi) for _ in range(rows)]
    if all(c == 0 for c in contexts):
        contexts[0] = 1
    window = int(rng.choice([0, 0, 1, 64, 128, int(rng.integers(2, 400))]))
    wl = Workload("random", rows=rows, q_heads=hq, kv_heads=hkv, head_dim=d, ctx_lo=1,
                  ctx_hi=hi, window=window, sinks=bool(rng.integers(0, 2)))
    lay = layout_from_contexts(wl, contexts, seed=seed)
    batch = make_batch(wl, seed=8000 + seed, device=DEV, layout=lay)
    batch.v_pool.mul_(0.25)
    batch.v_new.mul_(0.25)
    kernel = int(rng.choice([pgd.KERNEL_AUTO, pgd.KERNEL_TENSOR_CORE, pgd.KERNEL_CUDA_CORE]))
    pps = int(rng.choice([0, 0, 1, 2, 5]))
    layout = int(rng.choice([pgd.PAGE_MAJOR, pgd.HEAD_MAJOR]))
    run_and_check(batch, window=window, layout=layout, pages_per_split=pps, kernel=kernel,
                  what=f"seed {seed}: {hq}/{hkv} d{d} w{window} k{kernel} pps{pps} "
                       f"layout{layout} ctx {contexts}")


@pytest.mark.parametrize("seed", range(48))
def test_random_prefill(seed):
    rng = np.random.default_rng(9000 + seed)
    hq, hkv = heads(rng)
    d = int(rng.choice([64, 128]))
    rows = int(rng.integers(1, 5))
    prefix = [int(rng.choice([0, rng.integers(0, 64), rng.integers(0, 2000)])) for _ in range(rows)]
    chunks = [int(rng.choice([1, rng.integers(1, 70), rng.integers(60, 300)])) for _ in range(rows)]
    window = int(rng.choice([0, 0, 1, 128, int(rng.integers(2, 300))]))
    wl = PrefillWorkload("random", rows=rows, q_heads=hq, kv_heads=hkv, head_dim=d, prefix_lo=0,
                         prefix_hi=2000, chunk=0, window=window, sinks=bool(rng.integers(0, 2)))
    b = make_prefill_batch(wl, 9500 + seed, DEV, prefix=prefix, chunks=chunks)
    b.v_pool.mul_(0.25)
    b.v_new = b.v_new * 0.25
    kernel = int(rng.choice([pgd.KERNEL_AUTO, pgd.KERNEL_TENSOR_CORE, pgd.KERNEL_PREFILL_TILED,
                             pgd.KERNEL_PREFILL_UMMA]))
    layout = int(rng.choice([pgd.PAGE_MAJOR, pgd.HEAD_MAJOR]))
    prefill_check(b, window=window, layout=layout, kernel=kernel,
                  what=f"seed {seed}: {hq}/{hkv} d{d} w{window} k{kernel} layout{layout} "
                       f"prefix {prefix} chunks {chunks}")


@pytest.mark.parametrize("seed", range(24))
def test_random_prefill_pair(seed):
    """The paired-SM tcgen05 prefill (head_dim 128) on seeded random groups,
    prefixes, chunks, windows, sinks and layouts."""
    rng = np.random.default_rng(9700 + seed)
    hq, hkv = heads(rng)
    rows = int(rng.integers(1, 5))
    prefix = [int(rng.choice([0, rng.integers(0, 64), rng.integers(0, 2000)])) for _ in range(rows)]
    chunks = [int(rng.choice([1, rng.integers(1, 70), rng.integers(60, 300)])) for _ in range(rows)]
    window = int(rng.choice([0, 0, 1, 128, int(rng.integers(2, 300))]))
    wl = PrefillWorkload("random_pair", rows=rows, q_heads=hq, kv_heads=hkv, head_dim=128,
                         prefix_lo=0, prefix_hi=2000, chunk=0, window=window,
                         sinks=bool(rng.integers(0, 2)))
    b = make_prefill_batch(wl, 9900 + seed, DEV, prefix=prefix, chunks=chunks)
    b.v_pool.mul_(0.25)
    b.v_new = b.v_new * 0.25
    layout = int(rng.choice([pgd.PAGE_MAJOR, pgd.HEAD_MAJOR]))
    prefill_check(b, window=window, layout=layout, kernel=pgd.KERNEL_PREFILL_PAIR,
                  what=f"seed {seed}: {hq}/{hkv} w{window} layout{layout} prefix {prefix} "
                       f"chunks {chunks}")


@pytest.mark.parametrize("seed", range(24))
def test_random_prefill_key_parts(seed):
    """AUTO's key parts (few work items, tables of 16 pages or more) on seeded
    random groups, prefixes, chunks, windows, sinks and layouts."""
    rng = np.random.default_rng(9800 + seed)
    hq, hkv = heads(rng)
    d = int(rng.choice([64, 128]))
    rows = int(rng.integers(1, 4))
    prefix = [int(rng.integers(0, 3000)) for _ in range(rows)]
    prefix[0] = int(rng.integers(1100, 3000))  # a table of 16 pages or more
    chunks = [int(rng.choice([int(rng.integers(8, 70)), int(rng.integers(60, 300))]))
              for _ in range(rows)]
    window = int(rng.choice([0, 0, int(rng.integers(600, 2500))]))
    wl = PrefillWorkload("random_parts", rows=rows, q_heads=hq, kv_heads=hkv, head_dim=d,
                         prefix_lo=0, prefix_hi=3000, chunk=0, window=window,
                         sinks=bool(rng.integers(0, 2)))
    b = make_prefill_batch(wl, 9850 + seed, DEV, prefix=prefix, chunks=chunks)
    b.v_pool.mul_(0.25)
    b.v_new = b.v_new * 0.25
    layout = int(rng.choice([pgd.PAGE_MAJOR, pgd.HEAD_MAJOR]))
    prefill_check(b, window=window, layout=layout, fused=bool(rng.integers(0, 2)),
                  what=f"seed {seed}: {hq}/{hkv} d{d} w{window} layout{layout} prefix {prefix} "
                       f"chunks {chunks}")
