"""The bench's algorithmic work, counted by brute force on small cases: the
bytes a decode step and a prefill step must move at least once (the HBM
roofline's numerator) and the prefill FLOPs (the tensor roofline's)."""
import types

import numpy as np
import pytest

from bench import algorithmic_bytes, prefill_work
from pgd_inputs import PrefillWorkload, Workload


def attended(n, window):
    """Positions a query at position n attends: the definition, enumerated."""
    return [s for s in range(0, n + 1) if window <= 0 or s > n - window]


@pytest.mark.parametrize("window", [0, 1, 64, 128])
def test_decode_bytes_by_enumeration(window):
    wl = Workload("acct", rows=6, q_heads=14, kv_heads=2, head_dim=64, ctx_lo=1, ctx_hi=300,
                  window=window)
    positions = np.array([-1, 0, 5, 63, 64, 299])
    row = 2 * wl.kv_heads * wl.head_dim * 2  # one position's K and V over the kv heads
    kv = sum(len(attended(int(n), window)) for n in positions if n >= 0) * row
    q_out = 2 * len(positions) * wl.q_heads * wl.head_dim * 2
    append = 2 * int((positions >= 0).sum()) * row
    got = algorithmic_bytes(wl, positions)
    assert got == {"kv": kv, "q_out": q_out, "decode": kv + q_out, "append": append,
                   "step": kv + q_out + append}


@pytest.mark.parametrize("window", [0, 3, 128])
def test_prefill_work_by_enumeration(window):
    wl = PrefillWorkload("acct", rows=3, q_heads=8, kv_heads=2, head_dim=128, prefix_lo=0,
                         prefix_hi=10, chunk=4, window=window)
    # two chunks of row 0 (one gappy), one chunk of row 2, one token of row 1
    rows = np.array([0, 0, 0, 2, 2, 1, 0, 0], dtype=np.int32)
    positions = np.array([10, 11, 12, 0, 1, 7, 40, 41], dtype=np.int32)
    b = types.SimpleNamespace(positions_np=positions, rows_np=rows)
    row = 2 * wl.kv_heads * wl.head_dim * 2
    union = {}
    flops = 0
    for r, n in zip(rows.tolist(), positions.tolist()):
        keys = attended(n, window)
        union.setdefault(r, set()).update(keys)
        flops += len(keys) * wl.q_heads * wl.head_dim * 4
    kv = sum(len(u) for u in union.values()) * row
    tokens = len(positions)
    q_out = 2 * tokens * wl.q_heads * wl.head_dim * 2
    writes = 2 * tokens * row
    got = prefill_work(wl, b)
    assert got == {"kv": kv, "q_out": q_out, "writes": writes, "bytes": kv + q_out + writes,
                   "flops": flops, "tokens": tokens}
