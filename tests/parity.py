"""Helpers for the GPU parity tests: run one append + decode step through the
C ABI, build the oracle's inputs from the same seeded batch (never from the
CUDA path's results), and compare with the tolerance the target states:
max abs error 1e-2 and max rel error 2e-2 for bf16 output from fp32
accumulation (rel evaluated where |oracle| >= 1e-3)."""
from __future__ import annotations

import numpy as np
import torch

import paged_gqa_decode_gb300 as pgd
from pgd_inputs import Batch
from tests.oracle_side import HostCopy, oracle_step, pages_of_row, snapshot_rows  # noqa: F401

ABS_TOL = 1e-2
REL_TOL = 2e-2
REL_FLOOR = 1e-3


def gpu_step(batch: Batch, *, window: int, sinks, scale: float, layout: int = pgd.PAGE_MAJOR,
             pages_per_split: int = 0, kernel: int = pgd.KERNEL_AUTO) -> torch.Tensor:
    wl = batch.wl
    pgd.kv_append_paged(batch.k_new, batch.v_new, batch.table, batch.positions, batch.k_pool,
                        batch.v_pool, layout=layout)
    out = pgd.paged_decode_attention(batch.q, batch.k_pool, batch.v_pool, batch.table,
                                     batch.positions, sinks, window, scale,
                                     num_kv_heads=wl.kv_heads, layout=layout,
                                     pages_per_split=pages_per_split, kernel=kernel)
    status = pgd.get_device_error()
    assert status == pgd.OK, pgd.status_string(status)
    return out


def compare(got: torch.Tensor, want: np.ndarray, what: str = "") -> dict:
    g = got.float().cpu().numpy().astype(np.float64)
    assert g.shape == want.shape, (g.shape, want.shape)
    assert np.all(np.isfinite(g)), f"{what}: non-finite output"
    diff = np.abs(g - want)
    big = np.abs(want) >= REL_FLOOR
    rel = diff[big] / np.abs(want[big]) if big.any() else np.zeros(1)
    stats = {"max_abs": float(diff.max(initial=0.0)), "max_rel": float(rel.max(initial=0.0))}
    assert stats["max_abs"] <= ABS_TOL, f"{what}: max abs error {stats}"
    assert stats["max_rel"] <= REL_TOL, f"{what}: max rel error {stats}"
    return stats
