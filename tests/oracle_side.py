"""Oracle-side inputs for a batch: the pages of chosen rows copied out of
the seeded pool before the CUDA path runs, the oracle's own append, and its
decode.  Used by the parity tests and by the benchmark's CPU-baseline and
reference legs; it never imports the CUDA package."""
from __future__ import annotations

import dataclasses

import numpy as np
import torch

import oracle
from pgd_inputs import Batch, bf16_bits


@dataclasses.dataclass
class HostCopy:
    """Oracle-side inputs for a set of rows: their pages copied out of the
    pool BEFORE the CUDA path touched it, renumbered 0..k-1 in a compact pool
    (relabelling pages leaves the result unchanged), with the table
    rewritten to match."""
    rows: np.ndarray
    table: np.ndarray
    positions: np.ndarray
    k_pool: np.ndarray
    v_pool: np.ndarray
    num_pages: int


def pages_of_row(n: int, page_size: int = 64) -> int:
    return 0 if n < 0 else n // page_size + 1


def snapshot_rows(batch: Batch, rows, layout: int = oracle.PAGE_MAJOR) -> HostCopy:
    wl = batch.wl
    rows = np.asarray(rows, dtype=np.int64)
    table = batch.table.cpu().numpy()
    positions = batch.positions.cpu().numpy()
    used = []
    for b in rows:
        used.extend(int(p) for p in table[b, :pages_of_row(int(positions[b]))])
    uniq = sorted(set(used))
    remap = {p: i for i, p in enumerate(uniq)}
    ctable = np.zeros((len(rows), table.shape[1]), dtype=np.int32)
    for i, b in enumerate(rows):
        k = pages_of_row(int(positions[b]))
        ctable[i, :k] = [remap[int(p)] for p in table[b, :k]]
    idx = torch.tensor(uniq if uniq else [0], dtype=torch.long, device=batch.k_pool.device)
    tile = wl.page_size * wl.head_dim

    def gather(pool):
        if layout == oracle.PAGE_MAJOR:
            view = pool.view(-1, wl.kv_heads * tile)
            return bf16_bits(view.index_select(0, idx)).reshape(-1).copy()
        view = pool.view(wl.kv_heads, -1, tile)
        return bf16_bits(view.index_select(1, idx)).reshape(-1).copy()

    return HostCopy(rows, ctable, positions[rows].astype(np.int32), gather(batch.k_pool),
                    gather(batch.v_pool), max(len(uniq), 1))


def oracle_step(batch: Batch, host: HostCopy, *, window: int, sinks, scale: float,
                layout: int = oracle.PAGE_MAJOR, nthreads=None):
    """The oracle's own append (page_slots + write_tokens) followed by its
    decode, over the compact host pool."""
    wl = batch.wl
    slots = oracle.page_slots(host.table, host.positions, wl.page_size, host.num_pages)
    geo = dict(kv_heads=wl.kv_heads, head_dim=wl.head_dim, page_size=wl.page_size,
               num_pages=host.num_pages, layout=layout)
    k_new = bf16_bits(batch.k_new)[host.rows]
    v_new = bf16_bits(batch.v_new)[host.rows]
    oracle.write_tokens(host.k_pool, k_new, slots, **geo)
    oracle.write_tokens(host.v_pool, v_new, slots, **geo)
    sinks_np = None if sinks is None else sinks.detach().cpu().numpy().astype(np.float32)
    return oracle.decode_paged(bf16_bits(batch.q)[host.rows], host.k_pool, host.v_pool,
                               host.table, host.positions, kv_heads=wl.kv_heads,
                               page_size=wl.page_size, num_pages=host.num_pages, layout=layout,
                               sinks=sinks_np, window=window, scale=scale, nthreads=nthreads)


def snapshot_pages(k_pool: torch.Tensor, v_pool: torch.Tensor, table: np.ndarray, table_rows,
                   pages_per_row, *, kv_heads: int, head_dim: int, page_size: int = 64,
                   layout: int = oracle.PAGE_MAJOR):
    """Copies the first pages_per_row[i] pages of table rows table_rows[i] out
    of the pools into a compact pool (pages renumbered 0..k-1 in first-use
    order) and returns (k, v, compact table [len(table_rows), width],
    num_pages).  Relabelling pages leaves every oracle result unchanged."""
    uniq, remap = [], {}
    ctable = np.zeros((len(table_rows), table.shape[1]), dtype=np.int32)
    for i, (r, k) in enumerate(zip(table_rows, pages_per_row)):
        for j in range(int(k)):
            pg = int(table[r, j])
            if pg not in remap:
                remap[pg] = len(uniq)
                uniq.append(pg)
            ctable[i, j] = remap[pg]
    idx = torch.tensor(uniq if uniq else [0], dtype=torch.long, device=k_pool.device)
    tile = page_size * head_dim

    def gather(pool):
        if layout == oracle.PAGE_MAJOR:
            view = pool.view(-1, kv_heads * tile)
            return bf16_bits(view.index_select(0, idx)).reshape(-1).copy()
        view = pool.view(kv_heads, -1, tile)
        return bf16_bits(view.index_select(1, idx)).reshape(-1).copy()

    return gather(k_pool), gather(v_pool), ctable, max(len(uniq), 1)
