"""Seeded synthetic workloads for paged grouped-query decode attention.

This module serves both the CUDA path and the oracle with the same inputs.
It holds none of the method's arithmetic: it draws contexts, assigns pool
pages to rows, and fills tensors with seeded random values.  Slot
computation, the append, and attention itself live only in the two
implementations under test.

Workload shapes follow the model cards of the "Nest" zoo: Qwen2.5-0.5B
(14 query / 2 kv heads, head_dim 64), gpt-oss-20b (64 / 8, head_dim 64,
per-head sink logits, 128-position sliding window on alternating layers),
Mistral-7B-v0.3 (32 / 8, head_dim 128).  Pages hold 64 positions.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch

PAGE_SIZE = 64


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    rows: int
    q_heads: int
    kv_heads: int
    head_dim: int
    ctx_lo: int          # row contexts (positions attended before the window) ~ U[ctx_lo, ctx_hi]
    ctx_hi: int
    window: int = 0      # <= 0: full causal attention
    sinks: bool = False
    pool_pages: int | None = None   # None: pages needed + 10 % slack
    page_size: int = PAGE_SIZE

    @property
    def group(self) -> int:
        return self.q_heads // self.kv_heads

    @property
    def max_pages_per_row(self) -> int:
        return math.ceil(self.ctx_hi / self.page_size)

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The five single-layer workloads; the first finishes in the oracle in
# seconds, the last is the large serving batch (tens of GB of pool).
WORKLOADS = {
    "qwen_small": Workload("qwen_small", rows=4, q_heads=14, kv_heads=2, head_dim=64,
                           ctx_lo=1, ctx_hi=300, pool_pages=32),
    "qwen_serve": Workload("qwen_serve", rows=64, q_heads=14, kv_heads=2, head_dim=64,
                           ctx_lo=129, ctx_hi=640),
    "gptoss_full": Workload("gptoss_full", rows=64, q_heads=64, kv_heads=8, head_dim=64,
                            ctx_lo=512, ctx_hi=4096, sinks=True),
    "gptoss_sliding": Workload("gptoss_sliding", rows=128, q_heads=64, kv_heads=8,
                               head_dim=64, ctx_lo=1, ctx_hi=32768, window=128, sinks=True),
    "mistral_serve": Workload("mistral_serve", rows=256, q_heads=32, kv_heads=8,
                              head_dim=128, ctx_lo=1024, ctx_hi=32768),
}


@dataclasses.dataclass
class PageLayout:
    contexts: np.ndarray     # int64 [R]; row b's new token sits at contexts[b] - 1
    positions: np.ndarray    # int32 [R]
    table: np.ndarray        # int32 [R, max_pages_per_row]; unused entries 0
    num_pages: int
    pages_used: int


def layout_from_contexts(wl: Workload, contexts, seed: int, num_pages: int | None = None,
                         table: np.ndarray | None = None) -> PageLayout:
    """Row b's new token sits at contexts[b] - 1 (a context <= 0 makes the row
    inactive).  Unless a table is given, each row gets ceil(context /
    page_size) distinct pages taken in order from a random permutation of the
    pool, so tables are shuffled and no two rows share a page; unused table
    entries are 0."""
    rng = np.random.default_rng(seed)
    contexts = np.asarray(contexts, dtype=np.int64)
    need = [max(0, math.ceil(int(c) / wl.page_size)) for c in contexts]
    used = int(sum(need))
    if num_pages is None:
        num_pages = wl.pool_pages if wl.pool_pages is not None else max(1, math.ceil(used * 1.1))
    if table is None:
        if used > num_pages:
            raise ValueError(f"{wl.name}: rows need {used} pages, pool holds {num_pages}")
        order = rng.permutation(num_pages).astype(np.int32)
        width = max(wl.max_pages_per_row, max(need, default=1), 1)
        table = np.zeros((len(contexts), width), dtype=np.int32)
        taken = 0
        for b, k in enumerate(need):
            table[b, :k] = order[taken:taken + k]
            taken += k
    positions = np.where(contexts > 0, contexts - 1, -1).astype(np.int32)
    return PageLayout(contexts, positions, np.ascontiguousarray(table, dtype=np.int32),
                      int(num_pages), used)


def draw_layout(wl: Workload, seed: int) -> PageLayout:
    """Contexts ~ U[ctx_lo, ctx_hi], then pages as in layout_from_contexts."""
    rng = np.random.default_rng(seed)
    contexts = rng.integers(wl.ctx_lo, wl.ctx_hi + 1, size=wl.rows).astype(np.int64)
    return layout_from_contexts(wl, contexts, seed + 1)


@dataclasses.dataclass
class Batch:
    wl: Workload
    layout: PageLayout
    q: torch.Tensor          # bf16 [R, Hq, D]
    k_new: torch.Tensor      # bf16 [R, Hkv, D]
    v_new: torch.Tensor      # bf16 [R, Hkv, D]
    k_pool: torch.Tensor     # bf16, flat, num_pages * Hkv * page_size * D values
    v_pool: torch.Tensor
    sinks: torch.Tensor | None   # fp32 [Hq]
    table: torch.Tensor      # int32 [R, max_pages]
    positions: torch.Tensor  # int32 [R]


def make_batch(wl: Workload, seed: int, device: str | torch.device = "cpu",
               layout: PageLayout | None = None) -> Batch:
    """q, k, v and pool contents ~ N(0, 1) in bf16, sinks ~ N(0, 1) in fp32,
    all from one seeded torch generator on ``device``."""
    layout = layout if layout is not None else draw_layout(wl, seed)
    device = torch.device(device)
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    rows = len(layout.positions)

    def normal(*shape, dtype=torch.bfloat16):
        return torch.randn(*shape, generator=gen, device=device, dtype=dtype)

    pool_len = layout.num_pages * wl.kv_heads * wl.page_size * wl.head_dim
    q = normal(rows, wl.q_heads, wl.head_dim)
    k_new = normal(rows, wl.kv_heads, wl.head_dim)
    v_new = normal(rows, wl.kv_heads, wl.head_dim)
    k_pool = normal(pool_len)
    v_pool = normal(pool_len)
    sinks = normal(wl.q_heads, dtype=torch.float32) if wl.sinks else None
    table = torch.from_numpy(layout.table).to(device)
    positions = torch.from_numpy(layout.positions).to(device)
    return Batch(wl, layout, q, k_new, v_new, k_pool, v_pool, sinks, table, positions)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """The uint16 bit patterns of a bf16 tensor, as a host numpy array."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)



# ---------------------------------------------------------------------------
# Prefill: packed prompt chunks over the paged pool.

@dataclasses.dataclass(frozen=True)
class PrefillWorkload:
    """`rows` requests, each with `prefix` positions already cached
    (~ U[prefix_lo, prefix_hi]) and a chunk of `chunk` new prompt tokens;
    the chunks are packed end to end into one pass of rows * chunk tokens."""
    name: str
    rows: int
    q_heads: int
    kv_heads: int
    head_dim: int
    prefix_lo: int
    prefix_hi: int
    chunk: int
    window: int = 0
    sinks: bool = False
    page_size: int = PAGE_SIZE

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)

    @property
    def max_pages_per_row(self) -> int:
        return math.ceil((self.prefix_hi + self.chunk) / self.page_size)

    def replace(self, **kw) -> "PrefillWorkload":
        return dataclasses.replace(self, **kw)


PREFILL_WORKLOADS = {
    "mistral_prefill": PrefillWorkload("mistral_prefill", rows=8, q_heads=32, kv_heads=8,
                                       head_dim=128, prefix_lo=0, prefix_hi=8192, chunk=512),
    "gptoss_prefill_sliding": PrefillWorkload("gptoss_prefill_sliding", rows=8, q_heads=64,
                                              kv_heads=8, head_dim=64, prefix_lo=0,
                                              prefix_hi=8192, chunk=256, window=128,
                                              sinks=True),
}


@dataclasses.dataclass
class PrefillBatch:
    wl: PrefillWorkload
    prefix: np.ndarray       # int64 [R] cached positions before each chunk
    table_np: np.ndarray     # int32 [R, max_pages]
    rows_np: np.ndarray      # int32 [P] table row of each packed token
    positions_np: np.ndarray  # int32 [P]
    num_pages: int
    q: torch.Tensor          # bf16 [P, Hq, D]
    k_new: torch.Tensor      # bf16 [P, Hkv, D]
    v_new: torch.Tensor
    k_pool: torch.Tensor
    v_pool: torch.Tensor
    sinks: torch.Tensor | None
    table: torch.Tensor
    rows: torch.Tensor
    positions: torch.Tensor


def make_prefill_batch(wl: PrefillWorkload, seed: int, device: str | torch.device = "cpu",
                       prefix=None, chunks=None) -> PrefillBatch:
    """Prefix lengths ~ U[prefix_lo, prefix_hi] (or given); row r's chunk is
    positions prefix[r] .. prefix[r] + chunk[r] - 1, packed row after row.
    Pages per row cover prefix + chunk, shuffled as in draw_layout."""
    rng = np.random.default_rng(seed)
    if prefix is None:
        prefix = rng.integers(wl.prefix_lo, wl.prefix_hi + 1, size=wl.rows)
    prefix = np.asarray(prefix, dtype=np.int64)
    chunks = np.full(len(prefix), wl.chunk, dtype=np.int64) if chunks is None \
        else np.asarray(chunks, dtype=np.int64)
    lay = layout_from_contexts(Workload(wl.name, len(prefix), wl.q_heads, wl.kv_heads,
                                        wl.head_dim, 1, int((prefix + chunks).max())),
                               prefix + chunks, seed + 1)
    rows_np = np.concatenate([np.full(c, r, dtype=np.int32) for r, c in enumerate(chunks)])
    positions_np = np.concatenate([np.arange(p, p + c, dtype=np.int32)
                                   for p, c in zip(prefix, chunks)])
    device = torch.device(device)
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)

    def normal(*shape, dtype=torch.bfloat16):
        return torch.randn(*shape, generator=gen, device=device, dtype=dtype)

    tokens = len(rows_np)
    pool_len = lay.num_pages * wl.kv_heads * wl.page_size * wl.head_dim
    q = normal(tokens, wl.q_heads, wl.head_dim)
    k_new = normal(tokens, wl.kv_heads, wl.head_dim)
    v_new = normal(tokens, wl.kv_heads, wl.head_dim)
    k_pool = normal(pool_len)
    v_pool = normal(pool_len)
    sinks = normal(wl.q_heads, dtype=torch.float32) if wl.sinks else None
    return PrefillBatch(wl, prefix, lay.table, rows_np, positions_np, lay.num_pages, q, k_new,
                        v_new, k_pool, v_pool, sinks, torch.from_numpy(lay.table).to(device),
                        torch.from_numpy(rows_np).to(device),
                        torch.from_numpy(positions_np).to(device))


# ---------------------------------------------------------------------------
# decode_rows: dense per-row caches [Batch, KvHeads, MaxSeq, D].

ROWS_WORKLOADS = {
    # the pages' own serving setup: 64 fixed cache rows of 640 positions,
    # prompts of 128-512 tokens plus up to 128 new ones (gpt-oss heads, sinks)
    "gptoss_rows_serve": Workload("gptoss_rows_serve", rows=64, q_heads=64, kv_heads=8,
                                  head_dim=64, ctx_lo=129, ctx_hi=640, sinks=True),
    "mistral_rows": Workload("mistral_rows", rows=64, q_heads=32, kv_heads=8, head_dim=128,
                             ctx_lo=1024, ctx_hi=8192),
}


@dataclasses.dataclass
class RowsBatch:
    wl: Workload
    contexts: np.ndarray
    positions_np: np.ndarray
    max_seq: int
    q: torch.Tensor          # bf16 [R, Hq, D]
    k_new: torch.Tensor      # bf16 [R, Hkv, D]
    v_new: torch.Tensor
    cache_k: torch.Tensor    # bf16 [R, Hkv, MaxSeq, D]
    cache_v: torch.Tensor
    sinks: torch.Tensor | None
    positions: torch.Tensor


def make_rows_batch(wl: Workload, seed: int, device: str | torch.device = "cpu",
                    contexts=None, max_seq: int | None = None) -> RowsBatch:
    """Contexts ~ U[ctx_lo, ctx_hi] (or given); MaxSeq = ctx_hi rounded up to a
    whole number of 64-position pages; caches, q, k, v ~ N(0, 1) bf16."""
    rng = np.random.default_rng(seed)
    if contexts is None:
        contexts = rng.integers(wl.ctx_lo, wl.ctx_hi + 1, size=wl.rows)
    contexts = np.asarray(contexts, dtype=np.int64)
    if max_seq is None:
        max_seq = int(math.ceil(max(wl.ctx_hi, int(contexts.max())) / wl.page_size) * wl.page_size)
    rows = len(contexts)
    device = torch.device(device)
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)

    def normal(*shape, dtype=torch.bfloat16):
        return torch.randn(*shape, generator=gen, device=device, dtype=dtype)

    q = normal(rows, wl.q_heads, wl.head_dim)
    k_new = normal(rows, wl.kv_heads, wl.head_dim)
    v_new = normal(rows, wl.kv_heads, wl.head_dim)
    cache_k = normal(rows, wl.kv_heads, max_seq, wl.head_dim)
    cache_v = normal(rows, wl.kv_heads, max_seq, wl.head_dim)
    sinks = normal(wl.q_heads, dtype=torch.float32) if wl.sinks else None
    positions_np = np.where(contexts > 0, contexts - 1, -1).astype(np.int32)
    return RowsBatch(wl, contexts, positions_np, max_seq, q, k_new, v_new, cache_k, cache_v,
                     sinks, torch.from_numpy(positions_np).to(device))
