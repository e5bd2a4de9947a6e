"""Paged grouped-query decode attention for GB300 (sm_103a).

A thin binding over libpgd's C ABI (include/pgd.h): it turns torch tensors
into device pointers, sizes and the current CUDA stream, and nothing else.
Every step of the computation runs in the library's CUDA kernels; there is
no CPU or PyTorch fallback, and every call fails loudly if the library is
missing or the tensors are not on a CUDA device.

Entry points (same names as the C ABI, without the ``pgd_`` prefix):

- ``kv_append_paged``: write each row's new key and value at its page slot.
- ``paged_decode_attention``: grouped-query decode attention of each row over
  its pages, with optional per-head sink logits and sliding window.
- ``rope_append_paged``: rope_rows on q and k fused into the append.
- ``page_slots``, ``kv_write_slots``, ``paged_prefill_attention``: packed
  prompt tokens (prefill) and prompts plus decode steps in one pass.
- ``kv_append_rows``, ``decode_rows_attention``: the same step over dense
  per-row caches [Batch, KvHeads, MaxSeq, D] (decode_rows).
- ``paged_decode_workspace_bytes``, ``get_device_error``.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

import torch

PAGE_SIZE = 64
PAGE_MAJOR = 0
HEAD_MAJOR = 1
ROW_MAJOR = 2

OK, EINVAL, EUNSUPPORTED, ECUDA, EDEVICE_BOUNDS, EDEVICE_TIMEOUT, EWORKSPACE = range(7)

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "libpgd.so")

_lock = threading.Lock()
_lib = None


class PgdError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} (status {status})")


class Dims(ctypes.Structure):
    _fields_ = [(name, ctypes.c_int32) for name in (
        "rows", "num_q_heads", "num_kv_heads", "head_dim", "page_size", "num_pages",
        "max_pages_per_row", "layout")]


(KERNEL_AUTO, KERNEL_TENSOR_CORE, KERNEL_CUDA_CORE, KERNEL_PREFILL_TILED, KERNEL_PREFILL_UMMA,
 KERNEL_PREFILL_PAIR) = range(6)


class DecodeOptions(ctypes.Structure):
    _fields_ = [("pages_per_split", ctypes.c_int32), ("kernel", ctypes.c_int32)]


def load_library(path: str | None = None) -> ctypes.CDLL:
    """Loads libpgd.so (built by ``paged_gqa_decode_gb300.build``); raises if absent."""
    global _lib
    with _lock:
        if _lib is None:
            path = path or LIB_PATH
            if not os.path.exists(path):
                raise RuntimeError(
                    f"libpgd is not built ({path} missing): run "
                    "`python -c 'import __graft_entry__ as g; g.build()'`")
            lib = ctypes.CDLL(path)
            vp, i32 = ctypes.c_void_p, ctypes.c_int32
            dims_p = ctypes.POINTER(Dims)
            opts_p = ctypes.POINTER(DecodeOptions)
            lib.pgd_kv_append_paged.argtypes = [dims_p, vp, vp, vp, vp, vp, vp, vp]
            lib.pgd_kv_append_paged.restype = ctypes.c_int
            lib.pgd_rope_append_paged.argtypes = [dims_p, ctypes.c_float, vp, vp, vp, vp, vp,
                                                  vp, vp, vp, vp]
            lib.pgd_rope_append_paged.restype = ctypes.c_int
            lib.pgd_selftest_bounded_wait.argtypes = [vp, vp]
            lib.pgd_selftest_bounded_wait.restype = ctypes.c_int
            lib.pgd_page_slots.argtypes = [dims_p, i32, vp, vp, vp, vp, vp]
            lib.pgd_page_slots.restype = ctypes.c_int
            lib.pgd_kv_write_slots.argtypes = [dims_p, vp, vp, vp, vp, vp, vp]
            lib.pgd_kv_write_slots.restype = ctypes.c_int
            lib.pgd_paged_prefill_attention.argtypes = [dims_p, i32, vp, vp, vp, vp, vp, vp, vp,
                                                       i32, ctypes.c_float, vp, vp,
                                                       ctypes.c_size_t, opts_p, vp]
            lib.pgd_paged_prefill_attention.restype = ctypes.c_int
            lib.pgd_paged_prefill_step.argtypes = [dims_p, i32, vp, vp, vp, vp, vp, vp, vp, vp,
                                                   vp, i32, ctypes.c_float, vp, vp,
                                                   ctypes.c_size_t, opts_p, vp]
            lib.pgd_paged_prefill_step.restype = ctypes.c_int
            lib.pgd_prefill_step_kernel_count.argtypes = [dims_p, i32, i32, opts_p, vp]
            lib.pgd_prefill_step_kernel_count.restype = ctypes.c_int
            lib.pgd_paged_decode_workspace_bytes.argtypes = [dims_p, opts_p]
            lib.pgd_paged_decode_workspace_bytes.restype = ctypes.c_size_t
            lib.pgd_attention_kernel_count.argtypes = [dims_p, i32, i32, opts_p, vp]
            lib.pgd_attention_kernel_count.restype = ctypes.c_int
            lib.pgd_paged_decode_attention.argtypes = [dims_p, vp, vp, vp, vp, vp, vp, i32,
                                                      ctypes.c_float, vp, vp, ctypes.c_size_t,
                                                      opts_p, vp]
            lib.pgd_paged_decode_attention.restype = ctypes.c_int
            lib.pgd_paged_decode_step.argtypes = [dims_p, vp, vp, vp, vp, vp, vp, vp, vp, i32,
                                                  ctypes.c_float, vp, vp, ctypes.c_size_t,
                                                  opts_p, vp]
            lib.pgd_paged_decode_step.restype = ctypes.c_int
            lib.pgd_get_device_error.argtypes = [vp]
            lib.pgd_get_device_error.restype = ctypes.c_int
            lib.pgd_status_string.argtypes = [ctypes.c_int]
            lib.pgd_status_string.restype = ctypes.c_char_p
            lib.pgd_version.argtypes = []
            lib.pgd_version.restype = ctypes.c_int
            _lib = lib
    return _lib


def status_string(status: int) -> str:
    return load_library().pgd_status_string(status).decode()


def _stream_handle(stream: torch.cuda.Stream | None) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _ptr(t: torch.Tensor | None) -> int | None:
    return None if t is None else t.data_ptr()


def _check_cuda(*tensors: torch.Tensor | None) -> torch.device:
    device = None
    for t in tensors:
        if t is None:
            continue
        if not t.is_cuda:
            raise ValueError("paged_gqa_decode_gb300 runs on CUDA tensors only")
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous")
        if device is None:
            device = t.device
        elif t.device != device:
            raise ValueError("all tensors must be on one device")
    return device


def _dtype(t: torch.Tensor, dtype: torch.dtype, name: str) -> None:
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")


def make_dims(*, rows: int, num_q_heads: int, num_kv_heads: int, head_dim: int, num_pages: int,
              max_pages_per_row: int, layout: int = PAGE_MAJOR) -> Dims:
    return Dims(rows, num_q_heads, num_kv_heads, head_dim, PAGE_SIZE, num_pages,
                max_pages_per_row, layout)


def _pool_pages(pool: torch.Tensor, kv_heads: int, head_dim: int) -> int:
    per_page = kv_heads * PAGE_SIZE * head_dim
    if pool.numel() % per_page:
        raise ValueError(f"pool of {pool.numel()} values is not a whole number of pages")
    return pool.numel() // per_page


def kv_append_paged(k_new: torch.Tensor, v_new: torch.Tensor, table: torch.Tensor,
                    positions: torch.Tensor, k_pool: torch.Tensor, v_pool: torch.Tensor, *,
                    layout: int = PAGE_MAJOR, stream: torch.cuda.Stream | None = None) -> None:
    """Writes k_new/v_new (bf16 [R, Hkv, D]) into the pools at each row's slot:
    position positions[b] % 64 of page table[b][positions[b] // 64]."""
    dev = _check_cuda(k_new, v_new, table, positions, k_pool, v_pool)
    for t, n in ((k_new, "k_new"), (v_new, "v_new"), (k_pool, "k_pool"), (v_pool, "v_pool")):
        _dtype(t, torch.bfloat16, n)
    _dtype(table, torch.int32, "table")
    _dtype(positions, torch.int32, "positions")
    rows, hkv, d = k_new.shape
    if v_new.shape != k_new.shape or positions.shape != (rows,) or table.dim() != 2 \
            or table.shape[0] != rows or k_pool.shape != v_pool.shape:
        raise ValueError("inconsistent shapes")
    dims = make_dims(rows=rows, num_q_heads=hkv, num_kv_heads=hkv, head_dim=d,
                     num_pages=_pool_pages(k_pool, hkv, d), max_pages_per_row=table.shape[1],
                     layout=layout)
    with torch.cuda.device(dev):
        rc = load_library().pgd_kv_append_paged(
            ctypes.byref(dims), _ptr(k_new), _ptr(v_new), _ptr(table), _ptr(positions),
            _ptr(k_pool), _ptr(v_pool), _stream_handle(stream))
    if rc != OK:
        raise PgdError(rc, "kv_append_paged")


def paged_decode_workspace_bytes(dims: Dims, pages_per_split: int = 0) -> int:
    opts = DecodeOptions(pages_per_split, KERNEL_AUTO)
    return load_library().pgd_paged_decode_workspace_bytes(ctypes.byref(dims), ctypes.byref(opts))


def attention_kernel_count(dims: Dims, table_rows: int = 0, window: int = 0,
                           pages_per_split: int = 0, kernel: int = KERNEL_AUTO) -> int:
    """Kernels one paged_decode_attention (table_rows 0) or
    paged_prefill_attention (table_rows > 0) call with these arguments
    launches on the current device."""
    opts = DecodeOptions(pages_per_split, kernel)
    count = ctypes.c_int32(0)
    rc = load_library().pgd_attention_kernel_count(ctypes.byref(dims), int(table_rows),
                                                   int(window), ctypes.byref(opts),
                                                   ctypes.byref(count))
    if rc != OK:
        raise PgdError(rc, "attention_kernel_count")
    return count.value


def paged_decode_attention(q: torch.Tensor, k_pool: torch.Tensor, v_pool: torch.Tensor,
                           table: torch.Tensor, positions: torch.Tensor,
                           sinks: torch.Tensor | None = None, window: int = 0,
                           scale: float | None = None, *, num_kv_heads: int,
                           layout: int = PAGE_MAJOR, out: torch.Tensor | None = None,
                           workspace: torch.Tensor | None = None, pages_per_split: int = 0,
                           kernel: int = KERNEL_AUTO,
                           stream: torch.cuda.Stream | None = None) -> torch.Tensor:
    """Grouped-query decode attention of each row over its pages.

    q: bf16 [R, Hq, D]; pools: bf16 with num_kv_heads kv heads in ``layout``;
    table: int32 [R, max_pages]; positions: int32 [R]; sinks: fp32 [Hq] or
    None; window <= 0 for full attention.  Returns bf16 [R, Hq, D]."""
    return _decode(q, None, None, k_pool, v_pool, table, positions, sinks, window, scale,
                   num_kv_heads, layout, out, workspace, pages_per_split, kernel, stream)


def paged_decode_step(q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
                      k_pool: torch.Tensor, v_pool: torch.Tensor, table: torch.Tensor,
                      positions: torch.Tensor, sinks: torch.Tensor | None = None,
                      window: int = 0, scale: float | None = None, *, num_kv_heads: int,
                      layout: int = PAGE_MAJOR, out: torch.Tensor | None = None,
                      workspace: torch.Tensor | None = None, pages_per_split: int = 0,
                      kernel: int = KERNEL_AUTO,
                      stream: torch.cuda.Stream | None = None) -> torch.Tensor:
    """kv_append_paged then paged_decode_attention in one launch: each row's
    new K/V (bf16 [R, Hkv, D]) goes to its slot in the pools and the row
    attends over its pages, the new token included."""
    return _decode(q, k_new, v_new, k_pool, v_pool, table, positions, sinks, window, scale,
                   num_kv_heads, layout, out, workspace, pages_per_split, kernel, stream)


def _decode(q, k_new, v_new, k_pool, v_pool, table, positions, sinks, window, scale,
            num_kv_heads, layout, out, workspace, pages_per_split, kernel, stream):
    dev = _check_cuda(q, k_new, v_new, k_pool, v_pool, table, positions, sinks, out, workspace)
    _dtype(q, torch.bfloat16, "q")
    _dtype(k_pool, torch.bfloat16, "k_pool")
    _dtype(v_pool, torch.bfloat16, "v_pool")
    _dtype(table, torch.int32, "table")
    _dtype(positions, torch.int32, "positions")
    if sinks is not None:
        _dtype(sinks, torch.float32, "sinks")
    rows, hq, d = q.shape
    if positions.shape != (rows,) or table.dim() != 2 or table.shape[0] != rows \
            or k_pool.shape != v_pool.shape or (sinks is not None and sinks.shape != (hq,)):
        raise ValueError("inconsistent shapes")
    if k_new is not None:
        _dtype(k_new, torch.bfloat16, "k_new")
        _dtype(v_new, torch.bfloat16, "v_new")
        if k_new.shape != (rows, num_kv_heads, d) or v_new.shape != k_new.shape:
            raise ValueError("k_new and v_new must be [R, Hkv, D]")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dims = make_dims(rows=rows, num_q_heads=hq, num_kv_heads=num_kv_heads, head_dim=d,
                     num_pages=_pool_pages(k_pool, num_kv_heads, d),
                     max_pages_per_row=table.shape[1], layout=layout)
    opts = DecodeOptions(pages_per_split, kernel)
    lib = load_library()
    with torch.cuda.device(dev):
        if out is None:
            out = torch.empty_like(q)
        elif out.shape != q.shape or out.dtype != torch.bfloat16:
            raise ValueError("out must be bf16 shaped like q")
        need = lib.pgd_paged_decode_workspace_bytes(ctypes.byref(dims), ctypes.byref(opts))
        if workspace is None:
            workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
        tail = (_ptr(table), _ptr(positions), _ptr(sinks), int(window), float(scale), _ptr(out),
                _ptr(workspace), workspace.numel() * workspace.element_size(),
                ctypes.byref(opts), _stream_handle(stream))
        if k_new is None:
            rc = lib.pgd_paged_decode_attention(ctypes.byref(dims), _ptr(q), _ptr(k_pool),
                                                _ptr(v_pool), *tail)
            what = "paged_decode_attention"
        else:
            rc = lib.pgd_paged_decode_step(ctypes.byref(dims), _ptr(q), _ptr(k_new), _ptr(v_new),
                                           _ptr(k_pool), _ptr(v_pool), *tail)
            what = "paged_decode_step"
    if rc != OK:
        raise PgdError(rc, what)
    return out


def rope_append_paged(q: torch.Tensor | None, k_new: torch.Tensor, v_new: torch.Tensor,
                      table: torch.Tensor | None, positions: torch.Tensor, k_pool: torch.Tensor,
                      v_pool: torch.Tensor, *, theta: float, slots: torch.Tensor | None = None,
                      layout: int = PAGE_MAJOR, max_pages_per_row: int | None = None,
                      stream: torch.cuda.Stream | None = None) -> None:
    """rope_rows + append: rotates q (bf16 [R, Hq, D], in place) and k_new at
    positions[b] (base theta), writes rotated k and v into the pools at each
    row's slot (from the table, or the explicit slots)."""
    dev = _check_cuda(q, k_new, v_new, table, positions, slots, k_pool, v_pool)
    for t, n in ((k_new, "k_new"), (v_new, "v_new"), (k_pool, "k_pool"), (v_pool, "v_pool")):
        _dtype(t, torch.bfloat16, n)
    if q is not None:
        _dtype(q, torch.bfloat16, "q")
    _dtype(positions, torch.int32, "positions")
    rows, hkv, d = k_new.shape
    if v_new.shape != k_new.shape or positions.shape != (rows,) or k_pool.shape != v_pool.shape \
            or (q is not None and (q.shape[0] != rows or q.shape[2] != d)):
        raise ValueError("inconsistent shapes")
    width = table.shape[1] if table is not None else (max_pages_per_row or 1)
    dims = make_dims(rows=rows, num_q_heads=q.shape[1] if q is not None else hkv,
                     num_kv_heads=hkv, head_dim=d, num_pages=_pool_pages(k_pool, hkv, d),
                     max_pages_per_row=width, layout=layout)
    with torch.cuda.device(dev):
        rc = load_library().pgd_rope_append_paged(
            ctypes.byref(dims), float(theta), _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(table),
            _ptr(positions), _ptr(slots), _ptr(k_pool), _ptr(v_pool), _stream_handle(stream))
    if rc != OK:
        raise PgdError(rc, "rope_append_paged")


def page_slots(table: torch.Tensor, positions: torch.Tensor, rows: torch.Tensor | None = None, *,
               num_pages: int, stream: torch.cuda.Stream | None = None) -> torch.Tensor:
    """Pool position of each token: table[r][n // 64] * 64 + n % 64 with
    n = positions[p], r = rows[p] (rows None: r = p); -1 for n < 0."""
    dev = _check_cuda(table, positions, rows)
    _dtype(table, torch.int32, "table")
    _dtype(positions, torch.int32, "positions")
    if rows is not None:
        _dtype(rows, torch.int32, "rows")
        if rows.shape != positions.shape:
            raise ValueError("rows and positions must have one entry per token")
    elif table.shape[0] != positions.shape[0]:
        raise ValueError("without rows, the table needs one row per token")
    tokens = positions.shape[0]
    dims = make_dims(rows=tokens, num_q_heads=1, num_kv_heads=1, head_dim=64,
                     num_pages=num_pages, max_pages_per_row=table.shape[1])
    with torch.cuda.device(dev):
        slots = torch.empty(tokens, dtype=torch.int32, device=dev)
        rc = load_library().pgd_page_slots(ctypes.byref(dims), table.shape[0], _ptr(table),
                                           _ptr(rows), _ptr(positions), _ptr(slots),
                                           _stream_handle(stream))
    if rc != OK:
        raise PgdError(rc, "page_slots")
    return slots


def kv_write_slots(k_new: torch.Tensor, v_new: torch.Tensor, slots: torch.Tensor,
                   k_pool: torch.Tensor, v_pool: torch.Tensor, *, layout: int = PAGE_MAJOR,
                   stream: torch.cuda.Stream | None = None) -> None:
    """Writes token p's key and value (bf16 [P, Hkv, D]) at pool position slots[p]."""
    dev = _check_cuda(k_new, v_new, slots, k_pool, v_pool)
    for t, n in ((k_new, "k_new"), (v_new, "v_new"), (k_pool, "k_pool"), (v_pool, "v_pool")):
        _dtype(t, torch.bfloat16, n)
    _dtype(slots, torch.int32, "slots")
    tokens, hkv, d = k_new.shape
    if v_new.shape != k_new.shape or slots.shape != (tokens,) or k_pool.shape != v_pool.shape:
        raise ValueError("inconsistent shapes")
    dims = make_dims(rows=tokens, num_q_heads=hkv, num_kv_heads=hkv, head_dim=d,
                     num_pages=_pool_pages(k_pool, hkv, d), max_pages_per_row=1, layout=layout)
    with torch.cuda.device(dev):
        rc = load_library().pgd_kv_write_slots(ctypes.byref(dims), _ptr(k_new), _ptr(v_new),
                                               _ptr(slots), _ptr(k_pool), _ptr(v_pool),
                                               _stream_handle(stream))
    if rc != OK:
        raise PgdError(rc, "kv_write_slots")


def paged_prefill_attention(q: torch.Tensor, k_pool: torch.Tensor, v_pool: torch.Tensor,
                            table: torch.Tensor, rows: torch.Tensor, positions: torch.Tensor,
                            sinks: torch.Tensor | None = None, window: int = 0,
                            scale: float | None = None, *, num_kv_heads: int,
                            layout: int = PAGE_MAJOR, out: torch.Tensor | None = None,
                            workspace: torch.Tensor | None = None, pages_per_split: int = 0,
                            kernel: int = KERNEL_AUTO,
                            stream: torch.cuda.Stream | None = None) -> torch.Tensor:
    """Packed prompt tokens: token p (q bf16 [P, Hq, D]) attends over table row
    rows[p]'s pages up to positions[p].  Prompts and decode steps can share one
    call (a step of row b is a token with rows[p] = b).  Returns bf16 [P, Hq, D]."""
    return _prefill(q, None, None, k_pool, v_pool, table, rows, positions, sinks, window, scale,
                    num_kv_heads, layout, out, workspace, pages_per_split, kernel, stream)


def paged_prefill_step(q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
                       k_pool: torch.Tensor, v_pool: torch.Tensor, table: torch.Tensor,
                       rows: torch.Tensor, positions: torch.Tensor,
                       sinks: torch.Tensor | None = None, window: int = 0,
                       scale: float | None = None, *, num_kv_heads: int,
                       layout: int = PAGE_MAJOR, out: torch.Tensor | None = None,
                       workspace: torch.Tensor | None = None, pages_per_split: int = 0,
                       kernel: int = KERNEL_AUTO,
                       stream: torch.cuda.Stream | None = None) -> torch.Tensor:
    """The prefill call with the tokens' writes in it: token p's k_new / v_new
    (bf16 [P, Hkv, D]) go to its slot of table row rows[p] at positions[p],
    then every token attends as in paged_prefill_attention -- the same as
    page_slots + kv_write_slots + paged_prefill_attention.  Returns bf16
    [P, Hq, D]."""
    return _prefill(q, k_new, v_new, k_pool, v_pool, table, rows, positions, sinks, window,
                    scale, num_kv_heads, layout, out, workspace, pages_per_split, kernel, stream)


def _prefill(q, k_new, v_new, k_pool, v_pool, table, rows, positions, sinks, window, scale,
             num_kv_heads, layout, out, workspace, pages_per_split, kernel, stream):
    step = k_new is not None
    dev = _check_cuda(q, k_new, v_new, k_pool, v_pool, table, rows, positions, sinks, out,
                      workspace)
    _dtype(q, torch.bfloat16, "q")
    _dtype(k_pool, torch.bfloat16, "k_pool")
    _dtype(v_pool, torch.bfloat16, "v_pool")
    _dtype(table, torch.int32, "table")
    _dtype(rows, torch.int32, "rows")
    _dtype(positions, torch.int32, "positions")
    if sinks is not None:
        _dtype(sinks, torch.float32, "sinks")
    tokens, hq, d = q.shape
    if positions.shape != (tokens,) or rows.shape != (tokens,) or table.dim() != 2 \
            or k_pool.shape != v_pool.shape or (sinks is not None and sinks.shape != (hq,)):
        raise ValueError("inconsistent shapes")
    if step:
        if v_new is None:
            raise ValueError("k_new and v_new go together")
        _dtype(k_new, torch.bfloat16, "k_new")
        _dtype(v_new, torch.bfloat16, "v_new")
        if k_new.shape != (tokens, num_kv_heads, d) or v_new.shape != k_new.shape:
            raise ValueError("k_new and v_new are bf16 [P, Hkv, D]")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dims = make_dims(rows=tokens, num_q_heads=hq, num_kv_heads=num_kv_heads, head_dim=d,
                     num_pages=_pool_pages(k_pool, num_kv_heads, d),
                     max_pages_per_row=table.shape[1], layout=layout)
    opts = DecodeOptions(pages_per_split, kernel)
    lib = load_library()
    with torch.cuda.device(dev):
        if out is None:
            out = torch.empty_like(q)
        elif out.shape != q.shape or out.dtype != torch.bfloat16:
            raise ValueError("out must be bf16 shaped like q")
        need = lib.pgd_paged_decode_workspace_bytes(ctypes.byref(dims), ctypes.byref(opts))
        if workspace is None:
            workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
        ws = (_ptr(out), _ptr(workspace), workspace.numel() * workspace.element_size(),
              ctypes.byref(opts), _stream_handle(stream))
        tail = (_ptr(table), _ptr(rows), _ptr(positions), _ptr(sinks), int(window),
                float(scale))
        if step:
            rc = lib.pgd_paged_prefill_step(ctypes.byref(dims), table.shape[0], _ptr(q),
                                            _ptr(k_new), _ptr(v_new), _ptr(k_pool),
                                            _ptr(v_pool), *tail, *ws)
        else:
            rc = lib.pgd_paged_prefill_attention(ctypes.byref(dims), table.shape[0], _ptr(q),
                                                 _ptr(k_pool), _ptr(v_pool), *tail, *ws)
    if rc != OK:
        raise PgdError(rc, "paged_prefill_step" if step else "paged_prefill_attention")
    return out


def prefill_step_kernel_count(dims: Dims, table_rows: int, window: int = 0,
                              pages_per_split: int = 0, kernel: int = KERNEL_AUTO) -> int:
    """Kernels one paged_prefill_step call with these arguments launches on
    the current device."""
    opts = DecodeOptions(pages_per_split, kernel)
    count = ctypes.c_int32(0)
    rc = load_library().pgd_prefill_step_kernel_count(ctypes.byref(dims), int(table_rows),
                                                      int(window), ctypes.byref(opts),
                                                      ctypes.byref(count))
    if rc != OK:
        raise PgdError(rc, "prefill_step_kernel_count")
    return count.value


def _dense_dims(cache: torch.Tensor, rows: int, num_q_heads: int) -> Dims:
    if cache.dim() != 4 or cache.shape[2] % PAGE_SIZE:
        raise ValueError("dense caches are [Batch, KvHeads, MaxSeq, D] with MaxSeq % 64 == 0")
    batch, hkv, max_seq, d = cache.shape
    if rows > batch:
        raise ValueError("more rows than cache rows")
    per_row = max_seq // PAGE_SIZE
    return make_dims(rows=rows, num_q_heads=num_q_heads, num_kv_heads=hkv, head_dim=d,
                     num_pages=batch * per_row, max_pages_per_row=per_row, layout=ROW_MAJOR)


def kv_append_rows(k_new: torch.Tensor, v_new: torch.Tensor, positions: torch.Tensor,
                   cache_k: torch.Tensor, cache_v: torch.Tensor, *,
                   stream: torch.cuda.Stream | None = None) -> None:
    """write_rows: row b's new key and value (bf16 [R, Hkv, D]) go to position
    positions[b] of row b of the dense caches (bf16 [Batch, Hkv, MaxSeq, D])."""
    dev = _check_cuda(k_new, v_new, positions, cache_k, cache_v)
    for t, n in ((k_new, "k_new"), (v_new, "v_new"), (cache_k, "cache_k"), (cache_v, "cache_v")):
        _dtype(t, torch.bfloat16, n)
    _dtype(positions, torch.int32, "positions")
    if v_new.shape != k_new.shape or cache_k.shape != cache_v.shape \
            or positions.shape != (k_new.shape[0],):
        raise ValueError("inconsistent shapes")
    dims = _dense_dims(cache_k, k_new.shape[0], k_new.shape[1])
    with torch.cuda.device(dev):
        rc = load_library().pgd_kv_append_paged(
            ctypes.byref(dims), _ptr(k_new), _ptr(v_new), None, _ptr(positions), _ptr(cache_k),
            _ptr(cache_v), _stream_handle(stream))
    if rc != OK:
        raise PgdError(rc, "kv_append_rows")


def decode_rows_attention(q: torch.Tensor, cache_k: torch.Tensor, cache_v: torch.Tensor,
                          positions: torch.Tensor, sinks: torch.Tensor | None = None,
                          window: int = 0, scale: float | None = None, *,
                          out: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                          pages_per_split: int = 0, kernel: int = KERNEL_AUTO,
                          stream: torch.cuda.Stream | None = None) -> torch.Tensor:
    """decode_rows: row b's queries (q bf16 [R, Hq, D]) attend over row b of the
    dense caches (bf16 [Batch, Hkv, MaxSeq, D]) up to positions[b]."""
    return _decode_rows(q, None, None, cache_k, cache_v, positions, sinks, window, scale, out,
                        workspace, pages_per_split, kernel, stream)


def decode_rows_step(q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
                     cache_k: torch.Tensor, cache_v: torch.Tensor, positions: torch.Tensor,
                     sinks: torch.Tensor | None = None, window: int = 0,
                     scale: float | None = None, *, out: torch.Tensor | None = None,
                     workspace: torch.Tensor | None = None, pages_per_split: int = 0,
                     kernel: int = KERNEL_AUTO,
                     stream: torch.cuda.Stream | None = None) -> torch.Tensor:
    """kv_append_rows then decode_rows_attention in one launch."""
    return _decode_rows(q, k_new, v_new, cache_k, cache_v, positions, sinks, window, scale, out,
                        workspace, pages_per_split, kernel, stream)


def _decode_rows(q, k_new, v_new, cache_k, cache_v, positions, sinks, window, scale, out,
                 workspace, pages_per_split, kernel, stream):
    dev = _check_cuda(q, k_new, v_new, cache_k, cache_v, positions, sinks, out, workspace)
    _dtype(q, torch.bfloat16, "q")
    _dtype(cache_k, torch.bfloat16, "cache_k")
    _dtype(cache_v, torch.bfloat16, "cache_v")
    _dtype(positions, torch.int32, "positions")
    if sinks is not None:
        _dtype(sinks, torch.float32, "sinks")
    rows, hq, d = q.shape
    if cache_k.shape != cache_v.shape or positions.shape != (rows,) or cache_k.shape[3] != d \
            or (sinks is not None and sinks.shape != (hq,)):
        raise ValueError("inconsistent shapes")
    if k_new is not None:
        _dtype(k_new, torch.bfloat16, "k_new")
        _dtype(v_new, torch.bfloat16, "v_new")
        if k_new.shape != (rows, cache_k.shape[1], d) or v_new.shape != k_new.shape:
            raise ValueError("k_new and v_new must be [R, Hkv, D]")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dims = _dense_dims(cache_k, rows, hq)
    opts = DecodeOptions(pages_per_split, kernel)
    lib = load_library()
    with torch.cuda.device(dev):
        if out is None:
            out = torch.empty_like(q)
        need = lib.pgd_paged_decode_workspace_bytes(ctypes.byref(dims), ctypes.byref(opts))
        if workspace is None:
            workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
        tail = (None, _ptr(positions), _ptr(sinks), int(window), float(scale), _ptr(out),
                _ptr(workspace), workspace.numel() * workspace.element_size(),
                ctypes.byref(opts), _stream_handle(stream))
        if k_new is None:
            rc = lib.pgd_paged_decode_attention(ctypes.byref(dims), _ptr(q), _ptr(cache_k),
                                                _ptr(cache_v), *tail)
            what = "decode_rows_attention"
        else:
            rc = lib.pgd_paged_decode_step(ctypes.byref(dims), _ptr(q), _ptr(k_new), _ptr(v_new),
                                           _ptr(cache_k), _ptr(cache_v), *tail)
            what = "decode_rows_step"
    if rc != OK:
        raise PgdError(rc, what)
    return out


def selftest_bounded_wait(stream: torch.cuda.Stream | None = None) -> tuple[int, int, int]:
    """Runs the bounded-wait self-test (about 4 s): returns (device status,
    wait bits, abandoned-split bits); a correct run gives
    (EDEVICE_TIMEOUT, 0, 0)."""
    outcome = torch.full((2,), -1, dtype=torch.int32, device="cuda")
    rc = load_library().pgd_selftest_bounded_wait(_ptr(outcome), _stream_handle(stream))
    if rc != OK:
        raise PgdError(rc, "selftest_bounded_wait")
    status = get_device_error(stream)
    waits, abandoned = outcome.tolist()
    return status, int(waits), int(abandoned)


def get_device_error(stream: torch.cuda.Stream | None = None) -> int:
    """Synchronises the stream and returns (and clears) the device error word."""
    return load_library().pgd_get_device_error(_stream_handle(stream))
