"""fp64 CPU oracle for paged grouped-query decode attention (sink + window).

TEST INFRASTRUCTURE ONLY.  The test suite, the smoke check and the
benchmark's CPU-baseline leg may import this package; the product path
(``paged_gqa_decode_gb300``) never does, and this package never imports it.

The arithmetic lives in ``pgd_oracle.c`` (plain C, doubles, straight loops);
this module compiles it with gcc and marshals numpy arrays to it.  Arrays of
bf16 values are passed as their uint16 bit patterns.

Sources: Mistral 7B Instruct v0.3 model files, src/attention.linnet
(``decode_paged``: ``page_slots``, ``write_tokens``, ``paged_attention``);
GPT-OSS 20B model files, README "Attention sinks" and src/attention.linnet
(``SinkAttention.decode_rows``: the window mask and the sink).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

PAGE_MAJOR = 0
HEAD_MAJOR = 1

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pgd_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "liboracle.so")
# Test hook: the mutation tests point this at a deliberately broken build.
_LIB_OVERRIDE = os.environ.get("PGD_ORACLE_LIB")
_lock = threading.Lock()
_lib = None

_ERRORS = {1: "invalid argument", 2: "index out of range", 3: "out of memory"}


def build(force: bool = False) -> str:
    """Compiles the oracle into oracle/_build/liboracle.so (gcc, -O2, no fast-math)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(
            ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-o", tmp, _SRC, "-lm"],
            check=True,
        )
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(_LIB_OVERRIDE or build())
            p = ctypes.c_void_p
            i = ctypes.c_int
            lib.orc_page_slots.argtypes = [i, i, i, i, p, p, p]
            lib.orc_write_tokens.argtypes = [i, i, i, i, i, i, p, p, p]
            lib.orc_decode_rows.argtypes = [i, i, i, i, i, p, p, p, p, p, i, ctypes.c_float,
                                            p, p, p, i]
            lib.orc_decode_paged.argtypes = [i, i, i, i, i, i, i, i, p, p, p, p, p, p, i,
                                             ctypes.c_float, p, p, p, i]
            lib.orc_prefill_paged.argtypes = [i, i, i, i, i, i, i, i, i, p, p, p, p, p, p, p,
                                              i, ctypes.c_float, p, p, p, i]
            lib.orc_rope_table.argtypes = [i, ctypes.c_float, i, p, p]
            lib.orc_rope.argtypes = [i, i, i, ctypes.c_float, p, p, p]
            lib.orc_rope_table.restype = ctypes.c_int
            lib.orc_rope.restype = ctypes.c_int
            for fn in (lib.orc_page_slots, lib.orc_write_tokens, lib.orc_decode_rows,
                       lib.orc_decode_paged, lib.orc_prefill_paged):
                fn.restype = ctypes.c_int
            _lib = lib
    return _lib


def _check(rc: int, what: str) -> None:
    if rc != 0:
        raise ValueError(f"oracle {what}: {_ERRORS.get(rc, rc)}")


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def default_threads() -> int:
    return os.cpu_count() or 1


def page_slots(table: np.ndarray, positions: np.ndarray, page_size: int, num_pages: int) -> np.ndarray:
    """Pool position of each row's new token: table[b][n // P] * P + n % P (-1 if n < 0)."""
    table = _c(table, np.int32)
    positions = _c(positions, np.int32)
    rows, max_pages = table.shape
    slots = np.empty(rows, dtype=np.int64)
    _check(_load().orc_page_slots(rows, max_pages, page_size, num_pages, _ptr(table),
                                  _ptr(positions), _ptr(slots)), "page_slots")
    return slots


def write_tokens(pool: np.ndarray, kv_new: np.ndarray, slots: np.ndarray, *, kv_heads: int,
                 head_dim: int, page_size: int, num_pages: int, layout: int = PAGE_MAJOR) -> None:
    """Writes kv_new[b] (uint16 [rows, kv_heads, head_dim]) at slots[b] of ``pool`` in place."""
    assert pool.dtype == np.uint16 and pool.flags.c_contiguous
    kv_new = _c(kv_new, np.uint16)
    slots = _c(slots, np.int64)
    _check(_load().orc_write_tokens(kv_new.shape[0], kv_heads, head_dim, page_size, num_pages,
                                    layout, _ptr(slots), _ptr(kv_new), _ptr(pool)),
           "write_tokens")


def decode_rows(q, k, v, positions, sinks=None, window=0, scale=None, nthreads=None):
    """Decode attention over contiguous caches.

    q: uint16 [R, Hq, D]; k, v: uint16 [R, Hkv, L, D]; positions: int32 [R];
    sinks: float32 [Hq] or None.  Returns (out [R, Hq, D], lse [R, Hq],
    lse_real [R, Hq]) as float64.
    """
    q = _c(q, np.uint16)
    k = _c(k, np.uint16)
    v = _c(v, np.uint16)
    positions = _c(positions, np.int32)
    sinks = None if sinks is None else _c(sinks, np.float32)
    rows, hq, d = q.shape
    hkv, key_stride = k.shape[1], k.shape[2]
    if scale is None:
        scale = 1.0 / float(np.sqrt(d))
    out = np.empty((rows, hq, d), dtype=np.float64)
    lse = np.empty((rows, hq), dtype=np.float64)
    lse_real = np.empty((rows, hq), dtype=np.float64)
    _check(_load().orc_decode_rows(rows, hq, hkv, d, key_stride, _ptr(q), _ptr(k), _ptr(v),
                                   _ptr(positions), _ptr(sinks), int(window), float(scale),
                                   _ptr(out), _ptr(lse), _ptr(lse_real),
                                   nthreads or default_threads()), "decode_rows")
    return out, lse, lse_real


def decode_paged(q, k_pool, v_pool, table, positions, *, kv_heads, page_size=64, num_pages,
                 layout=PAGE_MAJOR, sinks=None, window=0, scale=None, nthreads=None):
    """Decode attention over a page pool (flat uint16 arrays in ``layout``).

    Row b attends over its positions 0..positions[b], found through
    table[b] (int32 [R, max_pages]).  Returns (out, lse, lse_real) as float64.
    """
    q = _c(q, np.uint16)
    k_pool = _c(k_pool, np.uint16)
    v_pool = _c(v_pool, np.uint16)
    table = _c(table, np.int32)
    positions = _c(positions, np.int32)
    sinks = None if sinks is None else _c(sinks, np.float32)
    rows, hq, d = q.shape
    max_pages = table.shape[1]
    if scale is None:
        scale = 1.0 / float(np.sqrt(d))
    expect = num_pages * kv_heads * page_size * d
    if k_pool.size != expect or v_pool.size != expect:
        raise ValueError(f"pool holds {k_pool.size} values, layout needs {expect}")
    out = np.empty((rows, hq, d), dtype=np.float64)
    lse = np.empty((rows, hq), dtype=np.float64)
    lse_real = np.empty((rows, hq), dtype=np.float64)
    _check(_load().orc_decode_paged(rows, hq, kv_heads, d, page_size, num_pages, max_pages,
                                    layout, _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(table),
                                    _ptr(positions), _ptr(sinks), int(window), float(scale),
                                    _ptr(out), _ptr(lse), _ptr(lse_real),
                                    nthreads or default_threads()), "decode_paged")
    return out, lse, lse_real


def prefill_paged(q, k_pool, v_pool, table, rows, positions, *, kv_heads, page_size=64,
                  num_pages, layout=PAGE_MAJOR, sinks=None, window=0, scale=None,
                  nthreads=None):
    """Paged prefill: token p (q uint16 [P, Hq, D]) attends over the pages of
    table row rows[p] up to positions[p], within the window, sink in the
    denominator.  Returns (out [P, Hq, D], lse [P, Hq], lse_real [P, Hq])."""
    q = _c(q, np.uint16)
    k_pool = _c(k_pool, np.uint16)
    v_pool = _c(v_pool, np.uint16)
    table = _c(table, np.int32)
    rows = _c(rows, np.int32)
    positions = _c(positions, np.int32)
    sinks = None if sinks is None else _c(sinks, np.float32)
    tokens, hq, d = q.shape
    table_rows, max_pages = table.shape
    if scale is None:
        scale = 1.0 / float(np.sqrt(d))
    expect = num_pages * kv_heads * page_size * d
    if k_pool.size != expect or v_pool.size != expect:
        raise ValueError(f"pool holds {k_pool.size} values, layout needs {expect}")
    out = np.empty((tokens, hq, d), dtype=np.float64)
    lse = np.empty((tokens, hq), dtype=np.float64)
    lse_real = np.empty((tokens, hq), dtype=np.float64)
    _check(_load().orc_prefill_paged(tokens, hq, kv_heads, d, page_size, num_pages, table_rows,
                                     max_pages, layout, _ptr(q), _ptr(k_pool), _ptr(v_pool),
                                     _ptr(table), _ptr(rows), _ptr(positions), _ptr(sinks),
                                     int(window), float(scale), _ptr(out), _ptr(lse),
                                     _ptr(lse_real), nthreads or default_threads()),
           "prefill_paged")
    return out, lse, lse_real


def rope_table(head_dim: int, theta: float, pos: int):
    """(cos, sin) uint16 bf16 bit patterns [head_dim / 2] at position pos."""
    c = np.empty(head_dim // 2, dtype=np.uint16)
    s = np.empty(head_dim // 2, dtype=np.uint16)
    _check(_load().orc_rope_table(head_dim, float(theta), int(pos), _ptr(c), _ptr(s)),
           "rope_table")
    return c, s


def rope(x, positions, theta: float):
    """rope_rows on x (uint16 bf16 bits [n, heads, D]) at positions [n]; bf16 out."""
    x = _c(x, np.uint16)
    positions = _c(positions, np.int32)
    n, heads, d = x.shape
    out = np.empty_like(x)
    _check(_load().orc_rope(n, heads, d, float(theta), _ptr(x), _ptr(positions), _ptr(out)),
           "rope")
    return out
