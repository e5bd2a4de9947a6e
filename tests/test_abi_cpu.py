"""The C ABI without a GPU: libpgd builds for sm_103a, loads, exports exactly
the symbols include/pgd.h declares, and rejects bad arguments on the host
before touching a device."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pgd.h")


@pytest.fixture(scope="module")
def lib():
    from paged_gqa_decode_gb300 import build
    path = build.build_library()
    import paged_gqa_decode_gb300 as pgd
    return pgd.load_library(path), path


def declared_symbols():
    text = open(HEADER).read()
    return set(re.findall(r"PGD_API\s+[\w\s\*]+?\b(pgd_\w+)\s*\(", text))


def test_header_declares_the_entry_points():
    assert declared_symbols() == {
        "pgd_kv_append_paged", "pgd_paged_decode_workspace_bytes", "pgd_paged_decode_attention",
        "pgd_get_device_error", "pgd_status_string", "pgd_version",
        "pgd_paged_decode_attention_static", "pgd_page_slots", "pgd_kv_write_slots",
        "pgd_paged_prefill_attention", "pgd_rope_append_paged", "pgd_selftest_bounded_wait",
        "pgd_attention_kernel_count", "pgd_paged_decode_step", "pgd_paged_prefill_step",
        "pgd_prefill_step_kernel_count"}


def test_library_exports_every_declared_symbol_and_nothing_else(lib):
    _, path = lib
    out = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True, text=True,
                         check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    assert declared_symbols() <= exported
    assert {s for s in exported if s.startswith("pgd_")} == declared_symbols()
    stray = {s for s in exported if not s.startswith("pgd_") and not s.startswith("_")}
    assert not stray, f"unexpected exports: {sorted(stray)[:10]}"


def test_status_strings_and_version(lib):
    import paged_gqa_decode_gb300 as pgd
    so, _ = lib
    assert so.pgd_version() >= 100
    for code in range(8):
        assert pgd.status_string(code) not in ("", "unknown status")
    assert pgd.status_string(99) == "unknown status"


def _dims(**kw):
    import paged_gqa_decode_gb300 as pgd
    base = dict(rows=2, num_q_heads=8, num_kv_heads=2, head_dim=64, num_pages=4,
                max_pages_per_row=3, layout=pgd.PAGE_MAJOR)
    base.update(kw)
    return pgd.make_dims(**base)


@pytest.mark.parametrize("kw,status", [
    (dict(num_q_heads=7), 1),          # Hq not a multiple of Hkv
    (dict(rows=-1), 1),
    (dict(num_kv_heads=0), 1),
    (dict(layout=5), 1),
    (dict(head_dim=96), 2),            # unsupported head_dim
    (dict(num_q_heads=32), 2),         # group of 16
    (dict(num_pages=2 ** 30), 2),      # pool rows beyond 32-bit TMA coordinates
])
def test_host_rejects_bad_dims_without_a_device(lib, kw, status):
    so, _ = lib
    d = _dims(**kw)
    rc = so.pgd_kv_append_paged(ctypes.byref(d), None, None, None, None, None, None, None)
    assert rc == status
    rc = so.pgd_paged_decode_attention(ctypes.byref(d), None, None, None, None, None, None, 0,
                                       0.125, None, None, 0, None, None)
    assert rc == status
    assert so.pgd_paged_decode_workspace_bytes(ctypes.byref(d), None) == 0
    rc = so.pgd_paged_decode_step(ctypes.byref(d), None, None, None, None, None, None, None,
                                  None, 0, 0.125, None, None, 0, None, None)
    assert rc == status
    count = ctypes.c_int32(-1)
    assert so.pgd_attention_kernel_count(ctypes.byref(d), 0, 0, None, ctypes.byref(count)) == status
    rc = so.pgd_paged_prefill_step(ctypes.byref(d), 2, None, None, None, None, None, None, None,
                                   None, None, 0, 0.125, None, None, 0, None, None)
    assert rc == status
    assert so.pgd_prefill_step_kernel_count(ctypes.byref(d), 2, 0, None,
                                            ctypes.byref(count)) == status


def test_bad_page_size_is_unsupported(lib):
    so, _ = lib
    d = _dims()
    d.page_size = 32
    assert so.pgd_kv_append_paged(ctypes.byref(d), None, None, None, None, None, None, None) == 2


def test_zero_rows_is_ok_and_null_pointers_are_rejected(lib):
    so, _ = lib
    d = _dims(rows=0)
    assert so.pgd_kv_append_paged(ctypes.byref(d), None, None, None, None, None, None, None) == 0
    d = _dims()
    assert so.pgd_kv_append_paged(ctypes.byref(d), None, None, None, None, None, None, None) == 1
    assert so.pgd_kv_append_paged(None, None, None, None, None, None, None, None) == 1
    assert so.pgd_attention_kernel_count(ctypes.byref(d), 0, 0, None, None) == 1
    buf = ctypes.create_string_buffer(64)   # any non-NULL host address: rejected before use
    assert so.pgd_paged_decode_step(ctypes.byref(d), buf, None, buf, buf, buf, buf, buf, None, 0,
                                    0.125, buf, buf, 64, None, None) == 1   # no k_new
    count = ctypes.c_int32(-1)
    assert so.pgd_attention_kernel_count(ctypes.byref(d), -1, 0, None, ctypes.byref(count)) == 1
    import paged_gqa_decode_gb300 as pgd
    opts = pgd.DecodeOptions(0, pgd.KERNEL_PREFILL_UMMA)   # a prefill kernel for a decode call
    assert so.pgd_attention_kernel_count(ctypes.byref(d), 0, 0, ctypes.byref(opts),
                                         ctypes.byref(count)) == 1
    pair = pgd.DecodeOptions(0, pgd.KERNEL_PREFILL_PAIR)
    d128 = _dims(head_dim=128)
    assert so.pgd_attention_kernel_count(ctypes.byref(d128), 0, 0, ctypes.byref(pair),
                                         ctypes.byref(count)) == 1   # decode call
    d64 = _dims(head_dim=64)
    assert so.pgd_attention_kernel_count(ctypes.byref(d64), 2, 0, ctypes.byref(pair),
                                         ctypes.byref(count)) == 1   # head_dim 128 only
    bad = pgd.DecodeOptions(0, pgd.KERNEL_PREFILL_PAIR + 1)
    assert so.pgd_attention_kernel_count(ctypes.byref(d), 2, 0, ctypes.byref(bad),
                                         ctypes.byref(count)) == 1   # no such kernel
    # the prefill step: rows, k_new and v_new are required; table_rows > 0
    assert so.pgd_paged_prefill_step(ctypes.byref(d), 2, buf, None, buf, buf, buf, buf, buf,
                                     buf, None, 0, 0.125, buf, buf, 64, None, None) == 1
    assert so.pgd_paged_prefill_step(ctypes.byref(d), 2, buf, buf, buf, buf, buf, buf, None,
                                     buf, None, 0, 0.125, buf, buf, 64, None, None) == 1
    assert so.pgd_prefill_step_kernel_count(ctypes.byref(d), 0, 0, None,
                                            ctypes.byref(count)) == 1
    assert so.pgd_prefill_step_kernel_count(ctypes.byref(d), 2, 0, None, None) == 1


def test_product_package_does_not_import_the_oracle():
    import ast
    pkg = os.path.join(ROOT, "paged_gqa_decode_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith(".py"):
                tree = ast.parse(open(os.path.join(dirpath, f)).read())
                for node in ast.walk(tree):
                    names = []
                    if isinstance(node, ast.Import):
                        names = [a.name for a in node.names]
                    elif isinstance(node, ast.ImportFrom):
                        names = [node.module or ""]
                    assert not any(n.split(".")[0] == "oracle" for n in names), f
            if f.endswith((".cu", ".cuh", ".h")):
                assert "oracle" not in open(os.path.join(dirpath, f)).read().lower(), f
