"""Builds libpgd.so in-tree (paged_gqa_decode_gb300/_build/) with nvcc for
sm_103a.  Each .cu is compiled in parallel, then linked into one shared
library whose only exported symbols are the C ABI of include/pgd.h."""
from __future__ import annotations

import concurrent.futures
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "libpgd.so")

SOURCES = ["pgd_api.cu", "kv_append.cu", "paged_decode_d64.cu", "paged_decode_d128.cu",
           "paged_prefill.cu", "paged_prefill_umma.cu", "paged_prefill_umma_d64.cu",
           "paged_prefill_pair.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-fvisibility=hidden",
         "-Xptxas", "-v", f"-I{INCLUDE}", f"-I{CSRC}"]


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libpgd")
    return path


def _inputs_newer_than(target: str) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(INCLUDE, "pgd.h"),
                                                                 __file__]
    return any(os.path.getmtime(d) > t for d in deps)


def _compile(src: str) -> tuple[str, str]:
    obj = os.path.join(BUILD, os.path.splitext(src)[0] + ".o")
    cmd = [nvcc(), *ARCH, *FLAGS, "-c", os.path.join(CSRC, src), "-o", obj]
    run = subprocess.run(cmd, capture_output=True, text=True)
    if run.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{run.stderr}")
    with open(os.path.join(BUILD, os.path.splitext(src)[0] + ".ptxas.txt"), "w") as f:
        f.write(run.stderr)
    return obj, run.stderr


def build_library(force: bool = False, verbose: bool = False) -> str:
    """Compiles and links libpgd.so if any source is newer than it."""
    os.makedirs(BUILD, exist_ok=True)
    if not force and not _inputs_newer_than(LIB):
        return LIB
    with concurrent.futures.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(_compile, SOURCES))
    objs = [o for o, _ in results]
    if verbose:
        for _, log in results:
            sys.stderr.write(log)
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [nvcc(), *ARCH, "-shared", "-Xlinker", "--exclude-libs,ALL", "-o", tmp, *objs]
    run = subprocess.run(cmd, capture_output=True, text=True)
    if run.returncode != 0:
        raise RuntimeError(f"link failed:\n{run.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build_library(force="--force" in sys.argv, verbose=True))
