"""Builds libbsa.so (the C-ABI library) in-tree for sm_103a.

    python -m block_sparse_attention_attn_gb300.build [--checks]

`--checks` builds the bounds-check variant libbsa_checks.so instead (the
kernels compiled with BSA_CHECKS=1: work items and list entries are validated
where they are read, a failure is recorded in the workspace header and
reported by bsa_check_status as 561002; selected with BSA_LIBRARY=checks).

Each translation unit is compiled in parallel with one ``-gencode``
(compute_103a -> sm_103a); the host API is compiled by nvcc as C++17 and the
CUDA runtime is linked statically, so the library needs only the driver
(libcuda, resolved at run time through the runtime's entry-point query).
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(ROOT, "_build")
LIB_DIR = os.path.join(HERE, "lib")
LIB_PATH = os.path.join(LIB_DIR, "libbsa.so")
LIB_CHECKS_PATH = os.path.join(LIB_DIR, "libbsa_checks.so")

SOURCES = ["bsa_api.cpp", "bsa_kernels.cu", "bsa_bwd.cu", "bsa_bwd_k64.cu", "bsa_bwd_dq.cu",
           "bsa_fwd.cu", "bsa_noalloc.cu"]
GENCODE = ["-gencode", "arch=compute_103a,code=sm_103a"]
COMMON = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-I" + INCLUDE, "-I" + CSRC]


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found")
    return cand


def _compile(src: str, verbose_ptxas: bool, bdir: str, extra: list) -> str:
    obj = os.path.join(bdir, os.path.splitext(src)[0] + ".o")
    cmd = [_nvcc(), *GENCODE, *COMMON, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
    if verbose_ptxas and src.endswith(".cu"):
        cmd += ["-Xptxas", "-v"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    if verbose_ptxas:
        sys.stderr.write(r.stderr)
    return obj


def _stale(lib: str) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(INCLUDE, "bsa.h")]
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose_ptxas: bool = False, checks: bool = False) -> str:
    """Compiles and links libbsa.so (with `checks`: libbsa_checks.so) if any
    source is newer; returns its path."""
    lib = LIB_CHECKS_PATH if checks else LIB_PATH
    if not force and not _stale(lib):
        return lib
    bdir = os.path.join(BUILD_DIR, "checks") if checks else BUILD_DIR
    extra = ["-DBSA_CHECKS=1"] if checks else []
    os.makedirs(bdir, exist_ok=True)
    os.makedirs(LIB_DIR, exist_ok=True)
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(s, verbose_ptxas, bdir, extra), SOURCES))
    tmp = lib + ".tmp"
    cmd = [_nvcc(), *GENCODE, "-shared", "-o", tmp, *objs, "-cudart", "static"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv,
                checks="--checks" in sys.argv))
