"""Builds the producer's C-ABI shared library for sm_103a with nvcc, in-tree.

Output: ``paged_kv_cache_msa_gb300/lib/libmsa_producer.so`` (git-ignored).  Run as
``python -m paged_kv_cache_msa_gb300.build`` or call ``build()``.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
SOURCES = [os.path.join(PKG, "csrc", n) for n in ("msa_producer.cu", "msa_indexer.cu", "msa_projection.cu")]
HEADERS = [os.path.join(PKG, "csrc", "msa_internal.h")]
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(PKG, "lib")
LIB_NAME = "libmsa_producer.so"
LIB_PATH = os.path.join(OUT_DIR, LIB_NAME)

ARCH = "-gencode=arch=compute_103a,code=sm_103a"


def cuda_home() -> str:
    for cand in (os.environ.get("CUDA_HOME"), os.environ.get("CUDA_PATH"), "/usr/local/cuda"):
        if cand and os.path.exists(os.path.join(cand, "bin", "nvcc")):
            return cand
    nvcc = shutil.which("nvcc")
    if nvcc:
        return os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))
    raise RuntimeError("nvcc not found: set CUDA_HOME")


def nvcc_command(out: str, verbose_ptxas: bool = False, extra=()) -> list:
    home = cuda_home()
    libdir = os.path.join(home, "lib64")
    cmd = [os.path.join(home, "bin", "nvcc"), "-O3", "-std=c++17", ARCH, "-lineinfo",
           "-Xcompiler", "-fPIC,-O2", "-shared", "-cudart", "shared", "-I", INCLUDE,
           "-I", os.path.join(PKG, "csrc"),
           "-Xlinker", f"-rpath,{libdir}", "-o", out, *SOURCES, *extra]
    if verbose_ptxas:
        cmd.insert(1, "-Xptxas=-v")
    return cmd


STAMP_PATH = LIB_PATH + ".defines"


def up_to_date(defines=()) -> bool:
    if not os.path.exists(LIB_PATH) or not os.path.exists(STAMP_PATH):
        return False
    with open(STAMP_PATH) as f:
        if f.read() != " ".join(defines):
            return False
    t = os.path.getmtime(LIB_PATH)
    deps = SOURCES + HEADERS + [os.path.join(INCLUDE, h) for h in ("msa_producer.h", "msa_projection.h")]
    deps.append(os.path.abspath(__file__))
    return all(os.path.getmtime(d) <= t for d in deps)


def build(force: bool = False, verbose: bool = False, defines=None) -> str:
    """Compiles the library unless it is newer than its sources and was built with
    the same defines; returns its path.  ``defines``: extra -D tuning macros (e.g.
    MSA_MIN_CTAS_PER_SM=4); by default the space-separated list in the
    MSA_BUILD_DEFINES environment variable (empty: the tuned defaults).  With
    MSA_NO_BUILD=1 an existing library is used as it is."""
    if defines is None:
        defines = tuple(os.environ.get("MSA_BUILD_DEFINES", "").split())
    if os.environ.get("MSA_NO_BUILD") == "1" and os.path.exists(LIB_PATH):
        return LIB_PATH
    if not force and up_to_date(defines):
        return LIB_PATH
    os.makedirs(OUT_DIR, exist_ok=True)
    tmp = LIB_PATH + f".{os.getpid()}.tmp"
    cmd = nvcc_command(tmp, verbose_ptxas=verbose, extra=[f"-D{d}" for d in defines])
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("nvcc failed:\n" + " ".join(cmd) + "\n" + r.stdout + r.stderr)
    if verbose:
        sys.stdout.write(r.stdout + r.stderr)
    os.replace(tmp, LIB_PATH)
    with open(STAMP_PATH, "w") as f:
        f.write(" ".join(defines))
    return LIB_PATH


CHECKED_LIB_PATH = os.path.join(OUT_DIR, "libmsa_producer_checked.so")


def build_checked(force: bool = False) -> str:
    """Compiles the checked library (-DMSA_CHECKED: every global store of the
    producer and projection kernels is checked against the extent of its
    destination, and a store outside it is skipped and counted) next to the normal
    one, and returns its path.  A diagnostic build; the product uses build()."""
    stamp = CHECKED_LIB_PATH + ".stamp"
    deps = SOURCES + HEADERS + [os.path.join(INCLUDE, h) for h in ("msa_producer.h", "msa_projection.h")]
    deps.append(os.path.abspath(__file__))
    if (not force and os.path.exists(CHECKED_LIB_PATH) and os.path.exists(stamp)
            and all(os.path.getmtime(d) <= os.path.getmtime(CHECKED_LIB_PATH) for d in deps)):
        return CHECKED_LIB_PATH
    os.makedirs(OUT_DIR, exist_ok=True)
    tmp = CHECKED_LIB_PATH + f".{os.getpid()}.tmp"
    cmd = nvcc_command(tmp, extra=["-DMSA_CHECKED"])
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("nvcc failed:\n" + " ".join(cmd) + "\n" + r.stdout + r.stderr)
    os.replace(tmp, CHECKED_LIB_PATH)
    with open(stamp, "w") as f:
        f.write("MSA_CHECKED")
    return CHECKED_LIB_PATH


if __name__ == "__main__":
    defs = [a[2:] for a in sys.argv[1:] if a.startswith("-D")]
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, defines=defs or None))
