"""Builds the producer's C-ABI shared library for sm_103a with nvcc, in-tree.

Output: ``paged_kv_cache_msa_gb300/lib/libmsa_producer.so`` (git-ignored).  Run as
``python -m paged_kv_cache_msa_gb300.build`` or call ``build()``.
"""
from __future__ import annotations

import hashlib
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
    """One nvcc command compiling and linking every source (kept for reference and
    as the digest's description of the flags; ``_compile`` runs the same flags per
    translation unit, in parallel, then links)."""
    return _nvcc_base(verbose_ptxas, extra) + ["-shared", "-o", out, *SOURCES] + _link_flags()


# Translation units of the normal build: the projection source once for its host
# code and once per kernel instantiation (see its "build units" section), so that
# the large kernels compile in parallel.  The checked build compiles each source once.
PROJECTION_UNITS = 9


def units(split: bool):
    out = []
    for src in SOURCES:
        if split and src.endswith("msa_projection.cu"):
            out += [(src, [f"-DMSA_PROJ_UNIT={k}"]) for k in range(PROJECTION_UNITS)]
        else:
            out.append((src, []))
    return out


def _nvcc_base(verbose_ptxas: bool = False, extra=()) -> list:
    home = cuda_home()
    cmd = [os.path.join(home, "bin", "nvcc"), "-O3", "-std=c++17", ARCH, "-lineinfo",
           "-Xcompiler", "-fPIC,-O2", "-I", INCLUDE, "-I", os.path.join(PKG, "csrc"), *extra]
    if verbose_ptxas:
        cmd.insert(1, "-Xptxas=-v")
    return cmd


def _link_flags() -> list:
    libdir = os.path.join(cuda_home(), "lib64")
    return ["-cudart", "shared", "-Xlinker", f"-rpath,{libdir}"]


DEPENDENCIES = SOURCES + HEADERS + [os.path.join(INCLUDE, h) for h in ("msa_producer.h", "msa_projection.h")]
STAMP_PATH = LIB_PATH + ".sha256"


def source_digest(defines=()) -> str:
    """SHA-256 over the bytes of every source and header the library is compiled
    from, this build script, the nvcc command line and the extra defines: a library
    is reused only when it was built from exactly these inputs (file times are not
    trusted: copies to another machine do not keep them reliably)."""
    h = hashlib.sha256()
    for path in DEPENDENCIES + [os.path.abspath(__file__)]:
        h.update(os.path.basename(path).encode())
        with open(path, "rb") as f:
            h.update(f.read())
    h.update(" ".join(nvcc_command("OUT", extra=[f"-D{d}" for d in defines])[1:]).encode())
    h.update(repr(units(True)).encode())
    return h.hexdigest()


def _fresh(lib: str, stamp: str, digest: str) -> bool:
    if not os.path.exists(lib) or not os.path.exists(stamp):
        return False
    with open(stamp) as f:
        return f.read().strip() == digest


def _compile(lib: str, stamp: str, digest: str, extra, verbose: bool = False,
             split: bool = True) -> None:
    """Compiles each translation unit to an object in parallel, then links them."""
    os.makedirs(OUT_DIR, exist_ok=True)
    tag = f"{os.path.basename(lib)}.{os.getpid()}"
    objs, procs = [], []
    for n, (src, unit_defs) in enumerate(units(split)):
        obj = os.path.join(OUT_DIR, f"{os.path.splitext(os.path.basename(src))[0]}.{n}.{tag}.o")
        cmd = _nvcc_base(verbose, list(extra) + unit_defs) + ["-c", "-o", obj, src]
        procs.append((cmd, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT,
                                            text=True)))
        objs.append(obj)
    failed, out = None, []
    for cmd, pr in procs:
        o, _ = pr.communicate()
        out.append(o)
        if pr.returncode != 0 and failed is None:
            failed = "nvcc failed:\n" + " ".join(cmd) + "\n" + o
    try:
        if failed:
            raise RuntimeError(failed)
        tmp = lib + f".{os.getpid()}.tmp"
        cmd = [os.path.join(cuda_home(), "bin", "nvcc"), ARCH, "-shared", "-o", tmp, *objs] + _link_flags()
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc link failed:\n" + " ".join(cmd) + "\n" + r.stdout + r.stderr)
    finally:
        for obj in objs:
            if os.path.exists(obj):
                os.remove(obj)
    if verbose:
        sys.stdout.write("".join(out))
    os.replace(tmp, lib)
    with open(stamp, "w") as f:
        f.write(digest)


def up_to_date(defines=()) -> bool:
    return _fresh(LIB_PATH, STAMP_PATH, source_digest(defines))


def build(force: bool = False, verbose: bool = False, defines=None) -> str:
    """Compiles the library unless the one on disk was built from the same sources
    and defines (a content hash, see ``source_digest``); returns its path.
    ``defines``: extra -D tuning macros (e.g. MSA_MIN_CTAS_PER_SM=4); by default the
    space-separated list in the MSA_BUILD_DEFINES environment variable (empty: the
    tuned defaults).  With MSA_NO_BUILD=1 an existing library is used as it is."""
    if defines is None:
        defines = tuple(os.environ.get("MSA_BUILD_DEFINES", "").split())
    if os.environ.get("MSA_NO_BUILD") == "1" and os.path.exists(LIB_PATH):
        return LIB_PATH
    digest = source_digest(defines)
    if force or not _fresh(LIB_PATH, STAMP_PATH, digest):
        _compile(LIB_PATH, STAMP_PATH, digest, [f"-D{d}" for d in defines], verbose)
    return LIB_PATH


CHECKED_LIB_PATH = os.path.join(OUT_DIR, "libmsa_producer_checked.so")


def build_checked(force: bool = False) -> str:
    """Compiles the checked library (-DMSA_CHECKED: every global store of the
    producer and projection kernels is checked against the extent of its
    destination, and a store outside it is skipped and counted) next to the normal
    one, and returns its path.  A diagnostic build; the product uses build()."""
    stamp = CHECKED_LIB_PATH + ".sha256"
    digest = source_digest(("MSA_CHECKED",))
    if force or not _fresh(CHECKED_LIB_PATH, stamp, digest):
        _compile(CHECKED_LIB_PATH, stamp, digest, ["-DMSA_CHECKED"], split=False)
    return CHECKED_LIB_PATH


STARVED_LIB_PATH = os.path.join(OUT_DIR, "libmsa_producer_starved.so")
STARVED_WAIT_LIMIT_NS = 50_000_000


def build_starved(force: bool = False) -> str:
    """Compiles the starved test library (-DMSA_STARVE, every bounded wait limited to
    STARVED_WAIT_LIMIT_NS): the projection's TMA warps and the query-run indexer's MMA
    thread issue nothing, so every wait on their barriers runs out with no copy or
    MMA in flight.  Only the tests of the timeout path load
    it; the product uses build()."""
    defs = ("MSA_STARVE", f"MSA_WAIT_LIMIT_NS={STARVED_WAIT_LIMIT_NS}ull")
    stamp = STARVED_LIB_PATH + ".sha256"
    digest = source_digest(defs)
    if force or not _fresh(STARVED_LIB_PATH, stamp, digest):
        _compile(STARVED_LIB_PATH, stamp, digest, [f"-D{d}" for d in defs])
    return STARVED_LIB_PATH


if __name__ == "__main__":
    defs = [a[2:] for a in sys.argv[1:] if a.startswith("-D")]
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, defines=defs or None))
