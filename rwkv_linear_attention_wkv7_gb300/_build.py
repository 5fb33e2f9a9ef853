"""Build libwkv7.so (the C-ABI CUDA library) in-tree with nvcc for sm_103a.

Each .cu under csrc/ is compiled to an object in parallel, then linked into
``libwkv7.so`` next to this file.  Rebuilds only when a source or header is
newer than the library.
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "libwkv7.so")
BUILD_DIR = os.path.join(ROOT, "_build")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
              "-Xptxas", "-warn-spills"]


def nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found; the CUDA toolkit is required to build libwkv7")
    return cand


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(INCLUDE, "*.h"))


# The files the two chunked kernels are compiled from (their measurements are
# keyed by a hash of these alone).
CHUNK_KERNEL_FILES = ("wkv7_chunk_fwd.cu", "wkv7_chunk_bwd.cu", "wkv7_chunk_bwd_exact.cuh", "wkv7_chunk_common.cuh",
                      "wkv7_mma.cuh", "wkv7_internal.cuh")


def source_hash(files=None) -> str:
    """Hash of every source and header the library is built from, or of the
    named csrc files only."""
    import hashlib
    h = hashlib.sha256()
    deps = _deps() if files is None else [os.path.join(CSRC, f) for f in files]
    for p in sorted(deps):
        h.update(os.path.basename(p).encode())
        with open(p, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def needs_build() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(p) > t for p in _deps())


def build(force: bool = False, verbose: bool = False, extra_flags=(), variant: str = "") -> str:
    """Build libwkv7.so, or with ``variant`` a separately named test build
    (libwkv7_<variant>.so, objects under _build/<variant>) compiled with
    ``extra_flags`` added (e.g. a -D switch only a test uses)."""
    lib = os.path.join(PKG, f"libwkv7_{variant}.so") if variant else LIB
    bdir = os.path.join(BUILD_DIR, variant) if variant else BUILD_DIR
    if not force and os.path.exists(lib) and not any(os.path.getmtime(p) > os.path.getmtime(lib) for p in _deps()):
        return lib
    os.makedirs(bdir, exist_ok=True)
    cc = nvcc()

    def compile_one(src):
        obj = os.path.join(bdir, os.path.basename(src) + ".o")
        cmd = [cc, *ARCH, *NVCC_FLAGS, *extra_flags, "-I", INCLUDE, "-I", CSRC, "-c", src, "-o", obj]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{res.stdout}\n{res.stderr}")
        if verbose and (res.stdout or res.stderr):
            print(res.stdout + res.stderr)
        return obj

    srcs = _sources()
    with ThreadPoolExecutor(max_workers=min(len(srcs), os.cpu_count() or 1)) as ex:
        objs = list(ex.map(compile_one, srcs))
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [cc, *ARCH, "-shared", "-o", tmp, *objs]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"link failed:\n{res.stdout}\n{res.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose=True))
