"""Build liblce.so in-tree (``chunked_lm_head_linear_gb300/_build/``) with nvcc for sm_103a.

Each translation unit compiles in its own nvcc process (in parallel), then one
link step produces the shared library. A stamp of the sources and flags skips
the rebuild when nothing changed.
"""
from __future__ import annotations

import hashlib
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "liblce.so")
# The bounds-checking debug build (-DLCE_CHECKS): every computed global index and
# TMA tile coordinate is checked in the kernels; a bad one sets a device status bit.
CHECKED_BUILD = os.path.join(BUILD, "checked")
CHECKED_LIB = os.path.join(CHECKED_BUILD, "liblce.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CFLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC,-O2", "--expt-relaxed-constexpr"]
INCLUDE = ["-I" + os.path.join(ROOT, "include")]
SOURCES = ["lce_kernels.cu", "lce_api.cu", "lce_noalloc.cu", "lce_rmsnorm.cu"]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build liblce.so")


def _stamp(extra=()) -> str:
    h = hashlib.sha256()
    for name in sorted(os.listdir(CSRC)) + ["../../include/lce.h"]:
        p = os.path.normpath(os.path.join(CSRC, name))
        if os.path.isfile(p):
            h.update(name.encode())
            with open(p, "rb") as f:
                h.update(f.read())
    h.update(" ".join(ARCH + CFLAGS + list(extra)).encode())  # not the checkout's path: same stamp anywhere
    return h.hexdigest()


def source_stamp() -> str:
    """Hash of the CUDA sources and build flags (identifies a kernel build)."""
    return _stamp()


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False, checks: bool = False) -> str:
    """Compile the CUDA library if its sources changed; return its path.
    ``checks``: the bounds-checking debug build, in its own directory."""
    out_dir = CHECKED_BUILD if checks else BUILD
    lib_path = CHECKED_LIB if checks else LIB
    os.makedirs(out_dir, exist_ok=True)
    extra = (["-Xptxas", "-v"] if ptxas_info else []) + (["-DLCE_CHECKS"] if checks else [])
    stamp = _stamp(extra)
    stamp_file = os.path.join(out_dir, "liblce.stamp")
    if (not force and os.path.exists(lib_path) and os.path.exists(stamp_file)
            and open(stamp_file).read() == stamp):
        return lib_path
    cc = nvcc()
    procs, objs = [], []
    for src in SOURCES:
        obj = os.path.join(out_dir, src.replace(".cu", ".o"))
        objs.append(obj)
        cmd = [cc, *ARCH, *CFLAGS, *INCLUDE, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            print(" ".join(cmd), flush=True)
        procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)))
    failed = []
    for src, p in procs:
        out, _ = p.communicate()
        if out and (verbose or p.returncode != 0 or ptxas_info):
            print(out, file=sys.stderr, flush=True)
        if p.returncode != 0:
            failed.append(src)
    if failed:
        raise RuntimeError(f"nvcc failed for {failed}")
    tmp = lib_path + f".{os.getpid()}.tmp"
    cmd = [cc, *ARCH, "-shared", "-o", tmp, *objs]
    subprocess.run(cmd, check=True)
    os.replace(tmp, lib_path)
    with open(stamp_file, "w") as f:
        f.write(stamp)
    return lib_path


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv,
                checks="--checks" in sys.argv))
