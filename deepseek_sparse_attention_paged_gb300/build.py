"""Builds ``libdsa_gb300.so`` (the C-ABI library) in-tree from ``csrc/*.cu`` with nvcc for sm_103a.

Each translation unit is compiled in parallel to ``_build/*.o`` and the objects are linked into a
shared library next to this file.  No torch headers are involved: the library's interface is the
plain C header ``include/dsa.h``.
"""
from __future__ import annotations

import glob
import hashlib
import os
import platform
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libdsa_gb300.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
              "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA library cannot be built")


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


STAMP = LIB + ".hash"


def _inputs_hash() -> str:
    """sha256 over every source and header the library is built from, the nvcc flags and nvcc's
    version line: the library is rebuilt whenever any of them differs from the last build's."""
    h = hashlib.sha256()
    deps = sorted(sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(INCLUDE, "*.h")))
    for p in deps:
        h.update(os.path.relpath(p, ROOT).encode())
        with open(p, "rb") as f:
            h.update(f.read())
    h.update(" ".join(ARCH + NVCC_FLAGS).replace(ROOT, "<root>").encode())
    try:
        v = subprocess.run([nvcc(), "--version"], stdout=subprocess.PIPE, stderr=subprocess.STDOUT).stdout
        h.update(v.strip().splitlines()[-1] if v.strip() else b"")
    except Exception:
        pass
    h.update(platform.machine().encode())
    return h.hexdigest()


def _stale(digest: str) -> bool:
    if not os.path.exists(LIB) or not os.path.exists(STAMP):
        return True
    with open(STAMP) as f:
        return f.read().strip() != digest


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False) -> str:
    """Compile and link the library unless the last build was made from the same sources, flags,
    compiler and machine type (a hash stored beside the library); returns the library path."""
    digest = _inputs_hash()
    if not force and not _stale(digest):
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    exe = nvcc()
    procs = []
    objs = []
    for src in sources():
        obj = os.path.join(BUILD, os.path.basename(src)[:-3] + ".o")
        objs.append(obj)
        cmd = [exe] + ARCH + NVCC_FLAGS + (["-Xptxas", "-v"] if ptxas_info else []) + ["-c", src, "-o", obj]
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
    failed = []
    for src, p in procs:
        out, _ = p.communicate()
        text = out.decode(errors="replace")
        if p.returncode != 0:
            failed.append((src, text))
        elif verbose or ptxas_info:
            sys.stderr.write(text)
    if failed:
        msg = "\n".join(f"--- {s}\n{t}" for s, t in failed)
        raise RuntimeError(f"nvcc failed:\n{msg}")
    tmp = LIB + f".tmp{os.getpid()}"
    link = [exe] + ARCH + ["-shared", "-o", tmp] + objs
    r = subprocess.run(link, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n" + r.stdout.decode(errors="replace"))
    os.replace(tmp, LIB)
    with open(STAMP + f".tmp{os.getpid()}", "w") as f:
        f.write(digest + "\n")
    os.replace(STAMP + f".tmp{os.getpid()}", STAMP)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv)
    print(LIB)
