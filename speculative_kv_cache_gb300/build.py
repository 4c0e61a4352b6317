"""Builds libig.so (the sm_103a kernels and the C ABI) in-tree, with nvcc and g++ only.

Each translation unit is compiled in parallel into ``_build/`` next to this file and the
objects are linked into ``libig.so`` beside it.  The library is reused only when a stamp written
beside it at link time matches a SHA-256 of everything the build depends on: the bytes of every
source and header, the compile and link commands, the compiler's version and the host machine
type (so a library that arrives with the sources, or one built for another CPU, is rebuilt).
Usage: ``python -m speculative_kv_cache_gb300.build [--force]``.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import hashlib
import os
import platform
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libig.so")
STAMP = LIB + ".sha256"
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-lineinfo", "-O3", "-std=c++17", "-Xcompiler", "-fPIC,-O3", "-Xptxas", "-v"]
CXX_FLAGS = ["-O3", "-std=c++17", "-fPIC", "-pthread"]
LINK_FLAGS = ["-shared", "-cudart", "shared"]


def _nvcc() -> str:
    for c in [os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"]:
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libig.so")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cpp")))


def _inputs():
    return _sources() + glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh")) + \
        glob.glob(os.path.join(ROOT, "include", "*.h")) + [os.path.abspath(__file__)]


def _tool_version(cmd) -> str:
    try:
        return subprocess.run(cmd, capture_output=True, text=True, timeout=60).stdout
    except (OSError, subprocess.SubprocessError):
        return "unknown"


def build_hash(nvcc: str | None = None) -> str:
    """SHA-256 of the build's inputs: file names and bytes, flags, tool versions, machine type."""
    h = hashlib.sha256()
    for p in sorted(set(_inputs())):
        h.update(os.path.relpath(p, ROOT).encode() + b"\0")
        with open(p, "rb") as f:
            h.update(f.read())
        h.update(b"\0")
    nvcc = nvcc or _nvcc()
    for part in (ARCH, NVCC_FLAGS, CXX_FLAGS, LINK_FLAGS):
        h.update(" ".join(part).encode() + b"\0")
    h.update(_tool_version([nvcc, "--version"]).encode())
    h.update(_tool_version(["g++", "--version"]).encode())
    h.update(platform.machine().encode())
    return h.hexdigest()


def up_to_date(digest: str | None = None) -> bool:
    if not (os.path.exists(LIB) and os.path.exists(STAMP)):
        return False
    with open(STAMP) as f:
        return f.read().strip() == (digest or build_hash())


def _compile(src: str, nvcc: str) -> str:
    obj = os.path.join(BUILD, os.path.basename(src) + ".o")
    if src.endswith(".cu"):
        cmd = [nvcc, *ARCH, *NVCC_FLAGS, "-c", src, "-o", obj]
    else:
        cmd = ["g++", *CXX_FLAGS, "-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"compile failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    with open(obj + ".log", "w") as f:
        f.write(r.stderr)
    return obj


def build(force: bool = False, verbose: bool = False) -> str:
    nvcc = _nvcc()
    digest = build_hash(nvcc)
    if not force and up_to_date(digest):
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    srcs = _sources()
    with cf.ThreadPoolExecutor(max_workers=min(len(srcs), os.cpu_count() or 4)) as ex:
        objs = list(ex.map(lambda s: _compile(s, nvcc), srcs))
    tmp = LIB + ".tmp"
    cmd = [nvcc, *ARCH, *LINK_FLAGS, "-o", tmp, *objs, "-lpthread"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    if os.path.exists(STAMP):
        os.remove(STAMP)
    os.replace(tmp, LIB)
    with open(STAMP, "w") as f:
        f.write(digest + "\n")
    if verbose:
        for o in objs:
            log = open(o + ".log").read()
            if log.strip():
                print(os.path.basename(o), "\n", log)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
