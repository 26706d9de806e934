"""Build the qkvp C-ABI library (libqkvp.so) in-tree for sm_103a.

Each CUDA translation unit is compiled by its own nvcc process (in parallel)
and the objects are linked into ``fp8_packed_reduced_gb300/libqkvp.so``.
Objects go to ``_build/`` at the repository root.  Incremental, by content:
each object and the library carry a stamp file with the SHA-256 of what they
were built from (the unit's source, every header, the compiler flags, the
nvcc version and the host machine type), and anything whose stamp does not
match the current sources is rebuilt, whatever the files' times say.
"""

from __future__ import annotations

import concurrent.futures as cf
import functools
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
LIB = os.path.join(PKG, "libqkvp.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-I" + INCLUDE, "-I" + CSRC]
LINK = ["-shared", "-cudart=static"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libqkvp.so")


def _sources():
    return sorted(f for f in os.listdir(CSRC) if f.endswith(".cu"))


def _headers():
    hs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    hs += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE)]
    return sorted(hs)


@functools.lru_cache(maxsize=None)
def _toolchain() -> str:
    r = subprocess.run([nvcc(), "--version"], capture_output=True, text=True)
    return r.stdout + platform.machine()


def _digest(paths, extra) -> str:
    h = hashlib.sha256()
    for p in paths:
        h.update(os.path.basename(p).encode())
        with open(p, "rb") as f:
            h.update(f.read())
    for e in extra:
        h.update(b"\0" + str(e).encode())
    h.update(_toolchain().encode())
    return h.hexdigest()


def _stamp_ok(target: str, digest: str) -> bool:
    stamp = target + ".sha256"
    if not (os.path.exists(target) and os.path.exists(stamp)):
        return False
    with open(stamp) as f:
        return f.read().strip() == digest


def _write_stamp(target: str, digest: str):
    with open(target + ".sha256", "w") as f:
        f.write(digest + "\n")


def _compile(src: str, extra, verbose: bool) -> str:
    obj = os.path.join(BUILD, src[:-3] + ".o")
    srcp = os.path.join(CSRC, src)
    digest = _digest([srcp, *_headers()], [*ARCH, *FLAGS, *extra])
    if _stamp_ok(obj, digest) and not extra:
        return obj
    cmd = [nvcc(), *ARCH, *FLAGS, *extra, "-c", srcp, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if verbose or r.returncode != 0:
        sys.stderr.write(r.stdout + r.stderr)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}")
    _write_stamp(obj, digest)
    return obj


def build(verbose: bool = False, ptxas_info: bool = False) -> str:
    """Compile every unit under csrc/ and link libqkvp.so; returns its path.
    Processes that build at once (the ranks of one job) take turns on a lock
    file: the first compiles, the others find the stamps current."""
    os.makedirs(BUILD, exist_ok=True)
    import fcntl
    with open(os.path.join(BUILD, ".lock"), "w") as lock:
        fcntl.flock(lock, fcntl.LOCK_EX)
        try:
            return _build_locked(verbose, ptxas_info)
        finally:
            fcntl.flock(lock, fcntl.LOCK_UN)


def _build_locked(verbose: bool, ptxas_info: bool) -> str:
    extra = ["-Xptxas", "-v"] if ptxas_info else []
    srcs = _sources()
    with cf.ThreadPoolExecutor(max_workers=len(srcs)) as ex:
        objs = list(ex.map(lambda s: _compile(s, extra, verbose or ptxas_info), srcs))
    digest = _digest(objs, [*ARCH, *LINK])
    if _stamp_ok(LIB, digest):
        return LIB
    tmp = LIB + ".tmp"
    cmd = [nvcc(), *ARCH, *LINK, "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        sys.stderr.write(r.stdout + r.stderr)
        raise RuntimeError("linking libqkvp.so failed")
    os.replace(tmp, LIB)
    _write_stamp(LIB, digest)
    return LIB


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, ptxas_info="--ptxas" in sys.argv))
