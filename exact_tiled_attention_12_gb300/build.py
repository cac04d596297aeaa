"""Builds libfa.so (the CUDA kernels and the C ABI) in-tree for sm_103a.

Each .cu file under csrc/ is compiled to an object in parallel, then nvcc
links them into ``libfa.so`` next to this file.  Objects go to ``_build/``.
Both directories' outputs are git-ignored.

A build is reused only when its key still matches: a hash of every source
and header, the compiler flags, the target arch and the host machine, kept
in ``_build/libfa.key``, and the ELF machine field of the existing
``libfa.so`` equal to this host's.  A library built elsewhere (another CPU
architecture, other flags) is rebuilt, never loaded as it is.
"""

from __future__ import annotations

import concurrent.futures as cf
import hashlib
import json
import os
import platform
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libfa.so")
KEY = os.path.join(BUILD, "libfa.key")
ARCH = "-gencode=arch=compute_103a,code=sm_103a"
CFLAGS = ["-O3", "-lineinfo", "-std=c++17", "--expt-relaxed-constexpr", "-Xcompiler", "-fPIC"]
# ELF e_machine values of the hosts this library is built on.
_ELF_MACHINE = {"x86_64": 62, "aarch64": 183, "arm64": 183}


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found (set NVCC or put CUDA's bin directory on PATH)")


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _compile(src: str, verbose: bool) -> str:
    obj = os.path.join(BUILD, os.path.basename(src)[:-3] + ".o")
    cmd = [nvcc(), ARCH] + CFLAGS + ["-I", os.path.join(ROOT, "include"), "-I", CSRC, "-c", src, "-o", obj]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
    if verbose and r.stderr:
        sys.stderr.write(r.stderr)
    return obj


def build_key() -> dict:
    """What a build depends on: sources and headers (by content), flags, arch, host."""
    h = hashlib.sha256()
    deps = sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC)) + [os.path.join(ROOT, "include", "fa.h")]
    for p in deps:
        h.update(os.path.basename(p).encode())
        with open(p, "rb") as f:
            h.update(f.read())
    return {"sources": h.hexdigest(), "arch": ARCH, "flags": CFLAGS, "machine": platform.machine()}


def elf_machine(path: str):
    """e_machine of an ELF file (None if it is not one): the CPU it was built for."""
    try:
        with open(path, "rb") as f:
            head = f.read(20)
    except OSError:
        return None
    if len(head) < 20 or head[:4] != b"\x7fELF":
        return None
    order = "little" if head[5] == 1 else "big"
    return int.from_bytes(head[18:20], order)


def _stale() -> bool:
    if not os.path.exists(LIB) or not os.path.exists(KEY):
        return True
    want = _ELF_MACHINE.get(platform.machine())
    if want is not None and elf_machine(LIB) != want:
        return True
    try:
        with open(KEY) as f:
            return json.load(f) != build_key()
    except (OSError, ValueError):
        return True


def build(force: bool = False, verbose: bool = False) -> str:
    """Compiles every kernel for sm_103a and links libfa.so; returns its path."""
    if not force and not _stale():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    srcs = sources()
    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 1))) as ex:
        objs = list(ex.map(lambda s: _compile(s, verbose), srcs))
    tmp = LIB + ".tmp"
    r = subprocess.run([nvcc(), ARCH, "-shared", "-o", tmp] + objs, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    with open(KEY, "w") as f:
        json.dump(build_key(), f)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
