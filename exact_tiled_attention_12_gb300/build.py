"""Builds libfa.so (the CUDA kernels and the C ABI) in-tree for sm_103a.

Each .cu file under csrc/ is compiled to an object in parallel, then nvcc
links them into ``libfa.so`` next to this file.  Objects go to ``_build/``.
``build(debug=True)`` makes ``libfa_debug.so`` the same way (objects in
``_build_debug/``) with FA_DEBUG_CHECKS defined: the kernels then check every
TMA coordinate, shared-memory operand and tensor-memory column range before
using it.  All of these outputs are git-ignored.

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
ARCH = "-gencode=arch=compute_103a,code=sm_103a"
CFLAGS = ["-O3", "-lineinfo", "-std=c++17", "--expt-relaxed-constexpr", "-Xcompiler", "-fPIC"]


class _Target:
    """Where one flavour of the library is built, and with which extra flags."""

    def __init__(self, debug: bool):
        self.debug = debug
        self.build = os.path.join(PKG, "_build_debug" if debug else "_build")
        self.lib = os.path.join(PKG, "libfa_debug.so" if debug else "libfa.so")
        self.key = os.path.join(self.build, "libfa.key")
        self.flags = CFLAGS + (["-DFA_DEBUG_CHECKS"] if debug else [])


RELEASE, DEBUG = _Target(False), _Target(True)
# Paths of the release build (kept as module attributes for callers and tests).
BUILD, LIB, KEY = RELEASE.build, RELEASE.lib, RELEASE.key
# ELF e_machine values of the hosts this library is built on.
_ELF_MACHINE = {"x86_64": 62, "aarch64": 183, "arm64": 183}


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found (set NVCC or put CUDA's bin directory on PATH)")


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _compile(src: str, verbose: bool, target: _Target = RELEASE) -> str:
    obj = os.path.join(target.build, os.path.basename(src)[:-3] + ".o")
    cmd = [nvcc(), ARCH] + target.flags + ["-I", os.path.join(ROOT, "include"), "-I", CSRC, "-c", src, "-o", obj]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
    if verbose and r.stderr:
        sys.stderr.write(r.stderr)
    return obj


def build_key(target: _Target = RELEASE) -> dict:
    """What a build depends on: sources and headers (by content), flags, arch, host."""
    h = hashlib.sha256()
    deps = sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC)) + [os.path.join(ROOT, "include", "fa.h")]
    for p in deps:
        h.update(os.path.basename(p).encode())
        with open(p, "rb") as f:
            h.update(f.read())
    return {"sources": h.hexdigest(), "arch": ARCH, "flags": target.flags, "machine": platform.machine()}


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


def _stale(target: _Target = None) -> bool:
    # The module attributes LIB / KEY name the release build (tests may point them elsewhere).
    lib, key = (LIB, KEY) if target is None or target is RELEASE else (target.lib, target.key)
    target = target or RELEASE
    if not os.path.exists(lib) or not os.path.exists(key):
        return True
    want = _ELF_MACHINE.get(platform.machine())
    if want is not None and elf_machine(lib) != want:
        return True
    try:
        with open(key) as f:
            return json.load(f) != build_key(target)
    except (OSError, ValueError):
        return True


def build(force: bool = False, verbose: bool = False, debug: bool = False) -> str:
    """Compiles every kernel for sm_103a and links libfa.so (libfa_debug.so
    with ``debug``); returns its path."""
    target = DEBUG if debug else RELEASE
    if not force and not _stale(target):
        return target.lib
    os.makedirs(target.build, exist_ok=True)
    srcs = sources()
    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 1))) as ex:
        objs = list(ex.map(lambda s: _compile(s, verbose, target), srcs))
    tmp = target.lib + ".tmp"
    r = subprocess.run([nvcc(), ARCH, "-shared", "-o", tmp] + objs, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, target.lib)
    with open(target.key, "w") as f:
        json.dump(build_key(target), f)
    return target.lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, debug="--debug" in sys.argv))
