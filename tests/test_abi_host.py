"""Host-side checks of the C ABI: the library builds and loads, exports every
function include/fa.h declares with the documented signatures, and rejects
invalid arguments before touching the GPU (these calls need no device)."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    import __graft_entry__

    __graft_entry__.build()
    import exact_tiled_attention_12_gb300 as fa

    return fa.lib()


def _declared():
    text = open(os.path.join(ROOT, "include", "fa.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return set(re.findall(r"\b(fa_[a-z0-9_]+)\s*\(", text))


def test_header_declares_the_expected_entry_points():
    assert _declared() >= {"fa_fwd", "fa_bwd", "fa_bwd_workspace_size", "fa_status_string", "fa_version",
                           "fa_bwd_prep", "fa_bwd_tiles", "fa_bwd_dq_finish", "fa_sync_status", "fa_fwd_kv",
                           "fa_fwd_kv_workspace_size", "fa_bwd_kv", "fa_bwd_kv_workspace_size", "fa_merge"}


def test_library_exports_every_declared_symbol(L):
    from exact_tiled_attention_12_gb300.binding import SIGNATURES

    for name in _declared():
        assert hasattr(L, name), name
        assert name in SIGNATURES, name


def test_status_strings(L):
    for code in range(7):
        s = L.fa_status_string(code).decode()
        assert s.startswith("FA_")
    assert L.fa_version() == 110


def test_workspace_size(L):
    # bf16: D and LSE2 (4 bytes per row each, padded to 256) + fp32 dQ accumulator
    rows, elems = 4 * 32 * 2048, 4 * 32 * 2048 * 128
    assert L.fa_bwd_workspace_size(4, 32, 2048, 128, 0) == 2 * rows * 4 + elems * 4
    assert L.fa_bwd_workspace_size(1, 1, 3, 64, 1) == 2 * 256
    # bf16 ragged N: whole 128-row tiles per head (200 -> 256 rows)
    assert L.fa_bwd_workspace_size(2, 1, 200, 64, 0) == 2 * (2 * 256 * 4) + 2 * 256 * 64 * 4
    assert L.fa_bwd_workspace_size(0, 1, 128, 64, 0) == 0
    assert L.fa_bwd_workspace_size(-1, 1, 128, 64, 0) == 0
    # d = 256 writes dQ directly: D and LSE2 only (200 -> 256 rows per head)
    assert L.fa_bwd_workspace_size(2, 3, 200, 256, 0) == 2 * (6 * 256 * 4)
    assert L.fa_bwd_workspace_size(2, 3, 200, 256, 2) == 2 * (6 * 256 * 4)


FAKE = ctypes.c_void_p(0x10000)       # 16-byte aligned, never dereferenced
ODD = ctypes.c_void_p(0x10008)        # 8-byte aligned only


def _fwd(L, ptr=FAKE, B=1, H=1, N=128, d=128, scale=0.1, causal=0, dtype=0, ws=None):
    return L.fa_fwd(ptr, FAKE, FAKE, FAKE, FAKE, B, H, N, d, scale, causal, dtype, ws, 0 if ws is None else 1, None)


@pytest.mark.parametrize("kwargs,code", [
    (dict(B=-1), 1), (dict(N=-5), 1), (dict(d=0), 1), (dict(scale=0.0), 1), (dict(scale=-1.0), 1),
    (dict(scale=float("nan")), 1), (dict(scale=float("inf")), 1), (dict(causal=2), 1), (dict(dtype=7), 1),
    (dict(ptr=ctypes.c_void_p(0)), 1),
    (dict(d=80), 2), (dict(d=256, dtype=1), 2), (dict(d=96, ws=ctypes.c_void_p(0x10010)), 4), (dict(B=300, H=300), 2), (dict(N=65535 * 128 + 1), 2),
    (dict(ptr=ODD), 3),
    (dict(ws=ctypes.c_void_p(0x10010)), 4),
    (dict(N=0), 0), (dict(B=0, ptr=ctypes.c_void_p(0)), 0), (dict(dtype=2, ws=ctypes.c_void_p(0x10010)), 4),
    (dict(dtype=2, ptr=ODD), 3), (dict(dtype=2, d=80), 2), (dict(dtype=3), 1),
    (dict(N=200, ws=ctypes.c_void_p(0x10010)), 4),   # ragged N passes the shape check
    (dict(d=256, ws=ctypes.c_void_p(0x10010)), 4),   # d = 256 passes the shape check (bf16, fp16)
    (dict(d=256, dtype=2, ws=ctypes.c_void_p(0x10010)), 4), (dict(d=192), 2), (dict(d=512), 2),
])
def test_forward_argument_checks(L, kwargs, code):
    assert _fwd(L, **kwargs) == code


def test_backward_argument_checks(L):
    args = [FAKE] * 9 + [1, 1, 128, 64, 0.125, 0, 0]
    # workspace missing, misaligned, too small
    assert L.fa_bwd(*args, None, 0, None) == 4
    assert L.fa_bwd(*args, ctypes.c_void_p(0x10010), 1 << 20, None) == 4
    assert L.fa_bwd(*args, ctypes.c_void_p(0x10000), 16, None) == 4
    # misaligned input checked before the workspace
    bad = [ODD] + [FAKE] * 8 + [1, 1, 128, 64, 0.125, 0, 0]
    assert L.fa_bwd(*bad, None, 0, None) == 3
    # stage entry points share the same checks
    assert L.fa_bwd_prep(FAKE, FAKE, FAKE, 1, 1, 128, 64, 0, None, 0, None) == 4
    assert L.fa_bwd_tiles(*([FAKE] * 7), 1, 1, 128, 64, 0.125, 0, 0, None, 0, None) == 4
    assert L.fa_bwd_dq_finish(FAKE, 1, 1, 100, 64, 0.125, 0, None, 0, None) == 4
    assert L.fa_bwd_dq_finish(FAKE, 1, 1, 100, 80, 0.125, 0, None, 0, None) == 2
    # d = 256 under the causal mask tiles the keys by 64 in the grid's second
    # dimension: 65,535 tiles are accepted (the missing workspace is then the
    # first error), one key more is refused before anything is queued
    edge = 65535 * 64
    for n, code in ((edge, 4), (edge + 1, 2)):
        assert L.fa_bwd(*([FAKE] * 9), 1, 1, n, 256, 0.0625, 1, 0, None, 0, None) == code
        assert L.fa_bwd_tiles(*([FAKE] * 7), 1, 1, n, 256, 0.0625, 1, 0, None, 0, None) == code
    # without the mask the key tiles run along the first dimension: accepted
    assert L.fa_bwd(*([FAKE] * 9), 1, 1, edge + 1, 256, 0.0625, 0, 0, None, 0, None) == 4


def _fwd_kv(L, Nq=128, Nk=256, causal=0, B=1, d=64, dtype=0):
    return L.fa_fwd_kv(FAKE, FAKE, FAKE, FAKE, FAKE, B, 1, Nq, Nk, d, 0.1, causal, dtype, ctypes.c_void_p(0x10010), 1,
                       None)


def test_kv_argument_checks(L):
    # shapes pass (a misaligned workspace is then the first error), so 4 means "accepted"
    assert _fwd_kv(L, 128, 256) == 4 and _fwd_kv(L, 1, 8192, causal=1) == 4 and _fwd_kv(L, 300, 77) == 4
    assert _fwd_kv(L, 256, 128, causal=1) == 2          # causal with more queries than keys
    assert _fwd_kv(L, 5, 0) == 1                        # queries with no key
    assert _fwd_kv(L, 0, 64) == 0 and _fwd_kv(L, 0, 0) == 0 and _fwd_kv(L, 5, 3, B=0) == 0
    # workspace of the backward depends on Nq only
    assert L.fa_bwd_kv_workspace_size(2, 1, 200, 4096, 64, 0) == L.fa_bwd_workspace_size(2, 1, 200, 64, 0)
    assert L.fa_bwd_kv_workspace_size(2, 1, 300, 100, 64, 0) > 0
    assert L.fa_bwd_kv_workspace_size(2, 1, 5, 0, 64, 0) == 0
    args = [FAKE] * 9 + [1, 1, 64, 128, 64, 0.125, 1, 0]
    assert L.fa_bwd_kv(*args, None, 0, None) == 4
    bad = [FAKE] * 9 + [1, 1, 128, 64, 64, 0.125, 1, 0]
    assert L.fa_bwd_kv(*bad, None, 0, None) == 2
    # Nq = 0: dk and dv are zero-filled, so they must be valid pointers
    none = [FAKE] * 7 + [ctypes.c_void_p(0), FAKE] + [1, 1, 0, 128, 64, 0.125, 0, 0]
    assert L.fa_bwd_kv(*none, None, 0, None) == 1


def test_merge_argument_checks(L):
    arr = (ctypes.c_void_p * 17)(*([0x10000] * 17))
    ok_parts = ctypes.cast(arr, ctypes.c_void_p)

    def merge(n=2, o=FAKE, B=1, N=4, d=64, dtype=0, parts=ok_parts, lparts=ok_parts):
        return L.fa_merge(parts, lparts, n, o, FAKE, B, 1, N, d, dtype, None)

    assert merge(n=0) == 1 and merge(n=17) == 1
    assert merge(d=300) == 2 and merge(d=0) == 1
    assert merge(parts=ctypes.c_void_p(0)) == 1
    assert merge(o=ODD) == 3
    odd = (ctypes.c_void_p * 2)(0x10000, 0x10008)
    assert merge(parts=ctypes.cast(odd, ctypes.c_void_p)) == 3
    assert merge(N=0) == 0 and merge(B=0) == 0
    null = (ctypes.c_void_p * 2)(0x10000, 0)
    assert merge(lparts=ctypes.cast(null, ctypes.c_void_p)) == 1


# ---------------------------------------------------------------- build key


def test_build_key_rejects_a_library_built_for_another_cpu(tmp_path, monkeypatch):
    """A libfa.so whose ELF machine is not this host's is rebuilt, not loaded,
    and so is one whose recorded key (sources, flags, arch, host) differs."""
    import json
    import platform

    import exact_tiled_attention_12_gb300.build as b

    lib, key = tmp_path / "libfa.so", tmp_path / "libfa.key"
    monkeypatch.setattr(b, "LIB", str(lib))
    monkeypatch.setattr(b, "KEY", str(key))
    assert b._stale()                                          # nothing built
    mine = b._ELF_MACHINE.get(platform.machine())
    if mine is None:
        pytest.skip("unknown host machine")
    other = 183 if mine == 62 else 62

    def elf(machine):
        head = bytearray(64)
        head[:4] = b"\x7fELF"
        head[4], head[5] = 2, 1                                # 64-bit, little endian
        head[18:20] = machine.to_bytes(2, "little")
        return bytes(head)

    lib.write_bytes(elf(mine))
    key.write_text(json.dumps(b.build_key()))
    assert b.elf_machine(str(lib)) == mine
    assert not b._stale()                                      # same host, same key
    lib.write_bytes(elf(other))
    assert b._stale()                                          # foreign CPU architecture
    lib.write_bytes(elf(mine))
    k = b.build_key()
    k["flags"] = k["flags"] + ["-G"]
    key.write_text(json.dumps(k))
    assert b._stale()                                          # other compiler flags
    key.write_text("not json")
    assert b._stale()
