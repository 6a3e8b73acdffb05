"""The C ABI library loads, exports every function include/*.h declares, and
rejects bad arguments on the host (no GPU needed: nothing here launches)."""
import ctypes
import glob
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
LIB = os.path.join(ROOT, "speculative_decoding_draft_online_gb300", "libspecverify.so")


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(spec_\w+)\s*\(", text, flags=re.M):
            names.add(m.group(1))
    return names


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(LIB):
        import __graft_entry__
        __graft_entry__.build()
    return ctypes.CDLL(LIB)


def test_header_declares_the_entry_points():
    names = declared_functions()
    for want in ("spec_verify", "spec_verify_ex", "spec_verify_tree", "spec_verify_guided", "spec_workspace_size",
                 "spec_workspace_init", "spec_random", "spec_strerror", "spec_abi_version", "spec_verify_noalloc",
                 "spec_test_force_stage_timeouts", "spec_probe_read"):
        assert want in names, names


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", LIB], capture_output=True, text=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    missing = declared_functions() - exported
    assert not missing, missing
    for name in declared_functions():
        getattr(lib, name)


def test_workspace_size(lib):
    lib.spec_workspace_size.restype = ctypes.c_size_t
    ws = lib.spec_workspace_size
    assert ws(64, 8, 128256, 0) > 0
    assert ws(0, 8, 128256, 0) == 0 and ws(1, 0, 10, 0) == 0 and ws(1, 1, 0, 0) == 0 and ws(1, 1, 10, 7) == 0
    # one 8-byte partial per 16 KB row tile (4096 fp32 elements) of every row with statistics
    assert ws(64, 8, 128256, 0) >= 64 * 16 * ((128256 + 4095) // 4096) * 8
    assert ws(64, 8, 128256, 0) % 256 == 0


def test_host_side_errors_return_before_any_launch(lib):
    vp = ctypes.c_void_p
    f = lib.spec_verify
    f.argtypes = [vp, vp, vp, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_float,
                  ctypes.c_uint64, vp, vp, vp, ctypes.c_size_t, vp]
    fake = vp(0x10000)                                  # never dereferenced: every call fails on the host
    ARG, ALIGN, UNSUP, WS = -1, -2, -5, -8
    assert f(None, fake, fake, 1, 1, 10, 0, 1.0, 0, fake, fake, fake, 1 << 20, None) == ARG       # no target
    assert f(fake, None, fake, 1, 1, 10, 0, 1.0, 0, fake, fake, fake, 1 << 20, None) == ARG       # no draft, T > 0
    assert f(fake, fake, fake, 0, 1, 10, 0, 1.0, 0, fake, fake, fake, 1 << 20, None) == ARG       # B = 0
    assert f(fake, fake, fake, 1, 0, 10, 0, 1.0, 0, fake, fake, fake, 1 << 20, None) == ARG       # k = 0
    assert f(fake, fake, fake, 1, 1, 10, 5, 1.0, 0, fake, fake, fake, 1 << 20, None) == ARG       # dtype
    assert f(fake, fake, fake, 1, 1, 10, 0, -1.0, 0, fake, fake, fake, 1 << 20, None) == ARG      # T < 0
    assert f(fake, fake, fake, 1, 1, 10, 0, float("inf"), 0, fake, fake, fake, 1 << 20, None) == ARG
    assert f(fake, fake, fake, 1, 5000, 10, 0, 1.0, 0, fake, fake, fake, 1 << 20, None) == UNSUP  # k too large
    assert f(vp(0x10001), fake, fake, 1, 1, 10, 0, 1.0, 0, fake, fake, fake, 1 << 20, None) == ALIGN
    assert f(fake, fake, fake, 1, 1, 10, 0, 1.0, 0, fake, fake, fake, 16, None) == WS            # too small
    assert f(fake, fake, fake, 1, 1, 10, 0, 1.0, 0, fake, fake, vp(0x10008), 1 << 20, None) == WS
    t = lib.spec_verify_tree
    t.argtypes = [vp, vp, vp, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_float,
                  vp, vp, vp, vp, vp, ctypes.c_size_t, vp]
    assert t(fake, fake, fake, 1, 3, 10, 0, 0.5, fake, fake, None, None, fake, 1 << 20, None) == UNSUP
    assert t(fake, fake, fake, 1, 5000, 10, 0, 0.0, fake, fake, None, None, fake, 1 << 20, None) == UNSUP
    assert t(fake, None, fake, 1, 3, 10, 0, 0.0, fake, fake, None, None, fake, 1 << 20, None) == ARG


def test_strerror_names_every_code(lib):
    lib.spec_strerror.restype = ctypes.c_char_p
    names = {c: lib.spec_strerror(c).decode() for c in range(-8, 1)}
    assert len(set(names.values())) == 9 and lib.spec_strerror(-99).decode() == "unknown status"


class _Aux(ctypes.Structure):
    _fields_ = [("p_draft", ctypes.c_void_p), ("q_draft", ctypes.c_void_p), ("lse", ctypes.c_void_p),
                ("status", ctypes.c_void_p), ("events", ctypes.c_void_p * 4),
                ("sequence_offset", ctypes.c_uint32), ("lenience", ctypes.c_float),
                ("stop_ids", ctypes.c_void_p), ("n_stop", ctypes.c_int32), ("n_committed", ctypes.c_void_p),
                ("match_mask", ctypes.c_void_p), ("n_match", ctypes.c_void_p), ("tail_runs", ctypes.c_void_p),
                ("top_k", ctypes.c_int32), ("top_p", ctypes.c_float)]


def test_abi_version_and_aux_layout(lib):
    assert lib.spec_abi_version() == (1 << 16) | 3
    # the 1.1 fields follow the 1.0 ones; the binding mirrors this layout
    assert _Aux.lenience.offset == _Aux.sequence_offset.offset + 4
    from speculative_decoding_draft_online_gb300 import _lib
    assert [f[0] for f in _lib._Aux._fields_] == [f[0] for f in _Aux._fields_]
    assert ctypes.sizeof(_lib._Aux) == ctypes.sizeof(_Aux)


def test_aux_and_guided_host_errors(lib):
    vp = ctypes.c_void_p
    f = lib.spec_verify_ex
    f.argtypes = [vp, vp, vp, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_float,
                  ctypes.c_uint64, vp, vp, vp, ctypes.c_size_t, vp, ctypes.POINTER(_Aux)]
    fake = vp(0x10000)
    ARG, ALIGN, UNSUP = -1, -2, -5

    def call(T=1.0, **kw):
        a = _Aux()
        for key, val in kw.items():
            setattr(a, key, val)
        return f(fake, fake, fake, 2, 3, 10, 0, T, 0, fake, fake, fake, 1 << 20, None, ctypes.byref(a))

    assert call(lenience=0.5) == ARG
    assert call(lenience=float("nan")) == ARG
    assert call(lenience=float("inf")) == ARG
    assert call(n_stop=-1) == ARG
    assert call(n_stop=2) == ARG                                    # no stop_ids
    assert call(n_stop=65, stop_ids=0x10000) == UNSUP
    assert call(n_stop=1, stop_ids=0x10002) == ALIGN
    assert call(match_mask=0x10000) == ARG                          # match outputs need greedy mode
    assert call(n_match=0x10000) == ARG
    assert call(tail_runs=0x10000) == ARG
    assert call(top_k=-1) == ARG
    assert call(top_p=-0.1) == ARG
    assert call(top_p=1.5) == ARG
    assert call(top_p=float("nan")) == ARG
    g = lib.spec_verify_guided
    g.argtypes = [vp, vp, vp, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                  vp, vp, vp, vp, vp, ctypes.c_size_t, vp]
    assert g(fake, fake, fake, 2, 3, -1, 10, 0, fake, fake, fake, None, fake, 1 << 20, None) == ARG   # L < 0
    assert g(fake, fake, None, 2, 3, 4, 10, 0, fake, fake, fake, None, fake, 1 << 20, None) == ARG    # no guide
    assert g(fake, fake, fake, 2, 3, 4, 10, 0, fake, fake, None, None, fake, 1 << 20, None) == ARG    # no n_committed
    assert g(fake, fake, vp(0x10002), 2, 3, 4, 10, 0, fake, fake, fake, None, fake, 1 << 20, None) == ALIGN
    assert g(fake, fake, fake, 2, 5000, 4, 10, 0, fake, fake, fake, None, fake, 1 << 20, None) == UNSUP
