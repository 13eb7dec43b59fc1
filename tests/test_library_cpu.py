"""The C-ABI library builds, loads, exports every symbol include/gdn.h declares,
and rejects bad arguments on the host before touching the GPU (CPU only)."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gdn.h")


@pytest.fixture(scope="module")
def lib():
    from gated_delta_rule_09_gb300 import build, _lib
    build.build()
    return _lib.load()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(gdn_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_entry_points():
    names = declared_functions()
    for n in ("gdn_chunk_fwd", "gdn_get_last_error", "gdn_get_device_status",
              "gdn_version", "gdn_last_launch_count"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    from gated_delta_rule_09_gb300 import _lib
    out = subprocess.run(["nm", "-D", "--defined-only", _lib.LIB_PATH],
                         capture_output=True, text=True, check=True).stdout
    exported = set(l.split()[-1] for l in out.splitlines() if l.strip())
    for name in declared_functions():
        assert name in exported, name
        assert hasattr(lib, name)
    assert set(declared_functions()) == set(_lib.SIGNATURES)


def test_wait_test_library_is_built_beside_it(lib):
    """build() also makes libgdn_waittest.so (the abort-path test build) with
    the same exports; nothing but its own test loads it."""
    from gated_delta_rule_09_gb300 import build
    assert os.path.exists(build.WAITTEST_LIB)
    out = subprocess.run(["nm", "-D", "--defined-only", build.WAITTEST_LIB],
                         capture_output=True, text=True, check=True).stdout
    exported = set(l.split()[-1] for l in out.splitlines() if l.strip())
    assert set(declared_functions()) <= exported


def test_header_compiles_as_c():
    # The header is plain C: it must compile without CUDA headers.
    src = '#include "gdn.h"\nint main(void){ return (int)GDN_OK + (int)GDN_BF16; }\n'
    p = subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.dirname(HEADER),
                        "-x", "c", "-", "-o", os.devnull], input=src, text=True,
                       capture_output=True)
    assert p.returncode == 0, p.stderr


def _call(lib, q=0x1000, k=0x100000, v=0x200000, la=0x300000, be=0x400000, S0=None,
          o=0x500000, Sf=None, B=1, H=1, T=16, dk=16, dv=16, C=16, cu=None, dtype=1):
    return lib.gdn_chunk_fwd(q, k, v, la, be, S0, o, Sf, B, H, T, dk, dv, C, cu, dtype, None)


def test_version(lib):
    assert lib.gdn_version() == 100


@pytest.mark.parametrize("kw,code", [
    (dict(C=48), 2), (dict(C=128), 2), (dict(dtype=7), 2), (dict(dk=129), 2),
    (dict(B=-1), 1), (dict(T=-5), 1), (dict(dk=0), 1), (dict(dv=0), 1),
    (dict(q=None), 1), (dict(o=None), 1), (dict(la=None), 1),
    (dict(q=0x1002), 1), (dict(o=0x500008), 1), (dict(la=0x300002), 1),
    (dict(o=0x1000), 1),                       # o aliases q
    (dict(Sf=0x100000), 1),                    # S_final overlaps k
    (dict(S0=0x600000, Sf=0x600040), 1),       # partial overlap of S0 / S_final
    (dict(cu=0x700000, B=0), 1),
])
def test_host_validation(lib, kw, code):
    st = _call(lib, **kw)
    assert st == code, (kw, st, lib.gdn_get_last_error())
    assert lib.gdn_get_last_error()  # a message is set


def test_empty_problem_is_a_no_op(lib):
    # No units: returns OK without any CUDA call (this host has no GPU).
    assert _call(lib, B=0) == 0
    assert _call(lib, H=0) == 0
    n = ctypes.c_int(5)
    assert lib.gdn_last_launch_count(ctypes.byref(n)) == 0


def test_python_binding_rejects_cpu_tensors():
    import torch
    import gated_delta_rule_09_gb300 as gdn
    x = torch.zeros(1, 4, 1, 16)
    with pytest.raises(TypeError):
        gdn.gdn_chunk_fwd(x, x, x, torch.zeros(1, 4, 1), torch.zeros(1, 4, 1))


def _dcall(lib, q=0x1000, k=0x100000, v=0x200000, la=0x300000, be=0x400000, Si=None,
           o=0x500000, So=0x600000, N=1, H=1, T=1, dk=16, dv=16, dtype=1):
    return lib.gdn_decode_step(q, k, v, la, be, Si, o, So, N, H, T, dk, dv, dtype, None)


@pytest.mark.parametrize("kw,code", [
    (dict(dtype=3), 2), (dict(dk=129), 2),
    (dict(N=-1), 1), (dict(T=-1), 1), (dict(dk=0), 1), (dict(dv=0), 1),
    (dict(So=None), 1), (dict(q=None), 1), (dict(o=None), 1), (dict(be=None), 1),
    (dict(k=0x100004), 1), (dict(So=0x600002), 1),
    (dict(o=0x200000), 1),                     # o aliases v
    (dict(So=0x400000), 1),                    # S_out overlaps beta
    (dict(Si=0x700000, So=0x700010), 1),       # partial overlap of S_in / S_out
])
def test_decode_host_validation(lib, kw, code):
    st = _dcall(lib, **kw)
    assert st == code, (kw, st, lib.gdn_get_last_error())
    assert lib.gdn_get_last_error()


def test_decode_empty_problem_is_a_no_op(lib):
    assert _dcall(lib, N=0) == 0
    assert _dcall(lib, H=0, So=None) == 0


def test_eta_entry_point_validation(lib):
    # eta is required when there is work; misaligned or overlapping eta is rejected
    f = lambda eta, o=0x500000: lib.gdn_chunk_fwd_eta(0x1000, 0x100000, 0x200000, 0x300000,
                                                       0x400000, eta, None, o, None, 1, 1, 16,
                                                       16, 16, 16, None, 1, None)
    assert f(None) == 1 and lib.gdn_get_last_error()
    assert f(0x700002) == 1
    assert f(0x500010) == 1      # eta inside o


def _scan_layout_bytes(nseg, H, dk, dv):
    """The scan workspace as the header describes it: segment boundaries,
    start states, segment final states and transitions, each 256-aligned."""
    a = lambda x: (x + 255) // 256 * 256
    return a((nseg + 1) * 4) + 2 * a(nseg * H * dv * dk * 4) + a(nseg * H * dk * dk * 4)


@pytest.mark.parametrize("segments,expect_P", [(3, 3), (16, 16), (100, 16), (1, 1)])
def test_scan_workspace_for_packed_sequences(lib, segments, expect_P):
    """Packed sequences (a non-NULL cu_seqlens; only its NULL-ness is read
    here) are cut into `segments` pieces each, capped at the chunks of the
    whole pack (1000 tokens = 16 chunks of 64); one piece needs no workspace."""
    B, H, T, dk, dv = 4, 2, 1000, 128, 128
    size = lib.gdn_chunk_fwd_scan_workspace_size(B, H, T, dk, dv, 64, 0x1000, segments)
    assert size == (0 if expect_P == 1 else _scan_layout_bytes(B * expect_P, H, dk, dv))


def test_scan_workspace_unpacked_has_no_empty_segment(lib):
    """Without cu_seqlens, B sequences of T tokens: 16 chunks asked for 5 pieces
    become ceil(16 / ceil(16 / 5)) = 4 pieces of 4 chunks."""
    B, H, T, dk, dv = 2, 2, 1024, 128, 128
    size = lib.gdn_chunk_fwd_scan_workspace_size(B, H, T, dk, dv, 64, None, 5)
    assert size == _scan_layout_bytes(B * 4, H, dk, dv)
