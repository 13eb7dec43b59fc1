"""ctypes loader for libgdn.so: the C ABI declared in include/gdn.h.

Loading fails loudly when the library is missing; there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libgdn.so")

GDN_OK = 0
GDN_ERR_INVALID_ARG = 1
GDN_ERR_UNSUPPORTED = 2
GDN_ERR_CUDA = 3
GDN_ERR_TIMEOUT = 4
GDN_ERR_RANGE = 5
GDN_F32 = 0
GDN_BF16 = 1
GDN_DEV_BAD_SEQLENS = 0x1
GDN_DEV_WAIT_TIMEOUT = 0x2
GDN_DEV_F16_RANGE = 0x4
GDN_DEV_F16_PRECISION = 0x8

# (name, restype, argtypes) for every entry point of include/gdn.h
_vp = ctypes.c_void_p
_i = ctypes.c_int
SIGNATURES = {
    "gdn_chunk_fwd": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                                     _i, _i, _i, _i, _i, _i, _vp, _i, _vp]),
    "gdn_chunk_fwd_eta": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                                         _i, _i, _i, _i, _i, _i, _vp, _i, _vp]),
    "gdn_chunk_fwd_scan_workspace_size": (ctypes.c_size_t, [_i, _i, _i, _i, _i, _i, _vp, _i]),
    "gdn_chunk_fwd_scan": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                                          _i, _i, _i, _i, _i, _i, _vp, _i, _i, _vp,
                                          ctypes.c_size_t, _vp]),
    "gdn_chunk_fwd_scan_noalloc": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                                                  _i, _i, _i, _i, _i, _i, _vp, _i, _i, _vp]),
    "gdn_ut_inverse": (ctypes.c_int, [_vp, _vp, _i, _i, _i, _vp]),
    "gdn_decode_step": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                                       _i, _i, _i, _i, _i, _i, _vp]),
    "gdn_get_device_status": (ctypes.c_int, [_vp, ctypes.POINTER(ctypes.c_uint)]),
    "gdn_get_last_error": (ctypes.c_char_p, []),
    "gdn_version": (ctypes.c_int, []),
    "gdn_last_launch_count": (ctypes.c_int, [ctypes.POINTER(ctypes.c_int)]),
}

_lib = None


class GdnError(RuntimeError):
    def __init__(self, status, msg):
        super().__init__("libgdn status %d: %s" % (status, msg))
        self.status = status


def load(path: str = LIB_PATH):
    """Load libgdn.so (build it first with ``gated_delta_rule_09_gb300.build``)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError("libgdn.so not found at %s: build it with "
                          "`python -c 'import __graft_entry__ as g; g.build()'`" % path)
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def check(status: int):
    if status != GDN_OK:
        raise GdnError(status, load().gdn_get_last_error().decode(errors="replace"))
