"""Oracle for the gated delta rule forward pass: TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its Python binding) never calls it and shares no code with it.

Contents
--------
``gdn_recurrence_f64``  the sequential fp64 recurrence in plain C
                        (``gdn_oracle.c``), called through ctypes.  This is the
                        oracle every GPU result is compared against.
``chunk_reference``     a second, independent fp64 statement of the chunkwise
                        (WY/UT-transform) form in numpy, used to localise
                        differences stage by stage (A, T, W, U, V_new).  It is
                        pinned against the recurrence; the GPU is never
                        compared against it alone.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``gdn_oracle.c`` with gcc into ``liboracle.so`` (in place)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + ".tmp.%d" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
           _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            dp = ctypes.POINTER(ctypes.c_double)
            lib.gdn_oracle_f64.restype = ctypes.c_int
            lib.gdn_oracle_f64.argtypes = [
                dp, dp, dp, dp, dp, dp, dp, dp, dp,
                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                ctypes.POINTER(ctypes.c_int32), ctypes.c_int]
            _lib = lib
    return _lib


def _f64(x):
    """Widen a numpy array or a (CPU) torch tensor exactly to contiguous fp64."""
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor, any float dtype; widening is exact
        x = x.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def gdn_recurrence_f64(q, k, v, log_alpha, beta, S0=None, cu_seqlens=None,
                       eta=None, n_threads=None):
    """Sequential fp64 gated delta rule over every (sequence, head).

    Follows the recurrence ``S_t = a_t S_{t-1}(I - b_t k_t k_t^T) + e_t v_t k_t^T``,
    ``o_t = S_t q_t`` ("从零开始的 GDN 推导", recurrent form, transposed so that
    S is d_v x d_k; "RNN的复兴03：现代RNN的并行计算", §二, separate write strength
    e = eta, default e = beta).

    Shapes: q,k [B,T,H,dk], v [B,T,H,dv], log_alpha/beta/eta [B,T,H],
    S0 [N,H,dv,dk] or None (zeros).  With ``cu_seqlens`` ([N+1] ints) the
    inputs are packed with B == 1 and N = len(cu_seqlens) - 1 sequences.

    Returns ``(o [B,T,H,dv], S_final [N,H,dv,dk])`` as fp64 numpy arrays.
    """
    lib = _load()
    q, k, v = _f64(q), _f64(k), _f64(v)
    log_alpha, beta, eta, S0 = _f64(log_alpha), _f64(beta), _f64(eta), _f64(S0)
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    assert k.shape == q.shape and v.shape == (B, T, H, dv)
    assert log_alpha.shape == (B, T, H) and beta.shape == (B, T, H)
    if eta is not None:
        assert eta.shape == (B, T, H)
    cu = None
    N = B
    Tk = T
    if cu_seqlens is not None:
        if hasattr(cu_seqlens, "detach"):
            cu_seqlens = cu_seqlens.detach().cpu().numpy()
        cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int32))
        assert B == 1
        N = len(cu) - 1
        Tk = T
    if S0 is not None:
        assert S0.shape == (N, H, dv, dk)
    o = np.zeros((B, T, H, dv), dtype=np.float64)
    S_final = np.zeros((N, H, dv, dk), dtype=np.float64)
    if n_threads is None:
        n_threads = os.cpu_count() or 1
    rc = lib.gdn_oracle_f64(
        _ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(beta), _ptr(eta),
        _ptr(S0), _ptr(o), _ptr(S_final), N, H, Tk, dk, dv,
        None if cu is None else cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
        int(n_threads))
    if rc != 0:
        raise ValueError("gdn_oracle_f64 failed with code %d" % rc)
    return o, S_final
