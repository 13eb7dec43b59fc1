"""GB300-native chunkwise forward pass of the gated delta rule.

The compute runs in libgdn.so (hand-written CUDA for sm_103a) behind the C ABI
of ``include/gdn.h``; this module only marshals torch CUDA tensors into that
call.  The library is loaded on first use, and every entry point raises
ImportError if it is missing: there is no fallback.
"""
from __future__ import annotations

import ctypes

import torch

from . import _lib
from ._lib import GdnError, GDN_BF16, GDN_F32  # noqa: F401

_DTYPES = {torch.float32: _lib.GDN_F32, torch.bfloat16: _lib.GDN_BF16}


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _need_cuda(name, t, dtype=None):
    if t is None:
        return
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError("%s must be a CUDA tensor" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if dtype is not None and t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))


def load():
    """Load libgdn.so now (raises ImportError if it has not been built)."""
    return _lib.load()


def _check_args(q, k, v, log_alpha, beta, eta, S0, o, S_final, packed):
    """Types, devices and shapes of one forward call; every tensor the kernels
    read or write is checked against the sizes the C call derives from q and v,
    so a wrongly shaped argument is refused here instead of being read or
    written past its end.  Returns (B, T, H, d_k, d_v, N)."""
    if q.dtype not in _DTYPES:
        raise TypeError("q/k/v dtype must be float32 or bfloat16, got %s" % q.dtype)
    for name, t in (("q", q), ("k", k), ("v", v)):
        _need_cuda(name, t, q.dtype)
    _need_cuda("log_alpha", log_alpha, torch.float32)
    _need_cuda("beta", beta, torch.float32)
    _need_cuda("eta", eta, torch.float32)
    _need_cuda("S0", S0, torch.float32)
    _need_cuda("o", o, q.dtype)
    _need_cuda("S_final", S_final, torch.float32)
    if q.dim() != 4 or k.shape != q.shape or v.dim() != 4 or v.shape[:3] != q.shape[:3]:
        raise ValueError("q, k must be [B,T,H,d_k] and v [B,T,H,d_v]")
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    if log_alpha.shape != (B, T, H) or beta.shape != (B, T, H):
        raise ValueError("log_alpha and beta must be [B,T,H] = %s" % ((B, T, H),))
    if eta is not None and eta.shape != (B, T, H):
        raise ValueError("eta must be [B,T,H] = %s" % ((B, T, H),))
    if packed is not None:
        _need_cuda("cu_seqlens", packed, torch.int32)
        if B != 1:
            raise ValueError("packed (cu_seqlens) inputs must have B == 1")
        if packed.dim() != 1 or packed.numel() < 2:
            raise ValueError("cu_seqlens must be a 1-D int32 tensor of N + 1 >= 2 offsets")
        N = packed.numel() - 1
    else:
        N = B
    if S0 is not None and S0.shape != (N, H, dv, dk):
        raise ValueError("S0 must be [N,H,d_v,d_k] = %s" % ((N, H, dv, dk),))
    if o is not None and o.shape != (B, T, H, dv):
        raise ValueError("o must be [B,T,H,d_v] = %s" % ((B, T, H, dv),))
    if S_final is not None and S_final.shape != (N, H, dv, dk):
        raise ValueError("S_final must be [N,H,d_v,d_k] = %s" % ((N, H, dv, dk),))
    return B, T, H, dk, dv, N


def gdn_chunk_fwd(q, k, v, log_alpha, beta, S0=None, o=None, S_final=None,
                  C=64, cu_seqlens=None, stream=None, want_final_state=True):
    """Chunkwise gated delta rule forward; returns ``(o, S_final)``.

    q, k [B,T,H,d_k] and v [B,T,H,d_v] (fp32 or bf16, one dtype);
    log_alpha, beta [B,T,H] fp32; S0 [N,H,d_v,d_k] fp32 or None.  With
    ``cu_seqlens`` (int32 CUDA tensor [N+1]) the inputs are packed with B == 1.
    ``o`` / ``S_final`` may be passed preallocated; otherwise they are
    allocated here.  Runs on ``stream`` (a torch.cuda.Stream, a raw handle, or
    None for the current torch stream).
    """
    return _chunk(q, k, v, log_alpha, beta, None, S0, o, S_final, C, cu_seqlens, stream,
                  want_final_state)


def gdn_chunk_fwd_eta(q, k, v, log_alpha, beta, eta, S0=None, o=None, S_final=None,
                      C=64, cu_seqlens=None, stream=None, want_final_state=True):
    """``gdn_chunk_fwd`` with a write strength ``eta`` [B,T,H] fp32 separate
    from the erase strength ``beta``: S_t = alpha S (I - beta k k^T) + eta v k^T."""
    if eta is None:
        raise ValueError("eta is required (use gdn_chunk_fwd for eta = beta)")
    return _chunk(q, k, v, log_alpha, beta, eta, S0, o, S_final, C, cu_seqlens, stream,
                  want_final_state)


def _chunk(q, k, v, log_alpha, beta, eta, S0, o, S_final, C, cu_seqlens, stream,
           want_final_state):
    B, T, H, dk, dv, N = _check_args(q, k, v, log_alpha, beta, eta, S0, o, S_final, cu_seqlens)
    lib = _lib.load()
    if o is None:
        o = torch.empty((B, T, H, dv), dtype=q.dtype, device=q.device)
    if S_final is None and want_final_state:
        S_final = torch.empty((N, H, dv, dk), dtype=torch.float32, device=q.device)
    handle = ctypes.c_void_p(_stream_handle(stream, q.device))
    with torch.cuda.device(q.device):
        if eta is None:
            st = lib.gdn_chunk_fwd(
                _ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(beta), _ptr(S0),
                _ptr(o), _ptr(S_final), N, H, T, dk, dv, int(C), _ptr(cu_seqlens),
                _DTYPES[q.dtype], handle)
        else:
            st = lib.gdn_chunk_fwd_eta(
                _ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(beta), _ptr(eta), _ptr(S0),
                _ptr(o), _ptr(S_final), N, H, T, dk, dv, int(C), _ptr(cu_seqlens),
                _DTYPES[q.dtype], handle)
    _lib.check(st)
    return o, S_final


def gdn_chunk_fwd_scan(q, k, v, log_alpha, beta, S0=None, o=None, S_final=None, C=64,
                       segments=0, workspace=None, stream=None, cu_seqlens=None):
    """``gdn_chunk_fwd`` with each sequence cut into ``segments`` pieces that
    run in parallel (0 = chosen by the library); returns ``(o, S_final)``.
    ``cu_seqlens`` (int32 CUDA tensor [N+1]) packs N sequences along the
    token axis as in ``gdn_chunk_fwd``.  ``workspace`` is a uint8 CUDA tensor
    of at least ``gdn_chunk_fwd_scan_workspace_size(...)`` bytes, allocated
    here if None."""
    B, T, H, dk, dv, N = _check_args(q, k, v, log_alpha, beta, None, S0, o, S_final, cu_seqlens)
    lib = _lib.load()
    if o is None:
        o = torch.empty((B, T, H, dv), dtype=q.dtype, device=q.device)
    if S_final is None:
        S_final = torch.empty((N, H, dv, dk), dtype=torch.float32, device=q.device)
    with torch.cuda.device(q.device):
        need = gdn_chunk_fwd_scan_workspace_size(N, H, T, dk, dv, C, segments,
                                                 packed=cu_seqlens is not None)
        if workspace is None:
            workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
        _need_cuda("workspace", workspace, torch.uint8)
        st = lib.gdn_chunk_fwd_scan(
            _ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(beta), _ptr(S0), _ptr(o),
            _ptr(S_final), N, H, T, dk, dv, int(C), _ptr(cu_seqlens), _DTYPES[q.dtype],
            int(segments), _ptr(workspace), workspace.numel(),
            ctypes.c_void_p(_stream_handle(stream, q.device)))
    _lib.check(st)
    return o, S_final


def gdn_chunk_fwd_scan_noalloc(q, k, v, log_alpha, beta, S0=None, o=None, S_final=None, C=64,
                               segments=0, stream=None, cu_seqlens=None):
    """``gdn_chunk_fwd_scan`` on the library's fixed device scratch (no
    workspace, nothing allocated by the call; o and S_final must then be
    passed in to allocate nothing at all).  Calls overlapping in time race."""
    B, T, H, dk, dv, N = _check_args(q, k, v, log_alpha, beta, None, S0, o, S_final, cu_seqlens)
    lib = _lib.load()
    if o is None:
        o = torch.empty((B, T, H, dv), dtype=q.dtype, device=q.device)
    if S_final is None:
        S_final = torch.empty((N, H, dv, dk), dtype=torch.float32, device=q.device)
    with torch.cuda.device(q.device):
        st = lib.gdn_chunk_fwd_scan_noalloc(
            _ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(beta), _ptr(S0), _ptr(o),
            _ptr(S_final), N, H, T, dk, dv, int(C), _ptr(cu_seqlens), _DTYPES[q.dtype],
            int(segments), ctypes.c_void_p(_stream_handle(stream, q.device)))
    _lib.check(st)
    return o, S_final


def gdn_chunk_fwd_scan_workspace_size(B, H, T, d_k, d_v, C=64, segments=0, packed=False):
    """Bytes of device workspace gdn_chunk_fwd_scan needs (0: none); ``B`` is
    the number of sequences and ``packed`` says whether they come packed
    (cu_seqlens; ``T`` is then the packed length)."""
    marker = ctypes.c_void_p(1) if packed else None  # only NULL-ness reaches the library
    return int(_lib.load().gdn_chunk_fwd_scan_workspace_size(B, H, T, d_k, d_v, int(C), marker,
                                                              int(segments)))


def _stream_handle(stream, device):
    if stream is None:
        return torch.cuda.current_stream(device).cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def gdn_decode_step(q, k, v, log_alpha, beta, S_in=None, o=None, S_out=None, stream=None):
    """Recurrent (token-by-token) gated delta rule; returns ``(o, S_out)``.

    q, k [N,T,H,d_k] and v [N,T,H,d_v] (fp32 or bf16, one dtype), or
    [N,H,d] for a single token; log_alpha, beta [N,T,H] (or [N,H]) fp32;
    S_in [N,H,d_v,d_k] fp32 or None (zeros).  ``S_out`` may be ``S_in`` for an
    in-place update; if None a new tensor is allocated.
    """
    if q.dtype not in _DTYPES:
        raise TypeError("q/k/v dtype must be float32 or bfloat16, got %s" % q.dtype)
    single = q.dim() == 3
    if single:
        q, k, v = q.unsqueeze(1), k.unsqueeze(1), v.unsqueeze(1)
        log_alpha, beta = log_alpha.unsqueeze(1), beta.unsqueeze(1)
    for name, t in (("q", q), ("k", k), ("v", v)):
        _need_cuda(name, t, q.dtype)
    _need_cuda("log_alpha", log_alpha, torch.float32)
    _need_cuda("beta", beta, torch.float32)
    _need_cuda("S_in", S_in, torch.float32)
    if q.dim() != 4 or k.shape != q.shape or v.dim() != 4 or v.shape[:3] != q.shape[:3]:
        raise ValueError("q, k must be [N,T,H,d_k] and v [N,T,H,d_v]")
    N, T, H, dk = q.shape
    dv = v.shape[-1]
    if log_alpha.shape != (N, T, H) or beta.shape != (N, T, H):
        raise ValueError("log_alpha and beta must be [N,T,H]")
    if S_in is not None and S_in.shape != (N, H, dv, dk):
        raise ValueError("S_in must be [N,H,d_v,d_k] = %s" % ((N, H, dv, dk),))
    if o is None:
        o = torch.empty((N, T, H, dv), dtype=q.dtype, device=q.device)
    elif single:
        o = o.unsqueeze(1)
    _need_cuda("o", o, q.dtype)
    if o.shape != (N, T, H, dv):
        raise ValueError("o must be [N,T,H,d_v] (or [N,H,d_v] for one token)")
    if S_out is None:
        S_out = torch.empty((N, H, dv, dk), dtype=torch.float32, device=q.device)
    _need_cuda("S_out", S_out, torch.float32)
    if S_out.shape != (N, H, dv, dk):
        raise ValueError("S_out must be [N,H,d_v,d_k] = %s" % ((N, H, dv, dk),))
    lib = _lib.load()
    with torch.cuda.device(q.device):
        st = lib.gdn_decode_step(
            _ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(beta), _ptr(S_in),
            _ptr(o), _ptr(S_out), N, H, T, dk, dv, _DTYPES[q.dtype],
            ctypes.c_void_p(_stream_handle(stream, q.device)))
    _lib.check(st)
    return (o.squeeze(1) if single else o), S_out


def gdn_ut_inverse(A, T=None, method=0, stream=None):
    """Batched T = (I + StrictLower(A))^{-1} for A [count, C, C] fp32 CUDA;
    method 0 forward substitution (CUDA cores), 1 doubling product (tensor
    cores).  Returns T."""
    lib = _lib.load()
    _need_cuda("A", A, torch.float32)
    if A.dim() != 3 or A.shape[1] != A.shape[2]:
        raise ValueError("A must be [count, C, C]")
    if T is None:
        T = torch.empty_like(A)
    _need_cuda("T", T, torch.float32)
    with torch.cuda.device(A.device):
        st = lib.gdn_ut_inverse(_ptr(A), _ptr(T), A.shape[0], A.shape[1], int(method),
                                ctypes.c_void_p(_stream_handle(stream, A.device)))
    _lib.check(st)
    return T


def gdn_get_device_status(stream=None):
    """Synchronise and return (then clear) the device status bits.  A timed-out
    wait or an fp16 overflow comes back as its bit (GDN_DEV_WAIT_TIMEOUT,
    GDN_DEV_F16_RANGE; the C call's GDN_ERR_TIMEOUT / GDN_ERR_RANGE), not as
    an exception."""
    handle = (torch.cuda.current_stream().cuda_stream if stream is None
              else getattr(stream, "cuda_stream", stream))
    flags = ctypes.c_uint(0)
    st = _lib.load().gdn_get_device_status(ctypes.c_void_p(handle), ctypes.byref(flags))
    if st not in (_lib.GDN_ERR_TIMEOUT, _lib.GDN_ERR_RANGE):
        _lib.check(st)
    return flags.value


def gdn_last_launch_count():
    """(kernels enqueued by the last gdn_chunk_fwd / gdn_chunk_fwd_scan /
    gdn_decode_step on this thread, path id: 0 fp32 chunk kernel, 1 tcgen05
    chunk kernel, 2 decode, 3 chunk-level scan)."""
    path = ctypes.c_int(-1)
    n = _lib.load().gdn_last_launch_count(ctypes.byref(path))
    return n, path.value


def gdn_version():
    return _lib.load().gdn_version()
