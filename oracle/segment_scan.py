"""Segment propagators and their scan, in fp64 (TEST INFRASTRUCTURE ONLY).

The state update of the gated delta rule is affine in the state: over any
run of tokens, S_end = S_start M + B, where (recurrent form of "从零开始的 GDN
推导", written with column vectors and S in R^{d_v x d_k})

  one token:   M = alpha (I - beta k k^T)   (d_k x d_k),   B = beta v k^T,
  a run:       M = M_1 M_2 ... M_n,  B = (((B_1 M_2) + B_2) M_3 + ...) + B_n.

Affine maps compose associatively ("Параллельность RNN?", §"Уровень 2:
рекуррентность линейна, и потому ассоциативна"), so a sequence cut into
segments can be evaluated by computing every segment's (M, B), scanning
x_{s+1} = x_s M_s + B_s for the state each segment starts from, and running
each segment from it.  This module states that decomposition with the oracle
recurrence as its only arithmetic step:

  B_s = the recurrence over the segment from the zero state,
  M_s = the recurrence over the segment with v = 0 from S0 = I (d_k x d_k):
        its rows evolve as x <- x M_t exactly.
"""
from __future__ import annotations

import numpy as np

from . import gdn_recurrence_f64


def _seq(x, lo, hi):
    return x[:, lo:hi]


def segment_propagator(q, k, v, log_alpha, beta):
    """(M [H, d_k, d_k], B [H, d_v, d_k]) of one run of tokens.

    q, k [1, n, H, d_k], v [1, n, H, d_v], log_alpha, beta [1, n, H] (any
    float arrays or tensors)."""
    q, k, v = (np.asarray(x, np.float64) for x in (q, k, v))
    log_alpha, beta = np.asarray(log_alpha, np.float64), np.asarray(beta, np.float64)
    H, dk = k.shape[2], k.shape[3]
    _, B = gdn_recurrence_f64(q, k, v, log_alpha, beta)
    eye = np.broadcast_to(np.eye(dk), (1, H, dk, dk)).copy()
    _, M = gdn_recurrence_f64(q, k, np.zeros(k.shape), log_alpha, beta, S0=eye)
    return M[0], B[0]


def segment_scan_f64(q, k, v, log_alpha, beta, segments, C=64, S0=None):
    """The forward pass of B sequences evaluated segment by segment.

    Each sequence of T tokens is cut into ``segments`` pieces of
    ceil(ceil(T / C) / segments) chunks; returns (o [B, T, H, d_v],
    S_final [B, H, d_v, d_k]) and the starting states [B, P, H, d_v, d_k]."""
    q, k, v = (np.asarray(x, np.float64) for x in (q, k, v))
    log_alpha, beta = np.asarray(log_alpha, np.float64), np.asarray(beta, np.float64)
    Bn, T, H, dk = k.shape
    dv = v.shape[3]
    nchunks = -(-T // C)
    per = -(-nchunks // segments) * C
    bounds = [(lo, min(lo + per, T)) for lo in range(0, T, per)]
    o = np.zeros((Bn, T, H, dv))
    S_final = np.zeros((Bn, H, dv, dk))
    starts = np.zeros((Bn, len(bounds), H, dv, dk))
    for b in range(Bn):
        sl = slice(b, b + 1)
        x = np.zeros((H, dv, dk)) if S0 is None else np.asarray(S0, np.float64)[b].copy()
        for s, (lo, hi) in enumerate(bounds):
            starts[b, s] = x
            args = [a[sl, lo:hi] for a in (q, k, v, log_alpha, beta)]
            M, Bs = segment_propagator(*args)
            x = np.einsum("hvi,hij->hvj", x, M) + Bs
        for s, (lo, hi) in enumerate(bounds):
            args = [a[sl, lo:hi] for a in (q, k, v, log_alpha, beta)]
            os_, Ss = gdn_recurrence_f64(*args, S0=starts[b, s][None])
            o[b, lo:hi] = os_[0]
            if s == len(bounds) - 1:
                S_final[b] = Ss[0]
    return o, S_final, starts
