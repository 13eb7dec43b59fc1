"""Chunkwise (WY / UT-transform) statement of the gated delta rule in fp64 numpy.

TEST INFRASTRUCTURE ONLY (see the package docstring).  This is the second,
independent formula used to localise a disagreement stage by stage; the oracle
proper is the sequential recurrence in ``gdn_oracle.c``.

It takes the steps of "从零开始的 GDN 推导" (§"总结", the four-step summary) in
that page's order, transposed to the orientation S in R^{d_v x d_k} used by the
library.  For one chunk of n tokens with incoming state S:

  g      = inclusive cumulative sum of log(alpha) inside the chunk; exp(g_i) is
           the page's gamma_{i+1} (§"推导 WY-representation", gamma_0 = 1).
  L      = StrictLower(B Gamma K K^T Gamma^{-1}),  L_ij = beta_i e^{g_i-g_j} k_i.k_j
           (§"UT transform").
  T      = (I + L)^{-1}, by forward substitution ("RNN的复兴03：现代RNN的并行计算",
           §2.3.1; that page writes the strictly lower matrix with the opposite
           sign, A = -L, and T = (E - A)^{-1}).
  W      = T B Gamma K,  U = T B V                      (§"S 的推导")
  V_new  = U - W S^T
  S_next = e^{g_C} S + V_new^T (K * e^{g_C - g})       (§"S 的推导": the page's
           gamma_C S_0 + gamma_C K^T Gamma^{-1}(U - W S_0), transposed)
  O      = Gamma Q S^T + (Lower(Q K^T) * e^{g_i - g_j}) V_new  (§"O 的推导";
           Lower keeps the diagonal)
"""
from __future__ import annotations

import numpy as np


def forward_substitution(A):
    """T = (E - A)^{-1} for a strictly lower triangular A.

    Column recursion of "RNN的复兴03：现代RNN的并行计算", §2.3.1:
    T[j,j] = 1, T[i,j] = sum_{m=j}^{i-1} A[i,m] T[m,j] for i > j, 0 above.
    """
    A = np.asarray(A, dtype=np.float64)
    C = A.shape[0]
    T = np.zeros((C, C), dtype=np.float64)
    for j in range(C):
        T[j, j] = 1.0
        for i in range(j + 1, C):
            T[i, j] = np.dot(A[i, j:i], T[j:i, j])
    return T


def chunk_step(q, k, v, log_alpha, beta, S):
    """One chunk of the chunkwise form.

    q,k [n,dk], v [n,dv], log_alpha/beta [n], S [dv,dk] (incoming state).
    Returns a dict with every stage: g, L, T, W, U, V_new, O, S_next.
    """
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    beta = np.asarray(beta, np.float64)
    g = np.cumsum(np.asarray(log_alpha, np.float64))
    n = k.shape[0]
    decay = np.exp(g[:, None] - g[None, :])            # e^{g_i - g_j}
    strict = np.tril(np.ones((n, n)), -1)
    causal = np.tril(np.ones((n, n)), 0)
    L = strict * (beta[:, None] * (k @ k.T) * decay)    # StrictLower(B Gamma K K^T Gamma^-1)
    T = forward_substitution(-L)                        # (I + L)^{-1}
    W = T @ (beta[:, None] * np.exp(g)[:, None] * k)   # T B Gamma K
    U = T @ (beta[:, None] * v)                         # T B V
    V_new = U - W @ S.T
    gC = g[-1] if n else 0.0
    S_next = np.exp(gC) * S + V_new.T @ (k * np.exp(gC - g)[:, None])
    O = np.exp(g)[:, None] * (q @ S.T) + (causal * (q @ k.T) * decay) @ V_new
    return dict(g=g, L=L, T=T, W=W, U=U, V_new=V_new, O=O, S_next=S_next)


def gdn_chunk_reference_f64(q, k, v, log_alpha, beta, S0=None, C=64,
                            cu_seqlens=None):
    """Whole forward pass by chunks; same shapes and result as the recurrence.

    Chunks never cross a sequence boundary; the last chunk of a sequence may be
    shorter than C and uses the same formulas with its own length.
    """
    q, k, v = (np.asarray(x, np.float64) for x in (q, k, v))
    log_alpha = np.asarray(log_alpha, np.float64)
    beta = np.asarray(beta, np.float64)
    B, T_len, H, dk = q.shape
    dv = v.shape[-1]
    if cu_seqlens is None:
        spans = [(b, 0, T_len) for b in range(B)]
    else:
        cu = [int(x) for x in cu_seqlens]
        spans = [(0, cu[n], cu[n + 1]) for n in range(len(cu) - 1)]
    N = len(spans)
    o = np.zeros((B, T_len, H, dv))
    S_final = np.zeros((N, H, dv, dk))
    for n, (b, s, e) in enumerate(spans):
        for h in range(H):
            S = np.zeros((dv, dk)) if S0 is None else np.array(S0[n, h], np.float64)
            for c0 in range(s, e, C):
                c1 = min(c0 + C, e)
                r = chunk_step(q[b, c0:c1, h], k[b, c0:c1, h], v[b, c0:c1, h],
                               log_alpha[b, c0:c1, h], beta[b, c0:c1, h], S)
                o[b, c0:c1, h] = r["O"]
                S = r["S_next"]
            S_final[n, h] = S
    return o, S_final


def ut_inverse_doubling(A):
    """(I + A)^{-1} for a strictly lower n x n A as the finite Neumann series of
    "RNN的复兴03：现代RNN的并行计算" (§2.3.2: A is nilpotent, A^n = 0), grouped as
    the doubling product (I - A)(I + A^2)(I + A^4)...: with X_0 = -A and
    X_k = X_{k-1}^2, the product of (I + X_k) over X_k != 0 holds every power
    (-A)^m, m < n, exactly once (binary expansion of m)."""
    A = np.asarray(A, np.float64)
    n = A.shape[0]
    X = -A
    T = np.eye(n) + X
    span = 2
    while span < n:
        X = X @ X
        T = T @ (np.eye(n) + X)
        span *= 2
    return T
