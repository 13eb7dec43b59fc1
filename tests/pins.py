"""Checks that pin a gated-delta-rule recurrence to what the pages and the
mathematics fix, independent of the implementation being checked.

Each ``check_*`` takes ``impl(q, k, v, log_alpha, beta, S0=None, eta=None,
cu_seqlens=None) -> (o, S_final)`` (fp64 numpy arrays in the oracle's layout:
q,k [B,T,H,dk], v [B,T,H,dv], gates [B,T,H], S [N,H,dv,dk]) and raises
AssertionError on a mismatch.  The tests run them on the C oracle and on
copies of it with planted mistakes, which must each fail at least one check.
"""
from __future__ import annotations

import numpy as np

TOL = 1e-11


def _rng(seed):
    return np.random.default_rng(seed)


def _unit(x):
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


def _close(a, b, tol=TOL, what=""):
    a = np.asarray(a)
    b = np.asarray(b)
    assert a.shape == b.shape, (what, a.shape, b.shape)
    scale = max(1.0, float(np.max(np.abs(b))) if b.size else 1.0)
    err = float(np.max(np.abs(a - b))) if a.size else 0.0
    assert err <= tol * scale, "%s: max abs err %.3e (scale %.3e)" % (what, err, scale)


def _transition(a, b, kk):
    """alpha (I - beta k k^T) as a dense matrix."""
    d = kk.shape[0]
    return a * (np.eye(d) - b * np.outer(kk, kk))


def check_brute_force_products(impl, seed=1, T=7, dk=5, dv=3):
    """S_t and o_t from explicit dense products, no recurrence loop.

    S_t = S0 Phi(1..t) + sum_tau eta_tau v_tau k_tau^T Phi(tau+1..t), with
    Phi(a..b) = prod_{s=a..b} alpha_s (I - beta_s k_s k_s^T) taken left to
    right ("RNN的复兴03：现代RNN的并行计算", §3.1 proof: 累积转移矩阵 and 累积更新项,
    here with the scalar gate of "从零开始的 GDN 推导" recurrent form), o_t = S_t q_t.
    dk != dv so a transposed state or readout cannot pass.
    """
    r = _rng(seed)
    q = r.standard_normal((1, T, 1, dk))
    k = _unit(r.standard_normal((1, T, 1, dk)))
    v = r.standard_normal((1, T, 1, dv))
    la = np.log(r.uniform(0.5, 1.0, (1, T, 1)))
    be = r.uniform(0.0, 1.5, (1, T, 1))
    S0 = r.standard_normal((1, 1, dv, dk))
    o, Sf = impl(q, k, v, la, be, S0=S0)
    a = np.exp(la[0, :, 0])
    b = be[0, :, 0]
    K = k[0, :, 0]
    V = v[0, :, 0]
    Q = q[0, :, 0]
    Phi = [_transition(a[s], b[s], K[s]) for s in range(T)]

    def prod(lo, hi):  # Phi(lo..hi) inclusive, 0-based; identity when empty
        M = np.eye(dk)
        for s in range(lo, hi + 1):
            M = M @ Phi[s]
        return M

    for t in range(T):
        St = S0[0, 0] @ prod(0, t)
        for tau in range(t + 1):
            St = St + b[tau] * np.outer(V[tau], K[tau]) @ prod(tau + 1, t)
        _close(o[0, t, 0], St @ Q[t], what="o_%d" % t)
    _close(Sf[0, 0], St, what="S_final")


def check_wy_identity(impl, seed=2, T=6, d=5):
    """prod_t (I - beta_t k_t k_t^T) = I - W^T K with the page's w_t recursion.

    "RNN的复兴03：现代RNN的并行计算", §2.1: w_t = beta_t k_t - beta_t
    sum_{tau<t} (k_tau^T k_t) w_tau.  With S0 = I, v = 0, alpha = 1 the
    recurrence's final state is exactly that product.
    """
    r = _rng(seed)
    k = _unit(r.standard_normal((1, T, 1, d)))
    be = r.uniform(0.0, 1.0, (1, T, 1))
    q = r.standard_normal((1, T, 1, d))
    v = np.zeros((1, T, 1, d))
    la = np.zeros((1, T, 1))
    S0 = np.eye(d)[None, None]
    _, Sf = impl(q, k, v, la, be, S0=S0)
    K = k[0, :, 0]
    b = be[0, :, 0]
    w = []
    for t in range(T):
        wt = b[t] * K[t]
        for tau in range(t):
            wt = wt - b[t] * np.dot(K[tau], K[t]) * w[tau]
        w.append(wt)
    W = np.array(w)
    P = np.eye(d)
    for t in range(T):
        P = P @ (np.eye(d) - b[t] * np.outer(K[t], K[t]))
    _close(P, np.eye(d) - W.T @ K, what="WY identity itself")
    _close(Sf[0, 0], np.eye(d) - W.T @ K, what="S_final vs I - W^T K")


def check_gated_product_expansion(impl, seed=3, T=6, d=4):
    """Gated product identity of "从零开始的 GDN 推导" (§ preceding the WY proof).

    prod_{i=t..0} alpha_i (I - E_i) = gamma_{t+1} I
        - sum_i gamma_{i+1} [prod_{j=t..i+1} alpha_j (I - E_j)] E_i,
    E_i = beta_i k_i k_i^T, gamma_i = alpha_0 ... alpha_{i-1}.  With v = 0 and
    S0 = I the recurrence's final state is the transpose of the left side.
    """
    r = _rng(seed)
    k = _unit(r.standard_normal((1, T, 1, d)))
    be = r.uniform(0.0, 1.0, (1, T, 1))
    la = np.log(r.uniform(0.6, 1.0, (1, T, 1)))
    q = r.standard_normal((1, T, 1, d))
    v = np.zeros((1, T, 1, d))
    _, Sf = impl(q, k, v, la, be, S0=np.eye(d)[None, None])
    a = np.exp(la[0, :, 0])
    b = be[0, :, 0]
    K = k[0, :, 0]
    E = [b[i] * np.outer(K[i], K[i]) for i in range(T)]
    gamma = np.concatenate([[1.0], np.cumprod(a)])   # gamma[i] = a_0..a_{i-1}
    t = T - 1
    rhs = gamma[t + 1] * np.eye(d)
    for i in range(t + 1):
        M = np.eye(d)
        for j in range(t, i, -1):          # reversed product j = t .. i+1
            M = M @ (a[j] * (np.eye(d) - E[j]))
        rhs = rhs - gamma[i + 1] * M @ E[i]
    _close(Sf[0, 0].T, rhs, what="gated product expansion")


def check_pure_decay(impl, seed=4, T=9, dk=4, dv=3):
    """beta = 0 (and eta = beta) leaves only the gate: S_t = gamma_t S0."""
    r = _rng(seed)
    q = r.standard_normal((1, T, 1, dk))
    k = _unit(r.standard_normal((1, T, 1, dk)))
    v = r.standard_normal((1, T, 1, dv))
    la = np.log(r.uniform(0.5, 1.0, (1, T, 1)))
    be = np.zeros((1, T, 1))
    S0 = r.standard_normal((1, 1, dv, dk))
    o, Sf = impl(q, k, v, la, be, S0=S0)
    g = np.cumsum(la[0, :, 0])
    for t in range(T):
        _close(o[0, t, 0], np.exp(g[t]) * S0[0, 0] @ q[0, t, 0], what="o_%d" % t)
    _close(Sf[0, 0], np.exp(g[-1]) * S0[0, 0], what="S_final")


def check_linear_attention(impl, seed=5, T=10, dk=4, dv=3):
    """alpha = 1, beta = 0, eta = 1, S0 = 0 gives O = (Q K^T * M) V.

    "从电路复杂性理论的角度分析大模型的可并行性和表达能力--Olmo Hybrid 系列",
    §前置知识 (类 RNN 模型训练): S_t = S_{t-1} + v_t k_t^T, o_t = S_t q_t,
    M the causal mask (diagonal included).
    """
    r = _rng(seed)
    q = r.standard_normal((1, T, 1, dk))
    k = r.standard_normal((1, T, 1, dk))
    v = r.standard_normal((1, T, 1, dv))
    o, _ = impl(q, k, v, np.zeros((1, T, 1)), np.zeros((1, T, 1)),
                eta=np.ones((1, T, 1)))
    Q, K, V = q[0, :, 0], k[0, :, 0], v[0, :, 0]
    M = np.tril(np.ones((T, T)))
    _close(o[0, :, 0], (Q @ K.T * M) @ V, what="linear attention")


def check_scalar_gated(impl, seed=6, T=10, dk=4, dv=3):
    """beta = 0, eta = 1, S0 = 0 gives O = ((Q K^T) * Gamma) V.

    Same page, §现代类 RNN 模型中的取舍 (the Mamba2 form S_t = a_t S_{t-1} +
    v_t k_t^T): Gamma_ij = gamma_i / gamma_j for i >= j, else 0, with
    gamma_j = a_1 ... a_j.
    """
    r = _rng(seed)
    q = r.standard_normal((1, T, 1, dk))
    k = r.standard_normal((1, T, 1, dk))
    v = r.standard_normal((1, T, 1, dv))
    la = np.log(r.uniform(0.5, 1.0, (1, T, 1)))
    o, _ = impl(q, k, v, la, np.zeros((1, T, 1)), eta=np.ones((1, T, 1)))
    gam = np.cumprod(np.exp(la[0, :, 0]))
    G = np.tril(gam[:, None] / gam[None, :])
    Q, K, V = q[0, :, 0], k[0, :, 0], v[0, :, 0]
    _close(o[0, :, 0], ((Q @ K.T) * G) @ V, what="scalar-gated closed form")


def check_retrieval(impl, seed=7, T=8, dk=6, dv=4):
    """Retrieval identities of the delta rule for unit-norm keys.

    Same page, §DeltaRule: writing (k, v) with beta = 1 onto a zero state
    gives S_1 k = v; in general v_new = beta v + (1 - beta) S_{t-1} k is what
    k_t reads back, so with the gate S_t k_t = alpha_t (1 - beta_t) S_{t-1} k_t
    + beta_t v_t.  Checked on every prefix of a random sequence.
    """
    r = _rng(seed)
    q = r.standard_normal((1, T, 1, dk))
    k = _unit(r.standard_normal((1, T, 1, dk)))
    v = r.standard_normal((1, T, 1, dv))
    la = np.log(r.uniform(0.5, 1.0, (1, T, 1)))
    be = r.uniform(0.0, 1.0, (1, T, 1))
    _, S1 = impl(q[:, :1], k[:, :1], v[:, :1], np.zeros((1, 1, 1)),
                 np.ones((1, 1, 1)))
    _close(S1[0, 0] @ k[0, 0, 0], v[0, 0, 0], what="S_1 k = v")
    S0 = r.standard_normal((1, 1, dv, dk))
    prev = S0[0, 0]
    for t in range(T):
        _, St = impl(q[:, :t + 1], k[:, :t + 1], v[:, :t + 1], la[:, :t + 1],
                     be[:, :t + 1], S0=S0)
        a, b, kt = np.exp(la[0, t, 0]), be[0, t, 0], k[0, t, 0]
        _close(St[0, 0] @ kt, a * (1 - b) * prev @ kt + b * v[0, t, 0],
               what="S_t k_t at t=%d" % t)
        prev = St[0, 0]


def check_contraction(impl, seed=8, T=12, dk=5, dv=4):
    """For beta in [0, 2] and unit k, ||I - beta k k^T||_2 <= 1, so
    ||S_t||_F <= alpha_t ||S_{t-1}||_F + beta_t ||v_t|| (extended DeltaNet
    range beta in (0, 2): same page, §扩展 DeltaNet)."""
    r = _rng(seed)
    q = r.standard_normal((1, T, 1, dk))
    k = _unit(r.standard_normal((1, T, 1, dk)))
    v = r.standard_normal((1, T, 1, dv))
    la = np.log(r.uniform(0.5, 1.0, (1, T, 1)))
    be = r.uniform(0.0, 2.0, (1, T, 1))
    S0 = 3.0 * r.standard_normal((1, 1, dv, dk))
    prev = np.linalg.norm(S0[0, 0])
    for t in range(T):
        _, St = impl(q[:, :t + 1], k[:, :t + 1], v[:, :t + 1], la[:, :t + 1],
                     be[:, :t + 1], S0=S0)
        cur = np.linalg.norm(St[0, 0])
        bound = np.exp(la[0, t, 0]) * prev + be[0, t, 0] * np.linalg.norm(v[0, t, 0])
        assert cur <= bound * (1 + 1e-12), ("contraction", t, cur, bound)
        prev = cur


def check_eta_write_strength(impl, seed=9, T=7, dk=4, dv=3):
    """Separate write strength: S_t = S_{t-1}(E - beta_t k k^T) + eta_t v k^T
    ("RNN的复兴03：现代RNN的并行计算", §一 state form), checked against the
    explicit product form of §3.1 with alpha = 1."""
    r = _rng(seed)
    q = r.standard_normal((1, T, 1, dk))
    k = _unit(r.standard_normal((1, T, 1, dk)))
    v = r.standard_normal((1, T, 1, dv))
    be = r.uniform(0.0, 1.0, (1, T, 1))
    et = r.uniform(0.0, 2.0, (1, T, 1))
    S0 = r.standard_normal((1, 1, dv, dk))
    o, Sf = impl(q, k, v, np.zeros((1, T, 1)), be, S0=S0, eta=et)
    K, V, Q = k[0, :, 0], v[0, :, 0], q[0, :, 0]
    b, e = be[0, :, 0], et[0, :, 0]
    H = [np.eye(dk) - b[s] * np.outer(K[s], K[s]) for s in range(T)]
    for t in range(T):
        P = np.eye(dk)
        for s in range(t + 1):
            P = P @ H[s]
        St = S0[0, 0] @ P
        for tau in range(t + 1):
            M = np.eye(dk)
            for s in range(tau + 1, t + 1):
                M = M @ H[s]
            St = St + e[tau] * np.outer(V[tau], K[tau]) @ M
        _close(o[0, t, 0], St @ Q[t], what="o_%d" % t)
    _close(Sf[0, 0], St, what="S_final")


def check_varlen_and_heads(impl, seed=10, H=3, dk=4, dv=5):
    """Packed sequences are independent: packing equals one call per sequence,
    heads are independent, and each sequence starts from its own S0."""
    r = _rng(seed)
    lens = [3, 0, 5, 1]
    Tt = sum(lens)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    q = r.standard_normal((1, Tt, H, dk))
    k = _unit(r.standard_normal((1, Tt, H, dk)))
    v = r.standard_normal((1, Tt, H, dv))
    la = np.log(r.uniform(0.5, 1.0, (1, Tt, H)))
    be = r.uniform(0.0, 1.0, (1, Tt, H))
    S0 = r.standard_normal((len(lens), H, dv, dk))
    o, Sf = impl(q, k, v, la, be, S0=S0, cu_seqlens=cu)
    for n in range(len(lens)):
        s, e = cu[n], cu[n + 1]
        if e == s:
            _close(Sf[n], S0[n], what="empty sequence keeps S0")
            continue
        for h in range(H):
            sl = (slice(None), slice(s, e), slice(h, h + 1))
            on, Sn = impl(q[sl], k[sl], v[sl], la[sl], be[sl],
                          S0=S0[n:n + 1, h:h + 1])
            _close(o[0, s:e, h], on[0, :, 0], what="o seq %d head %d" % (n, h))
            _close(Sf[n, h], Sn[0, 0], what="S seq %d head %d" % (n, h))


ALL_CHECKS = [
    check_brute_force_products,
    check_wy_identity,
    check_gated_product_expansion,
    check_pure_decay,
    check_linear_attention,
    check_scalar_gated,
    check_retrieval,
    check_contraction,
    check_eta_write_strength,
    check_varlen_and_heads,
]


def parse_expr(expr, A):
    """Evaluate 'A41 + A42*A21' style sums of products with A[i-1, j-1]."""
    expr = expr.strip()
    total = 0.0
    for term in expr.split("+"):
        val = 1.0
        for f in term.strip().split("*"):
            f = f.strip()
            if f == "1":
                continue
            if f == "0":
                val = 0.0
                continue
            assert f[0] == "A" and len(f) == 3, f
            val *= A[int(f[1]) - 1, int(f[2]) - 1]
        total += val
    return total


def read_golden(path):
    rows = []
    with open(path, encoding="utf-8") as fh:
        for line in fh:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            lhs, rhs = line.split("=")
            rows.append(([int(x) for x in lhs.split()], rhs.strip()))
    return rows
