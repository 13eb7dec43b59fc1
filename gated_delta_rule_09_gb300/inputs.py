"""Seeded synthetic inputs for the gated delta rule forward pass.

This module is shared by the tests, the benchmark and the smoke check; it
holds no step of the method itself, only the input distributions.  Every
tensor is drawn in fp64 from ``numpy.random.default_rng(seed)`` in a fixed
order (sequence lengths, q, k, v, beta, alpha or log alpha, S0, eta), normalised
in fp64 where a workload asks for unit-norm keys or queries, then rounded once
to the workload's dtype (round-to-nearest-even for bf16).  The oracle sees the
same rounded values widened back to fp64.

The named workloads:

==================  ==========================================================
``tiny_f32``        B1 H1 T64 d_k=d_v=16 C16, fp32.  q,v ~ N(0,1); k ~ N(0,1)
                    then unit norm; beta ~ U(0,1); alpha ~ U(0.9,1),
                    log alpha = ln alpha; S0 = explicit zeros.
``small_bf16``      B2 H4 T1024 d64 C64, bf16.  q,k ~ N(0,1) then unit norm;
                    v ~ N(0,1); beta = sigmoid(N(0,1));
                    log alpha = -softplus(N(0,1)) * 0.1; no S0.
``train_bf16``      B4 H16 T4096 d128 C64, bf16, same distributions as
                    ``small_bf16``; final state returned.
``varlen_bf16``     8 sequences packed through cu_seqlens, lengths drawn as
                    integers U[1024, 8192]; H32 d128 C64; same distributions;
                    per-sequence S0 ~ N(0, sd 0.02).
``wide_ungated_bf16`` B8 H8 T2048 d_k128 d_v256 C64; alpha == 1 (log alpha 0);
                    k ~ N(0,1) then unit norm; beta ~ U(0,1); q,v ~ N(0,1);
                    S0 ~ N(0, sd 0.02).
``hybrid_bf16``     B4 H16 T4096 d_k96 d_v192 C64 (the hybrid model's head
                    shape); beta ~ U(0,2) (the extended range); otherwise the
                    ``small_bf16`` distributions; no S0.
==================  ==========================================================

The decode batch (``decode_inputs``): 256 sequences x 16 heads, d_k = d_v =
128, bf16, one token each from a state S_in ~ N(0, sd 0.02), with the
``small_bf16`` distributions for q, k, v, beta and log alpha.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int                 # batch, or number of packed sequences when varlen
    H: int
    T: int                 # tokens per sequence (ignored when varlen)
    dk: int
    dv: int
    C: int
    dtype: str             # "f32" or "bf16"
    q_unit: bool           # normalise q per token
    beta_dist: str         # "uniform" | "uniform_0_2" | "sigmoid_normal"
    alpha_dist: str        # "uniform_0.9_1" | "softplus_0.1" | "one"
    s0: str                # "none" | "zeros" | "normal_0.02"
    varlen: bool = False
    len_lo: int = 0
    len_hi: int = 0
    eta_dist: str = "none"  # "none" | "uniform": a write strength separate from beta


WORKLOADS = {
    "tiny_f32": Workload("tiny_f32", 1, 1, 64, 16, 16, 16, "f32", False,
                         "uniform", "uniform_0.9_1", "zeros"),
    "small_bf16": Workload("small_bf16", 2, 4, 1024, 64, 64, 64, "bf16", True,
                           "sigmoid_normal", "softplus_0.1", "none"),
    "train_bf16": Workload("train_bf16", 4, 16, 4096, 128, 128, 64, "bf16", True,
                           "sigmoid_normal", "softplus_0.1", "none"),
    "varlen_bf16": Workload("varlen_bf16", 8, 32, 0, 128, 128, 64, "bf16", True,
                            "sigmoid_normal", "softplus_0.1", "normal_0.02",
                            varlen=True, len_lo=1024, len_hi=8192),
    "wide_ungated_bf16": Workload("wide_ungated_bf16", 8, 8, 2048, 128, 256, 64,
                                  "bf16", False, "uniform", "one", "normal_0.02"),
    "hybrid_bf16": Workload("hybrid_bf16", 4, 16, 4096, 96, 192, 64, "bf16", True,
                            "uniform_0_2", "softplus_0.1", "none"),
}

TORCH_DTYPE = {"f32": torch.float32, "bf16": torch.bfloat16}


def _unit(x):
    n = np.sqrt(np.sum(x * x, axis=-1, keepdims=True))
    return x / np.maximum(n, 1e-300)


def _sigmoid(x):
    return 1.0 / (1.0 + np.exp(-x))


def _softplus(x):
    return np.logaddexp(0.0, x)


def generate(w: Workload, seed: int = 0, lengths=None, S0: Optional[str] = None):
    """Draw the inputs of workload ``w``.

    Returns a dict of CPU torch tensors: q, k [B,T,H,dk] and v [B,T,H,dv] in
    the workload dtype; log_alpha, beta [B,T,H] fp32; S0 [N,H,dv,dk] fp32 or
    None; cu_seqlens int32 [N+1] or None; plus ``N`` and ``lengths``.
    ``lengths`` overrides the drawn sequence lengths of a varlen workload
    (still packed); ``S0`` overrides the workload's initial-state recipe.
    """
    rng = np.random.default_rng(seed)
    if w.varlen:
        if lengths is None:
            lengths = rng.integers(w.len_lo, w.len_hi + 1, size=w.B)
        lengths = [int(x) for x in lengths]
        N = len(lengths)
        Bt, Tt = 1, int(sum(lengths))
        cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    else:
        N, Bt, Tt = w.B, w.B, w.T
        lengths = [w.T] * w.B
        cu = None
    H, dk, dv = w.H, w.dk, w.dv
    q = rng.standard_normal((Bt, Tt, H, dk))
    if w.q_unit:
        q = _unit(q)
    k = _unit(rng.standard_normal((Bt, Tt, H, dk)))
    v = rng.standard_normal((Bt, Tt, H, dv))
    if w.beta_dist == "uniform":
        beta = rng.uniform(0.0, 1.0, (Bt, Tt, H))
    elif w.beta_dist == "uniform_0_2":
        beta = rng.uniform(0.0, 2.0, (Bt, Tt, H))
    else:
        beta = _sigmoid(rng.standard_normal((Bt, Tt, H)))
    if w.alpha_dist == "uniform_0.9_1":
        log_alpha = np.log(rng.uniform(0.9, 1.0, (Bt, Tt, H)))
    elif w.alpha_dist == "softplus_0.1":
        log_alpha = -_softplus(rng.standard_normal((Bt, Tt, H))) * 0.1
    else:
        log_alpha = np.zeros((Bt, Tt, H))
    s0 = w.s0 if S0 is None else S0
    if s0 == "zeros":
        S0t = np.zeros((N, H, dv, dk))
    elif s0 == "normal_0.02":
        S0t = rng.normal(0.0, 0.02, (N, H, dv, dk))
    else:
        S0t = None
    eta = rng.uniform(0.0, 1.0, (Bt, Tt, H)) if w.eta_dist == "uniform" else None
    dt = TORCH_DTYPE[w.dtype]
    out = dict(
        q=torch.from_numpy(q).to(dt),
        k=torch.from_numpy(k).to(dt),
        v=torch.from_numpy(v).to(dt),
        log_alpha=torch.from_numpy(log_alpha).to(torch.float32),
        beta=torch.from_numpy(beta).to(torch.float32),
        S0=None if S0t is None else torch.from_numpy(S0t).to(torch.float32),
        cu_seqlens=None if cu is None else torch.from_numpy(cu),
        eta=None if eta is None else torch.from_numpy(eta).to(torch.float32),
        N=N, lengths=lengths,
    )
    return out


def custom(B, H, T, dk, dv, C, dtype="bf16", seed=0, lengths=None,
           s0="none", alpha="softplus_0.1", beta="sigmoid_normal", q_unit=True, eta="none"):
    """Inputs of arbitrary shape with the small_bf16 distributions by default
    (``eta="uniform"`` adds a write strength eta ~ U(0,1), drawn last)."""
    w = Workload("custom", B if lengths is None else len(lengths), H, T, dk, dv,
                 C, dtype, q_unit, beta, alpha, s0, varlen=lengths is not None, eta_dist=eta)
    return generate(w, seed=seed, lengths=lengths)


def decode_inputs(seed=0, N=256, H=16, T=1, dk=128, dv=128, dtype="bf16"):
    """The decode batch: ``N`` sequences x ``H`` heads advancing ``T`` tokens
    from a state S_in ~ N(0, sd 0.02) (returned as ``S0``); the other tensors
    as ``custom`` draws them, laid out [N, T, H, *]."""
    return custom(N, H, T, dk, dv, 64, dtype=dtype, seed=seed, s0="normal_0.02")


def ut_matrices(count, C=64, scale=0.04, seed=0):
    """``count`` strictly lower C x C fp32 matrices with entries ~ N(0, scale^2)
    below the diagonal and zeros elsewhere (the UT-transform inverse's input;
    0.04 is the spread of beta_i e^{g_i - g_j} k_i.k_j for unit keys in 128
    dimensions, beta ~ 0.5 and in-chunk decay ~ 0.9)."""
    rng = np.random.default_rng(seed)
    a = rng.normal(0.0, scale, (count, C, C))
    a *= np.tril(np.ones((C, C)), -1)
    return torch.from_numpy(a).to(torch.float32)
