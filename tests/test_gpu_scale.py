"""Input scales on the tensor-core path: each case either matches the fp64
oracle within the bf16 bound or raises a device status bit; it never misses
silently.

The path converts bf16 inputs and the fp32 state to fp16 tensor-core
operands.  fp16 is exact for magnitudes in [2^-14, 65504]: far below it the
operands lose bits (GDN_DEV_F16_PRECISION), above it they overflow
(GDN_DEV_F16_RANGE).  The method is linear in (v, S0), so those two carry the
scale; the keys enter the erase term beta k k^T, so their norm is varied
with beta kept where the recurrence stays bounded (beta ||k||^2 <= 2: the
transition I - beta k k^T is then non-expansive, the Olmo page's condition
for beta in (0, 2) with unit keys)."""
import numpy as np
import pytest
import torch

from gated_delta_rule_09_gb300 import inputs as I
from oracle import gdn_recurrence_f64
from parity_util import TOL_BF16, dev, err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gdn():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import gated_delta_rule_09_gb300 as g
    return g


def bf16(x):
    return x.to(torch.bfloat16)


def check(gdn, x, expect_flag=None):
    """Run the tensor-core path on x and return (status, o error, S error).
    The call must either be within the bound or carry a status bit."""
    from gated_delta_rule_09_gb300 import _lib
    d = dev(x)
    o, S = gdn.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], S0=d["S0"], C=64)
    assert gdn.gdn_last_launch_count()[1] == 1  # the tensor-core kernel ran
    status = gdn.gdn_get_device_status()
    ro, rS = gdn_recurrence_f64(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], S0=x["S0"])
    eo = err(o.double().cpu().numpy(), ro, "bf16")
    es = err(S.double().cpu().numpy(), rS, "bf16", rounded=False)
    flags = _lib.GDN_DEV_F16_PRECISION | _lib.GDN_DEV_F16_RANGE
    within = np.isfinite(eo) and np.isfinite(es) and eo <= TOL_BF16 and es <= TOL_BF16
    assert within or (status & flags), ("silent miss", eo, es, status)
    if expect_flag is not None:
        assert status & expect_flag, (status, eo, es)
    return status, eo, es


def scaled(seed, scale):
    x = I.custom(1, 2, 320, 128, 128, 64, dtype="bf16", seed=seed, s0="normal_0.02")
    x["v"] = bf16(x["v"].float() * scale)
    x["S0"] = x["S0"] * scale
    return x


def test_tiny_values_and_state_are_flagged(gdn):
    """v and S0 of order 1e-6: every state-chain operand sits in fp16's
    subnormal range; the precision bit is required."""
    from gated_delta_rule_09_gb300 import _lib
    check(gdn, scaled(80, 1e-6), expect_flag=_lib.GDN_DEV_F16_PRECISION)


def test_small_but_normal_values_pass(gdn):
    """v and S0 of order 1e-2: still well inside fp16's normal range."""
    status, eo, es = check(gdn, scaled(81, 1e-2))
    assert status == 0 and eo <= TOL_BF16 and es <= TOL_BF16


def test_large_values_and_state(gdn):
    """v and S0 of order 1e3: the state and outputs grow to ~1e4, inside fp16's
    range; the result must be within the bound (or flagged)."""
    check(gdn, scaled(82, 1e3))


@pytest.mark.parametrize("norm", [0.25, 4.0])
def test_non_unit_keys(gdn, norm):
    """Keys of norm 4 (and 1/4) with beta ~ U(0, 2 / ||k||^2)."""
    x = I.custom(1, 2, 320, 128, 128, 64, dtype="bf16", seed=83, s0="normal_0.02")
    x["k"] = bf16(x["k"].float() * norm)
    x["beta"] = x["beta"] * min(1.0, 2.0 / norm ** 2)
    check(gdn, x)


def test_large_queries(gdn):
    """Queries scaled by 30: outputs scale with them; no operand leaves fp16."""
    x = I.custom(1, 2, 320, 128, 128, 64, dtype="bf16", seed=84, s0="normal_0.02")
    x["q"] = bf16(x["q"].float() * 30.0)
    status, eo, es = check(gdn, x)
    assert status == 0


def test_growing_gate_overflow_is_flagged(gdn):
    """log alpha > 0 is allowed.  One chunk whose last four tokens grow the
    gate by e^4 each, with q = k = 0 and beta = 0 there (so P, A and T'' stay
    in range): the state-update operand V_new e^{g_C - g} is ~e^16 times V_new
    and leaves fp16, while the exact final state (~5e6) is finite in fp32.
    The kernel cannot represent it and must say so."""
    from gated_delta_rule_09_gb300 import _lib
    x = I.custom(1, 1, 64, 128, 128, 64, dtype="bf16", seed=7)
    x["q"][:, 60:] = 0
    x["k"][:, 60:] = 0
    x["beta"][:, 60:] = 0
    x["log_alpha"][:, 60:] = 4.0
    check(gdn, x, expect_flag=_lib.GDN_DEV_F16_RANGE)


@pytest.mark.parametrize("lo,hi", [(0.0, 0.02), (-0.05, 0.03)])
def test_growing_gate_in_range(gdn, lo, hi):
    """log alpha ~ U(lo, hi) with lo >= 0 (the state grows ~e^0.64 a chunk)
    or of mixed sign: every decay factor the kernel splits or ships can then
    exceed 1.  Five chunks stay well inside fp16, so the result must be
    within the bound with a clean status."""
    x = I.custom(1, 2, 320, 128, 128, 64, dtype="bf16", seed=85, s0="normal_0.02")
    rng = np.random.default_rng(86)
    x["log_alpha"] = torch.from_numpy(rng.uniform(lo, hi, tuple(x["log_alpha"].shape))).to(torch.float32)
    status, eo, es = check(gdn, x)
    assert status == 0 and eo <= TOL_BF16 and es <= TOL_BF16, (status, eo, es)
