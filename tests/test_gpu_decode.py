"""GPU parity of the recurrent decode entry point (gdn_decode_step, through the
C ABI) against the fp64 oracle, which runs the same recurrence token by token
from the same initial state.  Metrics and tolerances: ``parity_util``."""
import numpy as np
import pytest
import torch

from gated_delta_rule_09_gb300 import inputs as I
from oracle import gdn_recurrence_f64
from parity_util import dev, err, tol

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gdn():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import gated_delta_rule_09_gb300 as g
    return g


def check(gdn, x, dtype, in_place=False, S_in="given"):
    d = dev(x)
    S0 = d["S0"] if S_in == "given" else None
    S_out = S0.clone() if (in_place and S0 is not None) else None
    o, S = gdn.gdn_decode_step(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"],
                               S_in=S_out if in_place else S0, S_out=S_out)
    assert gdn.gdn_last_launch_count() == (1, 2)
    assert gdn.gdn_get_device_status() == 0
    ro, rS = gdn_recurrence_f64(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"],
                                S0=x["S0"] if S_in == "given" else None)
    eo = err(o.double().cpu().numpy(), ro, dtype)
    es = err(S.double().cpu().numpy(), rS, dtype, rounded=False)
    assert np.isfinite(eo) and eo <= tol(dtype), ("o", eo)
    assert np.isfinite(es) and es <= tol(dtype), ("S_out", es)
    return o, S


@pytest.mark.parametrize("N,H,T,dk,dv,dtype", [
    (4, 16, 1, 128, 128, "bf16"),     # one decoding step, 8-row groups x 16
    (3, 2, 1, 128, 128, "f32"),
    (2, 3, 1, 96, 192, "bf16"),       # the hybrid-model head shape
    (2, 2, 1, 13, 7, "f32"),          # d_k not a multiple of 4: scalar lane layout; d_v < 8
    (2, 2, 1, 64, 61, "bf16"),        # ragged last row group
    (5, 3, 7, 128, 128, "bf16"),      # several tokens per call
    (1, 1, 64, 16, 16, "f32"),
    (2, 2, 3, 128, 256, "bf16"),
    (1, 1, 1, 1, 1, "f32"),
])
def test_decode_shapes(gdn, N, H, T, dk, dv, dtype):
    x = I.custom(N, H, T, dk, dv, 64, dtype=dtype, seed=N * 7 + T * 13 + dk + dv,
                 s0="normal_0.02")
    check(gdn, x, dtype)


def test_decode_zero_state_and_in_place(gdn):
    x = I.custom(3, 4, 2, 128, 128, 64, dtype="bf16", seed=11, s0="normal_0.02")
    check(gdn, x, "bf16", S_in=None)
    check(gdn, x, "bf16", in_place=True)


def test_decode_extended_beta(gdn):
    x = I.custom(2, 4, 5, 128, 128, 64, dtype="bf16", seed=12, s0="normal_0.02")
    x["beta"] = x["beta"] * 2.0
    check(gdn, x, "bf16")


def test_decode_zero_tokens_copies_state(gdn):
    x = I.custom(2, 3, 1, 64, 32, 64, dtype="f32", seed=13, s0="normal_0.02")
    d = dev(x)
    e = lambda t: t[:, :0].contiguous()
    o, S = gdn.gdn_decode_step(e(d["q"]), e(d["k"]), e(d["v"]), e(d["log_alpha"]),
                               e(d["beta"]), S_in=d["S0"])
    assert o.shape[1] == 0
    assert torch.equal(S, d["S0"])
    _, Z = gdn.gdn_decode_step(e(d["q"]), e(d["k"]), e(d["v"]), e(d["log_alpha"]), e(d["beta"]))
    assert torch.count_nonzero(Z) == 0


def test_prefill_then_decode_is_the_whole_recurrence(gdn):
    """gdn_chunk_fwd over the first tokens (tensor-core path), then one
    gdn_decode_step per remaining token carrying the state in place, equals
    the oracle over the whole sequence."""
    T0, T1 = 200, 6
    x = I.custom(2, 4, T0 + T1, 128, 128, 64, dtype="bf16", seed=14, s0="normal_0.02")
    d = dev(x)
    pre = {k: d[k][:, :T0].contiguous() for k in ("q", "k", "v", "log_alpha", "beta")}
    o_pre, S = gdn.gdn_chunk_fwd(pre["q"], pre["k"], pre["v"], pre["log_alpha"], pre["beta"],
                                 S0=d["S0"].clone(), C=64)
    assert gdn.gdn_last_launch_count()[1] == 1
    outs = [o_pre]
    for t in range(T0, T0 + T1):
        step = {k: d[k][:, t].contiguous() for k in ("q", "k", "v", "log_alpha", "beta")}
        o_t, S = gdn.gdn_decode_step(step["q"], step["k"], step["v"], step["log_alpha"],
                                     step["beta"], S_in=S, S_out=S)
        outs.append(o_t.unsqueeze(1))
    assert gdn.gdn_get_device_status() == 0
    o = torch.cat(outs, dim=1)
    ro, rS = gdn_recurrence_f64(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], S0=x["S0"])
    assert err(o.double().cpu().numpy(), ro, "bf16") <= tol("bf16")
    assert err(S.double().cpu().numpy(), rS, "bf16", rounded=False) <= tol("bf16")


def test_decode_serving_batch_full_size(gdn):
    """The benchmarked decode workload (256 sequences x 16 heads, d 128, one
    token, state in place), every output and state element compared."""
    x = I.decode_inputs(seed=0)
    check(gdn, x, "bf16", in_place=True)


def test_decode_deterministic(gdn):
    x = I.custom(4, 4, 3, 128, 128, 64, dtype="bf16", seed=15, s0="normal_0.02")
    d = dev(x)
    a = gdn.gdn_decode_step(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], S_in=d["S0"])
    b = gdn.gdn_decode_step(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], S_in=d["S0"])
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
