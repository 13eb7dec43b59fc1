"""GPU parity of the chunk-level scan (gdn_chunk_fwd_scan, through the C ABI)
against the fp64 oracle recurrence.  The scan must give the same result as
the plain forward pass whatever the number of segments.  Metrics and
tolerances: ``parity_util``."""
import ctypes

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


def check(gdn, x, segments, path=3):
    d = dev(x)
    o, S = gdn.gdn_chunk_fwd_scan(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"],
                                  S0=d["S0"], segments=segments)
    assert gdn.gdn_get_device_status() == 0
    assert gdn.gdn_last_launch_count()[1] == path
    ro, rS = gdn_recurrence_f64(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], S0=x["S0"])
    eo = err(o.double().cpu().numpy(), ro, "bf16")
    es = err(S.double().cpu().numpy(), rS, "bf16", rounded=False)
    assert np.isfinite(eo) and eo <= tol("bf16"), ("o", eo)
    assert np.isfinite(es) and es <= tol("bf16"), ("S_final", es)
    return o, S


@pytest.mark.parametrize("segments", [2, 3, 16, 40])
def test_scan_segments(gdn, segments):
    """1000 tokens (16 chunks, the last ragged): 2, 3 and 16 segments, and a
    request beyond the chunk count (clamped to 16)."""
    x = I.custom(2, 2, 1000, 128, 128, 64, dtype="bf16", seed=50 + segments, s0="normal_0.02")
    check(gdn, x, segments)


def test_scan_no_initial_state_and_extended_beta(gdn):
    x = I.custom(1, 3, 700, 128, 128, 64, dtype="bf16", seed=51, beta="uniform_0_2")
    check(gdn, x, 5)


def test_scan_hybrid_head_shape(gdn):
    """d_k = 96, d_v = 192: two value tiles plus the identity tile."""
    x = I.custom(1, 2, 640, 96, 192, 64, dtype="bf16", seed=52, s0="normal_0.02")
    check(gdn, x, 4)


def test_scan_one_segment_is_the_plain_pass(gdn):
    x = I.custom(1, 2, 300, 128, 128, 64, dtype="bf16", seed=53, s0="normal_0.02")
    d = dev(x)
    o1, S1 = gdn.gdn_chunk_fwd_scan(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"],
                                    S0=d["S0"], segments=1)
    assert gdn.gdn_last_launch_count()[1] == 1
    o2, S2 = gdn.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], S0=d["S0"])
    assert torch.equal(o1, o2) and torch.equal(S1, S2)


def test_scan_in_place_state(gdn):
    x = I.custom(2, 2, 512, 128, 128, 64, dtype="bf16", seed=54, s0="normal_0.02")
    d = dev(x)
    S = d["S0"].clone()
    o, S_out = gdn.gdn_chunk_fwd_scan(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"],
                                      S0=S, S_final=S, segments=4)
    assert S_out is S
    ro, rS = gdn_recurrence_f64(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], S0=x["S0"])
    assert err(o.double().cpu().numpy(), ro, "bf16") <= tol("bf16")
    assert err(S.double().cpu().numpy(), rS, "bf16", rounded=False) <= tol("bf16")


def test_scan_long_sequence_sampled(gdn):
    """One 65 536-token sequence x 4 heads with the library's segment count;
    every output is compared (the oracle finishes in about a second)."""
    x = I.custom(1, 4, 65536, 128, 128, 64, dtype="bf16", seed=55, s0="normal_0.02")
    need = gdn.gdn_chunk_fwd_scan_workspace_size(1, 4, 65536, 128, 128, 64, 0)
    assert need > 0
    check(gdn, x, 0)


def test_scan_rejects_small_workspace_and_fp32(gdn):
    from gated_delta_rule_09_gb300 import _lib
    x = I.custom(1, 1, 256, 128, 128, 64, dtype="bf16", seed=56)
    d = dev(x)
    need = gdn.gdn_chunk_fwd_scan_workspace_size(1, 1, 256, 128, 128, 64, 4)
    small = torch.empty(need - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(_lib.GdnError) as e:
        gdn.gdn_chunk_fwd_scan(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], segments=4,
                               workspace=small)
    assert e.value.status == _lib.GDN_ERR_INVALID_ARG
    xf = I.custom(1, 1, 256, 128, 128, 64, dtype="f32", seed=57)
    df = dev(xf)
    with pytest.raises(_lib.GdnError) as e:
        gdn.gdn_chunk_fwd_scan(df["q"], df["k"], df["v"], df["log_alpha"], df["beta"], segments=4)
    assert e.value.status == _lib.GDN_ERR_UNSUPPORTED


def check_packed(gdn, x, segments, fn=None):
    """Packed sequences (cu_seqlens) through the scan, against the oracle run
    sequence by sequence."""
    d = dev(x)
    fn = fn or gdn.gdn_chunk_fwd_scan
    o, S = fn(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], S0=d["S0"], segments=segments,
              cu_seqlens=d["cu_seqlens"])
    assert gdn.gdn_get_device_status() == 0
    # segments = 0: the library may choose one segment, the plain pass (path 1)
    assert gdn.gdn_last_launch_count()[1] in ((3,) if segments else (1, 3))
    ro, rS = gdn_recurrence_f64(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], S0=x["S0"],
                                cu_seqlens=x["cu_seqlens"])
    eo = err(o.double().cpu().numpy(), ro, "bf16")
    es = err(S.double().cpu().numpy(), rS, "bf16", rounded=False)
    assert np.isfinite(eo) and eo <= tol("bf16"), ("o", eo)
    assert np.isfinite(es) and es <= tol("bf16"), ("S_final", es)
    return o, S


@pytest.mark.parametrize("segments", [3, 8, 0])
def test_scan_packed_sequences(gdn, segments):
    """Packed ragged sequences, an empty one and one shorter than a chunk
    among them: every sequence is cut into the same number of segments (the
    short ones leave trailing segments empty), each from its own S0."""
    lens = [1, 64, 100, 1000, 0, 700, 130, 450]
    x = I.custom(1, 2, 0, 128, 128, 64, dtype="bf16", seed=70 + segments, lengths=lens,
                 s0="normal_0.02")
    check_packed(gdn, x, segments)


def test_scan_packed_matches_plain_packed_pass(gdn):
    """The packed scan and the plain packed forward pass agree (up to the
    rounding of the segment decomposition) on the varlen length mix."""
    lens = [1500, 640, 2100, 77]
    x = I.custom(1, 2, 0, 128, 128, 64, dtype="bf16", seed=74, lengths=lens, s0="normal_0.02")
    o, S = check_packed(gdn, x, 6)
    d = dev(x)
    o2, S2 = gdn.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], S0=d["S0"],
                               cu_seqlens=d["cu_seqlens"])
    rms = o2.float().pow(2).mean().sqrt().item()
    assert (o.float() - o2.float()).abs().max().item() <= 2e-2 * rms


def test_scan_packed_noalloc_is_the_workspace_entry(gdn):
    lens = [300, 1000, 5, 640]
    x = I.custom(1, 2, 0, 128, 128, 64, dtype="bf16", seed=75, lengths=lens, s0="normal_0.02")
    a = check_packed(gdn, x, 4, fn=gdn.gdn_chunk_fwd_scan_noalloc)
    b = check_packed(gdn, x, 4)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_scan_packed_bad_span_is_flagged(gdn):
    """An offset past the packed length: GDN_DEV_BAD_SEQLENS, and the other
    sequences are still right."""
    lens = [200, 300]
    x = I.custom(1, 2, 0, 128, 128, 64, dtype="bf16", seed=76, lengths=lens, s0="normal_0.02")
    d = dev(x)
    bad = d["cu_seqlens"].clone()
    bad[2] = 10 ** 6  # sequence 1 runs past T
    o, S = gdn.gdn_chunk_fwd_scan(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], S0=d["S0"],
                                  segments=3, cu_seqlens=bad)
    assert gdn.gdn_get_device_status() & 0x1
    ro, rS = gdn_recurrence_f64(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], S0=x["S0"],
                                cu_seqlens=x["cu_seqlens"])
    n0 = lens[0]
    eo = err(o[0, :n0].double().cpu().numpy(), ro[0, :n0], "bf16")
    es = err(S[0].double().cpu().numpy(), rS[0], "bf16", rounded=False)
    assert eo <= tol("bf16") and es <= tol("bf16"), (eo, es)


def test_scan_packed_hybrid_head_shape(gdn):
    """Packed sequences with d_k = 96, d_v = 192 through the scan: two value
    tiles plus the identity tile per segment, 96-wide transitions."""
    lens = [700, 130, 0, 1000]
    x = I.custom(1, 2, 0, 96, 192, 64, dtype="bf16", seed=77, lengths=lens, s0="normal_0.02",
                 beta="uniform_0_2")
    check_packed(gdn, x, 5)
