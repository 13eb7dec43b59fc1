"""GPU parity: libgdn's chunkwise forward (through its C ABI) against the
fp64 oracle.  Metrics and tolerances: ``parity_util``."""
import numpy as np
import pytest
import torch

from gated_delta_rule_09_gb300 import inputs as I
from oracle import gdn_recurrence_f64
from parity_util import TOL_BF16, TOL_F32, dev as _dev, err, half_ulp_bf16  # noqa: F401

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gdn():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import gated_delta_rule_09_gb300 as g
    return g


def run_and_check(gdn, x, C, dtype, S0=None, want_S=True, tol=None):
    d = _dev(x)
    S0_dev = d["S0"] if S0 is None else S0
    o, S = gdn.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"],
                             S0=S0_dev, C=C, cu_seqlens=d["cu_seqlens"],
                             want_final_state=want_S)
    assert gdn.gdn_get_device_status() == 0
    ro, rS = gdn_recurrence_f64(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"],
                                S0=x["S0"], cu_seqlens=x["cu_seqlens"])
    tol = tol or (TOL_F32 if dtype == "f32" else TOL_BF16)
    eo = err(o.double().cpu().numpy(), ro, dtype)
    if dtype == "bf16":  # the raw figure beside the net one (the bound is on the net one)
        print("o error: net of half a bf16 ulp %.4f, raw max|o-ref|/RMS %.4f"
              % (eo, err(o.double().cpu().numpy(), ro, dtype, rounded=False)))
    assert np.isfinite(eo) and eo <= tol, ("o", eo)
    if want_S:
        es = err(S.double().cpu().numpy(), rS, dtype, rounded=False)
        assert np.isfinite(es) and es <= tol, ("S_final", es)
    return o, S


@pytest.mark.parametrize("name", list(I.WORKLOADS))
def test_workload_full_size(gdn, name):
    """Every named workload at its full size, all outputs compared."""
    w = I.WORKLOADS[name]
    x = I.generate(w, seed=0)
    run_and_check(gdn, x, w.C, w.dtype)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("T,C", [(1, 16), (15, 16), (64, 16), (100, 32), (200, 64), (63, 64), (65, 64)])
def test_ragged_lengths(gdn, dtype, T, C):
    x = I.custom(2, 3, T, 32, 48, C, dtype=dtype, seed=T + C, s0="normal_0.02")
    run_and_check(gdn, x, C, dtype)


def tc_path_expected(dk, dv, C, dtype):
    """The tcgen05 kernel takes bf16, C = 64, d_k <= 128 and d_k, d_v
    multiples of 8 (zero-padded to 128-wide tiles); the rest is fp32 CUDA-core."""
    return dtype == "bf16" and C == 64 and dk % 8 == 0 and dk <= 128 and dv % 8 == 0


@pytest.mark.parametrize("dk,dv", [(16, 16), (64, 64), (128, 128), (64, 128), (128, 64),
                                   (128, 256), (96, 192), (40, 24), (8, 8), (128, 200),
                                   (72, 136), (100, 36), (20, 20)])
def test_head_dims(gdn, dk, dv):
    x = I.custom(1, 2, 300, dk, dv, 64, dtype="bf16", seed=dk * 1000 + dv, s0="normal_0.02")
    run_and_check(gdn, x, 64, "bf16")
    assert gdn.gdn_last_launch_count()[1] == (1 if tc_path_expected(dk, dv, 64, "bf16") else 0)


def test_hybrid_head_shape_extended_beta_varlen(gdn):
    """d_k = 96, d_v = 192 (two d_v tiles, the second half padding), beta in
    (0, 2), packed ragged sequences with an initial state: tensor-core path."""
    lens = [1, 64, 100, 255, 0, 129]
    x = I.custom(1, 6, 0, 96, 192, 64, dtype="bf16", seed=21, lengths=lens,
                 s0="normal_0.02", beta="uniform_0_2")
    assert float(x["beta"].max()) > 1.5
    run_and_check(gdn, x, 64, "bf16")
    assert gdn.gdn_last_launch_count() == (1, 1)


def test_varlen_edge_lengths(gdn):
    """Packed sequences with empty, length-1, sub-chunk and ragged lengths."""
    lens = [0, 1, 63, 64, 65, 130, 0, 7]
    x = I.custom(1, 4, 0, 128, 128, 64, dtype="bf16", seed=5, lengths=lens, s0="normal_0.02")
    run_and_check(gdn, x, 64, "bf16")


def test_extended_beta_range(gdn):
    """beta in (0, 2): the extended DeltaNet range (negative eigenvalues)."""
    x = I.custom(2, 2, 256, 64, 64, 64, dtype="bf16", seed=3)
    x["beta"] = x["beta"] * 2.0
    run_and_check(gdn, x, 64, "bf16")


def test_s0_none_equals_zeros_and_no_final_state(gdn):
    x = I.custom(1, 2, 130, 64, 64, 64, dtype="bf16", seed=4)
    d = _dev(x)
    o1, S1 = gdn.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], C=64)
    z = torch.zeros_like(S1)
    o2, S2 = gdn.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], S0=z, C=64)
    o3, S3 = gdn.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], C=64,
                               want_final_state=False)
    assert S3 is None
    assert torch.equal(o1, o2) and torch.equal(S1, S2) and torch.equal(o1, o3)


def test_in_place_state_and_resume(gdn):
    """S_final == S0 in place, and (T1) then (T2, S0 = S_final) equals (T1 + T2)."""
    x = I.custom(2, 2, 256, 64, 64, 64, dtype="bf16", seed=6, s0="normal_0.02")
    d = _dev(x)
    o_full, S_full = gdn.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"],
                                       S0=d["S0"], C=64)
    S = d["S0"].clone()
    cut = 128  # a chunk boundary, so the chunk grid is the same in both runs
    sl1 = lambda t: t[:, :cut].contiguous()
    sl2 = lambda t: t[:, cut:].contiguous()
    oa, _ = gdn.gdn_chunk_fwd(sl1(d["q"]), sl1(d["k"]), sl1(d["v"]), sl1(d["log_alpha"]),
                              sl1(d["beta"]), S0=S, S_final=S, C=64)
    ob, _ = gdn.gdn_chunk_fwd(sl2(d["q"]), sl2(d["k"]), sl2(d["v"]), sl2(d["log_alpha"]),
                              sl2(d["beta"]), S0=S, S_final=S, C=64)
    torch.cuda.synchronize()
    assert torch.equal(torch.cat([oa, ob], 1), o_full)
    assert torch.equal(S, S_full)


def test_deterministic(gdn):
    x = I.custom(2, 4, 500, 128, 128, 64, dtype="bf16", seed=7)
    d = _dev(x)
    a = gdn.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], C=64)
    b = gdn.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], C=64)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_guard_bands_untouched(gdn):
    """Writes stay inside o and S_final: canaries around both are unchanged."""
    x = I.custom(1, 3, 200, 64, 96, 64, dtype="bf16", seed=8)
    d = _dev(x)
    B, T, H, _ = d["q"].shape
    dv, dk = 96, 64
    pad = 4096
    ob = torch.full((2 * pad + B * T * H * dv,), float("nan"), dtype=torch.bfloat16, device="cuda")
    sb = torch.full((2 * pad + H * dv * dk,), -7.0, dtype=torch.float32, device="cuda")
    o = ob[pad:pad + B * T * H * dv].view(B, T, H, dv)
    S = sb[pad:pad + H * dv * dk].view(1, H, dv, dk)
    gdn.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], o=o, S_final=S, C=64)
    torch.cuda.synchronize()
    assert torch.isnan(ob[:pad].float()).all() and torch.isnan(ob[-pad:].float()).all()
    assert (sb[:pad] == -7.0).all() and (sb[-pad:] == -7.0).all()
    assert torch.isfinite(o.float()).all()


def test_bad_cu_seqlens_sets_device_status(gdn):
    """Malformed spans are skipped on the device and reported, not faulted."""
    x = I.custom(1, 2, 0, 32, 32, 16, dtype="bf16", seed=9, lengths=[10, 10])
    d = _dev(x)
    bad = torch.tensor([0, 15, 5], dtype=torch.int32, device="cuda")   # decreasing span
    gdn.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], C=16, cu_seqlens=bad)
    assert gdn.gdn_get_device_status() & 0x1
    past = torch.tensor([0, 10, 25], dtype=torch.int32, device="cuda")  # runs past T = 20
    gdn.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], C=16, cu_seqlens=past)
    assert gdn.gdn_get_device_status() & 0x1
    assert gdn.gdn_get_device_status() == 0  # cleared by the read


def test_sampled_outputs_at_full_size_train_shape(gdn):
    """The benchmark's launch (B4 H16 T4096 d128, C64, bf16): outputs of a few
    (sequence, head) units recomputed one by one by the oracle."""
    w = I.WORKLOADS["train_bf16"]
    x = I.generate(w, seed=1)
    d = _dev(x)
    o, S = gdn.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], C=64)
    o = o.double().cpu().numpy()
    S = S.double().cpu().numpy()
    for b, h in ((0, 0), (3, 15), (1, 7)):
        sl = (slice(b, b + 1), slice(None), slice(h, h + 1))
        ro, rS = gdn_recurrence_f64(x["q"][sl], x["k"][sl], x["v"][sl],
                                    x["log_alpha"][sl], x["beta"][sl])
        assert err(o[sl], ro, "bf16") <= TOL_BF16
        assert err(S[b:b + 1, h:h + 1], rS, "bf16", rounded=False) <= TOL_BF16


@pytest.mark.parametrize("dtype,dk,dv,C", [("bf16", 128, 128, 64), ("f32", 32, 48, 16),
                                           ("bf16", 96, 192, 64), ("bf16", 40, 36, 32)])
def test_write_strength_eta(gdn, dtype, dk, dv, C):
    """S_t = alpha S (I - beta k k^T) + eta v k^T with eta independent of beta,
    on both kernels, against the oracle's eta form."""
    x = I.custom(2, 3, 200, dk, dv, C, dtype=dtype, seed=31 + dk + C, s0="normal_0.02",
                 eta="uniform")
    d = _dev(x)
    o, S = gdn.gdn_chunk_fwd_eta(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], d["eta"],
                                 S0=d["S0"], C=C)
    assert gdn.gdn_get_device_status() == 0
    assert gdn.gdn_last_launch_count()[1] == (1 if tc_path_expected(dk, dv, C, dtype) else 0)
    ro, rS = gdn_recurrence_f64(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"],
                                S0=x["S0"], eta=x["eta"])
    tol = TOL_F32 if dtype == "f32" else TOL_BF16
    assert err(o.double().cpu().numpy(), ro, dtype) <= tol
    assert err(S.double().cpu().numpy(), rS, dtype, rounded=False) <= tol


@pytest.mark.parametrize("dtype,C", [("bf16", 64), ("f32", 32)])
def test_eta_equal_beta_is_gdn_chunk_fwd(gdn, dtype, C):
    x = I.custom(1, 4, 150, 64, 64, C, dtype=dtype, seed=33, s0="normal_0.02")
    d = _dev(x)
    a = gdn.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], S0=d["S0"], C=C)
    b = gdn.gdn_chunk_fwd_eta(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"],
                              d["beta"].clone(), S0=d["S0"], C=C)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_eta_linear_attention_limit(gdn):
    """alpha = 1, beta = 0, eta = 1: nothing is erased, every value is
    written, and the output is causal linear attention on top of S0 (the
    oracle is pinned to that closed form on the CPU)."""
    x = I.custom(2, 2, 130, 128, 128, 64, dtype="bf16", seed=34, s0="normal_0.02", alpha="one")
    x["beta"] = torch.zeros_like(x["beta"])
    eta = torch.ones_like(x["beta"])
    d = _dev(x)
    o, S = gdn.gdn_chunk_fwd_eta(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], eta.cuda(),
                                 S0=d["S0"], C=64)
    ro, rS = gdn_recurrence_f64(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"],
                                S0=x["S0"], eta=eta)
    assert err(o.double().cpu().numpy(), ro, "bf16") <= TOL_BF16
    assert err(S.double().cpu().numpy(), rS, "bf16", rounded=False) <= TOL_BF16


@pytest.mark.parametrize("dk,dv", [(128, 128), (40, 24)])
def test_final_state_unaligned_destination(gdn, dk, dv):
    """S_final only 4-byte aligned (a view one float into a buffer): the
    kernel's element-wise store path writes exactly what the 16-byte row
    path writes into an aligned buffer."""
    x = I.custom(1, 2, 200, dk, dv, 64, dtype="bf16", seed=30 + dk, s0="normal_0.02")
    d = _dev(x)
    _, S_al = gdn.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], S0=d["S0"], C=64)
    n = 2 * dv * dk
    buf = torch.full((n + 2,), -7.0, dtype=torch.float32, device="cuda")
    S_un = buf[1:1 + n].view(1, 2, dv, dk)
    assert S_un.data_ptr() % 16 != 0
    gdn.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], S0=d["S0"], S_final=S_un, C=64)
    assert gdn.gdn_get_device_status() == 0
    assert gdn.gdn_last_launch_count()[1] == 1
    assert torch.equal(S_un, S_al)
    assert buf[0].item() == -7.0 and buf[-1].item() == -7.0


@pytest.mark.parametrize("la", [-3.0, -1.5, -1.2])
def test_strong_in_chunk_decay(gdn, la):
    """Constant log alpha: a chunk decays by e^{63 |la|} from its first token to
    its last.  Past e^80 (la = -3.0, -1.5) the producer exponentiates every A
    and P entry on its own instead of splitting the factor around the middle
    of the chunk; la = -1.2 stays just inside the split form."""
    x = I.custom(1, 2, 300, 128, 128, 64, dtype="bf16", seed=41, s0="normal_0.02")
    x["log_alpha"] = torch.full_like(x["log_alpha"], la)
    run_and_check(gdn, x, 64, "bf16")
    assert gdn.gdn_last_launch_count()[1] == 1


def test_mixed_decay_per_token(gdn):
    """log alpha uniform in [-4, 0] per token: chunks on both sides of the
    split threshold in one call, ragged tail included."""
    x = I.custom(1, 3, 450, 128, 128, 64, dtype="bf16", seed=42, s0="normal_0.02")
    g = torch.Generator().manual_seed(42)
    x["log_alpha"] = -4.0 * torch.rand(x["log_alpha"].shape, generator=g, dtype=torch.float32)
    run_and_check(gdn, x, 64, "bf16")


def test_identical_keys_extended_beta(gdn):
    """Every token of a head has the same unit key and beta in (0, 2): A has
    all its sub-diagonal entries from one k.k, the most correlated input the
    UT transform meets; the state keeps one direction of k."""
    x = I.custom(1, 2, 300, 128, 128, 64, dtype="bf16", seed=43, s0="normal_0.02", beta="uniform_0_2")
    x["k"] = x["k"][:, :1].expand_as(x["k"]).contiguous()
    run_and_check(gdn, x, 64, "bf16")
    assert gdn.gdn_last_launch_count()[1] == 1


def test_zero_keys_pure_decay(gdn):
    """k = 0: nothing is erased or written (A = 0, T = I, W = 0), the state
    only decays and o_t = S_t q_t."""
    x = I.custom(1, 2, 200, 128, 128, 64, dtype="bf16", seed=44, s0="normal_0.02")
    x["k"] = torch.zeros_like(x["k"])
    run_and_check(gdn, x, 64, "bf16")


def repack(x, order):
    """The packed inputs of ``x`` with its sequences in ``order``."""
    cu = x["cu_seqlens"].tolist()
    pieces = lambda t: torch.cat([t[:, cu[i]:cu[i + 1]] for i in order], dim=1).contiguous()
    y = {kk: pieces(x[kk]) for kk in ("q", "k", "v", "log_alpha", "beta")}
    lens = [cu[i + 1] - cu[i] for i in order]
    y["cu_seqlens"] = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32)
    y["S0"] = x["S0"][list(order)].contiguous()
    return y


@pytest.mark.parametrize("how", ["reversed", "shuffled", "longest_last"])
def test_varlen_pack_order_is_bit_identical(gdn, how):
    """The full-size varlen workload packed in another sequence order: every
    sequence's outputs and final state are bit-identical to the given order's
    (the units are independent whatever slot or SM they land on; the kernel
    starts them longest first either way)."""
    w = I.WORKLOADS["varlen_bf16"]
    x = I.generate(w, seed=0)
    N = len(x["lengths"])
    order = {"reversed": list(range(N))[::-1],
             "shuffled": list(np.random.default_rng(5).permutation(N)),
             "longest_last": list(np.argsort(x["lengths"], kind="stable"))}[how]
    y = repack(x, order)
    dx, dy = _dev(x), _dev(y)
    ox, Sx = gdn.gdn_chunk_fwd(dx["q"], dx["k"], dx["v"], dx["log_alpha"], dx["beta"], S0=dx["S0"],
                               cu_seqlens=dx["cu_seqlens"])
    oy, Sy = gdn.gdn_chunk_fwd(dy["q"], dy["k"], dy["v"], dy["log_alpha"], dy["beta"], S0=dy["S0"],
                               cu_seqlens=dy["cu_seqlens"])
    assert gdn.gdn_get_device_status() == 0
    assert gdn.gdn_last_launch_count()[1] == 1
    cx, cy = x["cu_seqlens"].tolist(), y["cu_seqlens"].tolist()
    for j, i in enumerate(order):
        assert torch.equal(ox[:, cx[i]:cx[i + 1]], oy[:, cy[j]:cy[j + 1]]), (how, i)
        assert torch.equal(Sx[i], Sy[j]), (how, i)


@pytest.mark.parametrize("N", [256, 300])
def test_many_packed_sequences(gdn, N):
    """Many short packed sequences (ragged, some empty, some past a chunk):
    up to 256 are ranked longest first inside the kernel, more run in the
    given order; both against the oracle."""
    lens = [int(x) for x in np.random.default_rng(N).integers(0, 90, size=N)]
    x = I.custom(1, 1, 0, 64, 64, 64, dtype="bf16", seed=N, lengths=lens, s0="normal_0.02")
    run_and_check(gdn, x, 64, "bf16")
    assert gdn.gdn_last_launch_count()[1] == 1
