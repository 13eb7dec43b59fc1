"""The Python binding refuses wrongly shaped arguments before the library is
loaded or anything is launched (CPU only): every tensor the kernels read or
write is checked against the sizes the C call derives from q and v, so a
mis-shaped gate, state or output can never be read or written past its end."""
import pytest
import torch

import gated_delta_rule_09_gb300 as gdn


@pytest.fixture
def host_only(monkeypatch):
    """Device checks off (these are CPU tensors) and no library: any call that
    got past the argument checks would raise RuntimeError instead."""
    monkeypatch.setattr(gdn, "_need_cuda", lambda *a, **k: None)

    def no_load():
        raise RuntimeError("reached the library")

    monkeypatch.setattr(gdn._lib, "load", no_load)


def args(B=2, T=8, H=3, dk=16, dv=24):
    z = lambda *s: torch.zeros(*s, dtype=torch.float32)
    return dict(q=torch.zeros(B, T, H, dk, dtype=torch.bfloat16), k=torch.zeros(B, T, H, dk, dtype=torch.bfloat16),
                v=torch.zeros(B, T, H, dv, dtype=torch.bfloat16), log_alpha=z(B, T, H), beta=z(B, T, H)), (B, T, H, dk, dv)


FORWARD = [gdn.gdn_chunk_fwd, gdn.gdn_chunk_fwd_scan, gdn.gdn_chunk_fwd_scan_noalloc]


@pytest.mark.parametrize("fn", FORWARD)
@pytest.mark.parametrize("bad", ["log_alpha", "beta", "S0", "o", "S_final"])
def test_forward_entry_points_reject_bad_shapes(host_only, fn, bad):
    a, (B, T, H, dk, dv) = args()
    wrong = {"log_alpha": torch.zeros(B, T, H + 1), "beta": torch.zeros(B, T - 1, H),
             "S0": torch.zeros(B, H, dk, dv + 1), "o": torch.zeros(B, T, H, dv - 8, dtype=torch.bfloat16),
             "S_final": torch.zeros(B, H, dv, dk - 8)}
    a[bad] = wrong[bad]
    with pytest.raises(ValueError):
        fn(**a)


def test_forward_entry_point_accepts_right_shapes_until_the_library(host_only):
    a, (B, T, H, dk, dv) = args()
    a.update(S0=torch.zeros(B, H, dv, dk), o=torch.zeros(B, T, H, dv, dtype=torch.bfloat16),
             S_final=torch.zeros(B, H, dv, dk))
    for fn in FORWARD:
        with pytest.raises(RuntimeError, match="reached the library"):
            fn(**a)


def test_eta_shape_and_packed_offsets(host_only):
    a, (B, T, H, dk, dv) = args()
    with pytest.raises(ValueError):
        gdn.gdn_chunk_fwd_eta(eta=torch.zeros(B, T, H + 1), **a)
    p, _ = args(B=1)
    with pytest.raises(ValueError):  # packed inputs need N + 1 >= 2 offsets
        gdn.gdn_chunk_fwd(cu_seqlens=torch.zeros(1, dtype=torch.int32), **p)
    with pytest.raises(ValueError):  # the state is per packed sequence
        gdn.gdn_chunk_fwd(cu_seqlens=torch.tensor([0, 3, 8], dtype=torch.int32),
                          S0=torch.zeros(1, H, dv, dk), **p)
    with pytest.raises(ValueError):  # packed means B == 1
        gdn.gdn_chunk_fwd(cu_seqlens=torch.tensor([0, 8], dtype=torch.int32), **a)


@pytest.mark.parametrize("bad", ["o", "S_out", "S_in"])
def test_decode_rejects_bad_shapes(host_only, bad):
    N, T, H, dk, dv = 4, 2, 3, 16, 24
    a = dict(q=torch.zeros(N, T, H, dk, dtype=torch.bfloat16), k=torch.zeros(N, T, H, dk, dtype=torch.bfloat16),
             v=torch.zeros(N, T, H, dv, dtype=torch.bfloat16), log_alpha=torch.zeros(N, T, H),
             beta=torch.zeros(N, T, H))
    wrong = {"o": torch.zeros(N, T, H, dv + 8, dtype=torch.bfloat16), "S_out": torch.zeros(N, H, dv, dk + 8),
             "S_in": torch.zeros(N, H, dk, dv)}
    a[bad] = wrong[bad]
    with pytest.raises(ValueError):
        gdn.gdn_decode_step(**a)


@pytest.mark.parametrize("fn", [gdn.gdn_chunk_fwd_scan, gdn.gdn_chunk_fwd_scan_noalloc])
def test_packed_scan_argument_checks(host_only, fn):
    """The scan entry points take packed offsets with the rules of the plain
    pass: B == 1, states per packed sequence."""
    a, (B, T, H, dk, dv) = args(B=1)
    cu = torch.tensor([0, 3, 8], dtype=torch.int32)
    with pytest.raises(ValueError):  # S0 must be [N, H, d_v, d_k] with N = 2
        fn(cu_seqlens=cu, S0=torch.zeros(1, H, dv, dk), **a)
    b, _ = args(B=2)
    with pytest.raises(ValueError):  # packed means B == 1
        fn(cu_seqlens=torch.tensor([0, 8], dtype=torch.int32), **b)
    with pytest.raises(RuntimeError, match="reached the library"):
        fn(cu_seqlens=cu, S0=torch.zeros(2, H, dv, dk), **a)
