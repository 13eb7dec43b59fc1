"""The no-allocation scan entry point (gdn_chunk_fwd_scan_noalloc) against
the workspace entry point on the same inputs, two calls in a row (the second
reuses the fixed scratch the first wrote).  Collected last: it must pass on
its own and after every other test in the same process."""
import pytest
import torch

from gated_delta_rule_09_gb300 import inputs as I
from parity_util import dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gdn():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import gated_delta_rule_09_gb300 as g
    return g


def _run(gdn, fn, d, segments, **kw):
    o = torch.full(d["v"].shape, float("nan"), dtype=d["v"].dtype, device="cuda")
    B, T, H, dk = d["q"].shape
    S = torch.full((B, H, d["v"].shape[-1], dk), float("nan"), device="cuda")
    fn(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], S0=d["S0"], o=o, S_final=S,
       segments=segments, **kw)
    assert gdn.gdn_get_device_status() == 0
    return o, S


@pytest.mark.parametrize("seed,segments", [(61, 5), (62, 0)])
def test_noalloc_matches_workspace_entry_twice(gdn, seed, segments):
    xs = [I.custom(2, 2, 900, 128, 128, 64, dtype="bf16", seed=seed + i, s0="normal_0.02")
          for i in range(2)]
    for x in xs:  # two calls in a row on the fixed scratch
        d = dev(x)
        a = _run(gdn, gdn.gdn_chunk_fwd_scan_noalloc, d, segments)
        assert gdn.gdn_last_launch_count()[1] == 3
        b = _run(gdn, gdn.gdn_chunk_fwd_scan, d, segments)
        assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
        assert torch.isfinite(a[0].float()).all() and torch.isfinite(a[1]).all()


def test_noalloc_rejects_oversize(gdn):
    """A problem whose scratch exceeds the fixed 32 MiB is refused before any
    pointer is used (sizes passed straight through the C ABI)."""
    import ctypes
    from gated_delta_rule_09_gb300 import _lib
    B, H, T = 1, 64, 65536
    need = gdn.gdn_chunk_fwd_scan_workspace_size(B, H, T, 128, 128, 64, 64)
    assert need > (32 << 20)
    buf = torch.zeros(16, dtype=torch.float32, device="cuda")
    p = ctypes.c_void_p(buf.data_ptr())
    lib = _lib.load()
    st = lib.gdn_chunk_fwd_scan_noalloc(p, p, p, p, p, None, p, p, B, H, T, 128, 128, 64, None,
                                        _lib.GDN_BF16, 64, None)
    assert st == _lib.GDN_ERR_UNSUPPORTED
    assert b"fixed scratch" in lib.gdn_get_last_error()
