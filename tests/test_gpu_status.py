"""Device status bits of the tensor-core path (gdn_get_device_status): the
fp16 operand range check.  bf16 inputs and the fp32 state are converted to
fp16 for the MMAs; a value that does not fit must raise GDN_DEV_F16_RANGE
and nothing else, and ordinary inputs must leave the status clean."""
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


def run(gdn, d, S0=None):
    o, S = gdn.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], S0=S0)
    assert gdn.gdn_last_launch_count()[1] == 1  # the tensor-core kernel ran
    return gdn.gdn_get_device_status()


def test_status_clean_for_ordinary_inputs(gdn):
    d = dev(I.custom(1, 2, 300, 128, 128, 64, dtype="bf16", seed=70, s0="normal_0.02"))
    assert run(gdn, d, S0=d["S0"]) == 0


def test_f16_range_raised_by_large_values(gdn):
    """v scaled by 1e6: representable in bf16, far past the fp16 maximum.  The
    C status read reports it as GDN_ERR_RANGE with the bit in its flags."""
    import ctypes
    from gated_delta_rule_09_gb300 import _lib
    d = dev(I.custom(1, 2, 300, 128, 128, 64, dtype="bf16", seed=71))
    d["v"] = (d["v"].float() * 1e6).to(torch.bfloat16)
    assert run(gdn, d) == _lib.GDN_DEV_F16_RANGE
    gdn.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"])
    flags = ctypes.c_uint(0)
    st = _lib.load().gdn_get_device_status(ctypes.c_void_p(torch.cuda.current_stream().cuda_stream),
                                           ctypes.byref(flags))
    assert st == _lib.GDN_ERR_RANGE and flags.value == _lib.GDN_DEV_F16_RANGE


def test_f16_range_raised_by_large_initial_state(gdn):
    """An initial state of 1e5 leaves the fp16 range when the first chunk
    converts it for the MMAs; q, k, v stay ordinary."""
    from gated_delta_rule_09_gb300 import _lib
    d = dev(I.custom(1, 2, 300, 128, 128, 64, dtype="bf16", seed=72))
    S0 = torch.full((1, 2, 128, 128), 1e5, dtype=torch.float32, device="cuda")
    assert run(gdn, d, S0=S0) == _lib.GDN_DEV_F16_RANGE
