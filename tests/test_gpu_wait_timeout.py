"""The bounded-wait abort path of the tensor-core chunk kernel, run on purpose.

libgdn_waittest.so is the library with that kernel compiled under
GDN_WAIT_TEST: every wait gives up after 5 ms, and in the unit (sequence 0,
head 0, first d_v tile) the producer withholds one software arrival (the
"shipped" signal of chunk 1, an ordering signal between its pipelines), so the
next pipeline's wait runs out.  Withholding it leaves nothing asynchronous in
flight by itself.  The kernel must then raise GDN_DEV_WAIT_TIMEOUT (the C
status read returns GDN_ERR_TIMEOUT), wind down in milliseconds (the stalled
CTA gives up, its peer gives up on its own next wait, and both drain the
loads, shipments and MMAs they had issued before freeing their tensor
memory), leave every other unit's results exact to the
usual bound, and leave the device usable: the normal library's next call on
the same inputs passes parity with a clean status.
"""
import ctypes
import os
import time

import pytest
import torch

from gated_delta_rule_09_gb300 import inputs as I
from oracle import gdn_recurrence_f64
from parity_util import TOL_BF16, dev, err

pytestmark = pytest.mark.gpu

B, H, T = 2, 2, 640  # ten chunks per unit; unit (0, 0) is the one that stalls


@pytest.fixture(scope="module")
def gdn():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import gated_delta_rule_09_gb300 as g
    return g


def waittest_lib():
    from gated_delta_rule_09_gb300 import _lib
    path = os.path.join(os.path.dirname(_lib.LIB_PATH), "libgdn_waittest.so")
    assert os.path.exists(path), "libgdn_waittest.so is built by build(); it is missing"
    lib = ctypes.CDLL(path)
    for name, (res, args) in _lib.SIGNATURES.items():
        getattr(lib, name).restype = res
        getattr(lib, name).argtypes = args
    return lib


def check_units(o, S, ro, rS, skip):
    """Every (sequence, head) unit except `skip` within the bf16 bound."""
    for n in range(B):
        for h in range(H):
            if (n, h) == skip:
                continue
            eo = err(o[n, :, h], ro[n, :, h], "bf16")
            es = err(S[n, h], rS[n, h], "bf16", rounded=False)
            assert eo <= TOL_BF16 and es <= TOL_BF16, ((n, h), eo, es)


def test_withheld_arrival_times_out_and_device_recovers(gdn, monkeypatch):
    from gated_delta_rule_09_gb300 import _lib
    x = I.custom(B, H, T, 128, 128, 64, dtype="bf16", seed=90, s0="normal_0.02")
    d = dev(x)
    ro, rS = gdn_recurrence_f64(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], S0=x["S0"])
    assert gdn.gdn_get_device_status() == 0

    lib = waittest_lib()
    with monkeypatch.context() as m:  # the binding marshals into the test library
        m.setattr(_lib, "load", lambda *a, **k: lib)
        # warm-up (loads the test library's module): two chunks per unit, so
        # the withheld arrival of chunk 1 is never waited for and the call is clean
        w = dev(I.custom(1, 1, 128, 128, 128, 64, dtype="bf16", seed=92))
        gdn.gdn_chunk_fwd(w["q"], w["k"], w["v"], w["log_alpha"], w["beta"], C=64)
        assert gdn.gdn_get_device_status() == 0
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        o, S = gdn.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], S0=d["S0"], C=64)
        assert gdn.gdn_last_launch_count()[1] == 1  # the tensor-core kernel ran
        flags = ctypes.c_uint(0)
        handle = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
        st = lib.gdn_get_device_status(handle, ctypes.byref(flags))
        elapsed = time.perf_counter() - t0
    assert st == _lib.GDN_ERR_TIMEOUT, st
    assert flags.value & _lib.GDN_DEV_WAIT_TIMEOUT, flags.value
    assert elapsed < 1.0, elapsed  # 5 ms waits: the stalled unit winds down at once
    # the other units never waited on the stalled one
    check_units(o.double().cpu().numpy(), S.double().cpu().numpy(), ro, rS, skip=(0, 0))

    # the device is intact: the normal library, same inputs, every unit
    o2, S2 = gdn.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], S0=d["S0"], C=64)
    assert gdn.gdn_get_device_status() == 0
    check_units(o2.double().cpu().numpy(), S2.double().cpu().numpy(), ro, rS, skip=None)


def test_timeout_bit_reads_as_status_in_python(gdn, monkeypatch):
    """Through the Python binding the timeout is a returned bit, and the read
    clears it."""
    from gated_delta_rule_09_gb300 import _lib
    x = I.custom(1, 1, 256, 128, 128, 64, dtype="bf16", seed=91)
    d = dev(x)
    lib = waittest_lib()
    with monkeypatch.context() as m:
        m.setattr(_lib, "load", lambda *a, **k: lib)
        gdn.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["log_alpha"], d["beta"], C=64)
        assert gdn.gdn_get_device_status() & _lib.GDN_DEV_WAIT_TIMEOUT
        assert gdn.gdn_get_device_status() == 0
