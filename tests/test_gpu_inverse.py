"""GPU parity of the batched UT inverse (gdn_ut_inverse, both methods,
through the C ABI) against the fp64 forward substitution of the chunk
reference.

Tolerances, relative to the largest |T| of each matrix:
  method 0 (fp32 forward substitution): 1e-5.  Each entry is a sum of at
    most 63 products formed in fp32 (unit roundoff 6e-8); 1e-5 leaves a wide
    margin for the growth of |T| entries.
  method 1 (doubling product, fp16 operands, fp32 accumulation): 5e-3.  Each
    of the nine products rounds its operands to fp16 (unit roundoff 4.9e-4)
    and only the correction term Q X_k carries that rounding; with powers of
    A that shrink (|A| entries ~ 0.04) the total stays near 10 x 4.9e-4.
"""
import numpy as np
import pytest
import torch

from gated_delta_rule_09_gb300 import inputs as I
from oracle.chunk_reference import forward_substitution

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gdn():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import gated_delta_rule_09_gb300 as g
    return g


def rel_err(T, A):
    T = T.double().cpu().numpy()
    A = A.double().numpy()
    worst = 0.0
    for n in range(A.shape[0]):
        ref = forward_substitution(-A[n])
        worst = max(worst, np.abs(T[n] - ref).max() / np.abs(ref).max())
    return worst


@pytest.mark.parametrize("method,tol", [(0, 1e-5), (1, 5e-3)])
@pytest.mark.parametrize("C", [16, 32, 64])
def test_ut_inverse(gdn, method, tol, C):
    A = I.ut_matrices(257, C, 0.04, seed=C + method)
    T = gdn.gdn_ut_inverse(A.cuda(), method=method)
    assert gdn.gdn_get_device_status() == 0
    assert gdn.gdn_last_launch_count() == (1, 4 + method)
    e = rel_err(T, A)
    assert np.isfinite(e) and e <= tol, e
    Tc = T.cpu()
    assert torch.all(torch.diagonal(Tc, dim1=1, dim2=2) == 1)
    assert torch.all(torch.triu(Tc, 1) == 0)


def test_ut_inverse_larger_entries(gdn):
    """|A| entries ~ 0.2: forward substitution keeps fp32 accuracy; the
    doubling product's error is reported, not bounded tightly."""
    A = I.ut_matrices(64, 64, 0.2, seed=3)
    e0 = rel_err(gdn.gdn_ut_inverse(A.cuda(), method=0), A)
    e1 = rel_err(gdn.gdn_ut_inverse(A.cuda(), method=1), A)
    assert e0 <= 1e-5
    assert np.isfinite(e1) and e1 <= 5e-2, e1


def test_ut_inverse_argument_checks(gdn):
    from gated_delta_rule_09_gb300 import _lib
    A = torch.zeros(2, 48, 48, device="cuda")
    with pytest.raises(_lib.GdnError) as e:
        gdn.gdn_ut_inverse(A)
    assert e.value.status == _lib.GDN_ERR_UNSUPPORTED
    assert gdn.gdn_ut_inverse(torch.zeros(0, 64, 64, device="cuda")).shape[0] == 0
