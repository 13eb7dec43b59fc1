"""Every plausible mistake planted into a copy of the oracle's recurrence must
fail at least one pin (CPU only).  This shows the pins can tell a correct
recurrence from a near miss; the mistakes are planted here, never in the
CUDA path."""
import numpy as np
import pytest

import pins


def make_recurrence(mistake=None):
    def impl(q, k, v, log_alpha, beta, S0=None, eta=None, cu_seqlens=None):
        q, k, v = (np.asarray(x, np.float64) for x in (q, k, v))
        B, T, H, dk = q.shape
        dv = v.shape[-1]
        if cu_seqlens is None:
            spans = [(b, 0, T) for b in range(B)]
        else:
            cu = list(cu_seqlens)
            spans = [(0, cu[n], cu[n + 1]) for n in range(len(cu) - 1)]
        o = np.zeros((B, T, H, dv))
        Sf = np.zeros((len(spans), H, dv, dk))
        for n, (b, s, e) in enumerate(spans):
            for h in range(H):
                S = np.zeros((dv, dk)) if S0 is None else np.array(S0[n, h], np.float64)
                if mistake == "ignore_S0":
                    S = np.zeros((dv, dk))
                for t in range(s, e):
                    kt, qt, vt = k[b, t, h], q[b, t, h], v[b, t, h]
                    a = np.exp(log_alpha[b, t, h])
                    bt = beta[b, t, h]
                    et = bt if eta is None else eta[b, t, h]
                    if mistake == "eta_ignored":
                        et = bt
                    if mistake == "log_alpha_used_as_alpha":
                        a = log_alpha[b, t, h]
                    if mistake == "no_gate":
                        a = 1.0
                    prev = S
                    r = S @ kt
                    if mistake == "erase_from_undecayed_state":
                        S = a * S + np.outer(et * vt - bt * r, kt)
                    elif mistake == "gate_on_write":
                        S = a * (S + np.outer(et * vt - bt * r, kt))
                    elif mistake == "erase_sign_flipped":
                        S = a * S + np.outer(et * vt + a * bt * r, kt)
                    elif mistake == "beta_squared":
                        S = a * S + np.outer(et * vt - a * bt * bt * r, kt)
                    elif mistake == "write_with_query":
                        S = a * S + np.outer(et * vt - a * bt * r, qt)
                    else:
                        S = a * S + np.outer(et * vt - a * bt * r, kt)
                    if mistake == "output_from_previous_state":
                        o[b, t, h] = prev @ qt
                    elif mistake == "readout_transposed":
                        m = min(dk, dv)
                        qq = np.zeros(dv)
                        qq[:m] = qt[:m]
                        res = S.T @ qq
                        o[b, t, h] = 0.0
                        o[b, t, h, :m] = res[:m]
                    else:
                        o[b, t, h] = S @ qt
                Sf[n, h] = S
        return o, Sf
    return impl


MISTAKES = ["erase_from_undecayed_state", "gate_on_write", "erase_sign_flipped",
            "beta_squared", "write_with_query", "output_from_previous_state",
            "readout_transposed", "ignore_S0", "eta_ignored",
            "log_alpha_used_as_alpha", "no_gate"]


def test_python_copy_passes_all_pins():
    impl = make_recurrence(None)
    for check in pins.ALL_CHECKS:
        check(impl)


@pytest.mark.parametrize("mistake", MISTAKES)
def test_planted_mistake_is_caught(mistake):
    impl = make_recurrence(mistake)
    failed = []
    for check in pins.ALL_CHECKS:
        try:
            check(impl)
        except AssertionError:
            failed.append(check.__name__)
    assert failed, "planted mistake %r passed every pin" % mistake
