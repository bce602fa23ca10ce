"""Plant plausible mistakes in copies of the oracle (on the CPU) and check that the pins catch
every one of them.  A mutant that passes every pin would mean the pins leave that part of the
oracle unchecked."""
import inspect
import types

import pytest

from oracle import attention as orc
from tests.pins import ALL_CHECKS

MUTANTS = {
    "causal_off_by_one": ("ok &= j[None, :] <= diag", "ok &= j[None, :] < diag"),
    "causal_start_aligned": ("diag = i[:, None] + (kv_len - q_len)", "diag = i[:, None] + 0"),
    "window_w_plus_one": ("diag - window + 1", "diag - window"),
    "gqa_modulo_head_map": ("k[k0:k1, h // g],\n                                  v[k0:k1, h // g]",
                            "k[k0:k1, h % (hq // g)],\n                                  v[k0:k1, h % (hq // g)]"),
    "bias_scaled": ("s = s + bias_rows", "s = s + scale * bias_rows"),
    "lse_without_max": ("lse[live] = m[live] + np.log(l)", "lse[live] = np.log(l)"),
    "softmax_not_normalised": ("P[live] = e / l[:, None]", "P[live] = e"),
    "ds_sign": ("dS = P * (dP - Di[:, None])", "dS = P * (dP + Di[:, None])"),
    "dk_missing_scale": ("dk += scale * (dS[:, cols].T @ q[r0:r1])", "dk += (dS[:, cols].T @ q[r0:r1])"),
    "dq_missing_scale": ("dq[a] = scale * (dS[i - r0] @ k)", "dq[a] = (dS[i - r0] @ k)"),
    "dropped_rowdot": ("Di = (dout[r0:r1] * o).sum(axis=1)", "Di = 0.0 * (dout[r0:r1] * o).sum(axis=1)"),
    "dv_uses_ds": ("dv += P[:, cols].T @ dout[r0:r1]", "dv += dS[:, cols].T @ dout[r0:r1]"),
    "bias_head_ignored": ("b = bias[q0:q1, 0 if bias.shape[1] == 1 else h, : k1 - k0]\n            o, lse",
                          "b = bias[q0:q1, 0, : k1 - k0]\n            o, lse"),
    "bias_global_key_column": ("b = bias[q0:q1, 0 if bias.shape[1] == 1 else h, : k1 - k0]\n            o, lse",
                               "b = bias[q0:q1, 0 if bias.shape[1] == 1 else h, k0:k1]\n            o, lse"),
    "kv_offsets_from_cu_q": ("q0, q1, k0, k1 = cu_q[s], cu_q[s + 1], cu_kv[s], cu_kv[s + 1]\n        if q1 == q0:\n            continue\n        for h in range(hq):\n            b = None",
                             "q0, q1, k0, k1 = cu_q[s], cu_q[s + 1], cu_q[s], cu_q[s + 1]\n        if q1 == q0:\n            continue\n        for h in range(hq):\n            b = None"),
}


def _mutant(old, new):
    src = inspect.getsource(orc)
    assert src.count(old) >= 1, f"mutation site not found: {old!r}"
    mod = types.ModuleType("oracle_mutant")
    exec(compile(src.replace(old, new, 1), "oracle_mutant", "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name):
    mod = _mutant(*MUTANTS[name])
    failed = []
    for check in ALL_CHECKS:
        try:
            ok, _ = check(mod)
        except Exception:
            ok = False
        if not ok:
            failed.append(check.__name__)
    assert failed, f"no pin catches the planted mistake {name}"
