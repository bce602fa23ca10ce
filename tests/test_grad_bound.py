"""The derived gradient gate of the outlier-channel parity test (tests/parity.py,
grad_error_bound) is a real check: on CPU, with the oracle's own results standing in for a
correct GPU answer, planted mistakes of the kinds a wrong backward makes exceed it, and on
ordinary inputs the bound adds little to the stated tolerance."""
import numpy as np
import pytest
import torch

import workloads as W
from tests.parity import TOL, grad_error_bound, oracle_run


def _outliers(dtype):
    w = W.custom([200, 57], dtype=dtype, h_q=2, d_qk=128, causal=True)
    x = W.make_inputs(w, seed=21, with_dout=True)
    for t in ("q", "k"):
        y = x[t].float()
        y[..., 3] *= 300.0
        y[..., 77] *= -900.0
        x[t] = y.to(x[t].dtype)
    return w, x


def _rounded(a, dtype):
    dt = {"fp16": torch.float16, "bf16": torch.bfloat16}[dtype]
    return torch.from_numpy(np.asarray(a)).to(dt)


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_outlier_gate_catches_planted_mistakes(dtype):
    w, x = _outliers(dtype)
    ref = oracle_run(w, x)
    bound = grad_error_bound(w, x, _rounded(ref["out"], dtype))
    gate = {k: 3 * TOL[dtype] + bound[k] for k in ("dq", "dk", "dv")}
    for k in gate:
        assert np.all(np.isfinite(gate[k])), k
        # the correct answer rounded to the output type passes
        assert np.all(np.abs(_rounded(ref[k], dtype).double().numpy() - ref[k]) <= gate[k]), k
    # dV 25% too large (a mis-scaled accumulation) and dV from P that was not normalised by its
    # row sum twice (P^2 instead of P: an exponent taken against the wrong LSE) both fail
    assert np.any(np.abs(1.25 * ref["dv"] - ref["dv"]) > gate["dv"])
    # a dropped D term: dS = P dP instead of P (dP - D) -> dQ = scale sum_j P_ij dP_ij k_j
    from oracle import attention as orc
    q, k, v, do = (x[n].double().numpy() for n in ("q", "k", "v", "dout"))
    cu = x["cu_seqlens_q"].tolist()
    wrong = np.zeros_like(ref["dq"])
    for s in range(len(cu) - 1):
        a, b = cu[s], cu[s + 1]
        for h in range(w.h_q):
            ok = orc.visible(b - a, b - a, True, 0)
            P, _ = orc.softmax(orc.logits(q[a:b, h], k[a:b, h], w.softmax_scale, ok))
            wrong[a:b, h] = w.softmax_scale * ((P * (do[a:b, h] @ v[a:b, h].T)) @ k[a:b, h])
    assert np.any(np.abs(wrong - ref["dq"]) > gate["dq"])


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_bound_is_of_the_stated_tolerance_on_ordinary_inputs(dtype):
    """Without outliers the bound is of the order of the stated 3x tolerance (which was set to
    cover the same 16-bit roundings): the derived gate reduces to about the flat one."""
    w = W.custom([200, 57], dtype=dtype, h_q=2, d_qk=128, causal=True)
    x = W.make_inputs(w, seed=21, with_dout=True)
    ref = oracle_run(w, x)
    bound = grad_error_bound(w, x, _rounded(ref["out"], dtype))
    for k in ("dq", "dk", "dv"):
        assert bound[k].max() < 2 * 3 * TOL[dtype], (k, float(bound[k].max()))
        assert np.median(bound[k]) < 0.5 * 3 * TOL[dtype], (k, float(np.median(bound[k])))
