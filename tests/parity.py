"""Helpers shared by the GPU parity tests: run the CUDA path through the C ABI binding, run the
fp64 oracle on the same inputs, compare element by element."""
from __future__ import annotations

import numpy as np
import torch

from oracle import attention as orc

# max-abs error gates on O (3x on dQ/dK/dV); LSE is compared to 1e-3 absolute
TOL = {"fp16": 2e-3, "bf16": 1.5e-2, "fp32": 1e-5}
LSE_TOL = {"fp16": 1e-3, "bf16": 1e-3, "fp32": 1e-5}


def to_np(t):
    return t.detach().to("cpu", torch.float64).numpy()


def gpu_run(w, x, flags=0, backward=True, device="cuda"):
    import variable_length_flash_gb300 as vlf
    g = {k: (t.to(device) if isinstance(t, torch.Tensor) else t) for k, t in x.items()}
    out, lse = vlf.vlf_attn_varlen_fwd(g["q"], g["k"], g["v"], g["cu_seqlens_q"],
                                       g["cu_seqlens_kv"], w.max_seqlen_q, w.max_seqlen_kv,
                                       scale=w.scale, causal=w.causal, window=w.window,
                                       bias=g["bias"], flags=flags)
    res = {"out": out, "lse": lse}
    if backward:
        dq, dk, dv = vlf.vlf_attn_varlen_bwd(g["dout"], g["q"], g["k"], g["v"], out, lse,
                                             g["cu_seqlens_q"], g["cu_seqlens_kv"],
                                             w.max_seqlen_q, w.max_seqlen_kv, scale=w.scale,
                                             causal=w.causal, window=w.window, bias=g["bias"],
                                             flags=flags)
        res.update(dq=dq, dk=dk, dv=dv)
    status = vlf.vlf_check_error()
    assert status == 0, vlf.vlf_status_string(status)
    return res


def oracle_run(w, x, backward=True):
    O, L = orc.forward(x["q"], x["k"], x["v"], x["cu_seqlens_q"], x["cu_seqlens_kv"],
                       scale=w.softmax_scale, causal=w.causal, window=w.window, bias=x["bias"])
    ref = {"out": O, "lse": L}
    if backward:
        dq, dk, dv = orc.backward(x["q"], x["k"], x["v"], x["dout"], x["cu_seqlens_q"],
                                  x["cu_seqlens_kv"], scale=w.softmax_scale, causal=w.causal,
                                  window=w.window, bias=x["bias"])
        ref.update(dq=dq, dk=dk, dv=dv)
    return ref


def max_err(a, b):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    if a.size == 0:
        return 0.0
    same_inf = np.isinf(a) & np.isinf(b) & (np.sign(a) == np.sign(b))
    with np.errstate(invalid="ignore"):
        d = np.where(same_inf, 0.0, np.abs(a - b))
    d = np.nan_to_num(d, nan=np.inf)
    return float(d.max())


def compare(w, gpu, ref, keys=None):
    """Max-abs errors per output and whether each is within its gate.

    Returns {name: (err, limit)}; also reports the error of the oracle rounded to the output
    dtype (what output rounding alone costs) under name + '_rounding'.
    """
    tol = TOL[w.dtype]
    limits = {"out": tol, "lse": LSE_TOL[w.dtype], "dq": 3 * tol, "dk": 3 * tol, "dv": 3 * tol}
    dt = {"fp16": torch.float16, "bf16": torch.bfloat16, "fp32": torch.float32}[w.dtype]
    res = {}
    for k in keys or ref.keys():
        g = to_np(gpu[k]) if isinstance(gpu[k], torch.Tensor) else gpu[k]
        res[k] = (max_err(g, ref[k]), limits[k])
        if k != "lse":
            rounded = torch.from_numpy(np.asarray(ref[k])).to(dt).double().numpy()
            res[k + "_rounding"] = (max_err(rounded, ref[k]), float("inf"))
    return res


def assert_within(errs, label=""):
    bad = {k: v for k, v in errs.items() if not v[0] <= v[1]}
    assert not bad, f"{label} exceeds tolerance: {bad} (all: {errs})"
