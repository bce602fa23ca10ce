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


def gpu_run(w, x, flags=0, backward=True, device="cuda", bias_bands=None):
    """The CUDA path through the binding; bias_bands as the binding takes it (None: computed
    for a bias, False: none)."""
    import variable_length_flash_gb300 as vlf
    g = {k: (t.to(device) if isinstance(t, torch.Tensor) else t) for k, t in x.items()}
    if bias_bands is None and g["bias"] is not None:
        bias_bands = vlf.vlf_bias_bands(g["bias"], g["cu_seqlens_q"], g["cu_seqlens_kv"])
    out, lse = vlf.vlf_attn_varlen_fwd(g["q"], g["k"], g["v"], g["cu_seqlens_q"],
                                       g["cu_seqlens_kv"], w.max_seqlen_q, w.max_seqlen_kv,
                                       scale=w.scale, causal=w.causal, window=w.window,
                                       bias=g["bias"], flags=flags, bias_bands=bias_bands)
    res = {"out": out, "lse": lse}
    if backward:
        dq, dk, dv = vlf.vlf_attn_varlen_bwd(g["dout"], g["q"], g["k"], g["v"], out, lse,
                                             g["cu_seqlens_q"], g["cu_seqlens_kv"],
                                             w.max_seqlen_q, w.max_seqlen_kv, scale=w.scale,
                                             causal=w.causal, window=w.window, bias=g["bias"],
                                             flags=flags, bias_bands=bias_bands)
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


# unit roundoff of the 16-bit types P and dS enter the tensor cores in, and of the outputs
UNIT = {"fp16": 2.0 ** -11, "bf16": 2.0 ** -8, "fp32": 2.0 ** -24}


def grad_error_bound(w, x, out_gpu):
    """Element-wise first-order bound on |GPU - oracle| for dQ, dK, dV of a bias-free problem,
    from how the GPU forms them in floating point (the FlashAttention-2 backward of triton-msl
    part 2, "Beyond softmax": P = exp(S - LSE), D = rowsum(dO o O), dS = P (dP - D), fp32
    accumulation, P and dS rounded to the 16-bit input type before the tensor-core products).

    Logits.  An fp32 dot product of D_qk exact 16-bit products errs by at most
    Delta_ij = scale * D_qk * 2^-23 * sum_c |q_ic k_jc| (recursive summation, adds that may
    truncate).  The backward recomputes every logit with the same products in the same order as
    the forward, so the forward's LSE carries the same per-logit errors delta_ij; to first
    order P_ij then errs relatively by delta_ij - sum_k P_ik delta_ik, at most
    sum_{k != j} P_ik (Delta_ij + Delta_ik) (which vanishes for a one-hot row's winner), plus
    the roundings of the exponent argument at the magnitude of LSE and of the row max m_i
    (the base-2 row max, LSE's sum and conversion back to natural log, its fp32 store, the
    backward's conversion to base 2 and the two conversion constants: six fp32 roundings, each
    at most 2^-24 log2(e) max(|LSE_i|, |m_i|), so eta_i = 10 * 2^-24 max(|LSE_i|, |m_i|)), plus
    2^-21 for ex2.approx, plus u when P is rounded to 16 bits:
        |dP_ij| <= P_ij * (expm1(rho_ij) + u),  rho_ij = sum_{k!=j} P_ik (Delta_ij + Delta_ik)
                                                        + eta_i + 2^-21
    dP = dO.v    |ddP_ij| <= D_v 2^-23 sum_c |dO_ic v_jc|
    D = dO.O     |dD_i| <= sum_c |dO_ic| |O_gpu_ic - O_ic| + D_v 2^-23 sum_c |dO_ic O_ic|
                 (the GPU's D uses the O it stored)
    dS           |ddS_ij| <= |dP_ij| |dP_ij - D_i| + P_ij (|ddP_ij| + |dD_i|) + u |dS_ij|
    dQ_ic        <= scale sum_j |ddS_ij| |k_jc| + n_keys 2^-23 scale sum_j |dS_ij k_jc| + u |dQ_ic|
    dK_jc        <= scale sum_i |ddS_ij| |q_ic| + n_rows 2^-23 scale sum_i |dS_ij q_ic| + u |dK_jc|
    dV_jc        <= sum_i |dP_ij| |dO_ic| + n_rows 2^-23 sum_i |P_ij dO_ic| + u |dV_jc|
    with u the unit roundoff of the input type (P, dS and the outputs are rounded to it).
    Second-order terms are dropped.  Returns {"dq", "dk", "dv"}, arrays of the inputs' shapes
    (float64).  The parity gate of an element is the stated tolerance (3x the O gate) plus its
    bound.
    """
    q, k, v, do = (to_np(x[n]) for n in ("q", "k", "v", "dout"))
    o_gpu = to_np(out_gpu)
    cu_q = [int(t) for t in x["cu_seqlens_q"].tolist()]
    cu_k = [int(t) for t in x["cu_seqlens_kv"].tolist()]
    u = UNIT[w.dtype]
    sc = w.softmax_scale
    g = w.h_q // w.h_kv
    e23 = 2.0 ** -23
    bq, bk, bv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    dk_ref, dv_ref = np.zeros_like(k), np.zeros_like(v)  # the gradients themselves (u terms)
    for s in range(len(cu_q) - 1):
        a, b, c, d = cu_q[s], cu_q[s + 1], cu_k[s], cu_k[s + 1]
        if b == a or d == c:
            continue
        for h in range(w.h_q):
            qh, kh, vh, doh = q[a:b, h], k[c:d, h // g], v[c:d, h // g], do[a:b, h]
            ok = orc.visible(b - a, d - c, w.causal, w.window)
            lg = orc.logits(qh, kh, sc, ok)
            P, lse = orc.softmax(lg)
            O = P @ vh
            live = np.isfinite(lse)
            m = np.where(live, lg.max(axis=1), 0.0)
            Dl = sc * w.d_qk * e23 * (np.abs(qh) @ np.abs(kh).T)        # Delta_ij
            Dl = np.where(ok, Dl, 0.0)
            pd = (P * Dl).sum(axis=1)                                     # sum_k P_ik Delta_ik
            rho = (Dl * (1.0 - P) + (pd[:, None] - P * Dl)
                   + (10 * 2.0 ** -24 * np.maximum(np.where(live, np.abs(lse), 0.0),
                                                   np.abs(m)))[:, None]
                   + 2.0 ** -21)
            dPerr = P * (np.expm1(rho) + u)
            dP = doh @ vh.T
            ddP = w.d_v * e23 * (np.abs(doh) @ np.abs(vh).T)
            Di = (doh * O).sum(axis=1)
            dD = ((np.abs(doh) * np.abs(o_gpu[a:b, h] - O)).sum(axis=1)
                  + w.d_v * e23 * (np.abs(doh) * np.abs(O)).sum(axis=1))
            dS = P * (dP - Di[:, None])
            ddS = dPerr * np.abs(dP - Di[:, None]) + P * (ddP + dD[:, None]) + u * np.abs(dS)
            n_k, n_q = d - c, b - a
            dq = sc * (dS @ kh)
            bq[a:b, h] = (sc * (ddS @ np.abs(kh)) + n_k * e23 * sc * (np.abs(dS) @ np.abs(kh))
                          + u * np.abs(dq))
            bk[c:d, h // g] += sc * (ddS.T @ np.abs(qh)) + n_q * e23 * sc * (np.abs(dS).T @ np.abs(qh))
            bv[c:d, h // g] += dPerr.T @ np.abs(doh) + n_q * e23 * (P.T @ np.abs(doh))
            dk_ref[c:d, h // g] += sc * (dS.T @ qh)
            dv_ref[c:d, h // g] += P.T @ doh
    return {"dq": bq, "dk": bk + u * np.abs(dk_ref), "dv": bv + u * np.abs(dv_ref)}
