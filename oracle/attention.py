"""fp64 CPU oracle for fused variable-length attention, forward and backward.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports this module: only the tests,
``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg use it.  It shares no code with
the CUDA library (no kernels, headers, helpers or tables); the two meet only at the seeded input
generators in ``workloads``.

What it computes is the plain definition of the attention that the mtlattn 0.3.0 page
(pypi.org/project/mtlattn/0.3.0, section "Use") states for its ``varlen_attention`` call, written
out in float64 with no tiling, no online softmax and no fusion:

* packed ``cu_seqlens`` layout: q [total_q, H_q, D_qk], k [total_kv, H_kv, D_qk],
  v [total_kv, H_kv, D_v]; sequence s owns rows cu[s] .. cu[s+1]-1 (mtlattn page, "Use");
* query head h reads kv head h // (H_q / H_kv) (GQA/MQA, mtlattn page, "Use");
* logit = scale * (q . k) + bias, scale defaulting to 1/sqrt(D_qk) (mtlattn page, "Use");
* end-aligned causal rule: query i may see key j iff j <= i + (kv_len - q_len)
  (mtlattn page, "Use", causal=True);
* sliding window W: query i sees only the last W keys up to its causal diagonal, i.e.
  j >= i + (kv_len - q_len) - W + 1 (mtlattn page, "Use", window=W);
* additive fp32 bias indexed by global query row and sequence-local key, dim1 == 1 broadcast
  over heads, -inf meaning "masked" (mtlattn page, "Use", attn_bias);
* softmax over the visible keys, O = P V, and the log-sum-exp LSE = m + ln(sum exp(logit - m))
  that a FlashAttention-2 backward consumes (triton-msl part 2, "Beyond softmax");
* backward: the gradient of sum(O * dO) with the bias held constant
  (mtlattn page, "Use": the bias is treated as constant; triton-msl part 2, "Beyond softmax").

A row that sees no key (empty band, all-(-inf) bias) has O = 0 and LSE = -inf and contributes
nothing to any gradient.
"""
from __future__ import annotations

import numpy as np

NEG_INF = -np.inf


def visible(q_len: int, kv_len: int, causal: bool, window: int, rows=None) -> np.ndarray:
    """Boolean [n_rows, kv_len]: may sequence-local query row i attend sequence-local key j.

    Diagonal of row i is d_i = i + (kv_len - q_len) (end-aligned causal, mtlattn page "Use").
    causal: j <= d_i.  window W > 0: j >= d_i - W + 1 (the last W keys up to the diagonal).
    """
    i = np.arange(q_len, dtype=np.int64) if rows is None else np.asarray(rows, dtype=np.int64)
    j = np.arange(kv_len, dtype=np.int64)
    diag = i[:, None] + (kv_len - q_len)
    ok = np.ones((i.shape[0], kv_len), dtype=bool)
    if causal:
        ok &= j[None, :] <= diag
    if window > 0:
        ok &= j[None, :] >= diag - window + 1
    return ok


def logits(q_rows: np.ndarray, k: np.ndarray, scale: float, ok: np.ndarray,
           bias_rows=None) -> np.ndarray:
    """[n, kv_len] float64: scale * (q . k) + bias, -inf where the pair is not visible."""
    s = scale * (q_rows @ k.T)
    if bias_rows is not None:
        s = s + bias_rows
    return np.where(ok, s, NEG_INF)


def softmax(s: np.ndarray):
    """Row softmax of logits s (two passes: max, then exp/sum).  Returns (P, LSE).

    Rows with no finite logit get P = 0 and LSE = -inf.
    """
    m = s.max(axis=1) if s.shape[1] else np.full(s.shape[0], NEG_INF)
    live = np.isfinite(m)
    P = np.zeros_like(s)
    lse = np.full(s.shape[0], NEG_INF)
    if live.any():
        e = np.exp(s[live] - m[live, None])
        l = e.sum(axis=1)
        P[live] = e / l[:, None]
        lse[live] = m[live] + np.log(l)
    return P, lse


def head_forward(q_rows, rows, k, v, q_len, scale, causal=False, window=0, bias_rows=None):
    """Attention of one query head of one sequence, for the sequence-local ``rows``.

    q_rows [n, D_qk], k [kv_len, D_qk], v [kv_len, D_v] float64, bias_rows [n, kv_len] or None.
    Returns O [n, D_v], LSE [n].
    """
    ok = visible(q_len, k.shape[0], causal, window, rows)
    P, lse = softmax(logits(q_rows, k, scale, ok, bias_rows))
    return P @ v, lse


def _f64(x):
    if hasattr(x, "detach"):
        x = x.detach().to("cpu")
        import torch
        return x.to(torch.float64).numpy()
    return np.asarray(x, dtype=np.float64)


def _ints(x):
    if hasattr(x, "detach"):
        x = x.detach().to("cpu").numpy()
    return [int(t) for t in np.asarray(x)]


def forward(q, k, v, cu_q, cu_kv, scale=None, causal=False, window=0, bias=None):
    """Whole packed forward (small problems).  Returns O [total_q, H_q, D_v], LSE [H_q, total_q].

    bias: [total_q, 1 or H_q, max_kv] or None; row = global query, column = sequence-local key.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    bias = None if bias is None else _f64(bias)
    cu_q, cu_kv = _ints(cu_q), _ints(cu_kv)
    tq, hq, dqk = q.shape
    hkv, dv = v.shape[1], v.shape[2]
    g = hq // hkv
    scale = 1.0 / np.sqrt(dqk) if scale is None else scale
    O = np.zeros((tq, hq, dv))
    LSE = np.full((hq, tq), NEG_INF)
    for s in range(len(cu_q) - 1):
        q0, q1, k0, k1 = cu_q[s], cu_q[s + 1], cu_kv[s], cu_kv[s + 1]
        if q1 == q0:
            continue
        for h in range(hq):
            b = None
            if bias is not None:
                b = bias[q0:q1, 0 if bias.shape[1] == 1 else h, : k1 - k0]
            o, lse = head_forward(q[q0:q1, h], np.arange(q1 - q0), k[k0:k1, h // g],
                                  v[k0:k1, h // g], q1 - q0, scale, causal, window, b)
            O[q0:q1, h] = o
            LSE[h, q0:q1] = lse
    return O, LSE


def head_backward(q, k, v, dout, scale, causal=False, window=0, bias=None,
                  rows=None, cols=None, chunk=None):
    """Gradients of sum(O * dO) for one query head of one sequence.

    q [q_len, D_qk], k [kv_len, D_qk], v [kv_len, D_v], dout [q_len, D_v], bias [q_len, kv_len]
    (or a callable rows -> bias rows, for inputs too large to hold), all float64.
    rows: sequence-local query rows whose dQ is wanted (default: all).
    cols: sequence-local keys whose dK/dV contribution is wanted (default: all).
    chunk: optional number of query rows handled at a time; it only bounds memory (every row's
    softmax is still taken over its whole key range).

    With P = softmax(logits), D_i = sum_c dO_ic O_ic, dP_ij = dO_i . v_j,
    dS_ij = P_ij (dP_ij - D_i):  dQ_i = scale sum_j dS_ij k_j,  dK_j = scale sum_i dS_ij q_i,
    dV_j = sum_i P_ij dO_i.
    Returns dict with O, LSE (all rows), dq [len(rows), D_qk], dk [len(cols), D_qk],
    dv [len(cols), D_v].
    """
    q_len, kv_len = q.shape[0], k.shape[0]
    rows = np.arange(q_len) if rows is None else np.asarray(rows, dtype=np.int64)
    cols = np.arange(kv_len) if cols is None else np.asarray(cols, dtype=np.int64)
    chunk = q_len if chunk is None else chunk
    O = np.zeros((q_len, v.shape[1]))
    LSE = np.full(q_len, NEG_INF)
    dq = np.zeros((len(rows), q.shape[1]))
    dk = np.zeros((len(cols), k.shape[1]))
    dv = np.zeros((len(cols), v.shape[1]))
    row_pos = {int(r): a for a, r in enumerate(rows)}
    for r0 in range(0, q_len, max(chunk, 1)):
        r1 = min(q_len, r0 + chunk)
        idx = np.arange(r0, r1)
        ok = visible(q_len, kv_len, causal, window, idx)
        if bias is None:
            b = None
        elif callable(bias):
            b = bias(idx)
        else:
            b = bias[r0:r1]
        P, lse = softmax(logits(q[r0:r1], k, scale, ok, b))
        o = P @ v
        O[r0:r1], LSE[r0:r1] = o, lse
        Di = (dout[r0:r1] * o).sum(axis=1)
        dP = dout[r0:r1] @ v.T
        dS = P * (dP - Di[:, None])
        dk += scale * (dS[:, cols].T @ q[r0:r1])
        dv += P[:, cols].T @ dout[r0:r1]
        for i in idx:
            a = row_pos.get(int(i))
            if a is not None:
                dq[a] = scale * (dS[i - r0] @ k)
    return {"O": O, "LSE": LSE, "dq": dq, "dk": dk, "dv": dv}


def head_backward_rows(q_rows, rows, k, v, dout_rows, q_len, scale, causal=False, window=0,
                       bias_rows=None):
    """dQ of the sequence-local ``rows`` of one query head (plus their O and LSE).

    Every quantity dQ_i needs -- the row's softmax P_i, D_i = dO_i . O_i, dP_i = dO_i V^T and
    dS_i = P_i o (dP_i - D_i) -- belongs to row i alone, so this is the definition in
    head_backward restricted to the given rows.  q_rows [n, D_qk], dout_rows [n, D_v],
    bias_rows [n, kv_len] or None.  Returns O [n, D_v], LSE [n], dq [n, D_qk].
    """
    ok = visible(q_len, k.shape[0], causal, window, rows)
    P, lse = softmax(logits(q_rows, k, scale, ok, bias_rows))
    O = P @ v
    Di = (dout_rows * O).sum(axis=1)
    dS = P * (dout_rows @ v.T - Di[:, None])
    return O, lse, scale * (dS @ k)


def backward(q, k, v, dout, cu_q, cu_kv, scale=None, causal=False, window=0, bias=None):
    """Whole packed backward (small problems).  Returns dq, dk, dv (float64, input layouts).

    dK/dV of kv head g sum the contributions of every query head h with h // (H_q/H_kv) == g.
    """
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    bias = None if bias is None else _f64(bias)
    cu_q, cu_kv = _ints(cu_q), _ints(cu_kv)
    hq, hkv = q.shape[1], k.shape[1]
    g = hq // hkv
    scale = 1.0 / np.sqrt(q.shape[2]) if scale is None else scale
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    for s in range(len(cu_q) - 1):
        q0, q1, k0, k1 = cu_q[s], cu_q[s + 1], cu_kv[s], cu_kv[s + 1]
        if q1 == q0 or k1 == k0:
            continue
        for h in range(hq):
            b = None
            if bias is not None:
                b = bias[q0:q1, 0 if bias.shape[1] == 1 else h, : k1 - k0]
            r = head_backward(q[q0:q1, h], k[k0:k1, h // g], v[k0:k1, h // g], dout[q0:q1, h],
                              scale, causal, window, b)
            dq[q0:q1, h] = r["dq"]
            dk[k0:k1, h // g] += r["dk"]
            dv[k0:k1, h // g] += r["dv"]
    return dq, dk, dv
