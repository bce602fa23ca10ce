"""Checks that pin the fp64 oracle to things other than itself.

Each ``check_*`` takes an oracle module (``oracle.attention`` or a mutant of it) and returns
``(ok, message)``.  ``test_oracle_pins`` asserts they all pass on the real oracle;
``test_oracle_mutants`` plants plausible mistakes in copies of the oracle and asserts that at
least one check catches each.

Pins used (none re-types the oracle's own formula):
* hand-derived worked examples (``golden/worked_examples.json``);
* closed forms: one visible key returns its V row; identical keys return the mean of V;
  rows of P sum to 1; a constant bias shift leaves O unchanged and shifts LSE;
* brute-force masks written from the rule text, loop by loop;
* torch's own float64 CPU ``scaled_dot_product_attention`` (an independent routine) with an
  explicit boolean / float mask, and its autograd gradients;
* central finite differences of L = sum(O * dO) in float64;
* structure: varlen equals per-sequence dense, GQA equals K/V replicated over the group,
  split nope/rope dots summed equal the concatenated dot.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "worked_examples.json")


def _arr(x):
    return np.array([[[float(c) for c in h] for h in row] for row in x], dtype=np.float64)


def _cu(lens):
    return np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)


def _rng(seed):
    return np.random.default_rng(seed)


def _close(a, b, tol):
    a, b = np.asarray(a, dtype=np.float64), np.asarray(b, dtype=np.float64)
    if a.shape != b.shape:
        return False
    both_inf = np.isinf(a) & np.isinf(b) & (np.sign(a) == np.sign(b))
    with np.errstate(invalid="ignore"):
        d = np.where(both_inf, 0.0, np.abs(a - b))
    return bool(np.all(np.nan_to_num(d, nan=np.inf) <= tol))


# ---------------------------------------------------------------- worked examples
def check_worked_examples(orc):
    data = json.load(open(GOLDEN))
    for ex in data["examples"]:
        q, k, v = _arr(ex["q"]), _arr(ex["k"]), _arr(ex["v"])
        bias = None if ex["bias"] is None else _arr(ex["bias"])
        O, LSE = orc.forward(q, k, v, _cu(ex["lengths_q"]), _cu(ex["lengths_kv"]),
                             scale=ex["scale"], causal=ex["causal"], window=ex["window"],
                             bias=bias)
        if not _close(O, _arr(ex["O"]), 1e-12) or not _close(LSE, np.array(ex["LSE"]), 1e-12):
            return False, f"worked example {ex['name']}: O={O.tolist()} LSE={LSE.tolist()}"
    for ex in data["backward_examples"]:
        q, k, v, do = _arr(ex["q"]), _arr(ex["k"]), _arr(ex["v"]), _arr(ex["dout"])
        bias = None if ex["bias"] is None else _arr(ex["bias"])
        dq, dk, dv = orc.backward(q, k, v, do, _cu(ex["lengths_q"]), _cu(ex["lengths_kv"]),
                                  scale=ex["scale"], causal=ex["causal"], window=ex["window"],
                                  bias=bias)
        for name, got in (("dq", dq), ("dk", dk), ("dv", dv)):
            if not _close(got, _arr(ex[name]), 1e-12):
                return False, f"backward example {ex['name']}: {name}={got.tolist()}"
    return True, ""


# ---------------------------------------------------------------- brute-force masks
def brute_mask(q_len, kv_len, causal, window):
    """Mask written loop by loop from the rule text (end-aligned causal, last-W-keys window)."""
    m = [[True] * kv_len for _ in range(q_len)]
    for i in range(q_len):
        diag = i + (kv_len - q_len)          # the key aligned with query i
        for j in range(kv_len):
            if causal and j > diag:
                m[i][j] = False
            if window > 0:
                # the last `window` keys up to the diagonal: diag, diag-1, ..., diag-window+1
                last = [diag - t for t in range(window)]
                if j not in last:
                    m[i][j] = False
    return np.array(m, dtype=bool).reshape(q_len, kv_len)


def check_masks(orc):
    for q_len in (0, 1, 2, 5, 9):
        for kv_len in (0, 1, 3, 5, 12):
            for causal in (False, True):
                for window in (0, 1, 2, 3, 4, 20):
                    if window > 0 and not causal:
                        continue
                    got = orc.visible(q_len, kv_len, causal, window)
                    want = brute_mask(q_len, kv_len, causal, window)
                    if got.shape != want.shape or not np.array_equal(got, want):
                        return False, f"mask q={q_len} kv={kv_len} causal={causal} W={window}"
    # window without causal: only the lower bound of the band applies
    got = orc.visible(3, 6, False, 2)
    want = np.array([[j >= i + 3 - 1 for j in range(6)] for i in range(3)])
    if not np.array_equal(got, want):
        return False, "window without causal"
    return True, ""


# ---------------------------------------------------------------- closed forms
def check_single_key_and_identical_keys(orc):
    r = _rng(1)
    L, d = 6, 5
    q, k, v = r.standard_normal((L, 2, d)), r.standard_normal((L, 2, d)), r.standard_normal((L, 2, 3))
    cu = _cu([L])
    O, LSE = orc.forward(q, k, v, cu, cu, scale=0.7, causal=True)
    for h in range(2):
        # causal row 0 sees only key 0: O = v0 exactly, LSE = its logit
        logit = 0.7 * math.fsum(q[0, h, c] * k[0, h, c] for c in range(d))
        if not _close(O[0, h], v[0, h], 0.0) or abs(LSE[h, 0] - logit) > 1e-12:
            return False, "single visible key"
    # identical keys: O_i = mean of visible v_j, LSE_i = logit + ln(n_visible)
    kk = np.repeat(r.standard_normal((1, 1, d)), L, axis=0)
    O, LSE = orc.forward(q[:, :1], kk, v[:, :1], cu, cu, scale=0.3, causal=True)
    for i in range(L):
        want = np.mean(v[: i + 1, 0], axis=0)
        logit = 0.3 * math.fsum(q[i, 0, c] * kk[0, 0, c] for c in range(d))
        if not _close(O[i, 0], want, 1e-12) or abs(LSE[0, i] - (logit + math.log(i + 1))) > 1e-12:
            return False, f"identical keys row {i}"
    return True, ""


def check_rows_sum_to_one(orc):
    r = _rng(2)
    s = r.standard_normal((7, 9)) * 5
    s[2, :] = -np.inf          # a fully masked row
    s[3, ::2] = -np.inf
    P, lse = orc.softmax(s)
    live = np.isfinite(s).any(axis=1)
    if not np.allclose(P[live].sum(axis=1), 1.0, atol=1e-12, rtol=0):
        return False, "rows of P do not sum to 1"
    if np.any(P[~np.isfinite(s)] != 0) or np.isfinite(lse[2]):
        return False, "masked entries must be exactly 0, dead row LSE -inf"
    # LSE is the log of the partition function: sum_j exp(s_ij - LSE_i) == 1
    for i in np.nonzero(live)[0]:
        tot = math.fsum(math.exp(x - lse[i]) for x in s[i] if np.isfinite(x))
        if abs(tot - 1.0) > 1e-12:
            return False, "LSE is not log sum exp"
    return True, ""


def check_bias_shift(orc):
    r = _rng(3)
    lens = [5, 3]
    T = sum(lens)
    q, k, v = r.standard_normal((T, 2, 4)), r.standard_normal((T, 2, 4)), r.standard_normal((T, 2, 4))
    bias = r.standard_normal((T, 2, 5))
    cu = _cu(lens)
    O1, L1 = orc.forward(q, k, v, cu, cu, scale=0.5, bias=bias)
    c = np.array([0.75, -2.5])[None, :, None]
    O2, L2 = orc.forward(q, k, v, cu, cu, scale=0.5, bias=bias + c)
    if not _close(O1, O2, 1e-12) or not _close(L2 - L1, np.broadcast_to(c[0], L1.shape), 1e-12):
        return False, "constant bias shift must leave O unchanged and shift LSE by c"
    # -inf bias is a boolean mask: equals dropping those keys (here: keys j > 1 of sequence 0)
    b = np.zeros((T, 1, 5))
    b[:5, 0, 2:] = -np.inf
    O3, L3 = orc.forward(q, k, v, cu, cu, scale=0.5, bias=b)
    O4, L4 = orc.forward(q[:5], k[:2], v[:2], _cu([5]), _cu([2]), scale=0.5)
    if not _close(O3[:5], O4, 1e-12) or not _close(L3[:, :5], L4, 1e-12):
        return False, "-inf bias must equal masking those keys"
    return True, ""


# ---------------------------------------------------------------- structure
def check_varlen_equals_per_sequence(orc):
    r = _rng(4)
    lens = [3, 7, 1, 5]
    T = sum(lens)
    q, k, v = r.standard_normal((T, 2, 4)), r.standard_normal((T, 2, 4)), r.standard_normal((T, 2, 3))
    cu = _cu(lens)
    O, L = orc.forward(q, k, v, cu, cu, scale=0.5, causal=True)
    for s in range(len(lens)):
        a, b = cu[s], cu[s + 1]
        Os, Ls = orc.forward(q[a:b], k[a:b], v[a:b], _cu([b - a]), _cu([b - a]), 0.5, True)
        if not _close(O[a:b], Os, 0.0) or not _close(L[:, a:b], Ls, 0.0):
            return False, f"sequence {s} differs from its dense computation"
    # perturbing sequence 1 leaves the others bit-identical
    k2 = k.copy()
    k2[cu[1]:cu[2]] += 1.0
    O2, L2 = orc.forward(q, k2, v, cu, cu, scale=0.5, causal=True)
    other = np.ones(T, bool)
    other[cu[1]:cu[2]] = False
    if not np.array_equal(O[other], O2[other]) or np.array_equal(O[~other], O2[~other]):
        return False, "sequences leak into each other"
    return True, ""


def check_gqa_equals_replicated(orc):
    r = _rng(5)
    lens = [6, 4]
    T = sum(lens)
    hq, hkv = 6, 2
    q = r.standard_normal((T, hq, 4))
    k, v = r.standard_normal((T, hkv, 4)), r.standard_normal((T, hkv, 3))
    do = r.standard_normal((T, hq, 3))
    cu = _cu(lens)
    g = hq // hkv
    kr, vr = np.repeat(k, g, axis=1), np.repeat(v, g, axis=1)   # head h -> kv head h // g
    O1, L1 = orc.forward(q, k, v, cu, cu, 0.5, True)
    O2, L2 = orc.forward(q, kr, vr, cu, cu, 0.5, True)
    if not _close(O1, O2, 1e-13) or not _close(L1, L2, 1e-13):
        return False, "GQA forward != replicated K/V"
    dq1, dk1, dv1 = orc.backward(q, k, v, do, cu, cu, 0.5, True)
    dq2, dk2, dv2 = orc.backward(q, kr, vr, do, cu, cu, 0.5, True)
    dk2 = dk2.reshape(T, hkv, g, 4).sum(axis=2)
    dv2 = dv2.reshape(T, hkv, g, 3).sum(axis=2)
    if not (_close(dq1, dq2, 1e-12) and _close(dk1, dk2, 1e-12) and _close(dv1, dv2, 1e-12)):
        return False, "GQA backward != summed replicated-head gradients"
    return True, ""


def check_latent_split(orc):
    """nope (128) and rope (64) dots summed equal the concatenated 192-wide dot."""
    r = _rng(6)
    L = 5
    qn, qr = r.standard_normal((L, 1, 128)), r.standard_normal((L, 1, 64))
    kn, kr = r.standard_normal((L, 1, 128)), r.standard_normal((L, 1, 64))
    v = r.standard_normal((L, 1, 128))
    scale = 1.0 / math.sqrt(192.0)
    O, LSE = orc.forward(np.concatenate([qn, qr], 2), np.concatenate([kn, kr], 2), v,
                         _cu([L]), _cu([L]), scale=scale, causal=True)
    for i in range(L):
        lg = [scale * (math.fsum(qn[i, 0] * kn[j, 0]) + math.fsum(qr[i, 0] * kr[j, 0]))
              for j in range(i + 1)]
        m = max(lg)
        w = [math.exp(x - m) for x in lg]
        z = math.fsum(w)
        o = [math.fsum(w[j] * v[j, 0, c] for j in range(i + 1)) / z for c in range(128)]
        if not _close(O[i, 0], o, 1e-12) or abs(LSE[0, i] - (m + math.log(z))) > 1e-12:
            return False, f"latent split row {i}"
    return True, ""


# ---------------------------------------------------------------- torch float64 SDPA
def _torch_dense(q, k, v, cu_q, cu_kv, scale, causal, window, bias, dout=None):
    """Per-sequence torch SDPA in float64 with an explicit mask built from brute_mask."""
    import torch.nn.functional as F
    hq, hkv = q.shape[1], k.shape[1]
    g = hq // hkv
    tq = torch.tensor(q, requires_grad=dout is not None)
    tk = torch.tensor(k, requires_grad=dout is not None)
    tv = torch.tensor(v, requires_grad=dout is not None)
    outs = []
    for s in range(len(cu_q) - 1):
        a, b, c, d = cu_q[s], cu_q[s + 1], cu_kv[s], cu_kv[s + 1]
        mask = torch.tensor(brute_mask(b - a, d - c, causal, window))
        add = torch.zeros((hq, b - a, d - c), dtype=torch.float64)
        add = add.masked_fill(~mask, float("-inf"))
        if bias is not None:
            bb = torch.tensor(bias[a:b, :, : d - c]).permute(1, 0, 2)
            add = add + bb.expand(hq, -1, -1)
        qs = tq[a:b].permute(1, 0, 2)
        ks = tk[c:d].repeat_interleave(g, dim=1).permute(1, 0, 2)
        vs = tv[c:d].repeat_interleave(g, dim=1).permute(1, 0, 2)
        o = F.scaled_dot_product_attention(qs[None], ks[None], vs[None], attn_mask=add[None],
                                           scale=scale)[0]
        outs.append(o.permute(1, 0, 2))
    O = torch.cat(outs, 0)
    if dout is None:
        return O.detach().numpy()
    (O * torch.tensor(dout)).sum().backward()
    return O.detach().numpy(), tq.grad.numpy(), tk.grad.numpy(), tv.grad.numpy()


def _case(seed, lens_q, lens_kv, hq, hkv, d, dv, bias_heads=0):
    r = _rng(seed)
    tq, tk = sum(lens_q), sum(lens_kv)
    q = r.standard_normal((tq, hq, d))
    k = r.standard_normal((tk, hkv, d))
    v = r.standard_normal((tk, hkv, dv))
    do = r.standard_normal((tq, hq, dv))
    bias = None
    if bias_heads:
        bias = r.standard_normal((tq, bias_heads, max(lens_kv)))
    return q, k, v, do, bias


TORCH_CASES = [
    # lens_q, lens_kv, hq, hkv, d, dv, causal, window, bias_heads
    ([5, 9, 1], [5, 9, 1], 2, 2, 8, 8, False, 0, 0),
    ([5, 9, 1], [5, 9, 1], 4, 2, 8, 6, True, 0, 0),
    ([3, 8], [6, 8], 2, 1, 4, 4, True, 0, 0),          # cross, kv longer: end-aligned
    ([7, 2], [4, 5], 2, 2, 4, 4, True, 0, 0),          # cross, q longer: early rows see nothing
    ([12], [12], 2, 2, 4, 3, True, 3, 0),              # sliding window
    ([6, 5], [6, 7], 4, 1, 4, 4, False, 0, 1),         # broadcast bias, MQA
    ([6, 5], [6, 7], 2, 2, 4, 4, True, 2, 2),          # per-head bias + causal + window
]


def _finite_rows_only(O, ref):
    """torch SDPA returns NaN for rows with no visible key; the oracle's reading is O = 0."""
    bad = np.isnan(ref).any(axis=-1)
    return np.where(bad[..., None], 0.0, ref), bad


def check_torch_sdpa_forward(orc):
    for n, (lq, lk, hq, hkv, d, dv, causal, window, bh) in enumerate(TORCH_CASES):
        q, k, v, _, bias = _case(100 + n, lq, lk, hq, hkv, d, dv, bh)
        cq, ck = _cu(lq), _cu(lk)
        O, _ = orc.forward(q, k, v, cq, ck, scale=0.4, causal=causal, window=window, bias=bias)
        ref = _torch_dense(q, k, v, cq, ck, 0.4, causal, window, bias)
        ref, dead = _finite_rows_only(O, ref)
        if not _close(O, ref, 1e-12):
            return False, f"torch SDPA forward case {n}"
    return True, ""


def check_torch_autograd(orc):
    for n, (lq, lk, hq, hkv, d, dv, causal, window, bh) in enumerate(TORCH_CASES):
        q, k, v, do, bias = _case(200 + n, lq, lk, hq, hkv, d, dv, bh)
        cq, ck = _cu(lq), _cu(lk)
        # rows that see no key make torch's SDPA produce NaN (forward and backward); those
        # cases are pinned by check_dead_rows instead
        dead = ~np.concatenate([brute_mask(cq[s + 1] - cq[s], ck[s + 1] - ck[s], causal,
                                           window).any(axis=1) for s in range(len(lq))])
        if dead.any():
            continue
        _, tdq, tdk, tdv = _torch_dense(q, k, v, cq, ck, 0.4, causal, window, bias, dout=do)
        dq, dk, dv_ = orc.backward(q, k, v, do, cq, ck, scale=0.4, causal=causal,
                                   window=window, bias=bias)
        if not (_close(dq, tdq, 1e-11) and _close(dk, tdk, 1e-11) and _close(dv_, tdv, 1e-11)):
            return False, f"torch autograd case {n}"
    return True, ""


# ---------------------------------------------------------------- finite differences
def check_finite_differences(orc):
    cases = [([4, 3], [4, 3], 2, 1, 3, 2, True, 0, 0),
             ([5], [5], 2, 2, 3, 3, True, 2, 2),
             ([3, 2], [4, 2], 2, 2, 2, 2, False, 0, 1)]
    eps = 1e-6
    for n, (lq, lk, hq, hkv, d, dv, causal, window, bh) in enumerate(cases):
        q, k, v, do, bias = _case(300 + n, lq, lk, hq, hkv, d, dv, bh)
        cq, ck = _cu(lq), _cu(lk)

        def loss(q_, k_, v_):
            O, _ = orc.forward(q_, k_, v_, cq, ck, 0.6, causal, window, bias)
            return float(np.sum(O * do))

        dq, dk, dv_ = orc.backward(q, k, v, do, cq, ck, 0.6, causal, window, bias)
        for arr, grad in ((q, dq), (k, dk), (v, dv_)):
            for idx in np.ndindex(arr.shape):
                a = arr.copy()
                a[idx] += eps
                lp = loss(*(a if x is arr else x for x in (q, k, v)))
                a[idx] -= 2 * eps
                lm = loss(*(a if x is arr else x for x in (q, k, v)))
                fd = (lp - lm) / (2 * eps)
                if abs(fd - grad[idx]) > 1e-6 * max(1.0, abs(fd)):
                    return False, f"finite difference case {n} at {idx}: {fd} vs {grad[idx]}"
    return True, ""


# ---------------------------------------------------------------- degenerate rows
def check_dead_rows(orc):
    """Rows that see no key: O = 0, LSE = -inf, zero gradients, no NaN anywhere."""
    r = _rng(7)
    lens_q, lens_kv = [4, 2, 3], [2, 0, 3]
    q, k, v, do, _ = _case(8, lens_q, lens_kv, 2, 2, 3, 3)
    bias = r.standard_normal((9, 1, 3))
    bias[6, 0, :] = -np.inf                       # sequence 2, row 0: bias masks every key
    cq, ck = _cu(lens_q), _cu(lens_kv)
    O, L = orc.forward(q, k, v, cq, ck, 0.5, True, 0, bias)
    dq, dk, dv = orc.backward(q, k, v, do, cq, ck, 0.5, True, 0, bias)
    if any(np.isnan(x).any() for x in (O, dq, dk, dv)):
        return False, "NaN from an empty row"
    # sequence 0: q_len 4 > kv_len 2, rows 0,1 have diagonal < 0; sequence 1 has no keys
    for row in (0, 1, 4, 5, 6):
        if np.any(O[row] != 0) or np.any(np.isfinite(L[:, row])) or np.any(dq[row] != 0):
            return False, f"row {row} must be empty"
    return True, ""


def check_subset_and_chunks(orc):
    """The large-input form of the backward (row/col subsets, row chunks) equals the full one."""
    r = _rng(9)
    L = 11
    q, k, v, do = (r.standard_normal((L, 4)) for _ in range(4))
    bias = r.standard_normal((L, L))
    full = orc.head_backward(q, k, v, do, 0.5, True, 4, bias)
    rows, cols = [0, 5, 10], [1, 2, 9]
    part = orc.head_backward(q, k, v, do, 0.5, True, 4, lambda idx: bias[idx], rows, cols, chunk=3)
    ok = (_close(part["dq"], full["dq"][rows], 1e-12) and _close(part["dk"], full["dk"][cols], 1e-12)
          and _close(part["dv"], full["dv"][cols], 1e-12) and _close(part["O"], full["O"], 1e-12))
    if not ok:
        return False, "subset/chunked backward differs"
    # the row-local form used for sampled rows of large inputs
    O, L, dq = orc.head_backward_rows(q[rows], rows, k, v, do[rows], L, 0.5, True, 4, bias[rows])
    ok = (_close(O, full["O"][rows], 1e-12) and _close(L, full["LSE"][rows], 1e-12)
          and _close(dq, full["dq"][rows], 1e-12))
    return (ok, "" if ok else "row-local backward differs")


ALL_CHECKS = [check_worked_examples, check_masks, check_single_key_and_identical_keys,
              check_rows_sum_to_one, check_bias_shift, check_varlen_equals_per_sequence,
              check_gqa_equals_replicated, check_latent_split, check_torch_sdpa_forward,
              check_torch_autograd, check_finite_differences, check_dead_rows,
              check_subset_and_chunks]
