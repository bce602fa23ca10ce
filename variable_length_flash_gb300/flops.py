"""Work counting for throughput reports: unmasked (query, key, head) pairs and FLOPs.

Convention (the pages define none): a pair is counted when its logit is finite (visible under
causal/window and not masked by a -inf bias).  Per pair, the forward does QK^T and PV,
2 (D_qk + D_v) FLOPs; the backward does the five FlashAttention-2 products (S recompute, dV,
dP, dK, dQ), 2 (3 D_qk + 2 D_v) FLOPs.  Exponentials and masking are not counted, nor is any
recomputation a particular kernel split adds.
"""
from __future__ import annotations

import numpy as np

PREFIX_LEN = 8192


def visible_pairs(q_len: int, kv_len: int, causal: bool, window: int) -> int:
    """Pairs (i, j) of one sequence and one head that the causal/window rules leave visible."""
    if q_len <= 0 or kv_len <= 0:
        return 0
    i = np.arange(q_len, dtype=np.int64)
    diag = i + (kv_len - q_len)
    hi = np.minimum(diag, kv_len - 1) if causal else np.full(q_len, kv_len - 1)
    lo = np.maximum(diag - window + 1, 0) if window > 0 else np.zeros(q_len, np.int64)
    return int(np.clip(hi - lo + 1, 0, None).sum())


def prefix_lm_pairs(q_len: int, kv_len: int, prefix: int = PREFIX_LEN) -> int:
    """Pairs with a finite prefix-LM bias (key <= prefix - 1 or key <= query), single sequence."""
    i = np.arange(q_len, dtype=np.int64)
    return int(np.minimum(kv_len, np.maximum(prefix, i + 1)).sum())


def workload_pairs(w) -> int:
    """Unmasked pairs of a ``workloads.Workload`` summed over sequences and query heads."""
    total = 0
    for lq, lk in zip(w.lengths_q, w.lengths_kv):
        if w.bias is not None:
            assert not w.causal and w.window <= 0
            total += prefix_lm_pairs(lq, lk, w.meta.get("prefix", PREFIX_LEN))
        else:
            total += visible_pairs(lq, lk, w.causal, w.window)
    return total * w.h_q


def flops_per_pair(d_qk: int, d_v: int) -> dict:
    fwd = 2 * (d_qk + d_v)
    bwd = 2 * (3 * d_qk + 2 * d_v)
    return {"fwd": fwd, "bwd": bwd, "fwd_bwd": fwd + bwd,
            # per-kernel algorithmic counts of the backward's kernels
            "dkdv": 2 * (2 * d_qk + 2 * d_v),   # S recompute, dP, dV, dK
            "dq": 2 * (2 * d_qk + d_v)}         # S recompute, dP, dQ
