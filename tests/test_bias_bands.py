"""Bias bands (the keys an additive bias leaves each query row, include/vlf.h vlf_bias_bands):
the pass matches its definition computed here from the bias, and attention with the bands --
tiles and items the bias masks for every row skipped, 0 / -inf interval rows masked without
reading the bias -- matches the oracle on structured biases (prefix-LM masks, per-row interval
masks in varlen batches, ALiBi values, mixed rows), as does the same call without them."""
import numpy as np
import pytest
import torch

import workloads as W
from tests.parity import assert_within, compare, gpu_run, oracle_run

pytestmark = pytest.mark.gpu

NEG = float("-inf")


def band_definition(bias, cu_q, cu_kv):
    """Row and 64-row-block bands straight from the definition (numpy; ints exact)."""
    b = bias.numpy()
    tq, hb, _ = b.shape
    rows = np.zeros((hb, tq, 3), np.int64)
    blocks = {}
    for s in range(len(cu_q) - 1):
        q0, q1, kv = cu_q[s], cu_q[s + 1], cu_kv[s + 1] - cu_kv[s]
        for h in range(hb):
            for r in range(q0, q1):
                vals = b[r, h, :kv]
                fin = np.nonzero(~np.isneginf(vals))[0]
                if fin.size == 0:
                    rows[h, r] = (0, 0, 1)
                else:
                    lo, hi = int(fin[0]), int(fin[-1]) + 1
                    rows[h, r] = (lo, hi, int(np.all(vals[lo:hi] == 0.0)))
            for r0 in range(q0, q1, 64):
                # union of the rows' intervals; their intersection when all are pure, else -1s
                ent = rows[h, r0:min(r0 + 64, q1)]
                live = ent[ent[:, 1] > ent[:, 0]]
                lo, hi = (int(live[:, 0].min()), int(live[:, 1].max())) if live.size else (0, 0)
                if ent[:, 2].all():
                    ilo, ihi = int(ent[:, 0].max()), int(ent[:, 1].min())
                    blocks[(h, r0)] = (lo, hi, ilo, max(ihi, ilo))
                else:
                    blocks[(h, r0)] = (lo, hi, -1, -1)
    return rows, blocks


def _structured_bias(lengths_q, lengths_kv, heads, kind, seed, max_kv=None):
    g = torch.Generator("cpu").manual_seed(seed)
    tq = sum(lengths_q)
    mk = max_kv or max(lengths_kv)
    # columns past a sequence's keys hold finite garbage: the bands must ignore them
    bias = torch.randn((tq, heads, mk), generator=g)
    r0 = 0
    for lq, lk in zip(lengths_q, lengths_kv):
        i = torch.arange(lq)[:, None]
        j = torch.arange(lk)[None, :]
        if kind in ("prefix", "prefix_alibi"):
            allowed = (j <= lk // 3) | (j <= i + (lk - lq))
            allowed = allowed[:, None, :].expand(lq, heads, lk)
        else:  # per-row random intervals (not monotone in the row)
            a = torch.randint(0, lk + 1, (lq, heads, 1), generator=g)
            c = torch.randint(0, lk + 1, (lq, heads, 1), generator=g)
            lo, hi = torch.minimum(a, c), torch.maximum(a, c)
            jj = torch.arange(lk)[None, None, :]
            allowed = (jj >= lo) & (jj < hi)
        vals = torch.zeros((lq, heads, lk))
        if kind == "prefix_alibi":
            slope = torch.tensor([2.0 ** (-h - 1) for h in range(heads)])[None, :, None]
            vals = -slope * (i - j).abs().float()[:, None, :]
        if kind == "mixed":
            # every third row carries values inside its interval (not a pure interval)
            rowsel = (torch.arange(lq) % 3 == 0)[:, None, None]
            vals = torch.where(rowsel, torch.randn((lq, heads, lk), generator=g), vals)
        bias[r0:r0 + lq, :, :lk] = torch.where(allowed, vals, torch.full_like(vals, NEG))
        r0 += lq
    return bias.contiguous()


@pytest.mark.parametrize("kind", ["prefix", "intervals", "mixed"])
def test_bands_match_definition(kind):
    import variable_length_flash_gb300 as vlf
    lq = [300, 1, 64, 129, 0, 257]
    lk = [300, 5, 200, 129, 3, 400]
    bias = _structured_bias(lq, lk, 2, kind, seed=3, max_kv=404)
    bias[5, 1, :] = NEG                      # a row with no finite value
    bias[7, 0, 2] = float("nan")             # NaN counts as finite, and impure
    cu_q, cu_kv = W.cu_seqlens(lq), W.cu_seqlens(lk)
    bands = vlf.vlf_bias_bands(bias.cuda(), cu_q.cuda(), cu_kv.cuda())
    got = bands.view(torch.int32).view(2, 2, bias.shape[0], 4).cpu().numpy()
    rows, blocks = band_definition(bias, cu_q.tolist(), cu_kv.tolist())
    np.testing.assert_array_equal(got[0, :, :, :3], rows)
    for (h, r0), e in blocks.items():
        assert tuple(got[1, h, r0]) == e, (h, r0, got[1, h, r0], e)


CASES = [
    # (lengths_q, lengths_kv, dtype, h_q, h_kv, d_qk, d_v, causal, bias heads, kind, max_kv)
    ([700], [700], "fp16", 2, 2, 128, 128, False, 1, "prefix", None),
    ([700], [700], "bf16", 4, 4, 64, 64, False, 4, "prefix_alibi", None),
    ([300, 1, 129, 257], [300, 40, 129, 257], "bf16", 4, 2, 96, 96, True, 1, "intervals", None),
    ([260, 33], [260, 90], "bf16", 2, 2, 128, 128, False, 2, "mixed", None),
    ([400, 17], [400, 17], "fp16", 4, 2, 128, 128, False, 4, "prefix", None),
    # rows not 16-byte aligned (301 keys): bias values read row by row (bands narrow the tiles)
    ([301, 65], [301, 65], "bf16", 2, 2, 128, 128, False, 1, "prefix", None),
    # QK width 192 (bias read row by row in the backward)
    ([300], [300], "bf16", 2, 2, 192, 128, False, 1, "prefix", None),
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_parity_with_bands(case):
    lq, lk, dtype, hq, hkv, dqk, dv, causal, bh, kind, mk = CASES[case]
    w = W.custom(lq, lk, dtype=dtype, h_q=hq, h_kv=hkv, d_qk=dqk, d_v=dv, causal=causal)
    x = W.make_inputs(w, seed=50 + case, with_dout=True)
    x["bias"] = _structured_bias(lq, lk, bh, kind, seed=60 + case, max_kv=mk)
    ref = oracle_run(w, x)
    for bands in (None, False):
        gpu = gpu_run(w, x, bias_bands=bands)
        assert_within(compare(w, gpu, ref), f"bands case {case} ({kind}, bands={bands})")
