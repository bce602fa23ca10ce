"""GPU vs fp64 oracle at the benchmark workloads' full sizes, in the launch configuration bench.py
times (default flags, tensor-core path):

* O, LSE and dQ on seeded random query rows plus the last 4 rows of every sequence (the rows a
  32-bit index overflow would corrupt first), for a sample of query heads that includes the
  first and the last;
* dK and dV on whole (sequence, kv head) units -- every key of the unit, summed over the GQA
  group -- including the last sequence and the last kv head.  For the 49,152-token sequence the
  unit's keys are a seeded sample plus the prefix boundary and the last key (the oracle still
  takes every query row into each key's sum).

Inputs are drawn on the device with the seeded generators; the oracle receives host copies of
the input tensors and recomputes the bias rows on the host from the same fp64 formula.
"""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import attention as orc
from tests.parity import LSE_TOL, TOL, gpu_run, max_err

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

LARGE = ["dense4x4096_bf16_causal", "ragged64_gqa_window_bf16", "latent2x8192_bf16_causal",
         "long49152_fp16_bias_alibi", "long49152_fp16_bias_prefix", "dense4x4096_bf16_causal_d96",
         "dense4x4096_bf16_causal_d256"]


def _np(t):
    return t.detach().to("cpu", torch.float64).numpy()


def _head_sample(w, rng):
    heads = {0, w.h_q - 1}
    while len(heads) < min(4, w.h_q):
        heads.add(int(rng.integers(0, w.h_q)))
    return sorted(heads)


def _bias_rows(w, grows, head):
    """fp64 bias rows (global query rows `grows`) for query head `head`, from the generator."""
    hb = 0 if w.bias_heads == 1 else head
    b = W.bias_block(w, torch.as_tensor(np.asarray(grows), dtype=torch.int64), [hb])
    return b[:, 0, :].double().numpy()


@pytest.mark.parametrize("name", LARGE)
def test_full_size_workload(name):
    torch.cuda.empty_cache()
    w = W.workload(name)
    x = W.make_inputs(w, seed=0, device="cuda", with_dout=True)
    res = gpu_run(w, x)
    tol = TOL[w.dtype]
    rng = np.random.default_rng(2024)
    cu = [0]
    for L in w.lengths_q:
        cu.append(cu[-1] + L)
    g = w.h_q // w.h_kv
    scale = w.softmax_scale

    # ---------------------------------------------------------------- sampled rows: O, LSE, dQ
    rows = W.sample_rows(w, n_random=256, seed=3, tail=4)
    heads = _head_sample(w, rng)
    rows_t = torch.as_tensor(rows, dtype=torch.int64, device="cuda")
    q_rows = _np(x["q"][rows_t])
    do_rows = _np(x["dout"][rows_t])
    out_rows, dq_rows = _np(res["out"][rows_t]), _np(res["dq"][rows_t])
    lse_all = res["lse"]
    seq_of = np.searchsorted(np.asarray(cu), np.asarray(rows), side="right") - 1
    errs = {"out": 0.0, "lse": 0.0, "dq": 0.0}
    for s in sorted(set(seq_of.tolist())):
        sel = np.nonzero(seq_of == s)[0]
        local = np.asarray(rows)[sel] - cu[s]
        k0, k1 = cu[s], cu[s + 1]
        for h in heads:
            hk = h // g
            k = _np(x["k"][k0:k1, hk])
            v = _np(x["v"][k0:k1, hk])
            b = _bias_rows(w, np.asarray(rows)[sel], h) if w.bias else None
            O, L, dq = orc.head_backward_rows(q_rows[sel, h], local, k, v, do_rows[sel, h],
                                              k1 - k0, scale, w.causal, w.window, b)
            lse_gpu = lse_all[h, torch.as_tensor(np.asarray(rows)[sel], device="cuda")]
            errs["out"] = max(errs["out"], max_err(out_rows[sel, h], O))
            errs["lse"] = max(errs["lse"], max_err(_np(lse_gpu), L))
            errs["dq"] = max(errs["dq"], max_err(dq_rows[sel, h], dq))
    assert errs["out"] <= tol and errs["lse"] <= LSE_TOL[w.dtype] and errs["dq"] <= 3 * tol, errs

    # ---------------------------------------------------------------- dK / dV units
    n = w.num_seqs
    long_seq = max(w.lengths_q) > 20000
    units = {(n - 1, w.h_kv - 1)}
    if (n > 1 or w.h_kv > 1) and not long_seq:  # a 49k-token unit costs a minute of fp64 CPU
        units.add((int(rng.integers(0, n)), int(rng.integers(0, w.h_kv))))
    for s, hk in sorted(units):
        q0, q1 = cu[s], cu[s + 1]
        L = q1 - q0
        if long_seq:
            cols = set(rng.choice(L, 96, replace=False).tolist())
            cols |= {0, 8190, 8191, 8192, 8193, L - 2, L - 1}
            cols = sorted(c for c in cols if 0 <= c < L)
        else:
            cols = None
        k = _np(x["k"][q0:q1, hk])
        v = _np(x["v"][q0:q1, hk])
        dk = 0.0
        dv = 0.0
        for gh in range(g):
            h = hk * g + gh
            q = _np(x["q"][q0:q1, h])
            do = _np(x["dout"][q0:q1, h])
            bias = (lambda idx, h=h: _bias_rows(w, q0 + idx, h)) if w.bias else None
            r = orc.head_backward(q, k, v, do, scale, w.causal, w.window, bias, rows=[],
                                  cols=cols, chunk=2048 if long_seq else None)
            dk = dk + r["dk"]
            dv = dv + r["dv"]
        ck = slice(None) if cols is None else torch.as_tensor(cols, device="cuda")
        gdk = _np(res["dk"][q0:q1, hk][ck])
        gdv = _np(res["dv"][q0:q1, hk][ck])
        e_dk, e_dv = max_err(gdk, dk), max_err(gdv, dv)
        assert e_dk <= 3 * tol and e_dv <= 3 * tol, (name, s, hk, e_dk, e_dv)
    del x, res
    torch.cuda.empty_cache()


@pytest.mark.parametrize("name", ["decode64x8192_bf16_gqa", "decode4x32768_bf16_gqa"])
def test_decode_full_size_packing_exact(name):
    """The decode workloads at full size: the forward packs each kv head's 4 query heads into
    one tile; unsplit, the unpacked layout gives identical bits (every row's arithmetic is the
    same); in bench.py's configuration (the library's split of each cache: 2 and 9 parts)
    sampled sequences -- the last included, every head -- match the oracle."""
    import variable_length_flash_gb300 as vlf
    w = W.workload(name)
    x = W.make_inputs(w, seed=0, device="cuda", with_dout=False)
    args = (x["q"], x["k"], x["v"], x["cu_seqlens_q"], x["cu_seqlens_kv"], w.max_seqlen_q,
            w.max_seqlen_kv)
    out1, lse1 = vlf.vlf_attn_varlen_fwd(*args, scale=w.scale, causal=True, num_splits=1)
    out2, lse2 = vlf.vlf_attn_varlen_fwd(*args, scale=w.scale, causal=True, num_splits=1,
                                         flags=vlf.VLF_FLAG_NO_PACK)
    assert vlf.vlf_check_error() == 0
    assert torch.equal(out1, out2) and torch.equal(lse1, lse2)
    del out1, lse1, out2, lse2
    # the configuration bench.py times (the library's choice: each cache split in two parts)
    out, lse = vlf.vlf_attn_varlen_fwd(*args, scale=w.scale, causal=True)
    assert vlf.vlf_check_error() == 0
    rng = np.random.default_rng(0)
    seqs = sorted({0, w.num_seqs - 1} | set(int(s) for s in rng.integers(0, w.num_seqs, 4)))
    cq, ck = x["cu_seqlens_q"].tolist(), x["cu_seqlens_kv"].tolist()
    g = w.h_q // w.h_kv
    o_err = l_err = 0.0
    for s in seqs:
        for h in range(w.h_q):
            q = _np(x["q"][cq[s]:cq[s + 1], h])
            k = _np(x["k"][ck[s]:ck[s + 1], h // g])
            v = _np(x["v"][ck[s]:ck[s + 1], h // g])
            o_ref, l_ref = orc.head_forward(q, np.arange(q.shape[0]), k, v, q.shape[0],
                                            w.softmax_scale, True, 0)
            o_err = max(o_err, max_err(_np(out[cq[s]:cq[s + 1], h]), o_ref))
            l_err = max(l_err, max_err(_np(lse[h, cq[s]:cq[s + 1]]), l_ref))
    assert o_err <= TOL["bf16"] and l_err <= LSE_TOL["bf16"], (o_err, l_err)


def test_latent_shared_rope_full_size_equals_plain_calls():
    """latent2x8192_bf16_causal_shared_rope at full size through the split-operand calls (as
    bench.py times it) against the plain calls on the concatenated operands (checked against the
    oracle at full size on the latent workload): identical bits for every output; the shared rope
    key's gradient against the fp32 sum over the 128 heads of the plain call's rope gradients
    (each rounded to bf16 there, so the two differ by that rounding only)."""
    import variable_length_flash_gb300 as vlf
    torch.cuda.empty_cache()
    w = W.workload("latent2x8192_bf16_causal_shared_rope")
    x = W.make_inputs(w, seed=0, device="cuda", with_dout=True)
    ops = [x[n] for n in ("q_nope", "q_rope", "k_nope", "k_rope", "v")]
    cu = (x["cu_seqlens_q"], x["cu_seqlens_kv"], w.max_seqlen_q, w.max_seqlen_kv)
    out, lse = vlf.vlf_attn_varlen_fwd_latent(*ops, *cu, scale=w.scale, causal=True)
    grads = vlf.vlf_attn_varlen_bwd_latent(x["dout"], *ops, out, lse, *cu, scale=w.scale,
                                           causal=True)
    out_c, lse_c = vlf.vlf_attn_varlen_fwd(x["q"], x["k"], x["v"], *cu, scale=w.scale, causal=True)
    dq, dk, dv = vlf.vlf_attn_varlen_bwd(x["dout"], x["q"], x["k"], x["v"], out_c, lse_c, *cu,
                                         scale=w.scale, causal=True)
    assert vlf.vlf_check_error() == 0
    assert torch.equal(out, out_c) and torch.equal(lse, lse_c)
    assert torch.equal(grads[0], dq[..., :128]) and torch.equal(grads[1], dq[..., 128:])
    assert torch.equal(grads[2], dk[..., :128]) and torch.equal(grads[4], dv)
    ref = dk[..., 128:].float().sum(dim=1, keepdim=True)
    err = (grads[3].float() - ref).abs().max().item()
    assert err <= 1e-2 * ref.abs().max().item(), (err, ref.abs().max().item())
    del x, grads, dq, dk, dv
    torch.cuda.empty_cache()
