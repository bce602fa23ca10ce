"""Latent attention with split operands (triton-msl part 2, "Latent attention": a 128-wide nope
and a 64-wide rope query-key product, summed; output width 128), the rope key per kv head or
shared by all heads.  CPU: workspace arithmetic and the refusals the C ABI makes before touching
a device.  GPU: the split-operand calls against the fp64 oracle on the concatenated operands
(the shared rope key's gradient is the sum over heads of each head's), and bit-identity with
the concatenated-operand calls where the arithmetic is the same."""
import numpy as np
import pytest
import torch

import variable_length_flash_gb300 as vlf
import workloads as W
from tests.parity import LSE_TOL, TOL, max_err, oracle_run, to_np


def test_latent_workspace_size():
    f = vlf.vlf_attn_varlen_bwd_latent_workspace_size
    # row dot products [h_q, total_q] fp32, rounded up to 256 bytes
    assert f(100, 300, 4, 4, 4, torch.bfloat16) == 1792
    assert f(100, 300, 4, 1, 1, torch.bfloat16) == 1792           # one kv head: rope written directly
    # shared rope key over 4 kv heads: + per-head fp32 rope gradients [4, 300, 64]
    assert f(100, 300, 4, 4, 1, torch.bfloat16) == 1792 + 4 * 300 * 64 * 4
    assert f(-1, 300, 4, 4, 1, torch.bfloat16) == 0


def _fwd_latent_raw(**over):
    """A forward call with fake (aligned, never dereferenced) device addresses: only the host
    checks run, so it may be called without a GPU as long as a check refuses it."""
    a = dict(q_nope=0x10000, q_rope=0x20000, k_nope=0x30000, k_rope=0x40000, v=0x50000,
             cu_q=0x60000, cu_kv=0x70000, num_seqs=1, total_q=8, total_kv=8, max_q=8, max_kv=8,
             h_q=4, h_kv=2, rope_heads=1, d_nope=128, d_rope=64, d_v=128, dtype=1, scale=0.0,
             causal=0, window=0, bias=None, bias_heads=0, out=0x80000, lse=0x90000, stream=None,
             flags=0)
    a.update(over)
    return vlf._lib.vlf_attn_varlen_fwd_latent(*a.values())


def test_latent_refusals_without_gpu():
    assert _fwd_latent_raw(d_nope=96) == vlf.VLF_ERR_UNSUPPORTED       # only 128 / 64 / 128
    assert _fwd_latent_raw(d_rope=32) == vlf.VLF_ERR_UNSUPPORTED
    assert _fwd_latent_raw(d_v=64) == vlf.VLF_ERR_UNSUPPORTED
    assert _fwd_latent_raw(dtype=2) == vlf.VLF_ERR_UNSUPPORTED         # no fp32 split path
    assert _fwd_latent_raw(flags=vlf.VLF_FLAG_FORCE_SIMT) == vlf.VLF_ERR_UNSUPPORTED
    assert _fwd_latent_raw(rope_heads=3) == vlf.VLF_ERR_INVALID        # 1 or h_kv
    assert _fwd_latent_raw(k_rope=None) == vlf.VLF_ERR_INVALID
    assert _fwd_latent_raw(q_rope=0x20008) == vlf.VLF_ERR_ALIGN
    assert _fwd_latent_raw(h_kv=3) == vlf.VLF_ERR_INVALID              # 4 % 3


CASES = {
    # shared rope key, GQA 2, causal, ragged lengths with an empty and a one-token sequence
    "bf16_shared_rope_gqa": W.custom([129, 1, 300, 0, 64], dtype="bf16", h_q=4, h_kv=2, d_qk=192,
                                     d_v=128, causal=True, latent_split=(128, 64), rope_heads=1),
    # rope key per kv head, window
    "fp16_rope_per_head_window": W.custom([200, 77], dtype="fp16", h_q=2, h_kv=2, d_qk=192,
                                          d_v=128, causal=True, window=50,
                                          latent_split=(128, 64), rope_heads=2),
    # shared rope key over four kv heads, cross lengths, no mask
    "bf16_shared_rope_cross": W.custom([70, 140], [150, 33], dtype="bf16", h_q=4, h_kv=4,
                                       d_qk=192, d_v=128, causal=False, latent_split=(128, 64),
                                       rope_heads=1),
}


def _latent_run(w, g, bias=None):
    args = (g["q_nope"], g["q_rope"], g["k_nope"], g["k_rope"], g["v"])
    kw = dict(scale=w.scale, causal=w.causal, window=w.window, bias=bias)
    out, lse = vlf.vlf_attn_varlen_fwd_latent(*args, g["cu_seqlens_q"], g["cu_seqlens_kv"],
                                              w.max_seqlen_q, w.max_seqlen_kv, **kw)
    grads = vlf.vlf_attn_varlen_bwd_latent(g["dout"], *args, out, lse, g["cu_seqlens_q"],
                                           g["cu_seqlens_kv"], w.max_seqlen_q, w.max_seqlen_kv,
                                           **kw)
    assert vlf.vlf_check_error() == 0
    return out, lse, grads


def _expected(w, ref):
    """The split gradients from the oracle's gradients of the concatenated operands: the shared
    rope key's is the sum over kv heads (the broadcast's adjoint)."""
    dq, dk = ref["dq"], ref["dk"]
    dk_rope = dk[..., 128:]
    if w.rope_heads == 1:
        dk_rope = dk_rope.sum(axis=1, keepdims=True)
    return [dq[..., :128], dq[..., 128:], dk[..., :128], dk_rope, ref["dv"]]


def _check_against_oracle(w, x, label):
    g = {k: (t.cuda() if isinstance(t, torch.Tensor) else t) for k, t in x.items()}
    out, lse, grads = _latent_run(w, g)
    ref = oracle_run(w, x)
    tol = TOL[w.dtype]
    assert max_err(to_np(out), ref["out"]) <= tol, label
    assert max_err(to_np(lse), ref["lse"]) <= LSE_TOL[w.dtype], label
    names = ["dq_nope", "dq_rope", "dk_nope", "dk_rope", "dv"]
    for n, got, exp in zip(names, grads, _expected(w, ref)):
        # a shared rope key sums h_kv heads' gradients (their errors add)
        lim = 3 * tol * (w.h_kv if n == "dk_rope" and w.rope_heads == 1 else 1)
        assert max_err(to_np(got), exp) <= lim, (label, n, max_err(to_np(got), exp), lim)


@pytest.mark.gpu
@pytest.mark.parametrize("name", list(CASES))
def test_latent_split_matches_oracle(name):
    w = CASES[name]
    _check_against_oracle(w, W.make_inputs(w, seed=41, with_dout=True), name)


@pytest.mark.gpu
def test_latent_split_fuzz():
    """Random lengths (empty sequences included), GQA, rope key shared or per kv head, causal,
    window, dtype: every call matches the oracle."""
    rng = np.random.default_rng(77)
    for trial in range(8):
        n = int(rng.integers(1, 4))
        lq = [int(v) for v in rng.integers(0, 180, n)]
        lk = lq if rng.random() < 0.6 else [int(v) for v in rng.integers(0, 180, n)]
        if sum(lq) == 0 or sum(lk) == 0:
            continue
        hkv = int(rng.choice([1, 2, 4]))
        hq = hkv * int(rng.choice([1, 2]))
        w = W.custom(lq, lk, dtype=str(rng.choice(["fp16", "bf16"])), h_q=hq, h_kv=hkv, d_qk=192,
                     d_v=128, causal=bool(rng.random() < 0.6), window=int(rng.choice([0, 0, 9, 64])),
                     latent_split=(128, 64), rope_heads=1 if rng.random() < 0.6 else hkv)
        _check_against_oracle(w, W.make_inputs(w, seed=200 + trial, with_dout=True), f"fuzz {trial} {w}")


@pytest.mark.gpu
@pytest.mark.parametrize("name", list(CASES))
def test_latent_split_equals_concatenated(name):
    """The split-operand calls put the same values in shared memory as the concatenated calls:
    identical bits for every output but a shared rope key's gradient (summed in fp32 before
    rounding, where the concatenated call rounds each head's)."""
    w = CASES[name]
    x = W.make_inputs(w, seed=42, with_dout=True)
    g = {k: (t.cuda() if isinstance(t, torch.Tensor) else t) for k, t in x.items()}
    out, lse, grads = _latent_run(w, g)
    kw = dict(scale=w.scale, causal=w.causal, window=w.window)
    out_c, lse_c = vlf.vlf_attn_varlen_fwd(g["q"], g["k"], g["v"], g["cu_seqlens_q"],
                                           g["cu_seqlens_kv"], w.max_seqlen_q, w.max_seqlen_kv,
                                           **kw)
    dq, dk, dv = vlf.vlf_attn_varlen_bwd(g["dout"], g["q"], g["k"], g["v"], out_c, lse_c,
                                         g["cu_seqlens_q"], g["cu_seqlens_kv"], w.max_seqlen_q,
                                         w.max_seqlen_kv, **kw)
    assert torch.equal(out, out_c) and torch.equal(lse, lse_c)
    assert torch.equal(grads[0], dq[..., :128]) and torch.equal(grads[1], dq[..., 128:])
    assert torch.equal(grads[2], dk[..., :128]) and torch.equal(grads[4], dv)
    if w.rope_heads != 1 or w.h_kv == 1:
        assert torch.equal(grads[3], dk[..., 128:])


@pytest.mark.gpu
def test_latent_split_with_bias():
    w = W.custom([90, 1, 130], dtype="bf16", h_q=4, h_kv=2, d_qk=192, d_v=128, causal=True,
                 latent_split=(128, 64), rope_heads=1)
    x = W.make_inputs(w, seed=43, with_dout=True)
    gen = torch.Generator("cpu").manual_seed(44)
    b = torch.randn((w.total_q, w.h_q, w.max_seqlen_kv), generator=gen)
    b[torch.rand(b.shape, generator=gen) < 0.1] = float("-inf")
    x["bias"] = b.contiguous()
    g = {k: (t.cuda() if isinstance(t, torch.Tensor) else t) for k, t in x.items()}
    out, lse, grads = _latent_run(w, g, bias=g["bias"])
    ref = oracle_run(w, x)
    tol = TOL[w.dtype]
    assert max_err(to_np(out), ref["out"]) <= tol
    for n, got, exp in zip(range(5), grads, _expected(w, ref)):
        lim = 3 * tol * (w.h_kv if n == 3 else 1)
        assert max_err(to_np(got), exp) <= lim, (n, max_err(to_np(got), exp))


@pytest.mark.gpu
def test_latent_empty_problems():
    """No keys at all: O = 0, LSE = -inf, zero gradients; no queries: zero dK / dV."""
    w = W.custom([3, 2], [0, 0], dtype="bf16", h_q=2, h_kv=2, d_qk=192, d_v=128,
                 latent_split=(128, 64), rope_heads=1)
    x = W.make_inputs(w, seed=45, with_dout=True)
    g = {k: (t.cuda() if isinstance(t, torch.Tensor) else t) for k, t in x.items()}
    out, lse, grads = _latent_run(w, g)
    assert torch.count_nonzero(out) == 0 and bool(torch.all(lse == float("-inf")))
    assert all(torch.count_nonzero(t) == 0 for t in grads)
    w2 = W.custom([0, 0], [5, 9], dtype="fp16", h_q=2, h_kv=1, d_qk=192, d_v=128,
                  latent_split=(128, 64), rope_heads=1)
    x2 = W.make_inputs(w2, seed=46, with_dout=True)
    g2 = {k: (t.cuda() if isinstance(t, torch.Tensor) else t) for k, t in x2.items()}
    _, _, grads2 = _latent_run(w2, g2)
    assert all(torch.count_nonzero(t) == 0 for t in grads2)
