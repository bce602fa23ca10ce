"""The differentiable entry points (mtlattn 0.3.0, "Use": ``varlen_attention`` with window and
additive bias / bool mask, the flash_attn-compatible packed wrappers).  CPU: the argument
conversions and refusals.  GPU: autograd through the library's kernels against the fp64 oracle,
and the packed wrappers against direct calls of the C ABI (bit-identical: same kernels, same
values)."""
import pytest
import torch

import variable_length_flash_gb300 as vlf
import workloads as W
from variable_length_flash_gb300.functional import mask_to_bias, window_from_flash


def test_mask_to_bias():
    m = torch.tensor([[True, False], [False, True]])
    b = mask_to_bias(m)
    assert b.dtype == torch.float32
    assert b[0, 0] == 0 and b[1, 1] == 0
    assert b[0, 1] == float("-inf") and b[1, 0] == float("-inf")
    f = torch.ones(3, dtype=torch.float64)
    assert mask_to_bias(f).dtype == torch.float32


def test_window_from_flash():
    assert window_from_flash((-1, -1), True) == 0
    assert window_from_flash(None, False) == 0
    assert window_from_flash((4095, 0), True) == 4096       # the last 4096 keys
    assert window_from_flash((0, 0), True) == 1             # the diagonal alone
    assert window_from_flash((7, -1), False) == 8           # lower bound only
    for bad, causal in (((3, 2), True), ((3, 0), False), ((-1, 5), False)):
        with pytest.raises(vlf.VlfError):
            window_from_flash(bad, causal)


def test_refusals_without_gpu():
    x = torch.zeros(4, 3, 2, 64)
    cu = torch.tensor([0, 4], dtype=torch.int32)
    with pytest.raises(vlf.VlfError):
        vlf.flash_attn_varlen_qkvpacked_func(x, cu, 4, dropout_p=0.1)
    with pytest.raises(vlf.VlfError):
        vlf.flash_attn_varlen_qkvpacked_func(x, cu, 4, alibi_slopes=torch.ones(2))
    with pytest.raises(vlf.VlfError):
        vlf.flash_attn_varlen_qkvpacked_func(x[:, :2], cu, 4)   # not [T, 3, H, D]
    q = torch.zeros(4, 2, 64)
    b = torch.zeros(4, 1, 4, requires_grad=True)
    with pytest.raises(vlf.VlfError):
        vlf.varlen_attention(q, q, q, cu, cu, 4, attn_bias=b)


def _case(dtype="bf16", causal=True, window=0, h_q=4, h_kv=2, d=128):
    w = W.custom([70, 1, 140, 129], dtype=dtype, h_q=h_q, h_kv=h_kv, d_qk=d, causal=causal,
                 window=window)
    x = W.make_inputs(w, seed=21, device="cuda", with_dout=True)
    return w, x


@pytest.mark.gpu
@pytest.mark.parametrize("dtype,causal,window", [("bf16", True, 0), ("fp16", True, 33),
                                                 ("bf16", False, 0)])
def test_varlen_attention_autograd_matches_oracle(dtype, causal, window):
    from tests.parity import assert_within, compare, oracle_run, to_np
    w, x = _case(dtype, causal, window)
    q, k, v = (x[n].clone().requires_grad_(True) for n in ("q", "k", "v"))
    out = vlf.varlen_attention(q, k, v, x["cu_seqlens_q"], x["cu_seqlens_kv"], w.max_seqlen_q,
                               w.max_seqlen_kv, scale=w.scale, causal=causal, window=window)
    out.backward(x["dout"])
    assert vlf.vlf_check_error() == 0
    xc = {n: (t.cpu() if isinstance(t, torch.Tensor) else t) for n, t in x.items()}
    ref = oracle_run(w, xc)
    gpu = {"out": out, "dq": q.grad, "dk": k.grad, "dv": v.grad}
    assert_within(compare(w, gpu, ref, keys=["out", "dq", "dk", "dv"]), "varlen_attention")


@pytest.mark.gpu
def test_packed_wrappers_match_direct_calls():
    w, x = _case("bf16", True, 0, h_q=2, h_kv=2)
    cu = x["cu_seqlens_q"]
    out_ref, lse = vlf.vlf_attn_varlen_fwd(x["q"], x["k"], x["v"], cu, cu, w.max_seqlen_q,
                                           w.max_seqlen_kv, scale=w.scale, causal=True)
    dq, dk, dv = vlf.vlf_attn_varlen_bwd(x["dout"], x["q"], x["k"], x["v"], out_ref, lse, cu, cu,
                                         w.max_seqlen_q, w.max_seqlen_kv, scale=w.scale,
                                         causal=True)
    # qkv-packed: one tensor, gradient lands in its three slices
    qkv = torch.stack([x["q"], x["k"], x["v"]], dim=1).requires_grad_(True)
    out = vlf.flash_attn_varlen_qkvpacked_func(qkv, cu, w.max_seqlen_q, softmax_scale=w.scale,
                                               causal=True)
    out.backward(x["dout"])
    assert torch.equal(out, out_ref)
    assert torch.equal(qkv.grad[:, 0], dq) and torch.equal(qkv.grad[:, 1], dk)
    assert torch.equal(qkv.grad[:, 2], dv)
    # kv-packed
    qg = x["q"].clone().requires_grad_(True)
    kv = torch.stack([x["k"], x["v"]], dim=1).requires_grad_(True)
    out2 = vlf.flash_attn_varlen_kvpacked_func(qg, kv, cu, cu, w.max_seqlen_q, w.max_seqlen_kv,
                                               softmax_scale=w.scale, causal=True)
    out2.backward(x["dout"])
    assert torch.equal(out2, out_ref)
    assert torch.equal(qg.grad, dq) and torch.equal(kv.grad[:, 0], dk)
    assert torch.equal(kv.grad[:, 1], dv)
    # separate tensors, flash_attn window convention (left, 0) == window left + 1
    out3 = vlf.flash_attn_varlen_func(x["q"], x["k"], x["v"], cu, cu, w.max_seqlen_q,
                                      w.max_seqlen_kv, softmax_scale=w.scale, causal=True,
                                      window_size=(15, 0))
    out4, _ = vlf.vlf_attn_varlen_fwd(x["q"], x["k"], x["v"], cu, cu, w.max_seqlen_q,
                                      w.max_seqlen_kv, scale=w.scale, causal=True, window=16)
    assert torch.equal(out3, out4)
    assert vlf.vlf_check_error() == 0


@pytest.mark.gpu
def test_bool_mask_equals_additive_bias_and_oracle():
    from tests.parity import assert_within, compare, oracle_run
    w, x = _case("fp16", False, 0, h_q=4, h_kv=2, d=64)
    g = torch.Generator("cpu").manual_seed(3)
    mask = torch.rand((w.total_q, 1, w.max_seqlen_kv), generator=g) < 0.7
    mask[:, :, 0] = True                      # every row keeps a key
    mask_d = mask.cuda()
    q, k, v = (x[n].clone().requires_grad_(True) for n in ("q", "k", "v"))
    out = vlf.varlen_attention(q, k, v, x["cu_seqlens_q"], x["cu_seqlens_kv"], w.max_seqlen_q,
                               scale=w.scale, attn_bias=mask_d)
    out.backward(x["dout"])
    bias = torch.zeros(mask.shape).masked_fill_(~mask, float("-inf"))
    direct, _ = vlf.vlf_attn_varlen_fwd(x["q"], x["k"], x["v"], x["cu_seqlens_q"],
                                        x["cu_seqlens_kv"], w.max_seqlen_q, w.max_seqlen_kv,
                                        scale=w.scale, bias=bias.cuda())
    assert torch.equal(out.detach(), direct)
    xc = {n: (t.cpu() if isinstance(t, torch.Tensor) else t) for n, t in x.items()}
    xc["bias"] = bias
    ref = oracle_run(w, xc)
    gpu = {"out": out, "dq": q.grad, "dk": k.grad, "dv": v.grad}
    assert_within(compare(w, gpu, ref, keys=["out", "dq", "dk", "dv"]), "bool mask")


@pytest.mark.gpu
def test_latent_attention_autograd_equals_direct_calls():
    """latent_attention: autograd over the split-operand calls (a rope key shared by the heads
    gets the sum of their gradients)."""
    w = W.custom([70, 1, 130], dtype="bf16", h_q=4, h_kv=2, d_qk=192, d_v=128, causal=True,
                 latent_split=(128, 64), rope_heads=1)
    x = W.make_inputs(w, seed=22, device="cuda", with_dout=True)
    names = ("q_nope", "q_rope", "k_nope", "k_rope", "v")
    leaves = [x[n].clone().requires_grad_(True) for n in names]
    out = vlf.latent_attention(*leaves, x["cu_seqlens_q"], x["cu_seqlens_kv"], w.max_seqlen_q,
                               w.max_seqlen_kv, causal=True)
    out.backward(x["dout"])
    o, lse = vlf.vlf_attn_varlen_fwd_latent(*(x[n] for n in names), x["cu_seqlens_q"],
                                            x["cu_seqlens_kv"], w.max_seqlen_q, w.max_seqlen_kv,
                                            causal=True)
    grads = vlf.vlf_attn_varlen_bwd_latent(x["dout"], *(x[n] for n in names), o, lse,
                                           x["cu_seqlens_q"], x["cu_seqlens_kv"], w.max_seqlen_q,
                                           w.max_seqlen_kv, causal=True)
    assert vlf.vlf_check_error() == 0
    assert torch.equal(out.detach(), o)
    for leaf, g in zip(leaves, grads):
        assert torch.equal(leaf.grad, g)
