"""The backward entry point that allocates nothing (vlf_attn_varlen_bwd_noalloc).

It is for callers that cannot allocate device memory when they call -- a plugin whose enqueue
hook may not allocate, a service with its memory budget reserved up front, or code that must not
trigger the device-wide synchronisation cudaMalloc / cudaFree can cause.  Its workspace is a
fixed array inside the library, so this test checks that, called twice in a row through the C
ABI, it returns the same gradients as the regular entry point (which takes a caller-allocated
workspace).  Both run the same kernels on the same inputs, so the gradients must be identical
bit for bit; the second call draws new inputs, so a stale array would show.  This file is collected last so a failure here cannot
hide the result of any other test; it also passes when run alone in a fresh process.
"""
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu


def _inputs(w, seed):
    x = W.make_inputs(w, seed=seed, with_dout=True)
    return {k: (t.cuda() if isinstance(t, torch.Tensor) else t) for k, t in x.items()}


@pytest.mark.parametrize("case", ["bf16_gqa_causal", "fp16_latent_window"])
def test_noalloc_backward_matches_regular_twice(case):
    import variable_length_flash_gb300 as vlf
    if case == "bf16_gqa_causal":
        w = W.custom([300, 17, 129, 64], dtype="bf16", h_q=4, h_kv=2, d_qk=128, causal=True)
    else:
        w = W.custom([200, 1, 257], dtype="fp16", h_q=2, h_kv=1, d_qk=192, d_v=128, causal=True,
                     window=40)
    assert vlf.vlf_noalloc_scratch_bytes() >= 4 * w.h_q * w.total_q
    for call in range(2):
        g = _inputs(w, seed=40 + call)
        common = dict(scale=w.scale, causal=w.causal, window=w.window)
        out, lse = vlf.vlf_attn_varlen_fwd(g["q"], g["k"], g["v"], g["cu_seqlens_q"],
                                           g["cu_seqlens_kv"], w.max_seqlen_q, w.max_seqlen_kv,
                                           **common)
        ref = vlf.vlf_attn_varlen_bwd(g["dout"], g["q"], g["k"], g["v"], out, lse,
                                      g["cu_seqlens_q"], g["cu_seqlens_kv"], w.max_seqlen_q,
                                      w.max_seqlen_kv, **common)
        got = vlf.vlf_attn_varlen_bwd_noalloc(g["dout"], g["q"], g["k"], g["v"], out, lse,
                                              g["cu_seqlens_q"], g["cu_seqlens_kv"],
                                              w.max_seqlen_q, w.max_seqlen_kv, **common)
        assert vlf.vlf_check_error() == 0
        for name, a, b in zip(("dq", "dk", "dv"), got, ref):
            assert torch.isfinite(a).all(), (call, name)
            assert torch.equal(a, b), (call, name, float((a.double() - b.double()).abs().max()))


def test_noalloc_refuses_problems_beyond_its_array():
    import variable_length_flash_gb300 as vlf
    limit_floats = vlf.vlf_noalloc_scratch_bytes() // 4
    # h_q * total_q one past the array: refused on the host, nothing is read or launched
    total_q = limit_floats // 8 + 1
    st = vlf._lib.vlf_attn_varlen_bwd_noalloc(
        16, 16, 16, 16, 16, 16, 16, 16, 1, total_q, total_q, total_q, total_q, 8, 8, 64, 64,
        vlf.VLF_BF16, 0.0, 0, 0, None, 0, 16, 16, 16, None)
    assert st == vlf.VLF_ERR_UNSUPPORTED
