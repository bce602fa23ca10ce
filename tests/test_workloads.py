"""The seeded input generators: shapes, determinism and the long-context bias values."""
import math

import torch

import workloads as W


def test_named_workload_shapes():
    w = W.workload("varlen64_fp16_full")
    assert w.lengths_q == [17, 64, 100, 255] and w.total_q == 436 and w.d_qk == 64
    x = W.make_inputs(w)
    assert x["q"].shape == (436, 4, 64) and x["q"].dtype == torch.float16
    assert x["cu_seqlens_q"].tolist() == [0, 17, 81, 181, 436]
    w = W.workload("latent2x8192_bf16_causal")
    assert (w.d_qk, w.d_v, w.h_q, w.h_kv) == (192, 128, 128, 128)
    assert abs(w.softmax_scale - 1 / math.sqrt(192)) < 1e-15
    w = W.workload("ragged64_gqa_window_bf16")
    assert len(w.lengths_q) == 64 and all(128 <= L <= 8192 for L in w.lengths_q)
    assert (w.h_q, w.h_kv, w.window) == (32, 8, 4096)


def test_determinism():
    w = W.custom([5, 7], h_q=2, d_qk=16)
    a, b = W.make_inputs(w, seed=3), W.make_inputs(w, seed=3)
    assert all(torch.equal(a[k], b[k]) for k in ("q", "k", "v", "dout"))
    c = W.make_inputs(w, seed=4)
    assert not torch.equal(a["q"], c["q"])


def test_long_context_bias_values():
    w = W.workload("long49152_fp16_bias_alibi")
    rows = torch.tensor([0, 100, 10000, 49151])
    b = W.bias_block(w, rows, [0, 1, 2, 15])
    assert b.shape == (4, 4, 49152) and b.dtype == torch.float32
    # prefix keys 0..8191 always visible; beyond the prefix only keys <= query
    assert b[0, 0, 8191].item() == -8191.0 and b[0, 0, 8192].item() == float("-inf")
    assert b[2, 0, 10000].item() == 0.0 and b[2, 0, 10001].item() == float("-inf")
    assert b[2, 0, 0].item() == -10000.0
    # head 2: slope 2^(-8*2/16) = 1/2; head 1: 2^(-1/2); head 15: 2^(-7.5)
    assert b[1, 2, 0].item() == -50.0
    assert b[3, 1, 49151 - 3].item() == torch.tensor(-3 * 2 ** -0.5, dtype=torch.float32).item()
    assert b[3, 3, 0].item() == torch.tensor(-49151 * 2 ** -7.5, dtype=torch.float32).item()
    p = W.bias_block(W.workload("long49152_fp16_bias_prefix"), rows, [0])
    assert p.shape == (4, 1, 49152)
    assert p[1, 0, 8191].item() == 0.0 and p[1, 0, 8192].item() == float("-inf")
    assert p[3, 0, 49151].item() == 0.0


def test_sample_rows_include_sequence_tails():
    w = W.custom([5, 9, 3])
    rows = W.sample_rows(w, 4, seed=0, tail=2)
    for r in (3, 4, 12, 13, 15, 16):
        assert r in rows


def test_pair_counts_match_brute_force_masks():
    """The closed-form pair counter used for TFLOP/s equals counting the oracle's masks."""
    import numpy as np

    from oracle import attention as orc
    from variable_length_flash_gb300 import flops
    for q_len, kv_len in ((1, 1), (17, 17), (100, 255), (255, 100), (64, 64)):
        for causal, window in ((False, 0), (True, 0), (True, 1), (True, 7), (False, 5)):
            want = int(orc.visible(q_len, kv_len, causal, window).sum())
            assert flops.visible_pairs(q_len, kv_len, causal, window) == want
    # the forward-only varlen workload: sums of L^2 and L(L+1)/2 over {17, 64, 100, 255}, 4 heads
    assert flops.workload_pairs(W.workload("varlen64_fp16_full")) == 317_640
    assert flops.workload_pairs(W.workload("varlen64_fp16_causal")) == 159_692
    assert flops.workload_pairs(W.workload("dense4x4096_bf16_causal")) == 4 * 32 * 4096 * 4097 // 2
    # prefix-LM pairs: key <= 8191 or key <= query, counted from the generated bias
    w = W.workload("long49152_fp16_bias_prefix")
    rows = torch.arange(0, 49152, 997)
    b = W.bias_block(w, rows, [0])
    got = int(torch.isfinite(b).sum())
    want = int(sum(min(49152, max(8192, int(r) + 1)) for r in rows))
    assert got == want
    assert flops.workload_pairs(w) == 16 * sum(min(49152, max(8192, i + 1)) for i in range(49152))
    assert flops.flops_per_pair(128, 128) == {"fwd": 512, "bwd": 1280, "fwd_bwd": 1792,
                                              "dkdv": 1024, "dq": 768}
    assert flops.flops_per_pair(192, 128)["fwd_bwd"] == 2304
