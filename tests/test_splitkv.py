"""Split-KV forward (small-batch / decode shapes: each CTA's KV band cut into parts whose fp32
results a combine kernel merges by their log-sum-exps).  CPU: the workspace arithmetic and the
library's choice of part count.  GPU: explicit part counts -- packed decode tiles, unpacked
multi-tile rows, window, per-head bias, more parts than tiles (empty parts) -- against the fp64
oracle, the split forward against the unsplit one, and a backward fed by a split forward."""
import pytest
import torch

import variable_length_flash_gb300 as vlf
import workloads as W
from tests.parity import TOL, assert_within, compare, max_err, oracle_run, to_np


def test_split_workspace_size():
    # parts [S, Tq, H, Dv] fp32 and their LSEs [S, H, Tq] fp32, each rounded up to 256 bytes
    assert vlf.vlf_attn_varlen_fwd_split_workspace_size(4, 32, 128, 9) == 9 * 4 * 32 * 128 * 4 + 4608
    assert vlf.vlf_attn_varlen_fwd_split_workspace_size(3, 1, 64, 2) == 1536 + 256
    assert vlf.vlf_attn_varlen_fwd_split_workspace_size(5, 2, 64, 1) == 0
    assert vlf.vlf_attn_varlen_fwd_split_workspace_size(-1, 2, 64, 4) == 0


def test_num_splits_choice():
    f = vlf.vlf_fwd_num_splits
    bf16 = torch.bfloat16
    # 4 decode rows x 8 kv heads (packed tiles: 32 CTAs) on 152 SMs (304 slots): 9 parts
    assert f(4, 1, 32768, 32, 8, 128, 128, bf16, num_sms=152) == 9
    # between one and three waves with a partly empty last wave: 2 or 3 parts, whichever fills
    # its waves better (the fewer on a tie), parts of at least 16 tiles
    assert f(64, 1, 8192, 32, 8, 128, 128, bf16, num_sms=152) == 2    # 512 CTAs: .84 either way
    assert f(40, 1, 16384, 32, 8, 128, 128, bf16, num_sms=152) == 3   # 320: .70 vs .79
    assert f(48, 1, 8192, 32, 8, 128, 128, bf16, num_sms=152) == 3    # 384: .84 vs .95
    assert f(64, 1, 1984, 32, 8, 128, 128, bf16, num_sms=152) == 1    # 31 tiles
    assert f(40, 1, 2048, 32, 8, 128, 128, bf16, num_sms=152) == 2    # 32 tiles: 2 parts at most
    # whole waves, or three waves and more, are not split
    assert f(76, 1, 8192, 32, 8, 128, 128, bf16, num_sms=152) == 1
    assert f(114, 1, 8192, 32, 8, 128, 128, bf16, num_sms=152) == 1
    assert f(4, 4096, 4096, 32, 32, 128, 128, bf16, num_sms=152) == 1
    # parts of at least four 64-key tiles
    assert f(1, 1, 300, 8, 8, 128, 128, bf16, num_sms=152) == 1
    assert f(1, 1, 512, 8, 8, 128, 128, bf16, num_sms=152) == 2
    # width 256: one CTA per SM (152 slots)
    assert f(4, 1, 32768, 32, 8, 256, 256, bf16, num_sms=152) == 4
    # at most 64 parts
    assert f(1, 1, 1 << 20, 1, 1, 64, 64, bf16, num_sms=152) == 64
    # unpacked tiles: 2 row blocks x 4 heads
    assert f(1, 256, 65536, 4, 4, 128, 128, bf16, num_sms=152) == 38
    # shapes without a split path
    assert f(1, 1, 65536, 8, 8, 192, 128, bf16, num_sms=152) == 1
    assert f(1, 1, 65536, 8, 8, 128, 128, torch.float32, num_sms=152) == 1
    assert f(1, 1, 65536, 8, 8, 128, 128, bf16, flags=vlf.VLF_FLAG_FORCE_SIMT, num_sms=152) == 1
    assert f(1, 1, 65536, 8, 8, 256, 128, bf16, num_sms=152) == 1


CASES = {
    # packed decode tiles (G = 4), ragged caches, end-aligned causal
    "bf16_decode_gqa4": (W.custom([1, 1, 1, 1], [1000, 3000, 64, 2500], dtype="bf16", h_q=8,
                                  h_kv=2, d_qk=128, causal=True), (2, 5, 16)),
    # short queries, GQA 2, window across the part boundaries
    "fp16_shortq_window_d64": (W.custom([3, 17], [900, 2000], dtype="fp16", h_q=4, h_kv=2,
                                        d_qk=64, causal=True, window=700), (3, 7)),
    # unpacked tiles (no GQA), two row blocks in one sequence, no mask
    "bf16_d96_two_blocks": (W.custom([130, 5], [2000, 130], dtype="bf16", h_q=2, d_qk=96,
                                     causal=False), (3,)),
    # width 256 (one CTA per SM, 256-column O), packed decode tiles
    "bf16_d256_decode": (W.custom([1, 1, 2], [2000, 700, 3000], dtype="bf16", h_q=8, h_kv=2,
                                  d_qk=256, causal=True), (3, 9)),
    # more parts than the band has tiles: empty parts
    "bf16_parts_exceed_tiles": (W.custom([1, 2], [100, 40], dtype="bf16", h_q=4, h_kv=1,
                                         d_qk=128, causal=True), (8, 64)),
}


def _run(w, x, splits, with_lse=True):
    g = {k: (t.cuda() if isinstance(t, torch.Tensor) else t) for k, t in x.items()}
    out, lse = vlf.vlf_attn_varlen_fwd(g["q"], g["k"], g["v"], g["cu_seqlens_q"],
                                       g["cu_seqlens_kv"], w.max_seqlen_q, w.max_seqlen_kv,
                                       scale=w.scale, causal=w.causal, window=w.window,
                                       bias=g["bias"], num_splits=splits)
    assert vlf.vlf_check_error() == 0
    return {"out": out, "lse": lse}


@pytest.mark.gpu
@pytest.mark.parametrize("name", list(CASES))
def test_split_forward_matches_oracle(name):
    w, counts = CASES[name]
    x = W.make_inputs(w, seed=31, with_dout=False)
    ref = oracle_run(w, x, backward=False)
    one = _run(w, x, 1)
    for s in counts:
        gpu = _run(w, x, s)
        assert_within(compare(w, gpu, ref, keys=["out", "lse"]), f"{name} splits={s}")
        # the same softmax summed in another order: close to the unsplit result
        assert max_err(to_np(gpu["out"]), to_np(one["out"])) <= 2 * TOL[w.dtype]
        assert max_err(to_np(gpu["lse"]), to_np(one["lse"])) <= 1e-3


@pytest.mark.gpu
@pytest.mark.parametrize("heads", [1, 8])
def test_split_forward_with_bias(heads):
    w = W.custom([1, 3, 1], [700, 1200, 64], dtype="fp16", h_q=8, h_kv=2, d_qk=128, causal=True)
    x = W.make_inputs(w, seed=32, with_dout=False)
    g = torch.Generator("cpu").manual_seed(33)
    b = torch.randn((w.total_q, heads, w.max_seqlen_kv), generator=g)
    b[torch.rand(b.shape, generator=g) < 0.2] = float("-inf")
    x["bias"] = b.contiguous()
    ref = oracle_run(w, x, backward=False)
    for s in (4, 11):
        assert_within(compare(w, _run(w, x, s), ref, keys=["out", "lse"]), f"bias{heads} {s}")


@pytest.mark.gpu
def test_split_forward_auto_and_backward():
    """num_splits=None splits this shape (2 sequences x 2 kv heads of packed decode tiles); the
    backward of its output, fed its LSE, matches the oracle."""
    w = W.custom([1, 2], [3000, 1500], dtype="bf16", h_q=8, h_kv=2, d_qk=128, causal=True)
    assert vlf.vlf_fwd_num_splits(w.num_seqs, w.max_seqlen_q, w.max_seqlen_kv, w.h_q, w.h_kv,
                                  w.d_qk, w.d_v, torch.bfloat16) > 1
    x = W.make_inputs(w, seed=34, with_dout=True)
    g = {k: (t.cuda() if isinstance(t, torch.Tensor) else t) for k, t in x.items()}
    n0 = vlf.vlf_launch_count()
    out, lse = vlf.vlf_attn_varlen_fwd(g["q"], g["k"], g["v"], g["cu_seqlens_q"],
                                       g["cu_seqlens_kv"], w.max_seqlen_q, w.max_seqlen_kv,
                                       scale=w.scale, causal=True)
    assert vlf.vlf_launch_count() - n0 == 2  # the parts and their combine
    dq, dk, dv = vlf.vlf_attn_varlen_bwd(g["dout"], g["q"], g["k"], g["v"], out, lse,
                                         g["cu_seqlens_q"], g["cu_seqlens_kv"], w.max_seqlen_q,
                                         w.max_seqlen_kv, scale=w.scale, causal=True)
    assert vlf.vlf_check_error() == 0
    ref = oracle_run(w, x)
    assert_within(compare(w, {"out": out, "lse": lse, "dq": dq, "dk": dk, "dv": dv}, ref),
                  "auto split + backward")


@pytest.mark.gpu
def test_split_workspace_too_small_is_refused():
    w, _ = CASES["bf16_decode_gqa4"]
    x = W.make_inputs(w, seed=35, with_dout=False)
    g = {k: (t.cuda() if isinstance(t, torch.Tensor) else t) for k, t in x.items()}
    need = vlf.vlf_attn_varlen_fwd_split_workspace_size(w.total_q, w.h_q, w.d_v, 4)
    ws = torch.empty(need - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(vlf.VlfError) as e:
        vlf.vlf_attn_varlen_fwd(g["q"], g["k"], g["v"], g["cu_seqlens_q"], g["cu_seqlens_kv"],
                                w.max_seqlen_q, w.max_seqlen_kv, causal=True, num_splits=4,
                                workspace=ws)
    assert e.value.status == vlf.VLF_ERR_WORKSPACE
