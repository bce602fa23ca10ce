"""GPU vs fp64 oracle, every element, on small varlen problems that still span several tiles
and ragged tails: dtypes x {self, cross} x {causal, window, GQA/MQA, bias dim1 in {1, H}} x head
widths {64, 96, 128, 192/128, 256, odd}, lengths including 0, 1, 15-17, 127-129 and thousands of tiny
windows.  Also: tile skipping is exact (skip on/off give identical bits), bad cu_seqlens are
reported through the device error word, and the SIMT and tensor-core paths both pass."""
import numpy as np
import pytest
import torch

import workloads as W
from tests.parity import (TOL, assert_within, compare, gpu_run, grad_error_bound, oracle_run,
                          to_np)

pytestmark = pytest.mark.gpu

ODD = [1, 15, 16, 17, 127, 128, 129, 0, 300]

CASES = {
    "varlen64_fp16_full": W.workload("varlen64_fp16_full"),
    "varlen64_fp16_causal": W.workload("varlen64_fp16_causal"),
    "bf16_d128_gqa_causal_odd": W.custom(ODD, dtype="bf16", h_q=4, h_kv=2, d_qk=128, causal=True),
    "fp16_d128_full_odd": W.custom(ODD, dtype="fp16", h_q=2, d_qk=128),
    "bf16_latent_192_128": W.custom([129, 64, 1, 300], dtype="bf16", h_q=2, d_qk=192, d_v=128,
                                    causal=True, scale=1 / 192 ** 0.5),
    "fp16_d128_window16": W.custom([200, 33, 257], dtype="fp16", h_q=2, d_qk=128, causal=True,
                                   window=16),
    "bf16_d64_window1_tiny": W.custom([3, 1, 2, 5] * 6, dtype="bf16", h_q=2, d_qk=64, causal=True,
                                      window=1),
    "fp16_cross_causal": W.custom([5, 100, 64, 130], [70, 30, 64, 129], dtype="fp16", h_q=2,
                                  d_qk=64, causal=True),
    "bf16_cross_full": W.custom([5, 100], [70, 300], dtype="bf16", h_q=2, d_qk=128),
    "bf16_mqa_d128": W.custom([150, 77], dtype="bf16", h_q=8, h_kv=1, d_qk=128, causal=True),
    "fp32_d64_causal": W.custom([17, 64, 100], dtype="fp32", h_q=2, d_qk=64, causal=True),
    "fp32_d40_window": W.custom([50, 90], dtype="fp32", h_q=2, h_kv=1, d_qk=40, d_v=24,
                                causal=True, window=7),
    # fp32 on the tensor cores (products in three tf32 passes): widths 64 and 32, ragged tails,
    # GQA, windows, cross attention
    "fp32_d64_odd_gqa": W.custom(ODD, dtype="fp32", h_q=4, h_kv=2, d_qk=64, causal=True),
    "fp32_d32_window_cross": W.custom([5, 100, 300], [70, 130, 300], dtype="fp32", h_q=2,
                                      d_qk=32, causal=True, window=50),
    "fp32_d64_full_long": W.custom([700, 129], dtype="fp32", h_q=2, h_kv=1, d_qk=64),
    "fp32_d32_decode_mqa": W.custom([1, 3, 1], [200, 64, 1000], dtype="fp32", h_q=4, h_kv=1,
                                    d_qk=32, causal=True),
    "fp16_d96": W.custom([70, 129], dtype="fp16", h_q=2, d_qk=96, causal=True),
    "bf16_d96_gqa_window": W.custom([300, 1, 129, 64], dtype="bf16", h_q=6, h_kv=2, d_qk=96,
                                    causal=True, window=100),
    "fp16_d96_decode_gqa4": W.custom([1, 1, 3], [200, 1, 700], dtype="fp16", h_q=8, h_kv=2,
                                     d_qk=96, causal=True),
    # width 256: tensor-core forward (one CTA per SM, 256-column O) and backward (dV and dK
    # passes, dQ)
    "bf16_d256_gqa_causal": W.custom([129, 1, 300, 64], dtype="bf16", h_q=4, h_kv=2, d_qk=256,
                                     causal=True),
    "fp16_d256_decode_gqa4_window": W.custom([1, 2, 1], [700, 90, 1500], dtype="fp16", h_q=8,
                                             h_kv=2, d_qk=256, causal=True, window=600),
    "fp16_d256_gqa_window_long": W.custom([700, 300, 129], dtype="fp16", h_q=4, h_kv=2,
                                          d_qk=256, causal=True, window=200),
    "bf16_empty_seqs": W.custom([0, 5, 0, 130], [3, 5, 0, 130], dtype="bf16", h_q=2, d_qk=64,
                                causal=False),
    # decode-sized problems (the forward packs a kv head's G query heads into one tile)
    "bf16_decode_gqa4": W.custom([1] * 8, [5, 64, 65, 200, 1, 129, 1000, 3], dtype="bf16",
                                 h_q=8, h_kv=2, d_qk=128, causal=True),
    "fp16_decode_mqa16_window": W.custom([1, 2, 3, 1], [300, 17, 64, 1], dtype="fp16", h_q=16,
                                         h_kv=1, d_qk=64, causal=True, window=40),
    "bf16_shortq_gqa8": W.custom([16, 5, 16], [40, 300, 16], dtype="bf16", h_q=16, h_kv=2,
                                 d_qk=128, causal=True),
    "fp16_decode_gqa2_full": W.custom([1, 1, 2], [33, 700, 2], dtype="fp16", h_q=4, h_kv=2,
                                      d_qk=64, causal=False),
}


def _bias_case(dtype, heads, causal, d, window=0, lengths=(70, 1, 140)):
    w = W.custom(list(lengths), dtype=dtype, h_q=4, h_kv=2, d_qk=d, causal=causal, window=window)
    x = W.make_inputs(w, seed=11, with_dout=True)
    g = torch.Generator("cpu").manual_seed(12)
    b = torch.randn((w.total_q, heads, w.max_seqlen_kv), generator=g)
    b[torch.rand(b.shape, generator=g) < 0.1] = float("-inf")
    b[75, :, :] = float("-inf")          # a row that the bias masks completely
    x["bias"] = b.contiguous()
    return w, x


@pytest.mark.parametrize("name", sorted(CASES))
def test_parity_case(name):
    w = CASES[name]
    x = W.make_inputs(w, seed=5, with_dout=True)
    gpu = gpu_run(w, x)
    ref = oracle_run(w, x)
    assert_within(compare(w, gpu, ref), name)


@pytest.mark.parametrize("dtype,heads,causal,d,window,lengths", [
    ("fp16", 4, False, 64, 0, (70, 1, 140)), ("bf16", 1, True, 128, 0, (70, 1, 140)),
    ("fp16", 4, True, 128, 33, (70, 1, 140)), ("bf16", 4, False, 192, 0, (70, 1, 140)),
    ("fp32", 1, True, 64, 0, (70, 1, 140)),
    # max_seqlen_kv not a multiple of 4: bias rows are read row by row instead of through TMA
    ("bf16", 4, True, 128, 0, (70, 1, 141)),
    # enough items per CTA that both backward kernels' bias rings wrap several times
    ("fp16", 4, True, 96, 0, (300, 1, 257)), ("bf16", 1, False, 64, 0, (384, 129, 200)),
    # width 256: bias rows read by the softmax threads (no room for a bias ring)
    ("bf16", 4, True, 256, 0, (70, 1, 140))])
def test_parity_bias(dtype, heads, causal, d, window, lengths):
    """Bias tiles through TMA (D 64/128, rows 16-byte aligned), row by row otherwise, with the
    heads of a row block run together for a head-broadcast bias."""
    w, x = _bias_case(dtype, heads, causal, d, window, lengths)
    if d == 192:
        w.d_v = 128
        x["v"] = x["v"][:, :, :128].contiguous()
        x["dout"] = x["dout"][:, :, :128].contiguous()
    gpu = gpu_run(w, x)
    ref = oracle_run(w, x)
    assert_within(compare(w, gpu, ref), f"bias {dtype} {heads} {causal} {d}")


@pytest.mark.parametrize("heads", [1, 8])
def test_parity_bias_decode(heads):
    """A bias on a decode-sized problem (packed query heads: each row reads its own head's
    bias row)."""
    w = W.custom([1, 2, 1], [90, 7, 300], dtype="bf16", h_q=8, h_kv=2, d_qk=128, causal=True)
    x = W.make_inputs(w, seed=13, with_dout=True)
    g = torch.Generator("cpu").manual_seed(14)
    b = torch.randn((w.total_q, heads, w.max_seqlen_kv), generator=g)
    b[torch.rand(b.shape, generator=g) < 0.2] = float("-inf")
    x["bias"] = b.contiguous()
    gpu = gpu_run(w, x)
    ref = oracle_run(w, x)
    assert_within(compare(w, gpu, ref), f"decode bias {heads}")


def _outlier_case(dtype):
    """Transformer activations spike to 1e2-1e3 in a few channels (mtlattn 0.3.0,
    "Correctness": the outlier-channel overflow regression): channels 3 and 77 of q and k
    scaled by 300 and -900, so that logits reach 1e4-1e5 and the softmax rows are nearly
    one-hot."""
    w = W.custom([200, 57], dtype=dtype, h_q=2, d_qk=128, causal=True)
    x = W.make_inputs(w, seed=21, with_dout=True)
    for t in ("q", "k"):
        y = x[t].float()
        y[..., 3] *= 300.0
        y[..., 77] *= -900.0
        x[t] = y.to(x[t].dtype)
    return w, x


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_outlier_channels(dtype):
    """fp32 accumulation and the max subtraction keep every output finite and within its gate:
    O at the stated tolerance; LSE and the gradients within the stated tolerance plus their
    fp32 error bounds (the logits are ~1e4-1e5, where an fp32 logit is only good to ~1e-2)."""
    w, x = _outlier_case(dtype)
    gpu = gpu_run(w, x)
    for k in ("out", "lse", "dq", "dk", "dv"):
        assert torch.isfinite(gpu[k]).all(), k
    ref = oracle_run(w, x)
    errs = compare(w, gpu, ref, keys=["out"])
    assert_within(errs, f"outliers {dtype}")
    # LSE sits at |logit| ~ 1e4 here; an fp32 dot product of D terms carries an error of up to
    # D * 2^-24 * sum_c |q_c k_c| (standard bound for recursive summation), times the scale.
    q = x["q"].double().numpy()
    k = x["k"].double().numpy()
    lse_gpu = gpu["lse"].double().cpu().numpy()
    cu = x["cu_seqlens_q"].tolist()
    for s in range(len(cu) - 1):
        a, b = cu[s], cu[s + 1]
        for h in range(w.h_q):
            mag = np.abs(q[a:b, h]) @ np.abs(k[a:b, h]).T         # sum_c |q_ic k_jc|
            bound = 1e-3 + w.softmax_scale * w.d_qk * 2.0 ** -24 * mag.max(axis=1)
            err = np.abs(lse_gpu[h, a:b] - ref["lse"][h, a:b])
            assert np.all(err <= bound), (s, h, float(err.max()), float(bound.min()))
    # gradients, element by element: 3x the O tolerance plus the fp32 / 16-bit rounding bound
    # of each element (tests/parity.py, grad_error_bound)
    bound = grad_error_bound(w, x, gpu["out"])
    for key in ("dq", "dk", "dv"):
        err = np.abs(to_np(gpu[key]) - ref[key])
        gate = 3 * TOL[dtype] + bound[key]
        worst = np.unravel_index(int(np.argmax(err - gate)), err.shape)
        assert np.all(err <= gate), (key, worst, float(err[worst]), float(gate[worst]),
                                     float(ref[key][worst]))


@pytest.mark.parametrize("name", ["bf16_d128_gqa_causal_odd", "fp16_d128_window16",
                                  "varlen64_fp16_causal", "bf16_latent_192_128",
                                  "fp32_d32_window_cross"])
@pytest.mark.parametrize("simt", [False, True])
def test_tile_skipping_is_exact(name, simt):
    """Skipping fully masked KV tiles changes no bit of any output."""
    import variable_length_flash_gb300 as vlf
    w = CASES[name]
    x = W.make_inputs(w, seed=9, with_dout=True)
    base = vlf.VLF_FLAG_FORCE_SIMT if simt else 0
    a = gpu_run(w, x, flags=base)
    b = gpu_run(w, x, flags=base | vlf.VLF_FLAG_NO_SKIP)
    for k in a:
        assert torch.equal(a[k], b[k]), k


@pytest.mark.parametrize("w", [
    W.custom([2048, 1000], dtype="bf16", h_q=8, h_kv=2, d_qk=128, causal=True),
    W.custom([2048, 700], dtype="bf16", h_q=4, d_qk=192, d_v=128, causal=True, scale=1 / 192 ** 0.5),
    W.custom([1024, 300], dtype="bf16", h_q=4, d_qk=256, causal=True),
    W.custom([1500], dtype="fp16", h_q=4, d_qk=64),
], ids=["d128_gqa", "qk192", "d256", "d64_full"])
def test_backward_is_deterministic(w):
    """The kernels hand tiles and TMEM columns between warps through barriers only: repeated
    calls on the same inputs give identical bits (a missing wait shows up as a difference)."""
    x = W.make_inputs(w, seed=17, with_dout=True)
    runs = [gpu_run(w, x) for _ in range(4)]
    for r in runs[1:]:
        for k in runs[0]:
            assert torch.equal(runs[0][k], r[k]), k


def test_fp32_tensor_core_path_is_taken_and_matches_simt():
    """fp32 at widths 32 / 64 runs the three-pass tf32 forward and backward; they and the SIMT
    fp32-FMA kernels all meet the fp32 gates against the oracle."""
    import variable_length_flash_gb300 as vlf
    for d in (32, 64):
        assert vlf.vlf_fwd_path(4, 2, d, d, vlf.VLF_F32) == 1
        assert vlf.vlf_bwd_path(4, 2, d, d, vlf.VLF_F32) == 1
        assert vlf.vlf_fwd_path(4, 2, d, d, vlf.VLF_F32, flags=vlf.VLF_FLAG_FORCE_SIMT) == 0
    w = CASES["fp32_d64_odd_gqa"]
    x = W.make_inputs(w, seed=31, with_dout=True)
    ref = oracle_run(w, x)
    for flags in (0, vlf.VLF_FLAG_FORCE_SIMT):
        gpu = gpu_run(w, x, flags=flags)
        assert_within(compare(w, gpu, ref), f"fp32 flags={flags}")


@pytest.mark.parametrize("name", ["bf16_d128_gqa_causal_odd", "bf16_latent_192_128",
                                  "varlen64_fp16_full"])
def test_simt_path_parity(name):
    """The SIMT fp32-FMA kernels on 16-bit data (the tensor-core kernels' independent twin)."""
    import variable_length_flash_gb300 as vlf
    w = CASES[name]
    x = W.make_inputs(w, seed=6, with_dout=True)
    gpu = gpu_run(w, x, flags=vlf.VLF_FLAG_FORCE_SIMT)
    ref = oracle_run(w, x)
    assert_within(compare(w, gpu, ref), name + " simt")


def test_bad_cu_seqlens_reported_and_device_stays_usable():
    import variable_length_flash_gb300 as vlf
    w = W.custom([10, 20], dtype="bf16", h_q=2, d_qk=64)
    x = W.make_inputs(w, seed=1)
    dev = {k: (t.cuda() if isinstance(t, torch.Tensor) else t) for k, t in x.items()}
    for bad in ([0, 25, 20], [0, 10, 31], [1, 10, 30], [0, 10, 29]):
        cu = torch.tensor(bad, dtype=torch.int32, device="cuda")
        vlf.vlf_attn_varlen_fwd(dev["q"], dev["k"], dev["v"], cu, cu, 30, 30)
        assert vlf.vlf_check_error() == vlf.VLF_ERR_BAD_SEQLENS, bad
    # a sequence longer than max_seqlen_q is refused too (it would not be covered by the grid)
    vlf.vlf_attn_varlen_fwd(dev["q"], dev["k"], dev["v"], dev["cu_seqlens_q"],
                            dev["cu_seqlens_kv"], 12, 20)
    assert vlf.vlf_check_error() == vlf.VLF_ERR_BAD_SEQLENS
    # and the next good call works
    gpu = gpu_run(w, x, backward=False)
    ref = oracle_run(w, x, backward=False)
    assert_within(compare(w, gpu, ref), "after error")


def test_wait_timeout_reported_and_device_stays_usable():
    """The failure path without a fault: with VLF_FLAG_TEST_TIMEOUT the forward's producer never
    loads the query tile, the CTA's bounded waits run out (2 s), the kernel records
    VLF_ERR_TIMEOUT, drains and returns; the next call on the same context is correct."""
    import time
    import variable_length_flash_gb300 as vlf
    w = W.custom([64], dtype="bf16", h_q=1, d_qk=128)  # one CTA
    x = W.make_inputs(w, seed=2)
    dev = {k: (t.cuda() if isinstance(t, torch.Tensor) else t) for k, t in x.items()}
    assert vlf.vlf_check_error() == 0
    t0 = time.time()
    vlf.vlf_attn_varlen_fwd(dev["q"], dev["k"], dev["v"], dev["cu_seqlens_q"],
                            dev["cu_seqlens_kv"], w.max_seqlen_q, w.max_seqlen_kv,
                            flags=vlf.VLF_FLAG_TEST_TIMEOUT, num_splits=1)
    status = vlf.vlf_check_error()
    elapsed = time.time() - t0
    assert status == vlf.VLF_ERR_TIMEOUT, vlf.vlf_status_string(status)
    assert 1.5 < elapsed < 60, elapsed  # the 2 s limit ran out, once
    gpu = gpu_run(w, x, backward=False)
    ref = oracle_run(w, x, backward=False)
    assert_within(compare(w, gpu, ref), "after a timeout")


def test_refuses_grad_requiring_bias():
    import variable_length_flash_gb300 as vlf
    w = W.custom([8], dtype="bf16", h_q=2, d_qk=64)
    x = W.make_inputs(w, seed=1)
    dev = {k: (t.cuda() if isinstance(t, torch.Tensor) else t) for k, t in x.items()}
    b = torch.zeros((8, 1, 8), device="cuda", requires_grad=True)
    with pytest.raises(vlf.VlfError):
        vlf.vlf_attn_varlen_fwd(dev["q"], dev["k"], dev["v"], dev["cu_seqlens_q"],
                                dev["cu_seqlens_kv"], 8, 8, bias=b)


def test_fuzz_correct_or_refuse():
    """Random shapes and flags: every call either matches the oracle or is refused loudly."""
    import variable_length_flash_gb300 as vlf
    rng = np.random.default_rng(1234)
    widths = [(64, 64), (128, 128), (192, 128), (32, 32), (80, 48), (96, 96), (256, 256)]
    for trial in range(20):
        n = int(rng.integers(1, 5))
        if rng.random() < 0.25:  # decode-like: a few query rows against longer caches (split-KV)
            lq = [int(x) for x in rng.integers(1, 5, n)]
            lk = [int(x) for x in rng.integers(300, 2000, n)]
        else:
            lq = [int(x) for x in rng.integers(0, 200, n)]
            cross = rng.random() < 0.3
            lk = [int(x) for x in rng.integers(0, 200, n)] if cross else lq
        if sum(lq) == 0 or sum(lk) == 0:
            continue
        hkv = int(rng.choice([1, 2]))
        hq = hkv * int(rng.choice([1, 2, 4]))
        d, dv = widths[int(rng.integers(0, len(widths)))]
        dtype = str(rng.choice(["fp16", "bf16", "fp32"]))
        causal = bool(rng.random() < 0.6)
        window = int(rng.choice([0, 0, 1, 7, 64]))
        w = W.custom(lq, lk, dtype=dtype, h_q=hq, h_kv=hkv, d_qk=d, d_v=dv, causal=causal,
                     window=window)
        x = W.make_inputs(w, seed=100 + trial, with_dout=True)
        try:
            gpu = gpu_run(w, x)
        except vlf.VlfError:
            continue
        ref = oracle_run(w, x)
        assert_within(compare(w, gpu, ref), f"fuzz {trial} {w}")
