"""The C ABI without a GPU: the library loads, exports every function include/vlf.h declares,
refuses bad arguments before touching the device, and its tile scheduler's bands agree with
brute-force masks from the oracle."""
import ctypes
import os
import re

import numpy as np
import pytest

import variable_length_flash_gb300 as vlf
from oracle import attention as orc

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "vlf.h")


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(vlf_[a-z0-9_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported():
    names = declared_functions()
    assert "vlf_attn_varlen_fwd" in names and "vlf_attn_varlen_bwd" in names
    lib = ctypes.CDLL(vlf.LIB_PATH)
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing
    assert sorted(vlf.EXPORTS) == names


def test_status_strings_and_version():
    assert vlf.vlf_status_string(0) == "ok"
    assert "cu_seqlens" in vlf.vlf_status_string(vlf.VLF_ERR_BAD_SEQLENS)
    assert vlf.vlf_version() >= 100


def _fwd_raw(**kw):
    args = dict(q=16, k=16, v=16, cu_q=16, cu_kv=16, n=1, tq=4, tk=4, mq=4, mk=4, hq=2, hkv=1,
                dqk=64, dv=64, dtype=1, scale=0.0, causal=0, window=0, bias=None, bh=0, out=16,
                lse=16)
    args.update(kw)
    P = ctypes.c_void_p
    return vlf._lib.vlf_attn_varlen_fwd(
        P(args["q"]), P(args["k"]), P(args["v"]), P(args["cu_q"]), P(args["cu_kv"]), args["n"],
        args["tq"], args["tk"], args["mq"], args["mk"], args["hq"], args["hkv"], args["dqk"],
        args["dv"], args["dtype"], args["scale"], args["causal"], args["window"],
        P(args["bias"]) if args["bias"] else None, args["bh"], P(args["out"]), P(args["lse"]), None)


@pytest.mark.parametrize("kw,status", [
    (dict(hq=3, hkv=2), vlf.VLF_ERR_INVALID),          # H_q not a multiple of H_kv
    (dict(dtype=7), vlf.VLF_ERR_INVALID),
    (dict(dqk=0), vlf.VLF_ERR_INVALID),
    (dict(dqk=512), vlf.VLF_ERR_UNSUPPORTED),
    (dict(n=-1), vlf.VLF_ERR_INVALID),
    (dict(q=None), vlf.VLF_ERR_INVALID),
    (dict(q=24), vlf.VLF_ERR_ALIGN),
    (dict(out=8), vlf.VLF_ERR_ALIGN),
    (dict(bias=16, bh=3), vlf.VLF_ERR_INVALID),       # bias heads must be 1 or H_q
    (dict(n=0, tq=3), vlf.VLF_ERR_INVALID),
])
def test_host_refusals_before_any_launch(kw, status):
    # refused on the host: the (bogus) device pointers are never dereferenced
    assert _fwd_raw(**kw) == status


def test_workspace_size_query():
    n = vlf.vlf_attn_varlen_bwd_workspace_size(1000, 1000, 8, 2, 128, 128, vlf.VLF_BF16)
    assert n >= 1000 * 8 * 4 and n % 256 == 0          # D = rowsum(dO o O), [H_q, total_q] fp32
    assert vlf.vlf_attn_varlen_bwd_workspace_size(-1, 0, 8, 2, 128, 128, vlf.VLF_BF16) == 0


@pytest.mark.parametrize("q_len,kv_len", [(1, 1), (7, 7), (40, 40), (17, 64), (64, 17), (100, 255)])
@pytest.mark.parametrize("causal,window", [(False, 0), (True, 0), (True, 1), (True, 5), (True, 33),
                                           (False, 9)])
def test_scheduler_bands_match_brute_force(q_len, kv_len, causal, window):
    mask = orc.visible(q_len, kv_len, causal, window)
    for tile in (4, 16):
        for r0 in range(0, q_len, tile):
            r1 = min(q_len, r0 + tile)
            lo, hi = vlf.vlf_sched_kv_band(r0, r1, q_len, kv_len, causal, window)
            vis = np.nonzero(mask[r0:r1].any(axis=0))[0]
            if len(vis) == 0:
                assert hi <= lo or not mask[r0:r1, lo:hi].any()
            else:
                # the band holds every visible key and is tight at both ends
                assert lo == vis.min() and hi == vis.max() + 1, (r0, r1, lo, hi, vis)
        for j0 in range(0, kv_len, tile):
            j1 = min(kv_len, j0 + tile)
            lo, hi = vlf.vlf_sched_q_band(j0, j1, q_len, kv_len, causal, window)
            rows = np.nonzero(mask[:, j0:j1].any(axis=1))[0]
            if len(rows) == 0:
                assert hi <= lo or not mask[lo:hi, j0:j1].any()
            else:
                assert lo == rows.min() and hi == rows.max() + 1, (j0, j1, lo, hi, rows)


def test_scheduler_rejects_bad_ranges():
    with pytest.raises(vlf.VlfError):
        vlf.vlf_sched_kv_band(5, 5, 10, 10, True, 0)
    with pytest.raises(vlf.VlfError):
        vlf.vlf_sched_q_band(0, 11, 10, 10, True, 0)


def test_noalloc_array_holds_a_problem_at_its_limit():
    """A backward whose row-dot workspace is exactly the no-allocation entry point's array is
    within its limit (h_q * total_q = 8,388,608 fp32 values); one more row is beyond it."""
    limit_floats = vlf.vlf_noalloc_scratch_bytes() // 4
    assert limit_floats == 8 << 20
    for dtype in (vlf.VLF_F16, vlf.VLF_BF16, vlf.VLF_F32):
        at = vlf.vlf_attn_varlen_bwd_workspace_size(limit_floats // 8, limit_floats // 8, 8, 8,
                                                    128, 128, dtype)
        assert at == vlf.vlf_noalloc_scratch_bytes(), dtype
        past = vlf.vlf_attn_varlen_bwd_workspace_size(limit_floats // 8 + 1, 1, 8, 8, 128, 128,
                                                      dtype)
        assert past > vlf.vlf_noalloc_scratch_bytes(), dtype


def test_path_queries():
    """Which kernel family a shape gets (host-only): 16-bit widths 64/96/128/192-128/256 and
    fp32 widths 32/64 (forward and backward) on the tensor cores, everything else (and
    VLF_FLAG_FORCE_SIMT) on the SIMT fp32-FMA kernels."""
    for d, dv in ((64, 64), (96, 96), (128, 128), (192, 128), (256, 256)):
        for dt in (vlf.VLF_F16, vlf.VLF_BF16):
            assert vlf.vlf_fwd_path(8, 2, d, dv, dt) == 1
            assert vlf.vlf_bwd_path(8, 2, d, dv, dt) == 1
    for d in (32, 64):
        assert vlf.vlf_fwd_path(8, 2, d, d, vlf.VLF_F32) == 1
        assert vlf.vlf_bwd_path(8, 2, d, d, vlf.VLF_F32) == 1
    for d, dv in ((128, 128), (40, 24), (96, 96)):
        assert vlf.vlf_fwd_path(8, 2, d, dv, vlf.VLF_F32) == 0
        assert vlf.vlf_bwd_path(8, 2, d, dv, vlf.VLF_F32) == 0
    assert vlf.vlf_fwd_path(8, 2, 64, 64, vlf.VLF_F32, flags=vlf.VLF_FLAG_FORCE_SIMT) == 0
    assert vlf.vlf_fwd_path(8, 2, 80, 48, vlf.VLF_BF16) == 0
    assert vlf.vlf_fwd_path(3, 2, 64, 64, vlf.VLF_BF16) == vlf.VLF_ERR_INVALID
