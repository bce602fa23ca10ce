"""Python binding of libvlf.so: fused variable-length flash attention for GB300 (sm_103a).

Argument marshalling only.  Every step of the computation runs in the library's CUDA kernels;
PyTorch supplies device memory and the current stream.  There is no CPU fallback: importing
this package raises if the compiled library is missing.

The functions carry the names of the C entry points in ``include/vlf.h``:

* ``vlf_attn_varlen_fwd(q, k, v, cu_seqlens_q, cu_seqlens_kv, max_seqlen_q, ...)`` -> (out, lse)
* ``vlf_attn_varlen_bwd(dout, q, k, v, out, lse, cu_seqlens_q, cu_seqlens_kv, ...)``
  -> (dq, dk, dv)
* ``vlf_attn_varlen_bwd_workspace_size``, ``vlf_check_error``, ``vlf_status_string``,
  ``vlf_sched_kv_band``, ``vlf_sched_q_band``, ``vlf_version``.

The operation is the varlen attention of the mtlattn 0.3.0 page (section "Use"): packed
q/k/v [tokens, heads, head_dim] with int32 cu_seqlens, end-aligned causal, sliding window,
GQA/MQA, additive fp32 bias [total_q, H or 1, max_kv] (held constant in the backward; a bias
that requires grad is refused).
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libvlf.so")

VLF_F16, VLF_BF16, VLF_F32 = 0, 1, 2
VLF_OK = 0
VLF_ERR_INVALID, VLF_ERR_UNSUPPORTED, VLF_ERR_ALIGN, VLF_ERR_LAUNCH = -1, -2, -3, -4
VLF_ERR_TIMEOUT, VLF_ERR_BAD_SEQLENS, VLF_ERR_WORKSPACE = -5, -6, -7
VLF_FLAG_NO_SKIP = 1
VLF_FLAG_FORCE_SIMT = 2
VLF_FLAG_NO_PACK = 4
VLF_FLAG_TEST_TIMEOUT = 8  # testing: the forward's pipeline waits run out (VLF_ERR_TIMEOUT)

_DTYPE = {torch.float16: VLF_F16, torch.bfloat16: VLF_BF16, torch.float32: VLF_F32}

EXPORTS = ["vlf_attn_varlen_fwd", "vlf_attn_varlen_fwd_ex", "vlf_attn_varlen_bwd",
           "vlf_attn_varlen_bwd_ex", "vlf_attn_varlen_bwd_workspace_size", "vlf_check_error",
           "vlf_status_string", "vlf_sched_kv_band", "vlf_sched_q_band", "vlf_version",
           "vlf_launch_count", "vlf_fwd_path", "vlf_bwd_path", "vlf_attn_varlen_bwd_noalloc",
           "vlf_noalloc_scratch_bytes", "vlf_attn_varlen_fwd_split", "vlf_fwd_num_splits",
           "vlf_attn_varlen_fwd_split_workspace_size", "vlf_attn_varlen_fwd_latent",
           "vlf_attn_varlen_bwd_latent", "vlf_attn_varlen_bwd_latent_workspace_size",
           "vlf_bias_bands", "vlf_bias_bands_size"]
VLF_BWD_STAGES = 3
BWD_STAGE_NAMES = ["rowdot", "dkdv", "dq"]


class VlfError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"vlf status {status}: {vlf_status_string(status)}{': ' + what if what else ''}")


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is not built; run `python -c 'import __graft_entry__ as g; "
                          "g.build()'` (needs nvcc for sm_103a)")
    lib = ctypes.CDLL(LIB_PATH)
    P, I, F, Z, U = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t, ctypes.c_uint
    fwd = [P, P, P, P, P, I, I, I, I, I, I, I, I, I, I, F, I, I, P, I, P, P, P]
    lib.vlf_attn_varlen_fwd.argtypes = fwd
    lib.vlf_attn_varlen_fwd_ex.argtypes = fwd + [U, P]
    bwd = [P, P, P, P, P, P, P, P, I, I, I, I, I, I, I, I, I, I, F, I, I, P, I, P, P, P, P, Z, P]
    lib.vlf_attn_varlen_bwd.argtypes = bwd
    lib.vlf_attn_varlen_bwd_ex.argtypes = bwd + [U, P, I, P]
    for name in ("vlf_attn_varlen_fwd", "vlf_attn_varlen_fwd_ex", "vlf_attn_varlen_bwd",
                 "vlf_attn_varlen_bwd_ex"):
        getattr(lib, name).restype = I
    lib.vlf_attn_varlen_bwd_workspace_size.argtypes = [I, I, I, I, I, I, I]
    lib.vlf_attn_varlen_bwd_workspace_size.restype = Z
    lib.vlf_check_error.argtypes = [P]
    lib.vlf_check_error.restype = I
    lib.vlf_status_string.argtypes = [I]
    lib.vlf_status_string.restype = ctypes.c_char_p
    IP = ctypes.POINTER(ctypes.c_int)
    lib.vlf_sched_kv_band.argtypes = [I, I, I, I, I, I, IP, IP]
    lib.vlf_sched_kv_band.restype = I
    lib.vlf_sched_q_band.argtypes = [I, I, I, I, I, I, IP, IP]
    lib.vlf_sched_q_band.restype = I
    lib.vlf_version.argtypes = []
    lib.vlf_version.restype = I
    lib.vlf_attn_varlen_bwd_noalloc.argtypes = bwd[:23] + [P, P, P, P]  # ... bias_heads, dq, dk, dv, stream
    lib.vlf_attn_varlen_bwd_noalloc.restype = I
    lib.vlf_attn_varlen_fwd_split.argtypes = fwd[:22] + [I, P, Z, P, U, P]  # ..., out, lse, splits, ws, bytes, stream, flags, bands
    lib.vlf_attn_varlen_fwd_split.restype = I
    lib.vlf_fwd_num_splits.argtypes = [I, I, I, I, I, I, I, I, U, I]
    lib.vlf_fwd_num_splits.restype = I
    lib.vlf_attn_varlen_fwd_split_workspace_size.argtypes = [I, I, I, I]
    lib.vlf_attn_varlen_fwd_split_workspace_size.restype = Z
    lib.vlf_attn_varlen_fwd_latent.argtypes = [P] * 7 + [I] * 12 + [F, I, I, P, I, P, P, P, U]
    lib.vlf_attn_varlen_fwd_latent.restype = I
    lib.vlf_attn_varlen_bwd_latent_workspace_size.argtypes = [I] * 6
    lib.vlf_attn_varlen_bwd_latent_workspace_size.restype = Z
    lib.vlf_attn_varlen_bwd_latent.argtypes = ([P] * 10 + [I] * 12 + [F, I, I, P, I] + [P] * 6 +
                                               [Z, P, U, P, I])
    lib.vlf_attn_varlen_bwd_latent.restype = I
    lib.vlf_bias_bands_size.argtypes = [I, I]
    lib.vlf_bias_bands_size.restype = Z
    lib.vlf_bias_bands.argtypes = [P, I, P, P, I, I, I, P, Z, P]
    lib.vlf_bias_bands.restype = I
    lib.vlf_noalloc_scratch_bytes.argtypes = []
    lib.vlf_noalloc_scratch_bytes.restype = Z
    lib.vlf_launch_count.argtypes = []
    lib.vlf_launch_count.restype = ctypes.c_uint64
    for name in ("vlf_fwd_path", "vlf_bwd_path"):
        getattr(lib, name).argtypes = [I, I, I, I, I, I, U]
        getattr(lib, name).restype = I
    return lib


_lib = _load()
_fwd_ex = _lib.vlf_attn_varlen_fwd_ex  # (looked up once: the attribute lookup costs per call)


def _ptr(t):
    # (the argtypes are c_void_p: ctypes takes the integer address, None is NULL)
    return None if t is None else t.data_ptr()


_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(stream, like=None):
    """The handle of ``stream``, else of the current stream of ``like``'s device.  Asking torch
    for the raw handle avoids building a Stream object (microseconds per call)."""
    if stream is not None:
        return stream.cuda_stream
    if _raw_stream is not None and like is not None:
        return _raw_stream(like.get_device())
    return torch.cuda.current_stream().cuda_stream


def _check(status: int, what: str = ""):
    if status != VLF_OK:
        raise VlfError(status, what)


def vlf_status_string(status: int) -> str:
    return _lib.vlf_status_string(int(status)).decode()


def vlf_version() -> int:
    return _lib.vlf_version()


def vlf_launch_count() -> int:
    """Kernels launched by the library so far in this process."""
    return int(_lib.vlf_launch_count())


def vlf_fwd_path(h_q, h_kv, d_qk, d_v, dtype, bias_heads=0, flags=0) -> int:
    """1: tensor-core forward, 0: SIMT fp32-FMA forward, negative: refused."""
    dt = _DTYPE[dtype] if isinstance(dtype, torch.dtype) else int(dtype)
    return _lib.vlf_fwd_path(h_q, h_kv, d_qk, d_v, dt, bias_heads, flags)


def vlf_bwd_path(h_q, h_kv, d_qk, d_v, dtype, bias_heads=0, flags=0) -> int:
    """1: tensor-core backward, 0: SIMT fp32-FMA backward, negative: refused."""
    dt = _DTYPE[dtype] if isinstance(dtype, torch.dtype) else int(dtype)
    return _lib.vlf_bwd_path(h_q, h_kv, d_qk, d_v, dt, bias_heads, flags)


def vlf_check_error(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device error word."""
    return _lib.vlf_check_error(_stream(stream))


def vlf_sched_kv_band(r0, r1, q_len, kv_len, causal, window):
    lo, hi = ctypes.c_int(), ctypes.c_int()
    _check(_lib.vlf_sched_kv_band(r0, r1, q_len, kv_len, int(causal), int(window),
                                  ctypes.byref(lo), ctypes.byref(hi)), "kv band")
    return lo.value, hi.value


def vlf_sched_q_band(j0, j1, q_len, kv_len, causal, window):
    lo, hi = ctypes.c_int(), ctypes.c_int()
    _check(_lib.vlf_sched_q_band(j0, j1, q_len, kv_len, int(causal), int(window),
                                 ctypes.byref(lo), ctypes.byref(hi)), "q band")
    return lo.value, hi.value


def vlf_attn_varlen_bwd_workspace_size(total_q, total_kv, h_q, h_kv, d_qk, d_v, dtype) -> int:
    dt = _DTYPE[dtype] if isinstance(dtype, torch.dtype) else int(dtype)
    return int(_lib.vlf_attn_varlen_bwd_workspace_size(total_q, total_kv, h_q, h_kv, d_qk, d_v, dt))


def vlf_fwd_num_splits(num_seqs, max_seqlen_q, max_seqlen_kv, h_q, h_kv, d_qk, d_v, dtype,
                       flags=0, num_sms=0) -> int:
    """Parts the split-KV forward cuts each CTA's KV band into when left to choose (1: no
    split); ``num_sms`` <= 0 takes the current device's SM count."""
    dt = _DTYPE[dtype] if isinstance(dtype, torch.dtype) else int(dtype)
    return int(_lib.vlf_fwd_num_splits(num_seqs, max_seqlen_q, max_seqlen_kv, h_q, h_kv, d_qk, d_v,
                                       dt, flags, num_sms))


def vlf_attn_varlen_fwd_split_workspace_size(total_q, h_q, d_v, num_splits) -> int:
    return int(_lib.vlf_attn_varlen_fwd_split_workspace_size(total_q, h_q, d_v, num_splits))


def _events(evs):
    if evs is None:
        return None, 0
    handles = [e.cuda_event for e in evs]
    if not all(handles):
        raise VlfError(VLF_ERR_INVALID, "stage events must exist (torch creates them at their "
                       "first record())")
    arr = (ctypes.c_void_p * len(evs))(*[ctypes.c_void_p(h) for h in handles])
    _events.keep = arr  # keep alive for the duration of the call
    return ctypes.cast(arr, ctypes.c_void_p), len(evs)


def _max_len(cu):
    return int((cu[1:] - cu[:-1]).max().item()) if cu.numel() > 1 else 0


def _req(t, name, dtype=None):
    if t is None:
        raise VlfError(VLF_ERR_INVALID, f"{name} is None")
    if not t.is_cuda:
        raise VlfError(VLF_ERR_INVALID, f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise VlfError(VLF_ERR_INVALID, f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise VlfError(VLF_ERR_INVALID, f"{name} must be {dtype}, got {t.dtype}")
    return t


def _bias_args(bias, total_q, h_q):
    if bias is None:
        return None, 0
    if bias.requires_grad:
        raise VlfError(VLF_ERR_UNSUPPORTED, "the bias is treated as a constant; a bias that "
                       "requires grad is refused")
    _req(bias, "bias", torch.float32)
    if bias.dim() != 3 or bias.shape[0] != total_q or bias.shape[1] not in (1, h_q):
        raise VlfError(VLF_ERR_INVALID, "bias must be [total_q, 1 or H_q, max_seqlen_kv]")
    return bias, int(bias.shape[1])


def _fwd_checks(q, k, v, cu_seqlens_q, cu_seqlens_kv):
    """The forward's argument checks with a message for each failure (the slow path)."""
    _req(q, "q"), _req(k, "k", q.dtype), _req(v, "v", q.dtype)
    _req(cu_seqlens_q, "cu_seqlens_q", torch.int32), _req(cu_seqlens_kv, "cu_seqlens_kv", torch.int32)
    if q.dtype not in _DTYPE:
        raise VlfError(VLF_ERR_INVALID, f"unsupported dtype {q.dtype}")
    if q.dim() != 3 or k.dim() != 3 or v.dim() != 3:
        raise VlfError(VLF_ERR_INVALID, "q, k, v must be [tokens, heads, head_dim]")


def vlf_bias_bands_size(total_q, bias_heads) -> int:
    return int(_lib.vlf_bias_bands_size(int(total_q), int(bias_heads)))


def vlf_bias_bands(bias, cu_seqlens_q, cu_seqlens_kv, max_seqlen_kv=None, out=None, stream=None):
    """The bias bands of ``bias`` [total_q, 1 or H_q, max_seqlen_kv] (fp32, CUDA): per bias head
    and query row the keys from the first to the last finite value and whether the bias is 0
    throughout them, plus the same per 64-row block of each sequence (include/vlf.h).  Returns
    the uint8 CUDA buffer (``out`` when given) to pass as ``bias_bands`` to the forward and
    backward; it stays valid while the bias is unchanged."""
    _req(bias, "bias", torch.float32)
    _req(cu_seqlens_q, "cu_seqlens_q", torch.int32), _req(cu_seqlens_kv, "cu_seqlens_kv", torch.int32)
    if bias.dim() != 3:
        raise VlfError(VLF_ERR_INVALID, "bias must be [total_q, 1 or H_q, max_seqlen_kv]")
    tq, bh, mk = bias.shape
    if max_seqlen_kv is not None and int(max_seqlen_kv) != mk:
        raise VlfError(VLF_ERR_INVALID, "bias last dim must be max_seqlen_kv")
    need = vlf_bias_bands_size(tq, bh)
    if out is None:
        out = torch.empty(max(need, 16), dtype=torch.uint8, device=bias.device)
    st = _lib.vlf_bias_bands(bias.data_ptr(), bh, cu_seqlens_q.data_ptr(), cu_seqlens_kv.data_ptr(),
                             cu_seqlens_q.numel() - 1, tq, mk, out.data_ptr(), out.numel(),
                             _stream(stream, bias))
    _check(st, "vlf_bias_bands")
    return out


def _bands_arg(bias_bands, bias, cu_seqlens_q, cu_seqlens_kv, stream):
    """The bands pointer for a call: computed here for a bias when not given (None); False
    (or no bias) passes none."""
    if bias is None or bias_bands is False:
        return None
    if bias_bands is None:
        bias_bands = vlf_bias_bands(bias, cu_seqlens_q, cu_seqlens_kv, stream=stream)
    return bias_bands.data_ptr()


_SPLITS = {}  # (shape, device) -> the library's split-KV part count


def vlf_attn_varlen_fwd(q, k, v, cu_seqlens_q, cu_seqlens_kv, max_seqlen_q, max_seqlen_kv=None,
                        scale=None, causal=False, window=0, bias=None, out=None, lse=None,
                        stream=None, flags=0, num_splits=None, workspace=None, bias_bands=None):
    """Forward.  q [Tq,Hq,Dqk], k [Tkv,Hkv,Dqk], v [Tkv,Hkv,Dv] (fp16/bf16/fp32, CUDA,
    contiguous), cu_seqlens int32 [n+1].  Returns out [Tq,Hq,Dv] and lse fp32 [Hq,Tq].
    ``max_seqlen_kv=None`` reads it from cu_seqlens_kv (a host sync); the bias's last dim
    must equal max_seqlen_kv when a bias is given.  ``num_splits``: None lets the library
    decide whether to split each CTA's KV band (small-batch / decode shapes; the parts' fp32
    results go to ``workspace``, allocated here when not given), 1 never splits, k > 1 splits
    into k parts.  ``bias_bands``: for a bias, vlf_bias_bands's result for it (None: computed
    here, one extra pass; False: none, every tile's bias is read)."""
    # the common case's conditions in one pass (each tensor attribute costs ~0.1 us of host
    # time, which small problems pay per call); any failure takes the detailed checks
    dtype = q.dtype
    if not (dtype in _DTYPE and k.dtype is dtype and v.dtype is dtype and q.is_cuda and k.is_cuda
            and v.is_cuda and q.is_contiguous() and k.is_contiguous() and v.is_contiguous()
            and q.dim() == 3 and k.dim() == 3 and v.dim() == 3
            and cu_seqlens_q.dtype is torch.int32 and cu_seqlens_kv.dtype is torch.int32
            and cu_seqlens_q.is_cuda and cu_seqlens_kv.is_cuda
            and cu_seqlens_q.is_contiguous() and cu_seqlens_kv.is_contiguous()):
        _fwd_checks(q, k, v, cu_seqlens_q, cu_seqlens_kv)
    tq, hq, dqk = q.shape
    tk, hkv, dv = v.shape
    if k.shape != (tk, hkv, dqk):
        raise VlfError(VLF_ERR_INVALID, "k shape")
    if max_seqlen_kv is None:
        max_seqlen_kv = int(bias.shape[2]) if bias is not None else _max_len(cu_seqlens_kv)
    if bias is not None:
        if bias.shape[2] != max_seqlen_kv:
            raise VlfError(VLF_ERR_INVALID, "bias last dim must be max_seqlen_kv")
        bias, bh = _bias_args(bias, tq, hq)
        bias_p = bias.data_ptr()
        bands_p = _bands_arg(bias_bands, bias, cu_seqlens_q, cu_seqlens_kv, stream)
    else:
        bias_p, bh, bands_p = None, 0, None
    if out is None:
        out = torch.empty((tq, hq, dv), dtype=dtype, device=q.device)
    elif not (out.dtype is dtype and out.is_cuda and out.is_contiguous()):
        _req(out, "out", dtype)
    if lse is None:
        lse = torch.empty((hq, tq), dtype=torch.float32, device=q.device)
    elif not (lse.dtype is torch.float32 and lse.is_cuda and lse.is_contiguous()):
        _req(lse, "lse", torch.float32)
    nseq = cu_seqlens_q.numel() - 1
    dt = _DTYPE[dtype]
    dev = q.get_device()
    st_h = (stream.cuda_stream if stream is not None else
            _raw_stream(dev) if _raw_stream is not None else _stream(None, q))
    if num_splits is None:
        # the library's part count depends on the shape and the device alone: remembered per
        # (shape, device) so that a repeated call makes one foreign call, not two
        key = (nseq, int(max_seqlen_q), int(max_seqlen_kv), hq, hkv, dqk, dv, dt, int(flags), dev)
        num_splits = _SPLITS.get(key)
        if num_splits is None:
            num_splits = _lib.vlf_fwd_num_splits(nseq, int(max_seqlen_q), int(max_seqlen_kv), hq, hkv,
                                                 dqk, dv, dt, int(flags), 0)
            if len(_SPLITS) < 4096:
                _SPLITS[key] = num_splits
    if num_splits >= 2:
        need = vlf_attn_varlen_fwd_split_workspace_size(tq, hq, dv, int(num_splits))
        if workspace is None:
            workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
        _req(workspace, "workspace")
        st = _lib.vlf_attn_varlen_fwd_split(
            q.data_ptr(), k.data_ptr(), v.data_ptr(), cu_seqlens_q.data_ptr(),
            cu_seqlens_kv.data_ptr(), nseq, tq, tk, int(max_seqlen_q), int(max_seqlen_kv), hq, hkv,
            dqk, dv, dt, float(scale) if scale else 0.0, int(bool(causal)), int(window or 0), bias_p,
            bh, out.data_ptr(), lse.data_ptr(), int(num_splits), workspace.data_ptr(),
            workspace.numel() * workspace.element_size(), st_h, int(flags), bands_p)
        if st != VLF_OK:
            _check(st, "vlf_attn_varlen_fwd_split")
        return out, lse
    st = _fwd_ex(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), cu_seqlens_q.data_ptr(), cu_seqlens_kv.data_ptr(),
        nseq, tq, tk, int(max_seqlen_q), int(max_seqlen_kv), hq, hkv, dqk, dv, dt,
        float(scale) if scale else 0.0, 1 if causal else 0, int(window) if window else 0, bias_p,
        bh, out.data_ptr(), lse.data_ptr(), st_h, int(flags), bands_p)
    if st != VLF_OK:
        _check(st, "vlf_attn_varlen_fwd")
    return out, lse


def vlf_attn_varlen_bwd(dout, q, k, v, out, lse, cu_seqlens_q, cu_seqlens_kv, max_seqlen_q,
                        max_seqlen_kv=None, scale=None, causal=False, window=0, bias=None,
                        dq=None, dk=None, dv=None, workspace=None, stream=None, flags=0,
                        stage_events=None, bias_bands=None):
    """Backward: gradients of sum(out * dout) w.r.t. q, k, v (bias constant).
    Returns dq, dk, dv in the input dtype.  ``workspace`` (uint8 CUDA tensor of at least
    vlf_attn_varlen_bwd_workspace_size bytes) is allocated with torch when not given.
    ``stage_events``: optional list of VLF_BWD_STAGES + 1 ``torch.cuda.Event`` (timing) recorded
    before the first and after each backward kernel on the same stream."""
    for t, n in ((dout, "dout"), (q, "q"), (k, "k"), (v, "v"), (out, "out")):
        _req(t, n, q.dtype)
    _req(lse, "lse", torch.float32)
    _req(cu_seqlens_q, "cu_seqlens_q", torch.int32), _req(cu_seqlens_kv, "cu_seqlens_kv", torch.int32)
    tq, hq, dqk = q.shape
    tk, hkv, dvv = v.shape
    if max_seqlen_kv is None:
        max_seqlen_kv = int(bias.shape[2]) if bias is not None else _max_len(cu_seqlens_kv)
    bias, bh = _bias_args(bias, tq, hq)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    need = vlf_attn_varlen_bwd_workspace_size(tq, tk, hq, hkv, dqk, dvv, q.dtype)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    st = _lib.vlf_attn_varlen_bwd_ex(
        _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(dout), _ptr(cu_seqlens_q),
        _ptr(cu_seqlens_kv), cu_seqlens_q.numel() - 1, tq, tk, int(max_seqlen_q),
        int(max_seqlen_kv), hq, hkv, dqk, dvv, _DTYPE[q.dtype], float(scale) if scale else 0.0,
        int(bool(causal)), int(window or 0), _ptr(bias), bh, _ptr(dq), _ptr(dk), _ptr(dv),
        _ptr(workspace), workspace.numel(), _stream(stream, q), int(flags), *_events(stage_events),
        _bands_arg(bias_bands, bias, cu_seqlens_q, cu_seqlens_kv, stream))
    _check(st, "vlf_attn_varlen_bwd")
    return dq, dk, dv


def _latent_args(q_nope, q_rope, k_nope, k_rope, v):
    """Shapes of a split-operand latent call: (tq, hq, tk, hkv, rope_heads)."""
    _req(q_nope, "q_nope")
    for t, n in ((q_rope, "q_rope"), (k_nope, "k_nope"), (k_rope, "k_rope"), (v, "v")):
        _req(t, n, q_nope.dtype)
    if any(t.dim() != 3 for t in (q_nope, q_rope, k_nope, k_rope, v)):
        raise VlfError(VLF_ERR_INVALID, "latent operands must be [tokens, heads, width]")
    tq, hq, _ = q_nope.shape
    tk, hkv, _ = k_nope.shape
    if tuple(q_rope.shape[:2]) != (tq, hq) or k_rope.shape[0] != tk or tuple(v.shape[:2]) != (tk, hkv):
        raise VlfError(VLF_ERR_INVALID, "latent operand shapes disagree")
    return tq, hq, tk, hkv, int(k_rope.shape[1])


def vlf_attn_varlen_fwd_latent(q_nope, q_rope, k_nope, k_rope, v, cu_seqlens_q, cu_seqlens_kv,
                               max_seqlen_q, max_seqlen_kv=None, scale=None, causal=False,
                               window=0, bias=None, out=None, lse=None, stream=None, flags=0):
    """Latent attention forward with split operands (q_nope [Tq,H,128], q_rope [Tq,H,64],
    k_nope [Tkv,Hkv,128], k_rope [Tkv,1 or Hkv,64], v [Tkv,Hkv,128]); equals the forward on the
    concatenated operands.  Returns out [Tq,H,128] and lse fp32 [H,Tq]."""
    tq, hq, tk, hkv, rh = _latent_args(q_nope, q_rope, k_nope, k_rope, v)
    _req(cu_seqlens_q, "cu_seqlens_q", torch.int32), _req(cu_seqlens_kv, "cu_seqlens_kv", torch.int32)
    if max_seqlen_kv is None:
        max_seqlen_kv = int(bias.shape[2]) if bias is not None else _max_len(cu_seqlens_kv)
    bias, bh = _bias_args(bias, tq, hq)
    dv = v.shape[2]
    if out is None:
        out = torch.empty((tq, hq, dv), dtype=q_nope.dtype, device=q_nope.device)
    if lse is None:
        lse = torch.empty((hq, tq), dtype=torch.float32, device=q_nope.device)
    st = _lib.vlf_attn_varlen_fwd_latent(
        _ptr(q_nope), _ptr(q_rope), _ptr(k_nope), _ptr(k_rope), _ptr(v), _ptr(cu_seqlens_q),
        _ptr(cu_seqlens_kv), cu_seqlens_q.numel() - 1, tq, tk, int(max_seqlen_q),
        int(max_seqlen_kv), hq, hkv, rh, q_nope.shape[2], q_rope.shape[2], dv,
        _DTYPE[q_nope.dtype], float(scale) if scale else 0.0, int(bool(causal)), int(window or 0),
        _ptr(bias), bh, _ptr(out), _ptr(lse), _stream(stream, q_nope), int(flags))
    _check(st, "vlf_attn_varlen_fwd_latent")
    return out, lse


def vlf_attn_varlen_bwd_latent_workspace_size(total_q, total_kv, h_q, h_kv, rope_heads, dtype) -> int:
    dt = _DTYPE[dtype] if isinstance(dtype, torch.dtype) else int(dtype)
    return int(_lib.vlf_attn_varlen_bwd_latent_workspace_size(total_q, total_kv, h_q, h_kv,
                                                              rope_heads, dt))


def vlf_attn_varlen_bwd_latent(dout, q_nope, q_rope, k_nope, k_rope, v, out, lse, cu_seqlens_q,
                               cu_seqlens_kv, max_seqlen_q, max_seqlen_kv=None, scale=None,
                               causal=False, window=0, bias=None, grads=None, workspace=None,
                               stream=None, flags=0, stage_events=None):
    """Latent attention backward with split operands.  Returns (dq_nope, dq_rope, dk_nope,
    dk_rope, dv); a shared rope key (k_rope with one head) gets the sum of every head's
    gradient.  ``grads``: optional preallocated 5-tuple in that order."""
    tq, hq, tk, hkv, rh = _latent_args(q_nope, q_rope, k_nope, k_rope, v)
    for t, n in ((dout, "dout"), (out, "out")):
        _req(t, n, q_nope.dtype)
    _req(lse, "lse", torch.float32)
    _req(cu_seqlens_q, "cu_seqlens_q", torch.int32), _req(cu_seqlens_kv, "cu_seqlens_kv", torch.int32)
    if max_seqlen_kv is None:
        max_seqlen_kv = int(bias.shape[2]) if bias is not None else _max_len(cu_seqlens_kv)
    bias, bh = _bias_args(bias, tq, hq)
    if grads is None:
        grads = tuple(torch.empty_like(t) for t in (q_nope, q_rope, k_nope, k_rope, v))
    need = vlf_attn_varlen_bwd_latent_workspace_size(tq, tk, hq, hkv, rh, q_nope.dtype)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q_nope.device)
    st = _lib.vlf_attn_varlen_bwd_latent(
        _ptr(q_nope), _ptr(q_rope), _ptr(k_nope), _ptr(k_rope), _ptr(v), _ptr(out), _ptr(lse),
        _ptr(dout), _ptr(cu_seqlens_q), _ptr(cu_seqlens_kv), cu_seqlens_q.numel() - 1, tq, tk,
        int(max_seqlen_q), int(max_seqlen_kv), hq, hkv, rh, q_nope.shape[2], q_rope.shape[2],
        v.shape[2], _DTYPE[q_nope.dtype], float(scale) if scale else 0.0, int(bool(causal)),
        int(window or 0), _ptr(bias), bh, *[_ptr(g) for g in grads], _ptr(workspace),
        workspace.numel(), _stream(stream, q_nope), int(flags), *_events(stage_events))
    _check(st, "vlf_attn_varlen_bwd_latent")
    return grads


def vlf_noalloc_scratch_bytes() -> int:
    return int(_lib.vlf_noalloc_scratch_bytes())


def vlf_attn_varlen_bwd_noalloc(dout, q, k, v, out, lse, cu_seqlens_q, cu_seqlens_kv,
                                max_seqlen_q, max_seqlen_kv=None, scale=None, causal=False,
                                window=0, bias=None, dq=None, dk=None, dv=None, stream=None):
    """Backward through the entry point that allocates nothing on the device: the library keeps
    the row-dot workspace in a fixed array of its own (vlf_noalloc_scratch_bytes() bytes per
    GPU), for callers that cannot allocate device memory when they call.  Calls that overlap on
    the GPU share that array and race; problems with h_q * total_q above the array's size are
    refused.  The gradient outputs are allocated here with torch only when not passed in."""
    for t, n in ((dout, "dout"), (q, "q"), (k, "k"), (v, "v"), (out, "out")):
        _req(t, n, q.dtype)
    _req(lse, "lse", torch.float32)
    _req(cu_seqlens_q, "cu_seqlens_q", torch.int32), _req(cu_seqlens_kv, "cu_seqlens_kv", torch.int32)
    tq, hq, dqk = q.shape
    tk, hkv, dvv = v.shape
    if max_seqlen_kv is None:
        max_seqlen_kv = int(bias.shape[2]) if bias is not None else _max_len(cu_seqlens_kv)
    bias, bh = _bias_args(bias, tq, hq)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    st = _lib.vlf_attn_varlen_bwd_noalloc(
        _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(dout), _ptr(cu_seqlens_q),
        _ptr(cu_seqlens_kv), cu_seqlens_q.numel() - 1, tq, tk, int(max_seqlen_q),
        int(max_seqlen_kv), hq, hkv, dqk, dvv, _DTYPE[q.dtype], float(scale) if scale else 0.0,
        int(bool(causal)), int(window or 0), _ptr(bias), bh, _ptr(dq), _ptr(dk), _ptr(dv),
        _stream(stream, q))
    _check(st, "vlf_attn_varlen_bwd_noalloc")
    return dq, dk, dv


__all__ = ["vlf_attn_varlen_fwd", "vlf_attn_varlen_bwd", "vlf_attn_varlen_bwd_workspace_size",
           "vlf_bias_bands", "vlf_bias_bands_size",
           "vlf_check_error", "vlf_status_string", "vlf_sched_kv_band", "vlf_sched_q_band",
           "vlf_version", "vlf_launch_count", "vlf_fwd_path", "vlf_bwd_path",
           "vlf_attn_varlen_bwd_noalloc", "vlf_noalloc_scratch_bytes", "VlfError",
           "LIB_PATH", "EXPORTS"]

# differentiable entry points (autograd over the two calls above)
from .functional import (flash_attn_varlen_func, flash_attn_varlen_kvpacked_func,  # noqa: E402
                         flash_attn_varlen_qkvpacked_func, latent_attention, varlen_attention)

__all__ += ["varlen_attention", "latent_attention", "flash_attn_varlen_func", "flash_attn_varlen_qkvpacked_func",
            "flash_attn_varlen_kvpacked_func"]
