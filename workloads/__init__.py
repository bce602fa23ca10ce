"""Seeded synthetic inputs for the variable-length attention workloads.

This module only *draws* inputs: sequence lengths, packed Q/K/V/dO tensors, cu_seqlens and the
additive bias of the long-context workload.  It holds none of the attention arithmetic and is the
one module shared by the fp64 oracle side (tests) and the CUDA side (tests, bench, smoke).

Workloads (named by what they are; the shapes are the benchmark configurations of the method):

* ``varlen64_fp16_full`` / ``varlen64_fp16_causal`` -- 4 packed sequences of lengths
  {17, 64, 100, 255}, H_q = H_kv = 4, head_dim 64, fp16, forward only.
* ``dense4x4096_bf16_causal`` -- B=4 x L=4096 packed, H=32, head_dim 128, causal, bf16.
* ``ragged64_gqa_window_bf16`` -- 64 lengths ~ U{128..8192}, H_q=32, H_kv=8, head_dim 128,
  causal, window 4096, bf16.
* ``latent2x8192_bf16_causal`` -- B=2 x 8192, 128 heads, QK width 192 (128 "nope" ++ 64 "rope"),
  V/output width 128, causal, scale 1/sqrt(192), bf16.
* ``long49152_fp16_bias_alibi`` / ``long49152_fp16_bias_prefix`` -- one sequence of 49,152
  tokens, H=16, head_dim 128, q/k/v ~ N(0, 0.5^2), fp16, additive fp32 bias: prefix-LM 0/-inf
  plus per-head ALiBi (per-head bias tensor), or the prefix-LM part alone broadcast over heads.
* ``decode64x8192_bf16_gqa`` / ``decode4x32768_bf16_gqa`` -- one new query row per sequence
  against a cache of 8192 (64 sequences) or 32,768 tokens (4 sequences), H_q=32, H_kv=8, head
  dim 128, end-aligned causal, bf16, forward only.
* ``dense4x4096_bf16_causal_d96`` -- the dense configuration at head width 96.
* ``dense4x4096_bf16_causal_d256`` -- the dense configuration at head width 256.
* ``dense4x4096_fp32_causal_d64`` -- the dense configuration with fp32 data at head width 64.
* ``latent2x8192_bf16_causal_shared_rope`` -- the latent configuration with split operands and
  one rope key [tokens, 1, 64] shared by all 128 heads.

Draw order: the ragged lengths come from a CPU ``torch.Generator`` seeded with ``seed``; the
tensors from a generator on the target device seeded with ``seed``, in the order q, k, v, dout,
each drawn in fp32 as N(0,1) * sigma and rounded once (round-to-nearest-even) to the workload
dtype.  The latent workload draws q_nope, q_rope, k_nope, k_rope, v, dout and
concatenates nope ++ rope along the head dimension.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional

import torch

DTYPES = {"fp16": torch.float16, "bf16": torch.bfloat16, "fp32": torch.float32}

PREFIX_LEN = 8192          # prefix-LM: every query sees keys 0..8191
ALIBI_HEADS = 16


@dataclass
class Workload:
    name: str
    dtype: str
    lengths_q: list
    lengths_kv: list
    h_q: int
    h_kv: int
    d_qk: int
    d_v: int
    causal: bool
    window: int = 0                       # <= 0: no window
    scale: Optional[float] = None         # None: 1/sqrt(d_qk)
    sigma: float = 1.0
    bias: Optional[str] = None            # None | "alibi_prefix" (per head) | "prefix" (broadcast)
    latent_split: Optional[tuple] = None  # (nope, rope) widths of the QK head
    rope_heads: Optional[int] = None      # latent: heads of the rope key (None: h_kv; 1: shared)
    backward: bool = True
    meta: dict = field(default_factory=dict)

    @property
    def num_seqs(self) -> int:
        return len(self.lengths_q)

    @property
    def total_q(self) -> int:
        return int(sum(self.lengths_q))

    @property
    def total_kv(self) -> int:
        return int(sum(self.lengths_kv))

    @property
    def max_seqlen_q(self) -> int:
        return int(max(self.lengths_q)) if self.lengths_q else 0

    @property
    def max_seqlen_kv(self) -> int:
        return int(max(self.lengths_kv)) if self.lengths_kv else 0

    @property
    def softmax_scale(self) -> float:
        return self.scale if self.scale is not None else 1.0 / math.sqrt(self.d_qk)

    @property
    def bias_heads(self) -> int:
        if self.bias is None:
            return 0
        return self.h_q if self.bias == "alibi_prefix" else 1


def ragged_lengths(n: int, lo: int, hi: int, gen: torch.Generator) -> list:
    """n lengths uniform on the integers lo..hi inclusive, from ``gen`` (drawn first)."""
    return [int(x) for x in torch.randint(lo, hi + 1, (n,), generator=gen)]


def workload(name: str, seed: int = 0) -> Workload:
    """The named benchmark workload (lengths of the ragged one depend on ``seed``)."""
    if name in ("varlen64_fp16_full", "varlen64_fp16_causal"):
        lens = [17, 64, 100, 255]
        return Workload(name, "fp16", lens, lens, 4, 4, 64, 64,
                        causal=name.endswith("causal"), scale=1.0 / 8.0, backward=False)
    if name == "dense4x4096_bf16_causal":
        lens = [4096] * 4
        return Workload(name, "bf16", lens, lens, 32, 32, 128, 128, causal=True)
    if name == "dense4x4096_bf16_causal_d96":
        # the dense configuration at head width 96 (a width the pages list beside 64/128/256)
        lens = [4096] * 4
        return Workload(name, "bf16", lens, lens, 32, 32, 96, 96, causal=True)
    if name == "dense4x4096_fp32_causal_d64":
        # the dense configuration with fp32 inputs at head width 64 (fp32 is supported data)
        lens = [4096] * 4
        return Workload(name, "fp32", lens, lens, 32, 32, 64, 64, causal=True)
    if name == "dense4x4096_bf16_causal_d256":
        # the dense configuration at head width 256
        lens = [4096] * 4
        return Workload(name, "bf16", lens, lens, 32, 32, 256, 256, causal=True)
    if name == "ragged64_gqa_window_bf16":
        g = torch.Generator("cpu").manual_seed(seed)
        lens = ragged_lengths(64, 128, 8192, g)
        return Workload(name, "bf16", lens, lens, 32, 8, 128, 128, causal=True, window=4096)
    if name == "latent2x8192_bf16_causal":
        lens = [8192] * 2
        return Workload(name, "bf16", lens, lens, 128, 128, 192, 128, causal=True,
                        scale=1.0 / math.sqrt(192.0), latent_split=(128, 64))
    if name == "latent2x8192_bf16_causal_shared_rope":
        # the latent configuration with its operands split as produced and one rope key shared
        # by every head (the form the split-operand calls take)
        lens = [8192] * 2
        return Workload(name, "bf16", lens, lens, 128, 128, 192, 128, causal=True,
                        scale=1.0 / math.sqrt(192.0), latent_split=(128, 64), rope_heads=1)
    if name == "decode64x8192_bf16_gqa":
        # one new query row per sequence against an 8192-token cache (end-aligned causal: the
        # row sees every key), GQA 4, forward only
        return Workload(name, "bf16", [1] * 64, [8192] * 64, 32, 8, 128, 128, causal=True,
                        backward=False)
    if name == "decode4x32768_bf16_gqa":
        # a small batch of decode steps against long caches (4 rows x 8 kv heads: too few
        # CTAs to fill the GPU unless each cache is split), GQA 4, forward only
        return Workload(name, "bf16", [1] * 4, [32768] * 4, 32, 8, 128, 128, causal=True,
                        backward=False)
    if name in ("long49152_fp16_bias_alibi", "long49152_fp16_bias_prefix"):
        lens = [49152]
        return Workload(name, "fp16", lens, lens, 16, 16, 128, 128, causal=False, sigma=0.5,
                        bias="alibi_prefix" if name.endswith("alibi") else "prefix")
    if name in ("long12288_fp16_bias_alibi", "long12288_fp16_bias_prefix"):
        # the long-context workload at a quarter of the length (prefix 2048, the same share of
        # the sequence), small enough for profiler captures of its kernels
        lens = [12288]
        return Workload(name, "fp16", lens, lens, 16, 16, 128, 128, causal=False, sigma=0.5,
                        bias="alibi_prefix" if name.endswith("alibi") else "prefix",
                        meta={"prefix": 2048})
    raise KeyError(name)


WORKLOADS = ["varlen64_fp16_full", "varlen64_fp16_causal", "dense4x4096_bf16_causal",
             "ragged64_gqa_window_bf16", "latent2x8192_bf16_causal",
             "long49152_fp16_bias_alibi", "long49152_fp16_bias_prefix", "decode64x8192_bf16_gqa",
             "dense4x4096_bf16_causal_d96", "decode4x32768_bf16_gqa", "dense4x4096_bf16_causal_d256",
             "latent2x8192_bf16_causal_shared_rope", "dense4x4096_fp32_causal_d64",
             "long12288_fp16_bias_alibi", "long12288_fp16_bias_prefix"]


def custom(lengths_q, lengths_kv=None, *, dtype="bf16", h_q=4, h_kv=None, d_qk=64, d_v=None,
           causal=False, window=0, scale=None, sigma=1.0, bias=None, latent_split=None,
           rope_heads=None, name="custom") -> Workload:
    """A small ad-hoc workload for tests (same draw rules as the named ones)."""
    lengths_kv = list(lengths_q) if lengths_kv is None else list(lengths_kv)
    return Workload(name, dtype, list(lengths_q), lengths_kv, h_q, h_kv or h_q, d_qk,
                    d_v or d_qk, causal, window, scale, sigma, bias, latent_split, rope_heads)


def cu_seqlens(lengths) -> torch.Tensor:
    """int32 [n+1] cumulative lengths, starting at 0."""
    out = torch.zeros(len(lengths) + 1, dtype=torch.int32)
    if len(lengths):
        out[1:] = torch.cumsum(torch.tensor(lengths, dtype=torch.int64), 0).to(torch.int32)
    return out


def _normal(shape, sigma, dtype, gen, device):
    x = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    if sigma != 1.0:
        x.mul_(sigma)
    return x.to(dtype)


def alibi_slopes(heads: int = ALIBI_HEADS) -> torch.Tensor:
    """fp64 per-head ALiBi slopes: head h (0-based) gets 2^(-8 h / heads).

    Computed on the host in fp64 so that every device and the oracle see the same bits.
    """
    return torch.tensor([2.0 ** (-8.0 * h / heads) for h in range(heads)], dtype=torch.float64)


def bias_block(w: Workload, rows: torch.Tensor, heads, device="cpu") -> torch.Tensor:
    """fp32 bias values for global query ``rows`` (1-D int64) and ``heads`` (list of bias heads).

    Returns [len(rows), len(heads), max_seqlen_kv].  Only the single-sequence long workload
    carries a bias, so the global row is also the sequence-local row.  Entry (i, h, j) is
    -inf unless j <= PREFIX_LEN-1 or j <= i; allowed entries get 0 ("prefix") or
    -slope_h * |i - j| ("alibi_prefix"), evaluated in fp64 and rounded once to fp32.
    """
    assert w.bias is not None and w.num_seqs == 1
    n_kv = w.max_seqlen_kv
    i = rows.to(device=device, dtype=torch.int64)[:, None]
    j = torch.arange(n_kv, device=device, dtype=torch.int64)[None, :]
    allowed = (j <= w.meta.get("prefix", PREFIX_LEN) - 1) | (j <= i)
    out = torch.empty((rows.numel(), len(heads), n_kv), dtype=torch.float32, device=device)
    dist = (i - j).abs().to(torch.float64)
    slopes = alibi_slopes(w.h_q).to(device)
    for a, h in enumerate(heads):
        if w.bias == "alibi_prefix":
            val = (-(slopes[h] * dist)).to(torch.float32)
        else:
            val = torch.zeros(dist.shape, dtype=torch.float32, device=device)
        out[:, a, :] = torch.where(allowed, val, torch.full_like(val, float("-inf")))
    return out


def make_bias(w: Workload, device="cpu", chunk_rows: int = 1024) -> Optional[torch.Tensor]:
    """The whole bias tensor [total_q, bias_heads, max_seqlen_kv] fp32 (None if no bias)."""
    if w.bias is None:
        return None
    hb = w.bias_heads
    out = torch.empty((w.total_q, hb, w.max_seqlen_kv), dtype=torch.float32, device=device)
    heads = list(range(hb))
    for r0 in range(0, w.total_q, chunk_rows):
        r1 = min(w.total_q, r0 + chunk_rows)
        out[r0:r1] = bias_block(w, torch.arange(r0, r1), heads, device=device)
    return out


def make_inputs(w: Workload, seed: int = 0, device="cpu", with_dout: Optional[bool] = None,
                with_bias: bool = True) -> dict:
    """Packed inputs of ``w`` drawn from a generator seeded with ``seed`` on ``device``.

    Returns q [Tq,Hq,Dqk], k [Tkv,Hkv,Dqk], v [Tkv,Hkv,Dv] (workload dtype), dout [Tq,Hq,Dv]
    (if the workload has a backward or ``with_dout``), cu_seqlens_q/kv int32 on ``device``,
    and bias fp32 [Tq, bias_heads, max_kv] or None.  A latent workload also returns its parts
    q_nope, q_rope, k_nope, k_rope (k_rope with ``rope_heads`` heads; q / k are their
    concatenations, the rope key broadcast over the kv heads).
    """
    dt = DTYPES[w.dtype]
    gen = torch.Generator(device).manual_seed(seed)
    tq, tk = w.total_q, w.total_kv
    if w.latent_split is not None:
        nope, rope = w.latent_split
        qn = _normal((tq, w.h_q, nope), w.sigma, dt, gen, device)
        qr = _normal((tq, w.h_q, rope), w.sigma, dt, gen, device)
        kn = _normal((tk, w.h_kv, nope), w.sigma, dt, gen, device)
        kr = _normal((tk, w.rope_heads or w.h_kv, rope), w.sigma, dt, gen, device)
        q = torch.cat([qn, qr], dim=2).contiguous()
        k = torch.cat([kn, kr.expand(tk, w.h_kv, rope)], dim=2).contiguous()
        split = {"q_nope": qn, "q_rope": qr, "k_nope": kn, "k_rope": kr}
    else:
        q = _normal((tq, w.h_q, w.d_qk), w.sigma, dt, gen, device)
        k = _normal((tk, w.h_kv, w.d_qk), w.sigma, dt, gen, device)
        split = {}
    v = _normal((tk, w.h_kv, w.d_v), w.sigma, dt, gen, device)
    want_dout = w.backward if with_dout is None else with_dout
    dout = _normal((tq, w.h_q, w.d_v), 1.0, dt, gen, device) if want_dout else None
    return {
        "q": q, "k": k, "v": v, "dout": dout,
        "cu_seqlens_q": cu_seqlens(w.lengths_q).to(device),
        "cu_seqlens_kv": cu_seqlens(w.lengths_kv).to(device),
        "bias": make_bias(w, device=device) if (with_bias and w.bias is not None) else None,
        **split,
    }


def sample_rows(w: Workload, n_random: int, seed: int = 0, tail: int = 4) -> list:
    """Global query rows to check at full size: the last ``tail`` rows of every sequence plus
    ``n_random`` seeded random rows (sorted, unique)."""
    g = torch.Generator("cpu").manual_seed(seed + 7919)
    cu = [0]
    for L in w.lengths_q:
        cu.append(cu[-1] + L)
    rows = set()
    for s, L in enumerate(w.lengths_q):
        for t in range(min(tail, L)):
            rows.add(cu[s + 1] - 1 - t)
    if w.total_q:
        for r in torch.randint(0, w.total_q, (n_random,), generator=g).tolist():
            rows.add(int(r))
    return sorted(rows)
