"""Benchmark: varlen flash attention forward + backward on one GB300 (or N replicas).

One step = one pass of the whole hot path over one batch: forward (out, lse) then backward
(row-dot pre-pass, dK/dV, dQ).  The headline workload is the dense causal configuration B=4 x
L=4096, H=32, head_dim 128, bf16, packed as 4 cu_seqlens segments (inputs synthetic, seeded,
resident in HBM; each of q/k/v/out/dout is 134 MB, larger than the 129 MB L2, so no flush is
needed between steps).

Prints ONE JSON line (rank 0):
  value        fwd+bwd TFLOP/s over unmasked pairs (whole job, all ranks), CUDA-event timed
  fwd_tflops   forward-only TFLOP/s from the same timed region
  e2e          same metric through the C ABI with pinned host buffers, H2D/D2H inside the timing
  roofline     dominant kernel: algorithmic FLOPs (or bytes) per launch / its mean event time
  cpu_baseline the fp64 oracle (test infrastructure) on a bounded sample, host cores
  clocks       nvidia-smi samples taken during the timed region (and the sustained run before it)
  sustained    the same step repeated for >= 1 s right before the timed steps (clock evidence)
  configs      the other benchmark configurations, each timed the same way on its own inputs:
               the 436-token forward (latency per call), the ragged GQA + window batch, the
               latent head, the 49,152-token sequence with a per-head and a head-broadcast bias,
               and the widened rows (decode shapes, head widths 96 / 256, shared rope key)

``--impl reference`` times the fp64 CPU oracle on the same workload instead (rank 0 only); that
arm never loads the compiled library.  Multi-GPU (torchrun): every rank runs its own replica of
the headline workload (weak scaling; the ranks exchange nothing in the data path; a barrier and
a max-reduce of the timing only); the other configurations run at N = 1 only.
"""
from __future__ import annotations

import argparse
import importlib.util
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

import workloads as W  # noqa: E402


def _load_flops():
    """The pair / FLOP counting module, loaded by its path: importing the package would load the
    compiled library, which the reference arm must not touch."""
    path = os.path.join(ROOT, "variable_length_flash_gb300", "flops.py")
    spec = importlib.util.spec_from_file_location("vlf_flops", path)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


F = _load_flops()

WORKLOAD = "dense4x4096_bf16_causal"
# (workload, timed steps, warm-up steps) of the other configurations in the line's "configs"
CONFIGS = [
    ("ragged64_gqa_window_bf16", 10, 3),
    ("latent2x8192_bf16_causal", 10, 3),
    ("long49152_fp16_bias_alibi", 3, 3),
    ("long49152_fp16_bias_prefix", 3, 3),
    ("latent2x8192_bf16_causal_shared_rope", 10, 3),
    ("dense4x4096_bf16_causal_d96", 20, 5),
    ("dense4x4096_bf16_causal_d256", 20, 5),
    ("decode64x8192_bf16_gqa", 50, 5),
    ("decode4x32768_bf16_gqa", 50, 5),
    ("dense4x4096_fp32_causal_d64", 5, 3),
]
LATENCY_CONFIGS = ["varlen64_fp16_full", "varlen64_fp16_causal"]
SUSTAIN_S = 1.2  # length of the sustained run before the timed steps


# ------------------------------------------------------------------------------ helpers
def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    dev = torch.device("cuda", torch.cuda.current_device()) if torch.cuda.is_available() else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return {"hbm_gbs": d.get("hbm_gbs"), "bf16_tflops": d.get("bf16_tflops"),
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


def ncu_traffic(role: str, workload: str):
    """DRAM bytes per launch (read + write) that one ncu capture measured for this kernel on
    this workload, or None if there is no capture or the kernel's sources changed since."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(path):
        return None
    rec = json.load(open(path))
    for entry in rec.get("captures", [rec]):
        k = entry.get("kernels", {}).get(role)
        if k is None or entry.get("workload") != workload:
            continue
        h = hashlib.sha256()
        for f in k["source_files"]:
            fp = os.path.join(ROOT, "variable_length_flash_gb300", "csrc", f)
            if not os.path.exists(fp):
                return None
            h.update(open(fp, "rb").read())
        if h.hexdigest() != k["source_sha256"]:
            return None
        return k["dram_bytes_per_launch"] * k.get("scale_to_workload", 1.0)
    return None


def l2_bytes_of(dev=None) -> int:
    if not torch.cuda.is_available():
        return 0
    return int(torch.cuda.get_device_properties(dev if dev is not None else 0).L2_cache_size)


def input_bytes(w) -> int:
    """Bytes of a step's inputs (q, k, v, dout, bias), from the workload's shape alone."""
    eb = {"fp16": 2, "bf16": 2, "fp32": 4}[w.dtype]
    if w.latent_split is not None and w.rope_heads is not None:
        nope, rope = w.latent_split
        qk = (w.total_q * w.h_q + w.total_kv * w.h_kv) * nope + (w.total_q * w.h_q + w.total_kv * w.rope_heads) * rope
    else:
        qk = (w.total_q * w.h_q + w.total_kv * w.h_kv) * w.d_qk
    n = qk + w.total_kv * w.h_kv * w.d_v + (w.total_q * w.h_q * w.d_v if w.backward else 0)
    bias = w.total_q * w.bias_heads * w.max_seqlen_kv * 4 if w.bias is not None else 0
    return n * eb + bias


def config_of(w, world: int, l2: int) -> dict:
    """The line's ``config``: the workload and how it is timed (shared by both arms)."""
    ib = input_bytes(w)
    flush = ib < 2 * l2
    return {"workload": w.name, "lengths": sorted(set(w.lengths_q)),
            "lengths_kv": sorted(set(w.lengths_kv)), "num_seqs": w.num_seqs, "h_q": w.h_q,
            "h_kv": w.h_kv, "d_qk": w.d_qk, "d_v": w.d_v, "causal": w.causal,
            "window": w.window, "bias": w.bias, "unmasked_pairs": F.workload_pairs(w),
            "step": "fwd+bwd" if w.backward else "fwd",
            "parallelism": f"replicas x{world}",
            "l2": (f"inputs {ib / 1e6:.1f} MB < 2 x L2: L2 flushed between timed steps (a "
                   f"{2 * l2 / 1e6:.0f} MB write), per-step events" if flush else
                   f"inputs {ib / 1e6:.0f} MB > 2 x L2 ({l2 / 1e6:.0f} MB): streamed from HBM, "
                   "no flush")}


class ClockSampler:
    """nvidia-smi SM clock / throttle-reason samples every 100 ms while running, each stamped
    with the host time it arrived; ``summary(t0, t1)`` keeps those taken between t0 and t1."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index, self.rows, self.proc, self.thread = index, [], None, None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 8:
                self.rows.append((time.time(), parts))

    def stop(self):
        if self.proc is None:
            return
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)

    def summary(self, t0: float, t1: float):
        if self.proc is None:
            return None
        rows = [r for t, r in self.rows if t0 <= t <= t1]

        def num(s):
            try:
                return float(s)
            except ValueError:
                return None
        sm = [x for x in (num(r[0]) for r in rows) if x is not None]
        mx = [x for x in (num(r[1]) for r in rows) if x is not None]
        pw = [x for x in (num(r[2]) for r in rows) if x is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[4:8]) if v == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows), "power_w_max": max(pw) if pw else None,
                "window_s": round(t1 - t0, 3)}


def peak_for(clocks, peaks):
    """The tensor roof for a kernel timed inside this run: the burst figure while the SM clock
    held its maximum with no power cap, the sustained (power-capped) figure otherwise."""
    if clocks and clocks.get("sm_mhz") and clocks.get("sm_max_mhz") and \
            clocks["sm_mhz"] >= 0.97 * clocks["sm_max_mhz"] and "sw_power_cap" not in clocks["reasons"]:
        return peaks["bf16_tflops"], "burst"
    if clocks and clocks.get("sm_mhz"):
        return peaks["bf16_tflops_sustained"], "sustained"
    return peaks["bf16_tflops"], "burst (no clock samples)"


# ------------------------------------------------------------------------------ CPU oracle
def oracle_sample(w, x_cpu, units: int):
    """Time the fp64 oracle on `units` (sequence, head) units of the workload, fwd + bwd (the
    forward alone for workloads without a backward).  Returns (seconds, pairs) -- test
    infrastructure, run only for the CPU baseline."""
    import numpy as np

    from oracle import attention as orc
    cu, ck = x_cpu["cu_seqlens_q"].tolist(), x_cpu["cu_seqlens_kv"].tolist()
    pairs, t0 = 0, time.perf_counter()
    for u in range(units):
        s, h = u % w.num_seqs, (u * 7) % w.h_q
        a, b = cu[s], cu[s + 1]
        c, d = ck[s], ck[s + 1]
        g = w.h_q // w.h_kv
        q = x_cpu["q"][a:b, h].double().numpy()
        k = x_cpu["k"][c:d, h // g].double().numpy()
        v = x_cpu["v"][c:d, h // g].double().numpy()
        if w.backward:
            do = x_cpu["dout"][a:b, h].double().numpy()
            orc.head_backward(q, k, v, do, w.softmax_scale, w.causal, w.window)
        else:
            orc.head_forward(q, np.arange(b - a), k, v, b - a, w.softmax_scale, w.causal, w.window)
        pairs += F.visible_pairs(b - a, d - c, w.causal, w.window)
    del np
    return time.perf_counter() - t0, pairs


def cpu_inputs(w):
    """Host copies of the workload's inputs (drawn on the host generator)."""
    return W.make_inputs(w, seed=0, device="cpu")


def run_reference(args, rank, world):
    if rank != 0:
        return
    w = W.workload(args.workload)
    fpp = F.flops_per_pair(w.d_qk, w.d_v)["fwd_bwd" if w.backward else "fwd"]
    what = "fwd+bwd" if w.backward else "fwd"
    x = cpu_inputs(w)
    for _ in range(args.warmup):
        oracle_sample(w, x, 1)
    times, pairs = [], 0
    for _ in range(args.steps):
        dt, p = oracle_sample(w, x, 1)
        times.append(dt)
        pairs += p
    total = sum(times)
    value = pairs * fpp / total / 1e12
    cores = os.cpu_count()
    sample = (f"{args.steps} x one (sequence, head) unit of {w.name} "
              f"({w.lengths_q[0]} rows, {what}, fp64 numpy; BLAS threads = host cores)")
    line = {"impl": "reference", "metric": f"attention TFLOP/s {what} (unmasked pairs)",
            "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1000 * total / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded N(0,1))", "config": config_of(w, world, l2_bytes_of()),
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


# ------------------------------------------------------------------------------ GPU arm
class Problem:
    """One workload's device inputs, results and the calls of one step through the library."""

    def __init__(self, vlf, w, dev, seed, flags=0):
        self.vlf, self.w, self.dev, self.flags = vlf, w, dev, flags
        x = W.make_inputs(w, seed=seed, device=dev, with_dout=True)
        self.latent_api = w.latent_split is not None and w.rope_heads is not None
        self.in_names = (("q_nope", "q_rope", "k_nope", "k_rope", "v") if self.latent_api
                         else ("q", "k", "v"))
        self.grad_of = dict(zip(("dq_nope", "dq_rope", "dk_nope", "dk_rope", "dv") if self.latent_api
                                else ("dq", "dk", "dv"), self.in_names))
        if self.latent_api:
            del x["q"], x["k"]  # the concatenated operands are not used
        self.x = x
        dt = x["v"].dtype
        self.dt = dt
        out = torch.empty((w.total_q, w.h_q, w.d_v), dtype=dt, device=dev)
        lse = torch.empty((w.h_q, w.total_q), dtype=torch.float32, device=dev)
        self.res = {"out": out, "lse": lse}
        if w.backward:
            self.res.update({g: torch.empty_like(x[n]) for g, n in self.grad_of.items()})
        ws_bytes = (vlf.vlf_attn_varlen_bwd_latent_workspace_size(
            w.total_q, w.total_kv, w.h_q, w.h_kv, w.rope_heads, dt) if self.latent_api else
            vlf.vlf_attn_varlen_bwd_workspace_size(w.total_q, w.total_kv, w.h_q, w.h_kv, w.d_qk,
                                                   w.d_v, dt))
        self.ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
        self.kw = dict(scale=w.scale, causal=w.causal, window=w.window, bias=x["bias"])
        # small-batch / decode shapes split each CTA's KV band (the library's choice); the parts'
        # workspace is allocated once, outside the timed region
        self.n_split = vlf.vlf_fwd_num_splits(w.num_seqs, w.max_seqlen_q, w.max_seqlen_kv, w.h_q,
                                              w.h_kv, w.d_qk, w.d_v, dt)
        self.fws = [torch.empty(max(1, vlf.vlf_attn_varlen_fwd_split_workspace_size(
            w.total_q, w.h_q, w.d_v, self.n_split)), dtype=torch.uint8, device=dev)
            for _ in range(2)]
        # a bias: its bands (which keys it leaves each row) are computed once per step, for the
        # forward and the backward, into a buffer allocated here
        self.bands = None
        if x["bias"] is not None:
            self.bands = torch.empty(max(16, vlf.vlf_bias_bands_size(w.total_q, w.bias_heads)),
                                     dtype=torch.uint8, device=dev)
        # per-step timing stages (consecutive events)
        self.stages = ((["bands"] if self.bands is not None else []) + ["fwd"] +
                       (list(vlf.BWD_STAGE_NAMES) if w.backward else []))

    def run(self, d=None, r=None, fw=None, st=None, ev=None, stream=None):
        """One step on inputs d into results r (the problem's own when None) on stream st (the
        current one when None); ev: per-stage timing events recorded on ``stream``."""
        vlf, w = self.vlf, self.w
        d = self.x if d is None else d
        r = self.res if r is None else r
        fw = self.fws[0] if fw is None else fw
        ops = [d[n] for n in self.in_names]
        cu = (d["cu_seqlens_q"], d["cu_seqlens_kv"], w.max_seqlen_q, w.max_seqlen_kv)
        kw = dict(self.kw, bias=d["bias"] if "bias" in d else self.kw["bias"], flags=self.flags)
        e = 1  # the next timing event to record after a stage
        if self.bands is not None:
            vlf.vlf_bias_bands(kw["bias"], d["cu_seqlens_q"], d["cu_seqlens_kv"], out=self.bands,
                               stream=st)
            kw["bias_bands"] = self.bands
            if ev is not None:
                ev[e].record(stream)
            e += 1
        if self.latent_api:
            vlf.vlf_attn_varlen_fwd_latent(*ops, *cu, out=r["out"], lse=r["lse"], stream=st, **kw)
        else:
            vlf.vlf_attn_varlen_fwd(*ops, *cu, out=r["out"], lse=r["lse"], stream=st,
                                    workspace=fw, num_splits=self.n_split, **kw)
        if not w.backward:
            if ev is not None:
                ev[e].record(stream)
            return
        sev = None if ev is None else ev[e:]
        if self.latent_api:
            vlf.vlf_attn_varlen_bwd_latent(d["dout"], *ops, r["out"], r["lse"], *cu,
                                           grads=tuple(r[g] for g in self.grad_of),
                                           workspace=self.ws, stream=st, stage_events=sev, **kw)
        else:
            vlf.vlf_attn_varlen_bwd(d["dout"], *ops, r["out"], r["lse"], *cu, dq=r["dq"],
                                    dk=r["dk"], dv=r["dv"], workspace=self.ws, stream=st,
                                    stage_events=sev, **kw)

    def algorithmic(self):
        """Per-kernel algorithmic FLOPs and bytes (the minimum each kernel moves: its tensors
        read and written once, plus the bias once per pass)."""
        w, x = self.w, self.x
        pairs = F.workload_pairs(w)
        fpp = F.flops_per_pair(w.d_qk, w.d_v)
        eb = x["v"].element_size()
        nq, nk = w.total_q * w.h_q, w.total_kv * w.h_kv
        q_b, k_b, v_b = nq * w.d_qk * eb, nk * w.d_qk * eb, nk * w.d_v * eb
        if self.latent_api:  # K as read: the nope parts and the (possibly shared) rope key
            k_b = (x["k_nope"].numel() + x["k_rope"].numel()) * eb
        o_b, row_b = nq * w.d_v * eb, 4 * nq                    # O (or dO), one fp32 per row
        bias_b = 0 if x["bias"] is None else x["bias"].numel() * 4
        flops = {"fwd": pairs * fpp["fwd"], "dkdv": pairs * fpp["dkdv"], "dq": pairs * fpp["dq"]}
        bytes_ = {"bands": bias_b,  # (at most: the pass stops scanning a row at its ends)
                  "fwd": q_b + k_b + v_b + o_b + row_b + bias_b,
                  "rowdot": 2 * o_b + row_b,
                  "dkdv": q_b + k_b + v_b + o_b + 2 * row_b + k_b + v_b + bias_b,
                  "dq": q_b + k_b + v_b + o_b + 2 * row_b + q_b + bias_b}
        return flops, bytes_


def roofline(prob, stage_ms, peaks, tensor_peak, dev):
    """The dominant stage's roofline: achieved algorithmic FLOP/s (or bytes/s) of its mean
    event-timed launch against the roof it is closer to."""
    vlf, w = prob.vlf, prob.w
    fwd_path = vlf.vlf_fwd_path(w.h_q, w.h_kv, w.d_qk, w.d_v, prob.dt)
    bwd_path = vlf.vlf_bwd_path(w.h_q, w.h_kv, w.d_qk, w.d_v, prob.dt)
    dom = max(stage_ms, key=stage_ms.get)
    flops_of, bytes_of = prob.algorithmic()
    tc = (fwd_path if dom == "fwd" else bwd_path) == 1
    sec = stage_ms[dom] * 1e-3
    hbm_frac = bytes_of[dom] / sec / 1e9 / peaks["hbm_gbs"]
    ten_roof = tensor_peak * (1.1 / 2.25) / 3.0 if w.dtype == "fp32" else tensor_peak
    ten_frac = flops_of.get(dom, 0) / sec / 1e12 / ten_roof
    if dom == "rowdot" or (tc and hbm_frac > ten_frac):
        roof = {"bound": "hbm", "achieved": bytes_of[dom] / sec / 1e9, "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "algorithmic_bytes": bytes_of[dom]}
    elif tc:
        roof = {"bound": "tensor", "achieved": flops_of[dom] / sec / 1e12, "peak": tensor_peak,
                "unit": "TFLOP/s", "algorithmic_flops": flops_of[dom]}
        if w.dtype == "fp32":
            # fp32 on the tensor cores: tf32 products (the bf16 roof x the nominal dense ratio
            # 1.1 / 2.25), three passes per product -- the roof of the algorithmic FLOPs
            roof["peak"] = tensor_peak * (1.1 / 2.25) / 3.0
    else:
        props = torch.cuda.get_device_properties(dev)
        alu_peak = props.multi_processor_count * 128 * 2 * 2070.0 * 1e6 / 1e12
        roof = {"bound": "alu", "achieved": flops_of[dom] / sec / 1e12, "peak": alu_peak,
                "unit": "TFLOP/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    if roof["bound"] == "tensor":
        roof["frac_of_burst"] = roof["achieved"] / peaks["bf16_tflops"]
    tr = ncu_traffic(dom, w.name) if tc or roof["bound"] == "hbm" else None
    roof["traffic"] = tr
    roof["kernel"] = dom
    roof["peak_source"] = peaks["source"] + (
        " (fp32 FMA: SMs x 128 lanes x 2 x 2070 MHz)" if roof["bound"] == "alu" else
        (" (tf32 = bf16 x 1.1/2.25 nominal ratio, / 3 passes per product)"
         if roof["bound"] == "tensor" and w.dtype == "fp32" else ""))
    return roof, {"fwd": "tcgen05" if fwd_path == 1 else "simt",
                  "bwd": "tcgen05" if bwd_path == 1 else "simt"}


def time_steps(prob, steps, stream, dev, world, flush_l2):
    """Time exactly ``steps`` steps (barrier + synchronize on both sides).  Returns the step
    time in ms (max over ranks), the per-stage mean times and the library launches counted."""
    vlf = prob.vlf
    n_ev = len(prob.stages) + 1
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(n_ev)] for _ in range(steps)]
    for row in evs:  # torch creates the CUDA event at its first record()
        for e in row:
            e.record(stream)
    flush_buf = torch.empty(2 * l2_bytes_of(dev), dtype=torch.uint8, device=dev) if flush_l2 else None
    barrier(world)
    torch.cuda.synchronize()
    n0 = vlf.vlf_launch_count()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    # the step time: events at the step boundaries only, so that a step's kernels follow one
    # another directly as in a user's call (an event recorded between two kernels keeps the
    # second from starting on the SMs the first one's last CTAs leave)
    t_start.record(stream)
    for i in range(steps):
        if flush_l2:
            flush_buf.zero_()  # (outside the step's own events)
        evs[i][0].record(stream)
        prob.run(stream=stream)
        evs[i][-1].record(stream)
    t_end.record(stream)
    torch.cuda.synchronize()
    launches = vlf.vlf_launch_count() - n0
    barrier(world)
    st = vlf.vlf_check_error()
    assert st == 0, vlf.vlf_status_string(st)
    if flush_l2:
        ms_step = max_over_ranks(statistics.mean(e[0].elapsed_time(e[-1]) for e in evs), world)
    else:
        ms_step = max_over_ranks(t_start.elapsed_time(t_end), world) / steps
    # the stage times: as many steps again, with an event between stages
    for i in range(steps):
        if flush_l2:
            flush_buf.zero_()
        evs[i][0].record(stream)
        prob.run(ev=evs[i], stream=stream)
    torch.cuda.synchronize()
    st = vlf.vlf_check_error()
    assert st == 0, vlf.vlf_status_string(st)
    stage_ms = {n: statistics.mean(e[i].elapsed_time(e[i + 1]) for e in evs)
                for i, n in enumerate(prob.stages)}
    return ms_step, stage_ms, launches


def measure(vlf, w, dev, world, steps, warmup, sampler, peaks, tensor_peak=None, seed=0,
            sustain_s=0.0):
    """Times ``steps`` steps of workload ``w`` after ``warmup`` (and, with sustain_s > 0, a
    sustained run of that many seconds right before the timed steps).  Returns the result
    record and the Problem (kept alive by the caller while it needs the buffers)."""
    stream = torch.cuda.current_stream()
    prob = Problem(vlf, w, dev, seed)
    for _ in range(warmup):
        prob.run()
    torch.cuda.synchronize()
    st = vlf.vlf_check_error()
    assert st == 0, vlf.vlf_status_string(st)
    flush = input_bytes(w) < 2 * l2_bytes_of(dev)
    t0 = time.time()
    sustained = None
    if sustain_s > 0:
        # the same step back to back for >= sustain_s seconds: the clocks it runs at are those
        # of a GPU under this load (the samples cover it and the timed steps after it)
        ms_guess, _, _ = time_steps(prob, 3, stream, dev, world, flush)
        n = max(3, int(math.ceil(sustain_s * 1e3 / ms_guess)))
        ms_s, _, _ = time_steps(prob, n, stream, dev, world, flush)
        sustained = {"steps": n, "ms_per_step": ms_s, "seconds": n * ms_s / 1e3}
    ms_step, stage_ms, launches = time_steps(prob, steps, stream, dev, world, flush)
    t1 = time.time()
    clocks = sampler.summary(t0, t1) if sampler else None
    if tensor_peak is None:
        tensor_peak, kind = peak_for(clocks, peaks)
    else:
        kind = "as the headline"
    pairs = F.workload_pairs(w)
    fpp = F.flops_per_pair(w.d_qk, w.d_v)
    step_flops = fpp["fwd_bwd"] if w.backward else fpp["fwd"]
    value = world * pairs * step_flops / (ms_step * 1e-3) / 1e12
    fwd_tflops = pairs * fpp["fwd"] / (stage_ms["fwd"] * 1e-3) / 1e12
    roof, paths = roofline(prob, stage_ms, peaks, tensor_peak, dev)
    if w.dtype == "fp32":
        # the same forward on the SIMT fp32-FMA kernels, for comparison with the tf32 passes
        prob.flags = vlf.VLF_FLAG_FORCE_SIMT
        _, st_simt, _ = time_steps(prob, max(2, steps // 2), stream, dev, world, flush)
        prob.flags = 0
    rec = {"workload": w.name, "step": "fwd+bwd" if w.backward else "fwd",
           "value": value, "unit": "TFLOP/s", "steps": steps, "warmup": warmup,
           "ms_per_step": ms_step, "fwd_tflops": fwd_tflops,
           "fwd_frac_of_peak": fwd_tflops / tensor_peak,
           "value_frac_of_peak": value / world / tensor_peak,
           "tensor_peak": tensor_peak, "tensor_peak_kind": kind,
           "fwd_frac_of_burst": fwd_tflops / peaks["bf16_tflops"],
           "value_frac_of_burst": value / world / peaks["bf16_tflops"],
           "stage_ms": stage_ms, "roofline": roof, "paths": paths, "kv_splits": prob.n_split,
           "clocks": clocks, "gpu_launches": launches,
           "l2": config_of(w, world, l2_bytes_of(dev))["l2"]}
    if w.dtype == "fp32":
        rec["fwd_tflops_simt"] = pairs * fpp["fwd"] / (st_simt["fwd"] * 1e-3) / 1e12
        rec["stage_ms_simt"] = st_simt
    if sustained is not None:
        sustained["value"] = world * pairs * step_flops / (sustained["ms_per_step"] * 1e-3) / 1e12
        rec["sustained"] = sustained
    return rec, prob


def latency(vlf, w, dev, calls=300, warmup=30):
    """Per-call latency of a tiny forward through the Python binding and the C ABI.
    device_us: event-timed call on an L2-flushed device (the flush keeps the GPU busy while
    the host enqueues the call, so only device time is seen); host_us: host time of the call
    (argument marshalling, the C ABI's checks and the launch, returning before the kernel
    ends); us_per_call: back-to-back calls, wall clock (host and device overlap)."""
    stream = torch.cuda.current_stream()
    prob = Problem(vlf, w, dev, seed=0)
    x, r = prob.x, prob.res
    args = (x["q"], x["k"], x["v"], x["cu_seqlens_q"], x["cu_seqlens_kv"], w.max_seqlen_q,
            w.max_seqlen_kv)
    kw = dict(scale=w.scale, causal=w.causal, window=w.window, out=r["out"], lse=r["lse"],
              num_splits=prob.n_split, workspace=prob.fws[0])
    fwd = vlf.vlf_attn_varlen_fwd

    def call():  # the public call as a user makes it
        fwd(*args, **kw)

    for _ in range(warmup):
        call()
    torch.cuda.synchronize()
    # back-to-back calls, inputs L2-resident
    t0 = time.perf_counter()
    for _ in range(calls):
        call()
    t1 = time.perf_counter()
    torch.cuda.synchronize()
    t2 = time.perf_counter()
    host_us = (t1 - t0) / calls * 1e6
    per_call = (t2 - t0) / calls * 1e6
    # device time per call, L2 flushed before each
    flush_buf = torch.empty(2 * l2_bytes_of(dev), dtype=torch.uint8, device=dev)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(calls)]
    n0 = vlf.vlf_launch_count()
    for a, b in ev:
        flush_buf.zero_()
        a.record(stream)
        call()
        b.record(stream)
    torch.cuda.synchronize()
    launches = (vlf.vlf_launch_count() - n0) / calls
    st = vlf.vlf_check_error()
    assert st == 0, vlf.vlf_status_string(st)
    dev_us = statistics.mean(a.elapsed_time(b) for a, b in ev) * 1e3
    pairs = F.workload_pairs(w)
    fl = pairs * F.flops_per_pair(w.d_qk, w.d_v)["fwd"]
    return {"workload": w.name, "step": "fwd", "us_per_call": per_call, "host_us": host_us,
            "device_us": dev_us, "launches_per_call": launches,
            "value": fl / (per_call * 1e-6) / 1e12, "device_tflops": fl / (dev_us * 1e-6) / 1e12,
            "unit": "TFLOP/s", "calls": calls, "warmup": warmup, "unmasked_pairs": pairs,
            "l2": "us_per_call / host_us: back-to-back calls, inputs L2-resident (0.9 MB); "
                  "device_us: L2 flushed before each call",
            "status": "latency-bound: far below the 60% forward target (a few microseconds of "
                      "work per call)"}


def e2e_measure(prob, steps, warmup, world, pairs, step_flops):
    """End to end through the public API with pinned host buffers: every step uploads its
    inputs and reads back all of its results (out, lse, dq, dk, dv) inside the timed region.
    Two device / host buffer sets and three streams pipeline the steps the way an input
    pipeline would: step k+1's upload and step k-1's read-back run on the copy engines while
    step k's kernels run.  (A bias, where a workload has one, stays resident like a weight.)"""
    x, w = prob.x, prob.w
    in_keys = prob.in_names + ("cu_seqlens_q", "cu_seqlens_kv") + (("dout",) if w.backward else ())
    res_like = prob.res
    host = {k: x[k].cpu().pin_memory() for k in in_keys}
    dset = [{k: torch.empty_like(x[k]) for k in in_keys} for _ in range(2)]
    rset = [{k: torch.empty_like(t) for k, t in res_like.items()} for _ in range(2)]
    hres = [{k: torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
             for k, t in res_like.items()} for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = sum(t.numel() * t.element_size() for t in hres[0].values())
    s_up, s_cmp, s_dn = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev_up = [torch.cuda.Event() for _ in range(2)]
    ev_cmp = [torch.cuda.Event() for _ in range(2)]
    ev_dn = [torch.cuda.Event() for _ in range(2)]
    cur = torch.cuda.current_stream()
    for e in ev_cmp + ev_dn:
        e.record(cur)  # both sets start free
    torch.cuda.synchronize()

    def e2e_step(step):
        i = step % 2
        d, r, h = dset[i], rset[i], hres[i]
        with torch.cuda.stream(s_up):
            s_up.wait_event(ev_cmp[i])  # the kernels of step - 2 are done with set i
            for k in in_keys:
                d[k].copy_(host[k], non_blocking=True)
            ev_up[i].record(s_up)
        s_cmp.wait_event(ev_up[i])
        s_cmp.wait_event(ev_dn[i])  # the read-back of step - 2 is done with set i
        prob.run(d=d, r=r, fw=prob.fws[i], st=s_cmp)
        ev_cmp[i].record(s_cmp)
        with torch.cuda.stream(s_dn):
            s_dn.wait_event(ev_cmp[i])
            for k in res_like:
                h[k].copy_(r[k], non_blocking=True)
            ev_dn[i].record(s_dn)

    for it in range(warmup):
        e2e_step(it)
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(s_up)
    for it in range(steps):
        e2e_step(it)
    b.record(s_dn)  # after the last read-back, which follows every other stream's work
    torch.cuda.synchronize()
    barrier(world)
    e2e_ms = max_over_ranks(a.elapsed_time(b), world) / steps
    return {"value": world * pairs * step_flops / (e2e_ms * 1e-3) / 1e12,
            "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": e2e_ms, "pipelined": "upload / kernels / read-back of consecutive "
                                                "steps overlap (3 streams, 2 buffer sets)"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=WORKLOAD)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="headline workload only (skip the other configurations)")
    ap.add_argument("--configs", default=None,
                    help="comma-separated subset of the other configurations to time")
    ap.add_argument("--sustain", type=float, default=SUSTAIN_S,
                    help="seconds of the sustained run before the timed steps (clock evidence)")
    ap.add_argument("--cpu-units", type=int, default=20,
                    help="(sequence, head) units of the workload for the CPU oracle baseline")
    args = ap.parse_args()
    rank, world, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    assert args.warmup >= 3, "at least 3 warm-up steps"

    import variable_length_flash_gb300 as vlf
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    w = W.workload(args.workload)
    peaks = load_peaks()
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)

    head, prob = measure(vlf, w, dev, world, args.steps, args.warmup, sampler, peaks,
                         sustain_s=args.sustain)
    pairs = F.workload_pairs(w)
    fpp = F.flops_per_pair(w.d_qk, w.d_v)
    step_flops = fpp["fwd_bwd"] if w.backward else fpp["fwd"]
    e2e = None if args.no_e2e else e2e_measure(prob, args.steps, args.warmup, world, pairs,
                                               step_flops)
    del prob
    torch.cuda.empty_cache()

    configs = {}
    if world == 1 and not args.no_configs:
        names = [c[0] for c in CONFIGS] + LATENCY_CONFIGS
        want = set(args.configs.split(",")) if args.configs else set(names)
        for name in LATENCY_CONFIGS:
            if name in want and name != w.name:
                configs[name] = latency(vlf, W.workload(name), dev)
        for name, steps, warm in CONFIGS:
            if name not in want or name == w.name:
                continue
            rec, p = measure(vlf, W.workload(name), dev, world, steps, warm, sampler, peaks,
                             tensor_peak=head["tensor_peak"])
            del p
            torch.cuda.empty_cache()
            configs[name] = rec
    sampler.stop()

    cpu = None
    if rank == 0 and world == 1 and args.cpu_units > 0:
        xc = cpu_inputs(w)
        secs, p = oracle_sample(w, xc, args.cpu_units)
        cpu = {"value": p * step_flops / secs / 1e12, "unit": "TFLOP/s",
               "cores": os.cpu_count(), "kind": "oracle",
               "sample": f"{args.cpu_units} (sequence, head) units of {w.name}, "
                         f"{'fwd' if not w.backward else 'fwd+bwd'}, fp64 numpy, {secs:.1f} s"}

    if rank == 0:
        line = {
            "metric": "attention TFLOP/s " + ("fwd+bwd" if w.backward else "fwd") + " (unmasked pairs)",
            "value": head["value"], "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": head["ms_per_step"], "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
            "data": "synthetic (seeded N(0,1))", "config": config_of(w, world, l2_bytes_of(dev)),
            "paths": dict(head["paths"], kv_splits=head["kv_splits"]),
            "fwd_tflops": head["fwd_tflops"], "fwd_frac_of_peak": head["fwd_frac_of_peak"],
            "fwd_bwd_frac_of_peak": head["value_frac_of_peak"],
            "tensor_peak": head["tensor_peak"], "tensor_peak_kind": head["tensor_peak_kind"],
            "fwd_frac_of_burst": head["fwd_frac_of_burst"],
            "fwd_bwd_frac_of_burst": head["value_frac_of_burst"],
            "stage_ms": head["stage_ms"], "roofline": head["roofline"], "cpu_baseline": cpu,
            "e2e": e2e, "clocks": head["clocks"], "sustained": head.get("sustained"),
            "gpu_launches": head["gpu_launches"], "configs": configs,
        }
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
