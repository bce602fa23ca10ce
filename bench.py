"""Benchmark: varlen flash attention forward + backward on one GB300 (or N replicas).

One step = one pass of the whole hot path over one batch: forward (out, lse) then backward
(row-dot pre-pass, dK/dV, dQ), on the dense causal workload B=4 x L=4096, H=32, head_dim 128,
bf16, packed as 4 cu_seqlens segments (inputs are synthetic, seeded, resident in HBM; each of
q/k/v/out/dout is 134 MB, larger than the 129 MB L2, so no flush is needed between steps).

Prints ONE JSON line (rank 0):
  value        fwd+bwd TFLOP/s over unmasked pairs (whole job, all ranks), CUDA-event timed
  fwd_tflops   forward-only TFLOP/s from the same timed region
  e2e          same metric through the C ABI with pinned host buffers, H2D/D2H inside the timing
  roofline     dominant kernel: algorithmic FLOPs per launch / its average event-timed duration
  cpu_baseline the fp64 oracle (test infrastructure) on a bounded sample, host cores
  clocks       nvidia-smi samples taken during the timed region

``--impl reference`` times the fp64 CPU oracle on the same workload instead (rank 0 only).
Multi-GPU (torchrun): every rank runs its own replica of the workload (weak scaling; the
ranks exchange nothing in the data path; a barrier and a max-reduce of the timing only).
"""
from __future__ import annotations

import argparse
import json
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
from variable_length_flash_gb300 import flops as F  # noqa: E402

WORKLOAD = "dense4x4096_bf16_causal"


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
    k = rec.get("kernels", {}).get(role)
    if k is None or rec.get("workload") != workload:
        return None
    h = hashlib.sha256()
    for f in k["source_files"]:
        fp = os.path.join(ROOT, "variable_length_flash_gb300", "csrc", f)
        if not os.path.exists(fp):
            return None
        h.update(open(fp, "rb").read())
    return k["dram_bytes_per_launch"] if h.hexdigest() == k["source_sha256"] else None


class ClockSampler:
    """nvidia-smi SM clock / throttle-reason samples every 200 ms while running."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index, self.rows, self.proc, self.thread = index, [], None, None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
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
                self.rows.append(parts)

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm = [float(r[0]) for r in self.rows if r[0].replace(".", "", 1).isdigit()]
        mx = [float(r[1]) for r in self.rows if r[1].replace(".", "", 1).isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in self.rows for n, v in zip(names, r[4:8]) if v == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(self.rows)}


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


def cpu_inputs(w, units):
    """Host copies of the sequences the CPU sample touches (drawn on the host generator)."""
    return W.make_inputs(w, seed=0, device="cpu")


def run_reference(args, rank, world):
    if rank != 0:
        return
    w = W.workload(args.workload)
    fpp = F.flops_per_pair(w.d_qk, w.d_v)["fwd_bwd" if w.backward else "fwd"]
    what = "fwd+bwd" if w.backward else "fwd"
    x = cpu_inputs(w, 1)
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
            "data": "synthetic", "config": {"workload": w.name},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


# ------------------------------------------------------------------------------ GPU arm
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=WORKLOAD)
    ap.add_argument("--no-e2e", action="store_true")
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
    stream = torch.cuda.current_stream()
    w = W.workload(args.workload)
    x = W.make_inputs(w, seed=rank, device=dev, with_dout=True)
    fpp = F.flops_per_pair(w.d_qk, w.d_v)
    pairs = F.workload_pairs(w)
    dt = x["q"].dtype
    # a latent workload with a given rope_heads goes through the split-operand calls (its
    # operands as produced, the rope key possibly shared); the others through the plain calls
    latent_api = w.latent_split is not None and w.rope_heads is not None
    in_names = ("q_nope", "q_rope", "k_nope", "k_rope", "v") if latent_api else ("q", "k", "v")
    grad_of = dict(zip(("dq_nope", "dq_rope", "dk_nope", "dk_rope", "dv") if latent_api
                       else ("dq", "dk", "dv"), in_names))
    if latent_api:
        del x["q"], x["k"]  # the concatenated operands are not used
    out = torch.empty((w.total_q, w.h_q, w.d_v), dtype=dt, device=dev)
    lse = torch.empty((w.h_q, w.total_q), dtype=torch.float32, device=dev)
    res0 = {"out": out, "lse": lse, **{g: torch.empty_like(x[n]) for g, n in grad_of.items()}}
    ws_bytes = (vlf.vlf_attn_varlen_bwd_latent_workspace_size(
        w.total_q, w.total_kv, w.h_q, w.h_kv, w.rope_heads, dt) if latent_api else
        vlf.vlf_attn_varlen_bwd_workspace_size(w.total_q, w.total_kv, w.h_q, w.h_kv, w.d_qk,
                                               w.d_v, dt))
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
    kw = dict(scale=w.scale, causal=w.causal, window=w.window, bias=x["bias"])
    # small-batch / decode shapes split each CTA's KV band (the library's choice); the parts'
    # workspace is allocated once, outside the timed region
    n_split = vlf.vlf_fwd_num_splits(w.num_seqs, w.max_seqlen_q, w.max_seqlen_kv, w.h_q, w.h_kv,
                                     w.d_qk, w.d_v, dt)
    fws = [torch.empty(max(1, vlf.vlf_attn_varlen_fwd_split_workspace_size(
        w.total_q, w.h_q, w.d_v, n_split)), dtype=torch.uint8, device=dev) for _ in range(2)]
    fkw = dict(num_splits=n_split)

    # a step is the forward and the backward; workloads without a backward (decode-sized,
    # latency-bound) time the forward alone
    fwd_only = not w.backward

    def run(d, r, fw, st=None, ev=None):
        """One step on inputs d into results r through the library's calls (on stream st, the
        current one when None); ev: per-stage timing events."""
        ops = [d[n] for n in in_names]
        cu = (d["cu_seqlens_q"], d["cu_seqlens_kv"], w.max_seqlen_q, w.max_seqlen_kv)
        if latent_api:
            vlf.vlf_attn_varlen_fwd_latent(*ops, *cu, out=r["out"], lse=r["lse"], stream=st, **kw)
        else:
            vlf.vlf_attn_varlen_fwd(*ops, *cu, out=r["out"], lse=r["lse"], stream=st,
                                    workspace=fw, **fkw, **kw)
        if fwd_only:
            if ev is not None:
                ev[1].record(stream)
            return
        sev = None if ev is None else ev[1:]
        if latent_api:
            vlf.vlf_attn_varlen_bwd_latent(d["dout"], *ops, r["out"], r["lse"], *cu,
                                           grads=tuple(r[g] for g in grad_of), workspace=ws,
                                           stream=st, stage_events=sev, **kw)
        else:
            vlf.vlf_attn_varlen_bwd(d["dout"], *ops, r["out"], r["lse"], *cu, dq=r["dq"],
                                    dk=r["dk"], dv=r["dv"], workspace=ws, stream=st,
                                    stage_events=sev, **kw)

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        run(x, res0, fws[0], ev=ev)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    st = vlf.vlf_check_error()
    assert st == 0, vlf.vlf_status_string(st)

    # events: per step [fwd start, bwd start(=fwd end), after rowdot, after dkdv, after dq]
    n_ev = 2 if fwd_only else 2 + vlf.VLF_BWD_STAGES
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(n_ev)] for _ in range(args.steps)]
    for row in evs:  # torch creates the CUDA event at its first record()
        for e in row:
            e.record(stream)
    sampler = ClockSampler(local)
    barrier(world)
    torch.cuda.synchronize()
    sampler.start()
    time.sleep(0.3)
    n0 = vlf.vlf_launch_count()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    # Inputs larger than L2 stream from HBM every step; smaller ones would stay in L2, so between
    # their timed steps a buffer twice the L2 size is overwritten (outside each step's events)
    # and the step time is the mean of the per-step event times.
    l2_bytes = torch.cuda.get_device_properties(dev).L2_cache_size
    in_bytes = sum(t.numel() * t.element_size() for t in [x[n] for n in in_names] +
                   [x["dout"], x["bias"]] if t is not None)
    flush = in_bytes < 2 * l2_bytes
    flush_buf = torch.empty(2 * l2_bytes, dtype=torch.uint8, device=dev) if flush else None
    t_start.record(stream)
    for i in range(args.steps):
        if flush:
            flush_buf.zero_()
        step(evs[i])
    t_end.record(stream)
    torch.cuda.synchronize()
    launches = vlf.vlf_launch_count() - n0
    barrier(world)
    clocks = sampler.stop()
    st = vlf.vlf_check_error()
    assert st == 0, vlf.vlf_status_string(st)
    if flush:
        ms_step = max_over_ranks(statistics.mean(e[0].elapsed_time(e[-1]) for e in evs), world)
    else:
        ms_step = max_over_ranks(t_start.elapsed_time(t_end), world) / args.steps
    stage_names = ["fwd"] + ([] if fwd_only else list(vlf.BWD_STAGE_NAMES))
    stage_ms = {n: statistics.mean(e[i].elapsed_time(e[i + 1]) for e in evs)
                for i, n in enumerate(stage_names)}
    fwd_ms = stage_ms["fwd"]
    step_flops = fpp["fwd"] if fwd_only else fpp["fwd_bwd"]
    value = world * pairs * step_flops / (ms_step * 1e-3) / 1e12
    fwd_tflops = pairs * fpp["fwd"] / (fwd_ms * 1e-3) / 1e12

    # roofline of the dominant kernel (one launch per stage per step)
    peaks = load_peaks()
    fwd_path = vlf.vlf_fwd_path(w.h_q, w.h_kv, w.d_qk, w.d_v, dt)
    bwd_path = vlf.vlf_bwd_path(w.h_q, w.h_kv, w.d_qk, w.d_v, dt)
    dom = max(stage_ms, key=stage_ms.get)
    flops_of = {"fwd": pairs * fpp["fwd"], "dkdv": pairs * fpp["dkdv"], "dq": pairs * fpp["dq"]}
    tc = (fwd_path if dom == "fwd" else bwd_path) == 1
    # Algorithmic bytes per kernel launch (the minimum it moves): its tensors read and written
    # once, plus the bias once per pass where there is one.
    eb = x["v"].element_size()
    nq, nk = w.total_q * w.h_q, w.total_kv * w.h_kv
    q_b, k_b, v_b = nq * w.d_qk * eb, nk * w.d_qk * eb, nk * w.d_v * eb
    if latent_api:  # K as read: the nope parts and the (possibly shared) rope key
        k_b = (x["k_nope"].numel() + x["k_rope"].numel()) * eb
    o_b, row_b = nq * w.d_v * eb, 4 * nq                    # O (or dO), one fp32 per row
    bias_b = 0 if x["bias"] is None else x["bias"].numel() * 4
    bytes_of = {"fwd": q_b + k_b + v_b + o_b + row_b + bias_b,
                "rowdot": 2 * o_b + row_b,
                "dkdv": q_b + k_b + v_b + o_b + 2 * row_b + k_b + v_b + bias_b,
                "dq": q_b + k_b + v_b + o_b + 2 * row_b + q_b + bias_b}
    # the bound is the roof the kernel is closer to: HBM for the row-dot, decode-sized forwards
    # and bias streaming, the tensor cores for the rest
    hbm_frac = bytes_of[dom] / (stage_ms[dom] * 1e-3) / 1e9 / peaks["hbm_gbs"]
    ten_frac = flops_of.get(dom, 0) / (stage_ms[dom] * 1e-3) / 1e12 / peaks["bf16_tflops"]
    if dom == "rowdot" or (tc and hbm_frac > ten_frac):
        achieved = bytes_of[dom] / (stage_ms[dom] * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "algorithmic_bytes": bytes_of[dom]}
    elif tc:
        achieved = flops_of[dom] / (stage_ms[dom] * 1e-3) / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"],
                "unit": "TFLOP/s"}
    else:
        props = torch.cuda.get_device_properties(dev)
        sm_max = (clocks or {}).get("sm_max_mhz") or 2070.0
        alu_peak = props.multi_processor_count * 128 * 2 * sm_max * 1e6 / 1e12
        achieved = flops_of[dom] / (stage_ms[dom] * 1e-3) / 1e12
        roof = {"bound": "alu", "achieved": achieved, "peak": alu_peak, "unit": "TFLOP/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["traffic"] = ncu_traffic(dom, w.name) if tc or roof["bound"] == "hbm" else None
    roof["kernel"] = dom
    roof["peak_source"] = peaks["source"] + (" (fp32 FMA: SMs x 128 lanes x 2 x max SM clock)"
                                             if roof["bound"] == "alu" else "")

    # end to end through the C ABI with pinned host buffers
    e2e = None
    if not args.no_e2e:
        # End to end through the public API with pinned host buffers: every step uploads its
        # inputs and reads back all of its results (out, lse, dq, dk, dv) inside the timed
        # region.  Two device / host buffer sets and three streams pipeline the steps the way an
        # input pipeline would: step k+1's upload and step k-1's read-back run on the copy
        # engines while step k's kernels run.  (The bias, where a workload has one, stays
        # resident like a weight.)
        in_keys = in_names + ("cu_seqlens_q", "cu_seqlens_kv") + (() if fwd_only else ("dout",))
        res_like = {"out": out, "lse": lse} if fwd_only else res0
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
        for e in ev_cmp + ev_dn:
            e.record(stream)  # both sets start free
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
            run(d, r, fws[i], st=s_cmp)
            ev_cmp[i].record(s_cmp)
            with torch.cuda.stream(s_dn):
                s_dn.wait_event(ev_cmp[i])
                for k in res_like:
                    h[k].copy_(r[k], non_blocking=True)
                ev_dn[i].record(s_dn)

        for it in range(args.warmup):
            e2e_step(it)
        torch.cuda.synchronize()
        barrier(world)
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(s_up)
        for it in range(args.steps):
            e2e_step(it)
        b.record(s_dn)  # after the last read-back, which follows every other stream's work
        torch.cuda.synchronize()
        barrier(world)
        e2e_ms = max_over_ranks(a.elapsed_time(b), world) / args.steps
        e2e = {"value": world * pairs * step_flops / (e2e_ms * 1e-3) / 1e12,
               "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": e2e_ms, "pipelined": "upload / kernels / read-back of consecutive "
                                                   "steps overlap (3 streams, 2 buffer sets)"}

    cpu = None
    if rank == 0 and world == 1 and args.cpu_units > 0:
        xc = cpu_inputs(w, args.cpu_units)
        secs, p = oracle_sample(w, xc, args.cpu_units)
        cpu = {"value": p * step_flops / secs / 1e12, "unit": "TFLOP/s",
               "cores": os.cpu_count(), "kind": "oracle",
               "sample": f"{args.cpu_units} (sequence, head) units of {w.name}, "
                         f"{'fwd' if fwd_only else 'fwd+bwd'}, fp64 numpy, {secs:.1f} s"}

    if rank == 0:
        line = {
            "metric": "attention TFLOP/s " + ("fwd" if fwd_only else "fwd+bwd") + " (unmasked pairs)",
            "value": value,
            "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": w.dtype, "data": "synthetic (seeded N(0,1))",
            "config": {"workload": w.name, "lengths": sorted(set(w.lengths_q)),
                       "num_seqs": w.num_seqs, "h_q": w.h_q, "h_kv": w.h_kv, "d_qk": w.d_qk,
                       "d_v": w.d_v, "causal": w.causal, "window": w.window,
                       "unmasked_pairs": pairs, "parallelism": f"replicas x{world}",
                       "l2": (f"inputs {in_bytes / 1e6:.1f} MB < 2 x L2: L2 flushed between "
                              f"timed steps (a {2 * l2_bytes / 1e6:.0f} MB write), per-step events"
                              if flush else f"inputs {in_bytes / 1e6:.0f} MB > 2 x L2 "
                              f"({l2_bytes / 1e6:.0f} MB): streamed from HBM, no flush"),
                       "fwd_path": "tcgen05" if fwd_path == 1 else "simt",
                       "kv_splits": n_split,
                       "bwd_path": "tcgen05" if bwd_path == 1 else "simt"},
            "fwd_tflops": fwd_tflops, "fwd_frac_of_peak": fwd_tflops / peaks["bf16_tflops"],
            "fwd_bwd_frac_of_peak": value / world / peaks["bf16_tflops"],
            "stage_ms": stage_ms, "roofline": roof, "cpu_baseline": cpu, "e2e": e2e,
            "clocks": clocks, "gpu_launches": launches,
        }
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
