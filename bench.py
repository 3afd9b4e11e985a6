"""Benchmark of the GDN chunked-prefill forward on GB300.

`python bench.py --gpus N --steps K --warmup W` prints one JSON line.

A step is one whole forward (every kernel of the path) over the 1 x 32768,
h_qk = 2, h_v = 8 workload (the first row of the FlashQLA pages' forward
benchmark table), seeded synthetic inputs resident in HBM, AutoCP planning.
The L2 cache (129 MB) is flushed by writing a 256 MB buffer before every
timed step; each step is timed with CUDA events on its stream.  `e2e`
repeats the measurement through the public call with pinned host buffers,
host-to-device copies of the inputs and device-to-host copies of o and the
final state inside the timed region.  Under torchrun (N > 1) every rank runs
an independent replica (the layer needs no collective) and the slowest
rank's time is used.

The line also carries, for every workload: its time and roofline fraction;
the AutoCP modes of the varlen workload (time and distance from exact); the
decode step over a batch of 256 states; `graphs`: microseconds per call of the
tiny forward and of the decode step, called eagerly and replayed from a CUDA
graph that captured 20 calls; the fp32 path's time on the headline
workload; the host planning time; the backward (`backward`: gdn_chunk_bwd with
its forward recompute on the headline and four other workloads, per-kernel
times, its roofline fraction, a training step of gdn_chunk_fwd(for_backward)
then gdn_chunk_bwd(reuse_forward), and its gradients against the float64
oracle's); and, from the CPU-baseline leg (which runs the float64 oracle on
the host cores anyway), the raw max|diff|/RMS of o and of the final state
against the oracle and the excess over bf16's half-ulp store rounding.

`--only NAME` times just one case (a workload name, `decode`, `graphs`, `f32`, `bwd` or
`bwd:NAME`) and prints a short line: the entry point of the ncu captures
under profiles/.

`--impl reference` times the float64 CPU oracle on the host cores instead,
one bounded sample of the same workload per step.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "GDN chunked-prefill fwd tokens/s at T=32768 (h_qk/h_v sweep); % of roofline"
HEADLINE = "T32768_h2x8"
SWEEP = ["T32768_h8x24_h0", "T32768_h16x16", "varlen4_T348160_h2x8", "batch8_T4096_h8x32"]
# FlashQLA on an NVIDIA H200, same workloads (pages' benchmark table), ms per call.
PAGES_H200_MS = {"T32768_h2x8": 0.310, "T32768_h8x24_h0": 0.659, "T32768_h16x16": 0.493}
FLUSH_BYTES = 256 << 20
C, D = 64, 128


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            m = json.load(f)
        return float(m["hbm_gbs"]), float(m["bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, 1900.0, "fallback"


def algorithmic(w):
    """Bytes and FLOPs one forward must move / do: q,k,v,g,beta read, o and the
    final state written (the initial state read when given); the chunked
    algorithm's contractions counted once."""
    T, hqk, hv, n = w.T, w.h_qk, w.h_v, w.n_seqs
    by = T * (2 * hqk * D * 2 + 2 * hv * D * 2 + 2 * hv * 4) + n * hv * D * D * 4
    if w.h0 is not None:
        by += n * hv * D * D * 4
    fl = T * (hv * (6 * C * D + 6 * D * D + C * C / 3) + hqk * 4 * C * D)
    return by, fl


def algorithmic_bwd(w):
    """Bytes and FLOPs the backward must move / do: q, k, v, g, beta and d_out
    read, dq, dk, dv, dg, dbeta written (h0, dh_T read and dh0 written per
    state); the forward's contractions once more (the recompute) plus the
    chunked backward's: per token and value head 12 d^2 + 14 C d + 2 C^2
    (K~D, Q^T dO, W^T dV', dO H^T, V' D^T, Y_U H^T; P^T dO, dO V'^T, (dP*Gam) K,
    (dP*Gam)^T Q, A^T dV', dV' V'^T, the symmetrised dKK K; A^T (dV' V'^T))."""
    T, hqk, hv, n = w.T, w.h_qk, w.h_v, w.n_seqs
    by = T * (2 * (2 * hqk * D * 2) + 3 * hv * D * 2 + 4 * hv * 4) + n * hv * D * D * 4 * 2
    if w.h0 is not None:
        by += n * hv * D * D * 4
    _, fl_fwd = algorithmic(w)
    fl = fl_fwd + T * hv * (12 * D * D + 14 * C * D + 2 * C * C)
    return by, fl


# Each kernel's share of the layer's algorithmic bytes (the inputs it reads
# and outputs it writes that the layer must move anyway): the WY kernel reads
# q, k, v, g and beta, the output scans write o and the states.  The chunk
# records the WY kernel writes and the scans read back, the context-parallel
# transitions and the combine are overhead and count zero.
KERNEL_SOURCE = {"wy": "gdn_wy.cu", "scan_out": "gdn_scan.cu", "scan_prep": "gdn_scan.cu",
                 "combine": "gdn_combine.cu", "chunk_map": "gdn_wy.cu"}


def kernel_bytes(name, w):
    """name's share of the algorithmic bytes: the WY kernel reads q, k, v, g
    and beta, the output scan writes o and the final state (and reads the
    initial state); the other kernels move only intermediate data."""
    T, hqk, hv, n = w.T, w.h_qk, w.h_v, w.n_seqs
    if name == "wy":  # q, k (once per query/key head), v, g, beta
        return T * (2 * hqk * D * 2 + hv * D * 2 + 2 * hv * 4)
    per_head_state = D * D * 4 * (2 if w.h0 is not None else 1)
    if name == "scan_out":  # o out, the final state, and the initial state when given
        return T * hv * D * 2 + n * hv * per_head_state
    return 0


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device):
        self.rows = []
        self.proc = None
        sel = []
        try:
            uuid = str(torch.cuda.get_device_properties(device).uuid)
            sel = ["-i", uuid if uuid.startswith("GPU-") else "GPU-" + uuid]
        except Exception:
            pass
        self.cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100",
                    *sel]

    def start(self):
        try:
            self.proc = subprocess.Popen(self.cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 9:
                self.rows.append(parts)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.t.join(timeout=5)
        num = lambda x: x.replace(".", "", 1).isdigit()
        sm = [float(r[1]) for r in self.rows if num(r[1])]
        mx = [float(r[2]) for r in self.rows if num(r[2])]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in self.rows for i in range(4) if r[5 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(self.rows)}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
    return world, rank, local


def max_over_ranks(x: float, world: int, device) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def time_gpu(name, steps, warmup, device, cp="auto", lambda_=0.0, trace=True, tol_rule="noise"):
    """Times the forward on one workload; returns a dict of measurements."""
    from gated_deltanet_linear_fwd_gb300 import (gdn_chunk_fwd, gdn_cp_head_modes, gdn_cp_plan,
                                                 gdn_get_device_status, gdn_set_trace_events, gdn_trace_last)
    from gated_deltanet_linear_fwd_gb300.inputs import workload
    w = workload(name)
    d = w.to(device)
    plan = gdn_cp_plan(T=w.T, h_qk=w.h_qk, h_v=w.h_v, cu_seqlens=w.cu_seqlens, mode=cp, lambda_=lambda_,
                       tol_rule=tol_rule)
    ws = torch.empty(max(plan.workspace_bytes, 256), dtype=torch.uint8, device=device)
    out = torch.empty_like(d.v)
    hT = torch.empty(w.n_seqs, w.h_v, D, D, dtype=torch.float32, device=device)
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream(device)

    def fwd():
        gdn_chunk_fwd(d.q, d.k, d.v, d.g, d.beta, d.h0, d.cu_seqlens, plan=plan, out=out, final_state=hT,
                      workspace=ws)

    for _ in range(warmup):
        flush.zero_()
        fwd()
    torch.cuda.synchronize(device)
    code, detail = gdn_get_device_status(ws)
    names = gdn_trace_last()
    n_k = len(names)
    # the timed steps run without events between the kernels (they would keep
    # each kernel from starting before the one before it has drained)
    per_step = []
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for _ in range(steps):
        flush.zero_()
        s0.record(stream)
        fwd()
        s1.record(stream)
        s1.synchronize()
        per_step.append(s0.elapsed_time(s1))
    # the per-kernel split: separate steps with a pair of events around every
    # kernel, on the stream it runs on (with warmup heads, the output scan of
    # those heads runs beside the exact heads' kernels, so the times overlap)
    per_kernel = [0.0] * n_k
    trace_steps = max(5, steps // 4) if trace else 0
    if trace:
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(2 * n_k)]
        for e in ev:
            e.record(stream)
        torch.cuda.synchronize(device)
        gdn_set_trace_events(ev)
        for _ in range(trace_steps):
            flush.zero_()
            fwd()
            torch.cuda.synchronize(device)
            for i in range(n_k):
                per_kernel[i] += ev[2 * i].elapsed_time(ev[2 * i + 1])
        gdn_set_trace_events([])
    code2, detail2 = gdn_get_device_status(ws)
    modes, _ = gdn_cp_head_modes(ws, plan)
    by, fl = algorithmic(w)
    return {"workload": name, "w": w, "plan": plan, "ms": statistics.mean(per_step),
            "ms_median": statistics.median(per_step),
            "kernel_ms": {n: t / trace_steps for n, t in zip(names, per_kernel)} if trace else {},
            "launches": n_k, "status": (code, detail, code2, detail2), "bytes": by, "flops": fl,
            "modes": modes.flatten().tolist(), "tokens": w.T}


VARLEN = "varlen4_T348160_h2x8"
BWD_SWEEP = ["T32768_h8x24_h0", "T32768_h16x16", "varlen4_T348160_h2x8", "batch8_T4096_h8x32"]


def time_bwd(name, steps, warmup, device, cp="auto"):
    """Times the backward (gdn_chunk_bwd, its forward recompute included) on one
    workload with seeded upstream gradients d_out and d_final_state."""
    from gated_deltanet_linear_fwd_gb300 import (gdn_bwd_workspace_bytes, gdn_chunk_bwd, gdn_cp_plan,
                                                 gdn_get_device_status, gdn_set_trace_events, gdn_trace_last)
    from gated_deltanet_linear_fwd_gb300.inputs import make_output_grads, workload
    w = workload(name)
    d = w.to(device)
    d_out, dhT = make_output_grads(w)
    d_out, dhT = d_out.to(device), dhT.to(device)
    plan = gdn_cp_plan(T=w.T, h_qk=w.h_qk, h_v=w.h_v, cu_seqlens=w.cu_seqlens, mode=cp)
    ws = torch.empty(gdn_bwd_workspace_bytes(plan), dtype=torch.uint8, device=device)
    grads = (torch.empty_like(d.q), torch.empty_like(d.k), torch.empty_like(d.v), torch.empty_like(d.g),
             torch.empty_like(d.beta), torch.empty(w.n_seqs, w.h_v, D, D, dtype=torch.float32, device=device))
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream(device)

    def bwd():
        gdn_chunk_bwd(d.q, d.k, d.v, d.g, d.beta, d_out, d.h0, dhT, d.cu_seqlens, plan=plan, grads=grads,
                      workspace=ws)

    for _ in range(warmup):
        flush.zero_()
        bwd()
    torch.cuda.synchronize(device)
    names = gdn_trace_last()
    per_step = []
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for _ in range(steps):
        flush.zero_()
        s0.record(stream)
        bwd()
        s1.record(stream)
        s1.synchronize()
        per_step.append(s0.elapsed_time(s1))
    n_k, trace_steps = len(names), max(3, steps // 4)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2 * n_k)]
    for e in ev:
        e.record(stream)
    torch.cuda.synchronize(device)
    gdn_set_trace_events(ev)
    per_kernel = [0.0] * n_k
    for _ in range(trace_steps):
        flush.zero_()
        bwd()
        torch.cuda.synchronize(device)
        for i in range(n_k):
            per_kernel[i] += ev[2 * i].elapsed_time(ev[2 * i + 1])
    gdn_set_trace_events([])
    code, detail = gdn_get_device_status(ws)
    by, fl = algorithmic_bwd(w)
    return {"workload": name, "ms": statistics.mean(per_step), "ms_median": statistics.median(per_step),
            "kernel_ms": {n: t / trace_steps for n, t in zip(names, per_kernel)}, "status": [code, detail],
            "bytes": by, "flops": fl, "tokens": w.T, "segments": plan.n_seg_total,
            "grads": [x.cpu() for x in grads]}


def time_train_step(name, steps, warmup, device, cp="auto"):
    """A training step as a user runs it: gdn_chunk_fwd(for_backward=True), then
    gdn_chunk_bwd(reuse_forward=True) on the same plan and workspace (no recompute);
    also the training forward alone."""
    from gated_deltanet_linear_fwd_gb300 import gdn_bwd_workspace_bytes, gdn_chunk_bwd, gdn_chunk_fwd, gdn_cp_plan
    from gated_deltanet_linear_fwd_gb300.inputs import make_output_grads, workload
    w = workload(name)
    d = w.to(device)
    d_out, dhT = make_output_grads(w)
    d_out, dhT = d_out.to(device), dhT.to(device)
    plan = gdn_cp_plan(T=w.T, h_qk=w.h_qk, h_v=w.h_v, cu_seqlens=w.cu_seqlens, mode=cp)
    ws = torch.empty(gdn_bwd_workspace_bytes(plan), dtype=torch.uint8, device=device)
    o, hT = torch.empty_like(d.v), torch.empty(w.n_seqs, w.h_v, D, D, dtype=torch.float32, device=device)
    grads = (torch.empty_like(d.q), torch.empty_like(d.k), torch.empty_like(d.v), torch.empty_like(d.g),
             torch.empty_like(d.beta), torch.empty(w.n_seqs, w.h_v, D, D, dtype=torch.float32, device=device))
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream(device)

    def fwd():
        gdn_chunk_fwd(d.q, d.k, d.v, d.g, d.beta, d.h0, d.cu_seqlens, plan=plan, out=o, final_state=hT,
                      workspace=ws, for_backward=True)

    def step():
        fwd()
        gdn_chunk_bwd(d.q, d.k, d.v, d.g, d.beta, d_out, d.h0, dhT, d.cu_seqlens, plan=plan, grads=grads,
                      workspace=ws, reuse_forward=True)

    res = {}
    for key, f in (("forward_train_ms", fwd), ("train_step_ms", step)):
        for _ in range(warmup):
            flush.zero_()
            f()
        ts = []
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        for _ in range(steps):
            flush.zero_()
            s0.record(stream)
            f()
            s1.record(stream)
            s1.synchronize()
            ts.append(s0.elapsed_time(s1))
        res[key] = statistics.mean(ts)
    return res


def backward_report(r, hbm, tfl):
    t_roof = max(r["bytes"] / (hbm * 1e9), r["flops"] / (tfl * 1e12))
    return {"workload": r["workload"], "ms": r["ms"], "tokens_per_s": r["tokens"] / (r["ms"] * 1e-3),
            "roofline_frac": t_roof * 1e3 / r["ms"], "roofline_ms": t_roof * 1e3,
            "bound": "tensor" if r["flops"] / (tfl * 1e12) > r["bytes"] / (hbm * 1e9) else "hbm",
            "kernels_ms": r["kernel_ms"], "segments": r["segments"], "device_status": r["status"]}


def backward_accuracy(r):
    """The float64 oracle's gradients (chunk-level derivation, pinned on the CPU to
    the autograd definition) against the GPU's, max|diff| / RMS(ref) per tensor."""
    import numpy as np
    from oracle import backward as OB
    from gated_deltanet_linear_fwd_gb300.inputs import make_output_grads, workload
    w = workload(r["workload"])
    d_out, dhT = make_output_grads(w)
    f = lambda t: None if t is None else t.double().numpy()
    t0 = time.perf_counter()
    ref = OB.grad_chunked(f(w.q), f(w.k), f(w.v), f(w.g), f(w.beta), f(w.h0), w.seq_offsets(), f(d_out), f(dhT))
    res = {}
    for n, x, y in zip(("dq", "dk", "dv", "dg", "dbeta", "dh0"), r["grads"], ref):
        g = x.double().numpy()
        rms = float(np.sqrt(np.mean(y * y)))
        diff = np.abs(g - y)
        res[n] = float(diff.max()) / rms
        if n in ("dq", "dk", "dv"):  # bf16 outputs: beyond the half ulp their store adds, as for o
            a = np.maximum(np.maximum(np.abs(y), np.abs(g)), np.finfo(np.float32).tiny)
            res[n + "_excess"] = float(np.maximum(diff - np.exp2(np.floor(np.log2(a)) - 8), 0).max()) / rms
    res["bar"] = 2e-2
    res["oracle_s"] = time.perf_counter() - t0
    return res


def compare_cp_modes(name, steps, device):
    """The same workload without context parallelism, with every head
    combined exactly, and in the automatic mode (warmup restarts where the
    gate bound allows) with the noise-floor tolerance (the default) and with
    the fixed one: time of each, and how far each mode's o and final state
    are from the exact ones (max |diff| / RMS of the exact result)."""
    from gated_deltanet_linear_fwd_gb300 import gdn_chunk_fwd, gdn_cp_plan
    from gated_deltanet_linear_fwd_gb300.inputs import workload
    cases = {"off": ("off", "noise"), "exact": ("exact", "noise"), "auto": ("auto", "noise"),
             "auto_fixed_tol": ("auto", "fixed")}
    res = {}
    for key, (cp, rule) in cases.items():
        t = time_gpu(name, steps, 3, device, cp, 0.0, trace=False, tol_rule=rule)
        res[key] = {"ms": t["ms"], "segments": t["plan"].n_seg_total, "head_modes": t["modes"]}
    w = workload(name)
    d = w.to(device)
    outs = {}
    for key, (cp, rule) in cases.items():
        plan = gdn_cp_plan(T=w.T, h_qk=w.h_qk, h_v=w.h_v, cu_seqlens=w.cu_seqlens, mode=cp, tol_rule=rule)
        outs[key] = gdn_chunk_fwd(d.q, d.k, d.v, d.g, d.beta, d.h0, d.cu_seqlens, plan=plan)
    rel = lambda a, b: float((a.float() - b.float()).abs().max() / b.float().pow(2).mean().sqrt())
    for cp in ("off", "auto", "auto_fixed_tol"):
        res[cp + "_vs_exact"] = {"o": rel(outs[cp][0], outs["exact"][0]),
                                 "final_state": rel(outs[cp][1], outs["exact"][1])}
    return res


DECODE_BATCH = (256, 2, 8)  # sequences, h_qk, h_v: one token each; 268 MB of state read and written per step


def time_decode(steps, warmup, device, hbm):
    """The one-token step over a batch of states (gdn_decode_step), L2 flushed
    before each step; HBM roofline on its bytes (state read + written, q/k/v/o)."""
    from gated_deltanet_linear_fwd_gb300 import gdn_decode_step
    from gated_deltanet_linear_fwd_gb300.inputs import make_inputs
    B, hqk, hv = DECODE_BATCH
    w = make_inputs(cu_seqlens=list(range(B + 1)), h_qk=hqk, h_v=hv, seed=5, with_h0=True)
    d = w.to(device)
    state = d.h0.clone()
    out = torch.empty_like(d.v)
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream(device)
    for _ in range(warmup):
        flush.zero_()
        gdn_decode_step(d.q, d.k, d.v, d.g, d.beta, state, out=out)
    times = []
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for _ in range(steps):
        flush.zero_()
        s0.record(stream)
        gdn_decode_step(d.q, d.k, d.v, d.g, d.beta, state, out=out)
        s1.record(stream)
        s1.synchronize()
        times.append(s0.elapsed_time(s1))
    ms = statistics.mean(times)
    by = B * hv * D * D * 4 * 2 + B * (2 * hqk * D + 2 * hv * D) * 2 + B * hv * 8
    return {"batch": B, "h_qk": hqk, "h_v": hv, "ms": ms, "tokens_per_s": B / (ms * 1e-3), "bytes": by,
            "achieved_gbs": by / (ms * 1e-3) / 1e9, "peak_gbs": hbm, "frac": by / (ms * 1e-3) / 1e9 / hbm,
            "dtype": "bf16 q/k/v/o, fp32 state"}


def time_e2e(name, steps, warmup, device, cp="auto"):
    """The same forward through the public call from pinned host buffers, as
    a serving loop would run it: every step copies its inputs host -> device,
    runs the forward and reads o and the final state back, with the copies of
    one step overlapping the forward of its neighbours (an input stream, the
    compute stream and an output stream; device and host buffers alternate
    between two sets).  The timed region starts before the first step's first
    copy and ends after the last step's last read."""
    from gated_deltanet_linear_fwd_gb300 import gdn_chunk_fwd, gdn_cp_plan
    from gated_deltanet_linear_fwd_gb300.inputs import workload
    w = workload(name)
    pin = lambda t: None if t is None else t.pin_memory()
    hin = [t for t in map(pin, (w.q, w.k, w.v, w.g, w.beta, w.h0))]
    dev = lambda t: None if t is None else torch.empty_like(t, device=device)
    din = [[dev(t) for t in hin] for _ in range(2)]
    dcu = None if w.cu_seqlens is None else w.cu_seqlens.to(device)
    plan = gdn_cp_plan(T=w.T, h_qk=w.h_qk, h_v=w.h_v, cu_seqlens=w.cu_seqlens, mode=cp)
    ws = torch.empty(max(plan.workspace_bytes, 256), dtype=torch.uint8, device=device)
    dout = [torch.empty_like(din[0][2]) for _ in range(2)]
    dhT = [torch.empty(w.n_seqs, w.h_v, D, D, dtype=torch.float32, device=device) for _ in range(2)]
    hout = [torch.empty(dout[0].shape, dtype=dout[0].dtype).pin_memory() for _ in range(2)]
    hhT = [torch.empty(dhT[0].shape, dtype=torch.float32).pin_memory() for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in hin if t is not None)
    d2h = hout[0].numel() * hout[0].element_size() + hhT[0].numel() * hhT[0].element_size()
    comp = torch.cuda.current_stream(device)
    s_in, s_out = torch.cuda.Stream(device), torch.cuda.Stream(device)
    ev = lambda: torch.cuda.Event()
    in_ready, in_free, done, out_free = ([ev(), ev()] for _ in range(4))
    used = [False, False]

    def step(k):
        b = k & 1
        with torch.cuda.stream(s_in):
            if used[b]:
                s_in.wait_event(in_free[b])  # the forward two steps back has read this set
            for src, dst in zip(hin, din[b]):
                if src is not None:
                    dst.copy_(src, non_blocking=True)
            in_ready[b].record(s_in)
        comp.wait_event(in_ready[b])
        if used[b]:
            comp.wait_event(out_free[b])  # its outputs two steps back have been read
        q, k_, v, g, beta, h0 = din[b]
        gdn_chunk_fwd(q, k_, v, g, beta, h0, dcu, plan=plan, out=dout[b], final_state=dhT[b], workspace=ws,
                      stream=comp)
        done[b].record(comp)
        in_free[b].record(comp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(done[b])
            hout[b].copy_(dout[b], non_blocking=True)
            hhT[b].copy_(dhT[b], non_blocking=True)
            out_free[b].record(s_out)
        used[b] = True

    for i in range(warmup):
        step(i)
    torch.cuda.synchronize(device)
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s0.record(comp)
    s_in.wait_event(s0)
    s_out.wait_event(s0)
    for i in range(steps):
        step(warmup + i)
    for b in range(2):
        comp.wait_event(out_free[b])
    s1.record(comp)
    s1.synchronize()
    ms = s0.elapsed_time(s1) / steps
    return {"ms": ms, "h2d": h2d, "d2h": d2h, "tokens": w.T}


def time_f32(name, steps, warmup, device):
    """The fp32 path (q, k, v, o in fp32) on a workload, L2 flushed before each step."""
    from gated_deltanet_linear_fwd_gb300 import gdn_chunk_fwd, gdn_cp_plan
    from gated_deltanet_linear_fwd_gb300.inputs import workload
    w = workload(name, dtype=torch.float32)
    d = w.to(device)
    plan = gdn_cp_plan(T=w.T, h_qk=w.h_qk, h_v=w.h_v, cu_seqlens=w.cu_seqlens, dtype=torch.float32)
    ws = torch.empty(max(plan.workspace_bytes, 256), dtype=torch.uint8, device=device)
    out = torch.empty_like(d.v)
    hT = torch.empty(w.n_seqs, w.h_v, D, D, dtype=torch.float32, device=device)
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream(device)
    fwd = lambda: gdn_chunk_fwd(d.q, d.k, d.v, d.g, d.beta, d.h0, d.cu_seqlens, plan=plan, out=out,
                                final_state=hT, workspace=ws)
    for _ in range(warmup):
        flush.zero_()
        fwd()
    times = []
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for _ in range(steps):
        flush.zero_()
        s0.record(stream)
        fwd()
        s1.record(stream)
        s1.synchronize()
        times.append(s0.elapsed_time(s1))
    ms = statistics.mean(times)
    return {"workload": name, "ms": ms, "tokens_per_s": w.T / (ms * 1e-3), "dtype": "f32 q/k/v/o",
            "kernel": "recurrence_f32"}


def planning_ms(name, repeats=20):
    """Host time of gdn_cp_plan with automatic lambda: the first call for these
    sequence lengths (the planner's search) and later calls (its cache)."""
    from gated_deltanet_linear_fwd_gb300 import gdn_cp_plan
    from gated_deltanet_linear_fwd_gb300.inputs import WORKLOADS
    spec = WORKLOADS[name]
    cu = spec.get("cu_seqlens")
    T = cu[-1] if cu else spec["n_tokens"]
    # an SM count no other call of this process plans for, so the first call searches
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count - 1
    t0 = time.perf_counter()
    gdn_cp_plan(T=T, h_qk=spec["h_qk"], h_v=spec["h_v"], cu_seqlens=cu, sm_count=sms)
    first = time.perf_counter() - t0
    t0 = time.perf_counter()
    for _ in range(repeats):
        gdn_cp_plan(T=T, h_qk=spec["h_qk"], h_v=spec["h_v"], cu_seqlens=cu, sm_count=sms)
    return {"workload": name, "first_ms": first * 1e3, "cached_ms": (time.perf_counter() - t0) / repeats * 1e3}


def gpu_outputs(name, device, cp="auto"):
    """o and the final state of one forward on a workload, on the host."""
    from gated_deltanet_linear_fwd_gb300 import gdn_chunk_fwd
    from gated_deltanet_linear_fwd_gb300.inputs import workload
    w = workload(name)
    d = w.to(device)
    o, hT = gdn_chunk_fwd(d.q, d.k, d.v, d.g, d.beta, d.h0, d.cu_seqlens, mode=cp)
    torch.cuda.synchronize(device)
    return o.cpu(), hT.cpu()


def compare(o_gpu, hT_gpu, ref):
    """max|diff| / RMS(ref) for o (raw, and beyond bf16's half-ulp store
    rounding) and for the final state."""
    import numpy as np
    ro, rh = ref
    g = o_gpu.double().numpy()
    rms = float(np.sqrt(np.mean(ro ** 2)))
    diff = np.abs(g - ro)
    a = np.maximum(np.maximum(np.abs(ro), np.abs(g)), np.finfo(np.float32).tiny)
    half_ulp = np.exp2(np.floor(np.log2(a)) - 8)
    hs = hT_gpu.double().numpy()
    return {"o_raw": float(diff.max()) / rms, "o_excess": float(np.maximum(diff - half_ulp, 0).max()) / rms,
            "final_state": float(np.abs(hs - rh).max() / np.sqrt(np.mean(rh ** 2))), "bar": 2e-2}


def cpu_baseline(name, budget_s=12.0):
    """The float64 oracle, as it stands, on this host's cores: a bounded sample
    (a prefix of the sequence, all heads) of the same workload."""
    import oracle
    from gated_deltanet_linear_fwd_gb300.inputs import workload
    w = workload(name)
    cores = oracle.default_threads()
    f = lambda t: t.double().numpy()
    tokens = 1024
    while True:
        t0 = time.perf_counter()
        oracle.recurrence(f(w.q[:tokens]), f(w.k[:tokens]), f(w.v[:tokens]), f(w.g[:tokens]),
                          f(w.beta[:tokens]), None if w.h0 is None else f(w.h0[:1]), [0, tokens])
        dt = time.perf_counter() - t0
        if dt * 4 > budget_s or tokens * 2 > w.T:
            break
        tokens *= 2
    return {"value": tokens / dt, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"first {tokens} tokens of {name}, all {w.h_v} value heads, one pass ({dt:.2f} s)"}


def oracle_accuracy(outputs):
    """The oracle over each whole workload (float64, host cores), against the
    GPU outputs taken from the same seeded inputs."""
    import oracle
    from gated_deltanet_linear_fwd_gb300.inputs import workload
    res = {}
    for name, (o, hT) in outputs.items():
        w = workload(name)
        f = lambda t: None if t is None else t.double().numpy()
        t0 = time.perf_counter()
        ref = oracle.recurrence(f(w.q), f(w.k), f(w.v), f(w.g), f(w.beta), f(w.h0), w.seq_offsets())
        res[name] = compare(o, hT, ref)
        res[name]["oracle_s"] = time.perf_counter() - t0
    return res


def traffic_from_profile(tag, source):
    """DRAM bytes per launch from the committed ncu summary, when it was taken
    on the current kernel source (its recorded source hash matches)."""
    path = os.path.join(ROOT, "profiles", f"{tag}.md")
    src = os.path.join(ROOT, "gated_deltanet_linear_fwd_gb300", "csrc", source)
    try:
        txt = open(path).read()
        digest = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    except OSError:
        return None
    vals = {}
    for line in txt.splitlines():
        line = line.strip()
        if line.startswith("- ") and ":" in line:
            k, v = line[2:].split(":", 1)
            vals[k.strip()] = v.strip().strip("`")
    if vals.get("source_sha256_16") != digest:
        return None
    try:
        return float(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def run_reference(args, world, rank):
    if rank != 0:
        return 0
    import oracle
    from gated_deltanet_linear_fwd_gb300.inputs import workload
    w = workload(HEADLINE)
    f = lambda t: t.double().numpy()
    tokens = 1024
    arrays = [f(x[:tokens]) for x in (w.q, w.k, w.v, w.g, w.beta)]
    for _ in range(args.warmup):
        oracle.recurrence(*arrays, None, [0, tokens])
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.recurrence(*arrays, None, [0, tokens])
    dt = (time.perf_counter() - t0) / args.steps
    value = tokens / dt
    cores = oracle.default_threads()
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": HEADLINE, "B": 1, "T": 32768, "h_qk": 2, "h_v": 8, "d_k": 128, "d_v": 128},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                             "sample": f"first {tokens} tokens of {HEADLINE}, all 8 value heads, per step"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def time_graphs(device, calls=200, per_graph=20):
    """Back-to-back calls, eager (each one a Python call through the C ABI) against the
    same calls captured once as a CUDA graph and replayed: microseconds per call for
    the tiny forward (T = 512, h 2/4) and for the decode step over 256 states, where
    launching, not the kernels, can set the pace."""
    from gated_deltanet_linear_fwd_gb300 import gdn_chunk_fwd, gdn_cp_plan, gdn_decode_step
    from gated_deltanet_linear_fwd_gb300.inputs import make_inputs, workload
    stream = torch.cuda.current_stream(device)

    def per_call_us(fn, n):
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s0.record(stream)
        for _ in range(n):
            fn()
        s1.record(stream)
        s1.synchronize()
        return s0.elapsed_time(s1) * 1e3 / n

    def measure(call):
        for _ in range(5):
            call()
        torch.cuda.synchronize(device)
        eager = per_call_us(call, calls)
        side = torch.cuda.Stream(device)
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            call()
        stream.wait_stream(side)
        torch.cuda.synchronize(device)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for _ in range(per_graph):
                call()
        graph.replay()
        torch.cuda.synchronize(device)
        replayed = per_call_us(graph.replay, calls // per_graph) / per_graph
        return {"eager_us_per_call": eager, "graph_us_per_call": replayed}

    res = {}
    w = workload("tiny_T512_h2x4")
    d = w.to(device)
    plan = gdn_cp_plan(T=w.T, h_qk=w.h_qk, h_v=w.h_v)
    ws = torch.empty(max(plan.workspace_bytes, 256), dtype=torch.uint8, device=device)
    out = torch.empty_like(d.v)
    hT = torch.empty(1, w.h_v, D, D, dtype=torch.float32, device=device)
    res["forward_tiny_T512_h2x4"] = measure(
        lambda: gdn_chunk_fwd(d.q, d.k, d.v, d.g, d.beta, None, None, plan=plan, out=out, final_state=hT, workspace=ws))
    B, hqk, hv = DECODE_BATCH
    w = make_inputs(cu_seqlens=list(range(B + 1)), h_qk=hqk, h_v=hv, seed=5, with_h0=True)
    d = w.to(device)
    state = d.h0.clone()
    out = torch.empty_like(d.v)
    res[f"decode_B{B}_h{hqk}x{hv}"] = measure(lambda: gdn_decode_step(d.q, d.k, d.v, d.g, d.beta, state, out=out))
    return res


def run_only(args, device, hbm):
    """One case alone, few steps: the command the ncu captures run."""
    if args.only == "decode":
        r = time_decode(args.steps, args.warmup, device, hbm)
    elif args.only == "graphs":
        r = time_graphs(device)
    elif args.only == "f32":
        r = time_f32(HEADLINE, args.steps, args.warmup, device)
    elif args.only.startswith("bwd"):
        name = args.only.split(":", 1)[1] if ":" in args.only else HEADLINE
        t = time_bwd(name, args.steps, args.warmup, device, args.cp)
        r = {"workload": name, "ms": t["ms"], "kernels_ms": t["kernel_ms"], "segments": t["segments"],
             "status": t["status"]}
    else:
        t = time_gpu(args.only, args.steps, args.warmup, device, args.cp, args.lambda_)
        r = {"workload": args.only, "ms": t["ms"], "kernels_ms": t["kernel_ms"], "segments": t["plan"].n_seg_total,
             "status": list(t["status"])}
    print(json.dumps({"only": args.only, **r}), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cp", default="auto", choices=["off", "exact", "warmup", "auto"])
    ap.add_argument("--lambda", dest="lambda_", type=float, default=0.0,
                    help="segment-length factor; 0 lets the planner choose")
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--only", default=None,
                    help="time just this case (a workload name, 'decode' or 'f32') and print a short line")
    args = ap.parse_args(argv)
    args.warmup = max(args.warmup, 3)
    world, rank, local = dist_setup()
    if args.impl == "reference":
        return run_reference(args, world, rank)

    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    hbm, tfl, peak_src = peaks()
    if args.only:
        return run_only(args, device, hbm)
    plan_t = planning_ms(HEADLINE) if rank == 0 else None
    barrier(world)
    torch.cuda.synchronize(device)
    clocks = ClockSampler(device)
    clocks.start()
    r = time_gpu(HEADLINE, args.steps, args.warmup, device, args.cp, args.lambda_)
    clk = clocks.stop()
    torch.cuda.synchronize(device)
    barrier(world)
    ms = max_over_ranks(r["ms"], world, device)
    value = world * r["tokens"] / (ms * 1e-3)
    kms = r["kernel_ms"]
    t_hbm = r["bytes"] / (hbm * 1e9)
    t_tc = r["flops"] / (tfl * 1e12)
    roof = None
    if kms:
        # the dominant kernel: its share of the algorithmic bytes over its average launch time
        top = max((k for k in kms if kernel_bytes(k, r["w"]) > 0), key=lambda k: kms[k])
        kb = kernel_bytes(top, r["w"])
        achieved = kb / (kms[top] * 1e-3) / 1e9
        roof = {"bound": "hbm", "kernel": top, "achieved": achieved, "peak": hbm, "unit": "GB/s",
                "frac": achieved / hbm, "traffic": traffic_from_profile(f"{top}_T32768_h2x8", KERNEL_SOURCE[top]),
                "peak_source": peak_src, "algorithmic_bytes": kb, "kernel_ms": kms[top],
                "kernel_share": kms[top] / sum(kms.values())}
    e2e = time_e2e(HEADLINE, max(20, args.steps // 10), 3, device, args.cp)
    e2e_ms = max_over_ranks(e2e["ms"], world, device)
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": value / (32768 / (PAGES_H200_MS[HEADLINE] * 1e-3)),
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": HEADLINE, "B": 1, "T": 32768, "h_qk": 2, "h_v": 8, "d_k": 128, "d_v": 128,
                   "chunk": 64, "cp": r["plan"].mode, "warmup_tol_rule": "noise", "segments": r["plan"].n_seg_total,
                   "head_modes": r["modes"], "l2": "flushed (256 MB write) before every timed step",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "roofline": roof,
        "layer_roofline": {"t_roofline_ms": max(t_hbm, t_tc) * 1e3, "bound": "hbm" if t_hbm >= t_tc else "tensor",
                           "frac": max(t_hbm, t_tc) * 1e3 / r["ms"], "peak_source": peak_src,
                           "bytes": r["bytes"], "flops": r["flops"]},
        "kernels_ms": kms,
        "gpu_launches": r["launches"] * args.steps,
        "clocks": clk,
        "e2e": {"value": world * e2e["tokens"] / (e2e_ms * 1e-3), "unit": "tokens/s",
                "h2d_bytes_per_step": e2e["h2d"], "d2h_bytes_per_step": e2e["d2h"]},
        "device_status": list(r["status"]),
        "vs_baseline_note": "vs FlashQLA on an H200 (pages' table, 0.310 ms): another machine, context only",
    }
    if not args.no_sweep and rank == 0:
        sweep = {}
        for name in SWEEP:
            s = time_gpu(name, max(20, args.steps // 20), 5, device, args.cp, args.lambda_)
            t_r = max(s["bytes"] / (hbm * 1e9), s["flops"] / (tfl * 1e12))
            sweep[name] = {"tokens_per_s": s["tokens"] / (s["ms"] * 1e-3), "ms": s["ms"], "cp": s["plan"].mode,
                           "segments": s["plan"].n_seg_total, "roofline_frac": t_r * 1e3 / s["ms"],
                           "kernels_ms": s["kernel_ms"], "head_modes": s["modes"]}
            if name in PAGES_H200_MS:
                sweep[name]["pages_h200_ms"] = PAGES_H200_MS[name]
            if name == VARLEN:  # AutoCP: exact combine for every head against the automatic warmup mode
                sweep[name]["modes"] = compare_cp_modes(name, max(20, args.steps // 20), device)
        line["sweep"] = sweep
    if not args.no_sweep and rank == 0:
        line["decode"] = time_decode(max(20, args.steps // 10), 5, device, hbm)
        line["graphs"] = time_graphs(device)
        f32 = time_f32(HEADLINE, max(5, args.steps // 50), 3, device)
        f32["vs_bf16_path"] = f32["ms"] / ms
        line["f32"] = f32
    if not args.no_sweep and rank == 0:
        rb = time_bwd(HEADLINE, max(10, args.steps // 50), 3, device, args.cp)
        line["backward"] = backward_report(rb, hbm, tfl)
        line["backward"]["vs_forward"] = rb["ms"] / ms
        line["backward"]["training"] = time_train_step(HEADLINE, max(10, args.steps // 50), 3, device, args.cp)
        line["backward"]["sweep"] = {n: backward_report(time_bwd(n, 5, 2, device, args.cp), hbm, tfl)
                                     for n in BWD_SWEEP}
        if not args.no_cpu_baseline:
            line["backward"]["accuracy"] = backward_accuracy(rb)
    if rank == 0:
        line["planning"] = plan_t
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(HEADLINE)
        names = [HEADLINE] + ([] if args.no_sweep else SWEEP)
        line["accuracy"] = oracle_accuracy({n: gpu_outputs(n, device, args.cp) for n in names})
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
