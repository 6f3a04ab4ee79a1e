"""Benchmark of the GB300 causal gated-linear-attention path.

Headline (value): long-context GLA prefill, B=1 H=32 L=65536 dk=128 dv=256,
chunk 64, bf16 q/k/v, fp32 log alpha, fp32 initial state ~N(0, 0.1), returns
the final state -- tokens/s for the whole job (all ranks).  One step is one
gla_fwd call over the whole batch (the fused cumsum-gate / intra-chunk /
inter-chunk / output kernel).  The same run also measures, each in its own
JSON object: the other prefill workloads ("configs": fp32 B1 H1 L256 d32,
elu+1 normalised B4 H8 L2048 d64, gated B8 H16 L4096 d128); the decode step
(256 sequences x H32, d128, fp32 state, 1024 consecutive steps on fresh
tokens) as state HBM GB/s; the 8-token hand-off on that state; the
long-context prefill with one gate per token; the delta rule (chunk form) and the backward
pass; and the end-to-end step through gla_fwd_host with host buffers.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gla|reference]

Under torchrun every rank runs an independent replica on its own seeded
inputs (no collective on the data path): "scaling": "weak".  Inputs are
larger than L2 (4.3 GB per prefill step, 537 MB of decode state), so no L2
flush is needed between timed iterations.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synth  # noqa: E402

METRIC = ("GLA prefill tokens/s & % bf16 tensor peak; decode-step state HBM GB/s (1×GB300)")
HEADLINE = synth.LONGCTX
DEC = synth.DECODE
C = 64


def prefill_flops(w) -> float:
    per_head = 2.0 * w.L * C * (w.dk + w.dv) + 4.0 * w.L * w.dk * w.dv
    return per_head * w.B * w.H


def prefill_bytes(w, final_state=True) -> float:
    """Algorithmic bytes: q, k, v, log alpha read once, out written once, init/final state
    (fp32 inputs and output for the fp32 workload, bf16 otherwise; no log alpha without a gate)."""
    BH, L = w.B * w.H, w.L
    es = 4 if w.dtype == "f32" else 2
    la_bytes = 0 if not w.gate else (4 if getattr(w, "scalar_gate", False) else 4 * w.dk)
    per_tok = es * (2 * w.dk + w.dv) + la_bytes + es * w.dv
    states = ((1 if w.init_std > 0 else 0) + (1 if final_state else 0)) * w.dk * w.dv * 4
    return float(BH * (L * per_tok + states))


def decode_multi_bytes(w) -> float:
    """Per call: fp32 state read + write once, and per token bf16 q/k/v, fp32 log alpha, bf16 out."""
    return float(w.B * w.H * (2 * w.dk * w.dv * 4 + w.L * (2 * w.dk * 2 + w.dv * 2 + w.dk * 4 + w.dv * 2)))


def delta_flops(w) -> float:
    """Delta rule per token and head: prediction S^T k, write k u^T, output S^T q (2 dk dv flops
    each), plus the gate's decay (dk dv)."""
    return float(w.B * w.H * w.L * (6 + (1 if w.gate else 0)) * w.dk * w.dv)


def bwd_flops(w) -> float:
    """Backward per token and state element: S_t = alpha S + k v^T (3 flops with the gate, 2
    without) and dq = S dout (2); G_t += q dout^T (2), dk = G v (2), dv = G^T k (2), and the
    decay of G in both reverse sweeps (1 each, with the gate)."""
    return float(w.B * w.H * w.L * (15 if w.gate else 12) * w.dk * w.dv)


def delta_bytes(w) -> float:
    """Delta rule, algorithmic bytes: q, k, v (bf16), beta, log alpha read once; out (bf16) written
    once; initial (if any) and final fp32 state."""
    BH, L = w.B * w.H, w.L
    per_tok = 2 * (2 * w.dk + w.dv) + 4 + (4 * w.dk if w.gate else 0) + 2 * w.dv
    states = ((1 if w.init_std > 0 else 0) + 1) * w.dk * w.dv * 4
    return float(BH * (L * per_tok + states))


def delta_chunk_flops(w) -> float:
    """Delta rule in chunk form, tensor-core flops per chunk and head: A = Kr Kh^T, P = Qh Kh^T,
    M V' and P U (2 C^2 d each), Kr S', Qh S' and Kh^T U (2 C dk dv each)."""
    per_chunk = 4 * 2 * C * C * w.dk + 3 * 2 * C * w.dk * w.dv
    return float(w.B * w.H * math.ceil(w.L / C) * per_chunk)


def bwd_bytes(w, dla=True) -> float:
    """Backward, algorithmic bytes: q, k, v, dout (bf16) and log alpha read once; dq, dk, dv (and
    dlog_alpha) written once in fp32."""
    BH, L = w.B * w.H, w.L
    per_tok = 2 * (2 * w.dk + 2 * w.dv) + (4 * w.dk if w.gate else 0) + 4 * (2 * w.dk + w.dv) + \
        (4 * w.dk if (dla and w.gate) else 0)
    return float(BH * L * per_tok)


def bwd_chunk_flops(w) -> float:
    """Backward in chunk form, tensor-core flops per chunk and head (the chunk algorithm's own
    products, with the state copies counted once): dq pass D = dO V^T (2 C^2 dv), dS = Kh^T V
    (2 C dk dv), dQ = S' dO^T + Kh^T D_m^T (2 C dk dv + 2 C^2 dk); dk/dv pass P = Qh Kh^T (2 C^2 dk),
    D (2 C^2 dv), dG = Qh^T dO (2 C dk dv), dK = G V^T + Qh^T D_m (2 C dk dv + 2 C^2 dk),
    dV = G^T Kh^T + dO^T P_m (2 C dk dv + 2 C^2 dv)."""
    Cc, dk, dv = C, w.dk, w.dv
    per_chunk = (2 * Cc * Cc * dv + 2 * Cc * dk * dv + 2 * Cc * dk * dv + 2 * Cc * Cc * dk) + \
        (2 * Cc * Cc * dk + 2 * Cc * Cc * dv + 2 * Cc * dk * dv + 2 * Cc * dk * dv + 2 * Cc * Cc * dk +
         2 * Cc * dk * dv + 2 * Cc * Cc * dv)
    return float(w.B * w.H * math.ceil(w.L / Cc) * per_chunk)


def fp32_alu_peak_tflops(peaks) -> float:
    """FP32 FMA peak from unit counts: SMs x 128 FP32 lanes x 2 flops x max SM clock."""
    import torch
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    return sms * 128 * 2 * peaks["sm_max_mhz"] * 1e6 / 1e12


def decode_bytes(NS, H, dk, dv) -> float:
    """Per step: fp32 state read + write, bf16 q/k/v, fp32 log alpha, fp32 out."""
    return float(NS * H * (2 * dk * dv * 4 + 2 * dk * 2 + dv * 2 + dk * 4 + dv * 4))


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return dict(hbm_gbs=float(d["hbm_gbs"]), bf16_tflops=float(d["bf16_tflops"]),
                    bf16_tflops_sustained=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                    sm_max_mhz=float(d.get("sm_max_mhz", 2070.0)), source="measured")
    return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0, sm_max_mhz=2070.0,
                source="fallback")


KERNEL_SOURCES = {
    "gla_delta_tc_kernel": ("gla_delta_tc.cu", "gla_ptx.cuh"),
    "gla_bwd_tc": ("gla_bwd_tc.cu", "gla_ptx.cuh"),  # the dq and dk/dv kernels together
    "gla_prefill_tc_kernel": ("gla_tc.cu", "gla_ptx.cuh"),
    "gla_decode_kernel": ("gla_decode.cu",),
    "gla_prefill_short_kernel": ("gla_short.cu",),
    "gla_prefill_tc_kernel_scalar_gate": ("gla_tc.cu", "gla_ptx.cuh"),
    "gla_delta_kernel": ("gla_delta.cu",),
    "gla_bwd_kernel": ("gla_bwd.cu",),
}


def kernel_source_hash(kernel: str, csrc: str | None = None) -> str:
    """Hash of a kernel's sources with comments and blank space removed (a comment edit
    does not change the kernel, so it does not void a recorded capture)."""
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(csrc or os.path.join(ROOT, "causal_gated_linear_gb300", "csrc"), f)) as fh:
            src = fh.read()
        src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
        src = re.sub(r"//[^\n]*", " ", src)
        h.update(" ".join(src.split()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on this source."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(kernel)
    if not e or e.get("source_hash") != kernel_source_hash(kernel):
        return None
    return e.get("bytes_per_launch")


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons; summary() keeps the
    samples whose timestamps fall inside the timed region (mark() brackets it)."""

    Q = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.window = None
        # raw samples go to $GLA_BENCH_CLOCKS_DIR (default: the system temp directory)
        d = os.environ.get("GLA_BENCH_CLOCKS_DIR") or tempfile.gettempdir()
        self.path = os.path.join(d, f"clocks_bench_{os.getpid()}.csv")

    def __enter__(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "20"], stdout=self.fh, stderr=subprocess.DEVNULL)
            # give nvidia-smi time to start sampling before the timed region
            t0 = time.perf_counter()
            while time.perf_counter() - t0 < 1.5 and os.path.getsize(self.path) == 0:
                time.sleep(0.01)
        except Exception:
            self.proc = None
        return self

    def mark(self, start: float, end: float):
        """Host wall-clock bounds (time.time()) of the timed region."""
        self.window = (start, end)

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        lo, hi = self.window if self.window else (-math.inf, math.inf)
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 10:
                    continue
                try:
                    ts = parts[0]
                    frac = float("0." + ts.rsplit(".", 1)[1]) if "." in ts else 0.0
                    t = time.mktime(time.strptime(ts.rsplit(".", 1)[0], "%Y/%m/%d %H:%M:%S")) + frac
                    if not (lo - 0.02 <= t <= hi + 0.02):
                        continue
                    sm.append(float(parts[2]))
                    mx.append(float(parts[3]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[6:10]):
                    if v.lower() == "active":
                        reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples in the timed region"],
                    "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(x: float, world: int, device=None) -> float:
    """Slowest rank's value (timing is max over ranks); `device` may be CPU under gloo."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank: float, steps: int, world: int, max_ms: float) -> float:
    """Whole-job throughput: units processed by all ranks / slowest rank's time."""
    return units_per_rank * world * steps / (max_ms / 1e3)


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ---------------------------------------------------------------------------- oracle leg

def oracle_sample(seconds_target: float = 10.0):
    """Time the fp64 oracle on a bounded sample of the prefill workload.

    Sample: `nh` heads x `Ls` tokens of the long-context shape (dk 128, dv 256),
    one OpenMP thread per head.  Returns (tokens/s of the full workload's
    token definition, cores, sample description, seconds).
    """
    import oracle
    cores = max(1, oracle.max_threads())
    nh = min(HEADLINE.H, max(1, cores))
    Ls = 256
    # grow the sample until it takes a noticeable fraction of the target
    while True:
        w = synth.with_shape(HEADLINE, B=1, H=nh, L=Ls)
        x = synth.make_prefill(w, heads=list(range(nh)))
        args = [synth.as_f64(x[n]) for n in ("q", "k", "v", "log_alpha", "init_state")]
        t0 = time.perf_counter()
        oracle.gla_fwd(*args, nthreads=cores)
        dt = time.perf_counter() - t0
        if dt >= seconds_target / 4 or Ls >= HEADLINE.L:
            break
        Ls = min(HEADLINE.L, Ls * max(2, int(math.ceil(seconds_target / 4 / max(dt, 1e-3)))))
    token_heads_per_s = nh * Ls / dt
    tps = token_heads_per_s / (HEADLINE.B * HEADLINE.H)   # tokens/s of the B*H workload
    desc = f"{nh} heads x {Ls} tokens of the B1 H32 L65536 dk128 dv256 workload, fp64, {cores} threads"
    return tps, cores, desc, dt


def oracle_single_thread(seconds_target: float = 3.0):
    """The oracle on one host thread: one head of the long-context shape for a bounded number of
    tokens, extrapolated to the whole B*H workload's tokens/s (labelled as extrapolated)."""
    import oracle
    Ls = 256
    while True:
        w = synth.with_shape(HEADLINE, B=1, H=1, L=Ls)
        x = synth.make_prefill(w, heads=[0])
        args = [synth.as_f64(x[n]) for n in ("q", "k", "v", "log_alpha", "init_state")]
        t0 = time.perf_counter()
        oracle.gla_fwd(*args, nthreads=1)
        dt = time.perf_counter() - t0
        if dt >= seconds_target / 4 or Ls >= HEADLINE.L:
            break
        Ls = min(HEADLINE.L, Ls * max(2, int(math.ceil(seconds_target / 4 / max(dt, 1e-3)))))
    tps = Ls / dt / (HEADLINE.B * HEADLINE.H)
    return tps, f"1 head x {Ls} tokens, 1 thread, extrapolated to the 32-head workload", dt


def run_reference(args):
    rank, world, local = dist_env()
    if rank != 0:
        return 0
    times = []
    cores, desc = None, None
    for i in range(args.warmup + args.steps):
        tps, cores, desc, dt = oracle_sample(seconds_target=args.ref_seconds)
        if i >= args.warmup:
            times.append(tps)
    v = statistics.median(times)
    line = {
        "impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": HEADLINE.name, "B": HEADLINE.B, "H": HEADLINE.H, "L": HEADLINE.L,
                   "dk": HEADLINE.dk, "dv": HEADLINE.dv, "chunk": C},
        "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": desc},
        "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------- GPU legs

def to_dev(x, device):
    import torch
    if x is None:
        return None
    if x.dtype == np.uint16:
        return torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).to(device)
    return torch.from_numpy(x).to(device)


def bench_prefill(args, device, rank, world):
    import torch

    import causal_gated_linear_gb300 as gla
    w = synth.with_shape(HEADLINE, seed=HEADLINE.seed + 1000 * rank)
    if args.L:  # reduced sequence length (profiling a small case); the line names it
        w = synth.with_shape(w, L=args.L, name=f"{HEADLINE.name}_L{args.L}")
    x = synth.make_prefill(w)
    BH = w.B * w.H
    q, k, v = (to_dev(x[n], device) for n in ("q", "k", "v"))
    la, s0 = to_dev(x["log_alpha"], device), to_dev(x["init_state"], device)
    out = torch.empty((w.B, w.H, w.L, w.dv), dtype=torch.bfloat16, device=device)
    fs = torch.empty((w.B, w.H, w.dk, w.dv), dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream(device)

    def step():
        st = gla.gla_fwd(q, k, v, la, s0, out, fs, w.B, w.H, w.L, w.dk, w.dv, C, stream=stream)
        if st != 0:
            raise RuntimeError(gla.gla_status_string(st))

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(device)
    gla.check(gla.gla_device_error(stream))
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    per = []
    with ClockSampler(device.index) as clk:
        barrier(world)
        torch.cuda.synchronize(device)
        t_wall = time.perf_counter()
        t_epoch = time.time()
        ev0.record(stream)
        evs = []
        for _ in range(args.steps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            step()
            b.record(stream)
            evs.append((a, b))
        ev1.record(stream)
        torch.cuda.synchronize(device)
        clk.mark(t_epoch, time.time())
        barrier(world)
        wall = time.perf_counter() - t_wall
    gla.check(gla.gla_device_error(stream))
    total_ms = ev0.elapsed_time(ev1)
    per = [a.elapsed_time(b) for a, b in evs]
    total_ms = max_over_ranks(total_ms, world, device)
    res = dict(total_ms=total_ms, per_launch_ms=statistics.mean(per), wall_s=wall, clocks=clk.summary())

    # the same workload with one gate per token (GLA_FLAG_SCALAR_GATE): q, k, v and states reused
    if args.scalar_calls > 0:
        ws = synth.with_shape(w, scalar_gate=True, name=w.name + "_scalar_gate")
        las = to_dev(synth.gate_log_alpha(ws), device)

        def sstep():
            st = gla.gla_fwd_ex(q, k, v, out, w.B, w.H, w.L, w.dk, w.dv, log_alpha=las, init_state=s0,
                                final_state=fs, flags=gla.FLAG_SCALAR_GATE, stream=stream)
            if st != 0:
                raise RuntimeError(gla.gla_status_string(st))

        for _ in range(2):
            sstep()
        torch.cuda.synchronize(device)
        sev = []
        for _ in range(args.scalar_calls):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            sstep()
            b.record(stream)
            sev.append((a, b))
        torch.cuda.synchronize(device)
        gla.check(gla.gla_device_error(stream))
        res["scalar"] = dict(w=ws, per_launch_ms=statistics.mean(a.elapsed_time(b) for a, b in sev),
                             calls=args.scalar_calls)
        del las

    # end to end through the public API with host buffers (pinned), copies inside the timed region:
    # gla_fwd_host copies each head group in, computes it and copies it out, overlapping the groups.
    # Consecutive steps alternate between two sets of device buffers and streams (as a caller
    # streaming batches would): a call overwrites its device inputs only after that set's earlier
    # kernels have read them, so with one set a step's copies could not overlap the previous step.
    if args.e2e:
        hq, hk, hv = (t.cpu().pin_memory() for t in (q, k, v))
        hla, hs0 = la.cpu().pin_memory(), s0.cpu().pin_memory()
        hout = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        hfs = torch.empty(fs.shape, dtype=fs.dtype).pin_memory()
        h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv, hla, hs0))
        d2h = hout.numel() * hout.element_size() + hfs.numel() * hfs.element_size()
        host = dict(q=hq, k=hk, v=hv, log_alpha=hla, init_state=hs0, out=hout, final_state=hfs)
        sets = []
        for b in range(2):
            devb = dict(q=torch.empty_like(q), k=torch.empty_like(k), v=torch.empty_like(v),
                        log_alpha=torch.empty_like(la), init_state=torch.empty_like(s0),
                        out=out if b == 0 else torch.empty_like(out), final_state=fs if b == 0 else torch.empty_like(fs))
            sets.append((devb, tuple(torch.cuda.Stream(device) for _ in range(3))))
        dv_, s_in = sets[0][0]["v"], sets[0][1][0]
        step_no = [0]
        last_in = [None]  # end of the previous step's host-to-device copies

        def e2e_step():
            devb, (si, sc, so) = sets[step_no[0] & 1]
            step_no[0] += 1
            # a step's inputs go over the link after the previous step's: each step's copies
            # finish as early as they can, so its outputs come back while the next step's
            # inputs are still going in (the two directions overlap; two steps' inputs sharing
            # the link would only delay both)
            if last_in[0] is not None:
                si.wait_event(last_in[0])
            st = gla.gla_fwd_host(host, devb, w.B, w.H, w.L, w.dk, w.dv, C, groups=args.e2e_groups,
                                  copy_in=si, compute=sc, copy_out=so)
            if st != 0:
                raise RuntimeError(gla.gla_status_string(st))
            ev = torch.cuda.Event()
            ev.record(si)
            last_in[0] = ev

        e2e_step()
        e2e_step()
        torch.cuda.synchronize(device)
        # the host link's own rate on these buffers: one timed copy of v in, one of out back
        c0, c1, c2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
        with torch.cuda.stream(s_in):
            c0.record(s_in)
            dv_.copy_(hv, non_blocking=True)
            c1.record(s_in)
            hout.copy_(out, non_blocking=True)
            c2.record(s_in)
        torch.cuda.synchronize(device)
        h2d_gbs = hv.numel() * hv.element_size() / (c0.elapsed_time(c1) / 1e3) / 1e9
        d2h_gbs = hout.numel() * hout.element_size() / (c1.elapsed_time(c2) / 1e3) / 1e9
        ne = args.steps
        barrier(world)
        torch.cuda.synchronize(device)
        # CUDA events: the start on the first step's copy-in stream, the end on a stream that
        # waits for the last work of both stream sets
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s_in)
        for _ in range(ne):
            e2e_step()
        join = torch.cuda.Stream(device)
        for _, streams in sets:
            for st_ in streams:
                ev = torch.cuda.Event()
                ev.record(st_)
                join.wait_event(ev)
        e1.record(join)
        torch.cuda.synchronize(device)
        e_ms = max_over_ranks(e0.elapsed_time(e1), world, device)
        gla.check(gla.gla_device_error())
        res["e2e"] = dict(ms_per_step=e_ms / ne, steps=ne, h2d=h2d, d2h=d2h, groups=args.e2e_groups,
                          h2d_gbs=h2d_gbs, d2h_gbs=d2h_gbs, buffer_sets=2)
        del hq, hk, hv, hla, hs0, hout, hfs, dv_, host, sets
    del q, k, v, la, s0, out, fs
    torch.cuda.empty_cache()
    return w, BH, res


CONFIG_LEGS = (  # (key, workload, writes the final state)
    ("fp32_small", synth.FP32_SMALL, True),
    ("elu_norm", synth.ELU_NORM, False),
    ("prefill", synth.PREFILL, True),
)


def bench_configs(args, device, rank):
    """The other prefill workloads, each timed launch by launch with CUDA events on the launching
    stream; L2 (129 MB) is flushed before every timed launch by writing a 256 MB buffer, so the
    workloads smaller than L2 (the fp32 and elu+1 ones) read their inputs from HBM too."""
    import torch

    import causal_gated_linear_gb300 as gla
    stream = torch.cuda.current_stream(device)
    flush = torch.empty(64 << 20, dtype=torch.float32, device=device)
    res = {}
    for key, w0, final in CONFIG_LEGS:
        w = synth.with_shape(w0, seed=w0.seed + 1000 * rank)
        x = synth.make_prefill(w)
        q, k, v = (to_dev(x[n], device) for n in ("q", "k", "v"))
        la, s0 = to_dev(x["log_alpha"], device), to_dev(x["init_state"], device)
        f32 = w.dtype == "f32"
        out = torch.empty((w.B, w.H, w.L, w.dv), dtype=torch.float32 if f32 else torch.bfloat16, device=device)
        fs = torch.empty((w.B, w.H, w.dk, w.dv), dtype=torch.float32, device=device) if final else None
        flags = (gla.FLAG_FEATURE_ELU1 if w.feature_elu1 else 0) | (gla.FLAG_NORMALIZE if w.normalize else 0)
        dt = gla.F32 if f32 else gla.BF16

        def call():
            r = gla.gla_fwd_ex(q, k, v, out, w.B, w.H, w.L, w.dk, w.dv, log_alpha=la, init_state=s0,
                               final_state=fs, in_dtype=dt, out_dtype=dt, flags=flags, stream=stream)
            if r != 0:
                raise RuntimeError(gla.gla_status_string(r))

        for _ in range(3):
            call()
        torch.cuda.synchronize(device)
        evs = []
        for _ in range(args.config_calls):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            call()
            b.record(stream)
            evs.append((a, b))
        torch.cuda.synchronize(device)
        gla.check(gla.gla_device_error(stream))
        res[key] = dict(w=w, final=final, ms=statistics.mean(a.elapsed_time(b) for a, b in evs),
                        calls=args.config_calls)
        del q, k, v, la, s0, out, fs, x
    del flush
    torch.cuda.empty_cache()
    return res


def bench_decode(args, device, rank):
    import torch

    import causal_gated_linear_gb300 as gla
    NS, H, dk, dv = DEC["NS"], DEC["H"], DEC["dk"], DEC["dv"]
    seed = DEC["seed"] + 1000 * rank
    st = to_dev(synth.decode_state(NS, H, dk, dv, DEC["state_std"], seed), device)
    n = args.decode_steps
    # one fresh token per (sequence, head) for every step, drawn on the device before the timed
    # region from a seeded generator with the workload's distributions: q, k, v ~ N(0, 1) in bf16,
    # log alpha = logsigmoid(N(4, 1.5)) in fp32 (10.5 MB per step)
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    tq = torch.randn((n, NS, H, dk), generator=g, device=device).to(torch.bfloat16)
    tk = torch.randn((n, NS, H, dk), generator=g, device=device).to(torch.bfloat16)
    tv = torch.randn((n, NS, H, dv), generator=g, device=device).to(torch.bfloat16)
    tla = torch.nn.functional.logsigmoid(
        torch.randn((n, NS, H, dk), generator=g, device=device) * DEC["gate_std"] + DEC["gate_mean"])
    out = torch.empty((NS, H, dv), dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream(device)

    def step(i):
        r = gla.gla_decode_step(tq[i], tk[i], tv[i], tla[i], st, out, NS, H, dk, dv, stream=stream)
        if r != 0:
            raise RuntimeError(gla.gla_status_string(r))

    for i in range(8):
        step(i)
    torch.cuda.synchronize(device)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for i in range(n):
        step(i)
    ev1.record(stream)
    torch.cuda.synchronize(device)
    gla.check(gla.gla_device_error(stream))
    ms = ev0.elapsed_time(ev1) / n
    del tq, tk, tv, tla
    torch.cuda.empty_cache()
    return dict(ms_per_step=ms, steps=n, NS=NS, H=H, dk=dk, dv=dv)


def bench_decode_multi(args, device, rank):
    """Several tokens per sequence per call (the prefill -> decode hand-off) through gla_fwd with
    the state advanced in place."""
    import torch

    import causal_gated_linear_gb300 as gla
    w = synth.with_shape(synth.DECODE_MULTI, seed=synth.DECODE_MULTI.seed + 1000 * rank)
    x = synth.make_prefill(w)
    q, k, v = (to_dev(x[n], device) for n in ("q", "k", "v"))
    la, st = to_dev(x["log_alpha"], device), to_dev(x["init_state"], device)
    out = torch.empty((w.B, w.H, w.L, w.dv), dtype=torch.bfloat16, device=device)
    stream = torch.cuda.current_stream(device)

    def call():
        r = gla.gla_fwd(q, k, v, la, st, out, st, w.B, w.H, w.L, w.dk, w.dv, C, stream=stream)
        if r != 0:
            raise RuntimeError(gla.gla_status_string(r))

    for _ in range(4):
        call()
    torch.cuda.synchronize(device)
    n = args.multi_calls
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(n):
        call()
    ev1.record(stream)
    torch.cuda.synchronize(device)
    gla.check(gla.gla_device_error(stream))
    return dict(w=w, ms_per_call=ev0.elapsed_time(ev1) / n, calls=n)


def bench_delta(args, device, rank):
    """The delta rule (gla_delta_fwd) on its workload: B8 H16 L4096 dk = dv = 128, gated."""
    import torch

    import causal_gated_linear_gb300 as gla
    w = synth.with_shape(synth.DELTA, seed=synth.DELTA.seed + 1000 * rank)
    if args.aux_L:  # reduced sequence length (profiling a small case); the line names it
        w = synth.with_shape(w, L=args.aux_L, name=f"{w.name}_L{args.aux_L}")
    x = synth.make_delta(w)
    q, k, v, b = (to_dev(x[n], device) for n in ("q", "k", "v", "beta"))
    la = to_dev(x["log_alpha"], device)
    out = torch.empty((w.B, w.H, w.L, w.dv), dtype=torch.bfloat16, device=device)
    fs = torch.empty((w.B, w.H, w.dk, w.dv), dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream(device)

    def call(flags=0):
        r = gla.gla_delta_fwd(q, k, v, b, out, w.B, w.H, w.L, w.dk, w.dv, log_alpha=la, final_state=fs,
                              flags=flags, stream=stream)
        if r != 0:
            raise RuntimeError(gla.gla_status_string(r))

    def timed(flags, n):
        for _ in range(2):
            call(flags)
        torch.cuda.synchronize(device)
        evs = []
        for _ in range(n):
            a, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            call(flags)
            e.record(stream)
            evs.append((a, e))
        torch.cuda.synchronize(device)
        gla.check(gla.gla_device_error(stream))
        return statistics.mean(a.elapsed_time(e) for a, e in evs)

    res = dict(w=w, ms=timed(0, args.delta_calls), calls=args.delta_calls)
    # the token-by-token fp32 kernel on the same workload, for comparison
    res["token_ms"] = timed(gla.FLAG_FORCE_SIMT, 2)
    return res


def bench_bwd(args, device, rank):
    """The backward pass (gla_bwd) on its workload: B8 H16 L4096 dk = dv = 128, bf16, gated;
    all of dq, dk, dv and dlog_alpha (the chunk form on the tensor cores; the recurrent fp32
    kernel timed beside it)."""
    import torch

    import causal_gated_linear_gb300 as gla
    w = synth.with_shape(synth.BWD, seed=synth.BWD.seed + 1000 * rank)
    if args.aux_L:  # reduced sequence length (profiling a small case); the line names it
        w = synth.with_shape(w, L=args.aux_L, name=f"{w.name}_L{args.aux_L}")
    x = synth.make_bwd(w)
    q, k, v, do = (to_dev(x[n], device) for n in ("q", "k", "v", "dout"))
    la = to_dev(x["log_alpha"], device)
    f32 = lambda *s: torch.empty(s, dtype=torch.float32, device=device)
    dq, dk, dv, dla = f32(w.B, w.H, w.L, w.dk), f32(w.B, w.H, w.L, w.dk), f32(w.B, w.H, w.L, w.dv), \
        f32(w.B, w.H, w.L, w.dk)
    stream = torch.cuda.current_stream(device)

    def call(flags=0):
        r = gla.gla_bwd(q, k, v, do, dq, dk, dv, w.B, w.H, w.L, w.dk, w.dv, log_alpha=la, dlog_alpha=dla,
                        flags=flags, stream=stream)
        if r != 0:
            raise RuntimeError(gla.gla_status_string(r))

    def timed(flags, n):
        for _ in range(2):
            call(flags)
        torch.cuda.synchronize(device)
        evs = []
        for _ in range(n):
            a, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            call(flags)
            e.record(stream)
            evs.append((a, e))
        torch.cuda.synchronize(device)
        gla.check(gla.gla_device_error(stream))
        return statistics.mean(a.elapsed_time(e) for a, e in evs)

    res = dict(w=w, ms=timed(0, args.bwd_calls), calls=args.bwd_calls)
    # the recurrent fp32 kernel on the same workload, for comparison
    res["recurrent_ms"] = timed(gla.FLAG_FORCE_SIMT, 2)
    return res


def run_gla(args):
    import torch
    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    import causal_gated_linear_gb300 as gla
    gla.load()
    peaks = load_peaks()

    w, BH, pre = bench_prefill(args, device, rank, world)
    cfgs = bench_configs(args, device, rank) if args.config_calls > 0 else {}
    dec = bench_decode(args, device, rank) if args.decode_steps > 0 else None
    mdec = bench_decode_multi(args, device, rank) if args.multi_calls > 0 else None
    dlt = bench_delta(args, device, rank) if args.delta_calls > 0 else None
    bwd = bench_bwd(args, device, rank) if args.bwd_calls > 0 else None

    ms = pre["total_ms"] / args.steps
    tokens = w.B * w.L
    value = job_throughput(tokens, args.steps, world, pre["total_ms"])
    flops = prefill_flops(w)
    abytes = prefill_bytes(w)
    lt = pre["per_launch_ms"] / 1e3
    ach_gbs = abytes / lt / 1e9
    tflops = flops / lt / 1e12
    traffic = recorded_traffic("gla_prefill_tc_kernel")
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "L": w.L, "dk": w.dk, "dv": w.dv, "chunk": C,
                   "inputs": "bf16 q/k/v, fp32 log alpha, fp32 init state, out bf16 + final state",
                   "l2": "inputs (4.3 GB/step) larger than L2: no flush", "parallelism": f"replicas x{world}"},
        "tflops": tflops,
        "tensor_frac": tflops / peaks["bf16_tflops"],
        "roofline": {"bound": "hbm", "achieved": ach_gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": ach_gbs / peaks["hbm_gbs"], "traffic": traffic,
                     "kernel": "gla_prefill_tc_kernel", "alg_bytes_per_launch": abytes,
                     "peak_source": peaks["source"]},
        "gpu_launches": args.steps,
        "clocks": pre["clocks"],
    }
    if cfgs:
        line["configs"] = {}
    for key, r in cfgs.items():
        cw = r["w"]
        cb = prefill_bytes(cw, final_state=r["final"])
        cf = prefill_flops(cw)
        sec = r["ms"] / 1e3
        gbs = cb / sec / 1e9
        line["configs"][key] = {
            "workload": cw.name, "ms_per_launch": r["ms"], "us_per_launch": r["ms"] * 1e3, "calls": r["calls"],
            "tokens_per_s": cw.B * cw.L / sec, "tflops": cf / sec / 1e12, "tensor_frac": cf / sec / 1e12 /
            peaks["bf16_tflops"], "dtype": cw.dtype, "l2": "flushed (256 MB write) before every timed launch",
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": gbs / peaks["hbm_gbs"], "alg_bytes_per_launch": cb,
                         "kernel": "gla_prefill_simt_kernel" if cw.dtype == "f32" else "gla_prefill_tc_kernel"}}
    if dec is not None:
        dbytes = decode_bytes(dec["NS"], dec["H"], dec["dk"], dec["dv"])
        gbs = dbytes / (dec["ms_per_step"] / 1e3) / 1e9
        line["decode"] = {"workload": DEC["name"], "ms_per_step": dec["ms_per_step"], "steps": dec["steps"],
                          "state_hbm_gbs": gbs, "unit": "GB/s",
                          "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                       "frac": gbs / peaks["hbm_gbs"],
                                       "traffic": recorded_traffic("gla_decode_kernel"),
                                       "kernel": "gla_decode_kernel", "alg_bytes_per_launch": dbytes},
                          "tokens_per_s": dec["NS"] * dec["H"] / (dec["ms_per_step"] / 1e3) / dec["H"],
                          "tokens": "a fresh token per (sequence, head) every step, all steps consecutive"}
    if "scalar" in pre:
        sw = pre["scalar"]["w"]
        sbytes = prefill_bytes(sw)
        sgbs = sbytes / (pre["scalar"]["per_launch_ms"] / 1e3) / 1e9
        line["scalar_gate"] = {
            "workload": sw.name, "ms_per_launch": pre["scalar"]["per_launch_ms"], "calls": pre["scalar"]["calls"],
            "tokens_per_s": sw.B * sw.L / (pre["scalar"]["per_launch_ms"] / 1e3),
            "roofline": {"bound": "hbm", "achieved": sgbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": sgbs / peaks["hbm_gbs"],
                         "traffic": recorded_traffic("gla_prefill_tc_kernel_scalar_gate"),
                         "kernel": "gla_prefill_tc_kernel (per-token gate)", "alg_bytes_per_launch": sbytes}}
    if dlt is not None:
        dw = dlt["w"]
        sec = dlt["ms"] / 1e3
        db = delta_bytes(dw)
        dgbs = db / sec / 1e9
        cfl = delta_chunk_flops(dw)
        line["delta"] = {
            "workload": dw.name, "ms_per_launch": dlt["ms"], "calls": dlt["calls"],
            "tokens_per_s": dw.B * dw.L / sec, "tflops": cfl / sec / 1e12,
            "tensor_frac": cfl / sec / 1e12 / peaks["bf16_tflops"],
            "path": "chunk form on the tensor cores (per-chunk triangular solve)",
            "roofline": {"bound": "hbm", "achieved": dgbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": dgbs / peaks["hbm_gbs"], "traffic": recorded_traffic("gla_delta_tc_kernel"),
                         "kernel": "gla_delta_tc_kernel", "alg_bytes_per_launch": db, "alg_flops_per_launch": cfl}}
        if "token_ms" in dlt:
            dfl = delta_flops(dw)
            apk = fp32_alu_peak_tflops(peaks)
            dtf = dfl / (dlt["token_ms"] / 1e3) / 1e12
            line["delta"]["token_by_token"] = {
                "ms_per_launch": dlt["token_ms"], "kernel": "gla_delta_kernel (GLA_FLAG_FORCE_SIMT)",
                "roofline": {"bound": "alu", "achieved": dtf, "peak": apk, "unit": "TFLOP/s", "frac": dtf / apk,
                             "alg_flops_per_launch": dfl,
                             "peak_source": "FP32 FMA: SMs x 128 lanes x 2 flops x max SM clock"}}
    if bwd is not None:
        bw = bwd["w"]
        bb = bwd_bytes(bw)
        sec = bwd["ms"] / 1e3
        gbs = bb / sec / 1e9
        bfl = bwd_chunk_flops(bw)
        line["backward"] = {
            "workload": bw.name, "ms_per_launch": bwd["ms"], "calls": bwd["calls"],
            "tokens_per_s": bw.B * bw.L / sec, "tflops": bfl / sec / 1e12,
            "tensor_frac": bfl / sec / 1e12 / peaks["bf16_tflops"],
            "path": "chunk form on the tensor cores (dq pass + dk/dv pass)",
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": gbs / peaks["hbm_gbs"],
                         "traffic": recorded_traffic("gla_bwd_tc"),
                         "kernel": "gla_bwd_dq_kernel + gla_bwd_dkdv_kernel", "alg_bytes_per_launch": bb,
                         "alg_flops_per_launch": bfl}}
        if "recurrent_ms" in bwd:
            rf = bwd_flops(bw)
            apk = fp32_alu_peak_tflops(peaks)
            rtf = rf / (bwd["recurrent_ms"] / 1e3) / 1e12
            line["backward"]["recurrent"] = {
                "ms_per_launch": bwd["recurrent_ms"], "kernel": "gla_bwd_kernel (GLA_FLAG_FORCE_SIMT)",
                "roofline": {"bound": "alu", "achieved": rtf, "peak": apk, "unit": "TFLOP/s", "frac": rtf / apk,
                             "alg_flops_per_launch": rf,
                             "peak_source": "FP32 FMA: SMs x 128 lanes x 2 flops x max SM clock"}}
    if mdec is not None:
        mw = mdec["w"]
        mbytes = decode_multi_bytes(mw)
        mgbs = mbytes / (mdec["ms_per_call"] / 1e3) / 1e9
        line["decode_multi"] = {
            "workload": mw.name, "tokens_per_call": mw.L, "ms_per_call": mdec["ms_per_call"],
            "calls": mdec["calls"], "tokens_per_s": mw.B * mw.L / (mdec["ms_per_call"] / 1e3),
            "state_hbm_gbs": mgbs, "unit": "GB/s",
            "roofline": {"bound": "hbm", "achieved": mgbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": mgbs / peaks["hbm_gbs"],
                         "traffic": recorded_traffic("gla_prefill_short_kernel"),
                         "kernel": "gla_prefill_short_kernel", "alg_bytes_per_launch": mbytes}}
    if "e2e" in pre:
        e = pre["e2e"]
        line["e2e"] = {"value": tokens * world / (e["ms_per_step"] / 1e3), "unit": "tokens/s",
                       "h2d_bytes_per_step": e["h2d"], "d2h_bytes_per_step": e["d2h"],
                       "ms_per_step": e["ms_per_step"], "steps": e["steps"], "api": "gla_fwd_host",
                       "head_groups": e["groups"], "device_buffer_sets": e["buffer_sets"],
                       "link": {"h2d_gbs": e["h2d_gbs"], "d2h_gbs": e["d2h_gbs"],
                                "h2d_floor_ms": e["h2d"] / e["h2d_gbs"] / 1e6}}
    if rank == 0 and world == 1 and args.cpu_baseline:
        tps, cores, desc, dt = oracle_sample(args.ref_seconds)
        tps1, desc1, dt1 = oracle_single_thread()
        line["cpu_baseline"] = {"value": tps, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                                "sample": desc, "seconds": dt,
                                "single_thread": {"value": tps1, "unit": "tokens/s", "cores": 1,
                                                  "extrapolated": True, "sample": desc1, "seconds": dt1}}
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="gla", choices=["gla", "reference"])
    ap.add_argument("--decode-steps", type=int, default=1024,
                    help="consecutive decode steps timed, each on fresh tokens (0: skip)")
    ap.add_argument("--config-calls", type=int, default=20,
                    help="timed launches of each of the fp32, elu+1 and B8 H16 prefill workloads (0: skip)")
    ap.add_argument("--delta-calls", type=int, default=3,
                    help="timed launches of the delta-rule workload (0: skip)")
    ap.add_argument("--bwd-calls", type=int, default=3,
                    help="timed launches of the backward workload (0: skip)")
    ap.add_argument("--scalar-calls", type=int, default=5,
                    help="timed launches of the long-context workload with one gate per token (0: skip)")
    ap.add_argument("--multi-calls", type=int, default=64,
                    help="timed calls of the 8-tokens-per-sequence hand-off workload (0: skip)")
    ap.add_argument("--no-e2e", dest="e2e", action="store_false")
    ap.add_argument("--e2e-groups", type=int, default=4,
                    help="head groups whose host copies gla_fwd_host overlaps with the computation")
    ap.add_argument("--no-cpu-baseline", dest="cpu_baseline", action="store_false")
    ap.add_argument("--ref-seconds", type=float, default=10.0)
    ap.add_argument("--L", type=int, default=0,
                    help="override the prefill sequence length (small cases for ncu captures)")
    ap.add_argument("--aux-L", type=int, default=0,
                    help="override the delta-rule and backward sequence length (small cases for ncu captures)")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)  # timing rule: at least 3 warm-up steps
    if args.impl == "reference":
        return run_reference(args)
    return run_gla(args)


if __name__ == "__main__":
    sys.exit(main())
