#!/usr/bin/env python
"""Benchmark of SANATAN p=1 attention on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step is one sanatan_chunk_fwd call over the layer-forward workload
(B=4, H=12, T=2048, d=dv=64, bf16 q/k/v): the whole prefill path (load,
feature map, intra-chunk scores, value products, state carry, segment scan,
normalisation, stores).  `value` is prefill tokens/s (B*T per step, all heads),
timed with CUDA events on the launching stream, L2 flushed (256 MiB write)
before every timed step.  The same line also carries the long-prefill,
decode, training and power-sharpened attention (p = 2) measurements (each
timed the same way), the roofline of
the dominant kernel, an end-to-end figure through the C ABI with pinned host
buffers, the float64 oracle timed on the host cores, and the SM clocks
sampled during the timed region.

Under torchrun (N > 1) every rank runs its own copy of the workload (the
sequences are independent: weak scaling, no collective on the data path);
`value` is the tokens of all ranks divided by the slowest rank's time.

`--impl reference` times the float64 oracle (the only reference this method
has) on the host cores, on bounded samples of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
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

from constant_state_recurrence_gb300 import workloads as W  # noqa: E402

PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")
KERNEL_SOURCES = {
    "sanatan_tc_kernel": os.path.join(ROOT, "constant_state_recurrence_gb300", "csrc", "chunk_tc.cu"),
    "pow_attn_kernel": os.path.join(ROOT, "constant_state_recurrence_gb300", "csrc",
                                    "chunk_pow_tc.cu"),
}

# Algorithmic work per token-head (d = dv = 64, F = 6d = 384, C = 64), the
# figures of the hot-path scope table: forward flops 2CF + 2C dv + 4F dv,
# forward bytes 3*64*2 (bf16 q, k, v) + 64*4 (o) + 4 (D); decode bytes per
# slot: read + write of S and z plus q, k, v, o.
FWD_FLOPS_PER_TOKEN_HEAD = 2 * 64 * 384 + 2 * 64 * 64 + 4 * 384 * 64        # 155,648
FWD_BYTES_PER_TOKEN_HEAD = 3 * 64 * 2 + 64 * 4 + 4                          # 644
BWD_FLOPS_PER_TOKEN_HEAD = 6 * 64 * 384 + 4 * 64 * 64 + 10 * 384 * 64       # 409,600
DECODE_BYTES_PER_SLOT = 2 * (384 * 64 + 384) * 4 + 4 * 64 * 4               # 200,704

FLUSH_BYTES = 256 << 20

# Both arms report this metric on the layer-forward workload (B=4 H=12 T=2048).
METRIC = "SANATAN p=1 prefill tokens/s"
POWER_P = 2          # power of the sharpened-attention leg (the pre-training stage's p)
ABLATION_P = 2       # power of the ablation-map leg
HARMONICS = 2        # harmonics of the harmonic-map leg
FP32_LANES_PER_SM = 128   # FP32 FMA lanes per SM (the CUDA-core peak of the harmonic leg)

# Data shard of this process: under torchrun every rank processes its own
# sequences (same gamma, omega, phi), set in main().
SHARD = 0


def peaks():
    try:
        with open(PEAKS_FILE) as f:
            p = json.load(f)
        return dict(hbm=float(p["hbm_gbs"]), bf16=float(p["bf16_tflops"]),
                    bf16_sustained=float(p["bf16_tflops_sustained"]),
                    sm_max_mhz=float(p.get("sm_max_mhz", 2070.0)), source="measured")
    except Exception:
        return dict(hbm=6800.0, bf16=1900.0, bf16_sustained=1700.0, sm_max_mhz=2070.0,
                    source="fallback")


def source_hash(path):
    with open(path, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def traffic_for(kernel, workload):
    """Per-launch DRAM bytes from a committed ncu summary, if the kernel source
    is unchanged since the counters were taken; otherwise None."""
    try:
        with open(TRAFFIC_FILE) as f:
            t = json.load(f)
        rec = t[kernel][workload]
        if rec["source_sha256_16"] != source_hash(KERNEL_SOURCES[kernel]):
            return None
        return float(rec["bytes_per_launch"])
    except Exception:
        return None


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples every 100 ms."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(self.gpu), "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.thread.join(timeout=2)

    def summary(self):
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
            except ValueError:
                continue
            for n, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}


def capture(step, i):
    """One CUDA graph of step(i): the library's launches on the capture stream."""
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step(i)
    return g


def timed_steps(step, steps, flush, stream, profile=None, per_step_inputs=False):
    """Run `steps` steps, each after an L2 flush; return per-step ms (whole
    step) and, if `profile` is given, per-step ms of the dominant kernel.

    Whole steps are replayed from CUDA graphs captured beforehand (one graph,
    or one per step when the steps read different inputs), so the device time
    is not stretched by host-side launch overhead; a graph holds exactly the
    launches of one eager call.  The dominant kernel is timed in a second,
    eager pass with events the library records right around its launch."""
    from constant_state_recurrence_gb300 import sanatan as S
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    graphs = [capture(step, i) for i in range(steps if per_step_inputs else 1)]
    if not per_step_inputs:
        flush.zero_()
        graphs[0].replay()  # the first replay uploads the graph
    torch.cuda.synchronize()
    for i in range(steps):
        flush.zero_()
        ev[i][0].record(stream)
        graphs[i if per_step_inputs else 0].replay()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    whole = [a.elapsed_time(b) for a, b in ev]
    kern = None
    if profile:
        kev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(steps)]
        for i in range(steps):
            flush.zero_()
            S.set_profile_events(*kev[i])
            step(i)
        S.set_profile_events(None, None)
        torch.cuda.synchronize()
        kern = [a.elapsed_time(b) for a, b in kev]
    return whole, kern


def prefill_case(w, dev, flush, steps, warmup, stream):
    from constant_state_recurrence_gb300 import sanatan as S
    x = W.make(w, device=dev, shard=SHARD)
    g = {n: x[n] for n in ("q", "k", "v", "gamma", "omega", "phi")}
    B, H, T = x["B"], x["H"], x["T"]
    o = torch.empty(B, H, T, 64, dtype=torch.float32, device=dev)
    D = torch.empty(B, H, T, dtype=torch.float32, device=dev)
    ws_n = S.chunk_fwd_workspace_size(B, H, T)
    ws = torch.empty(max(ws_n, 16), dtype=torch.uint8, device=dev)
    segs, launches = S.chunk_fwd_plan(B, H, T)

    def step(_i):
        S.sanatan_chunk_fwd(g["q"], g["k"], g["v"], g["gamma"], g["omega"], g["phi"], out=o,
                            D_out=D, workspace=ws)

    for _ in range(warmup):
        flush.zero_()
        step(0)
    torch.cuda.synchronize()
    S.device_status()
    return dict(step=step, B=B, H=H, T=T, segs=segs, launches=launches, x=x, o=o, D=D, ws=ws,
                g=g)


E2E_SLICES = (2, 4, 8, 12)  # sequence slices tried for the pipelined host-buffer forward (best
                            # reported)


def e2e_prefill(case, dev, steps, stream):
    """tokens/s through the public call with pinned host buffers, every step:
    H2D of q, k, v, the chunked forward, D2H of o.  The library's HostForward
    pipelines the B * H sequences in E2E_SLICES slices over three streams (copies in,
    attention, copies out), captured once as a CUDA graph for the fixed pinned
    host buffers and replayed every step; the unpipelined sequence on one stream
    is timed beside it."""
    from constant_state_recurrence_gb300 import sanatan as S
    g, o, D, ws = case["g"], case["o"], case["D"], case["ws"]
    hq, hk, hv = (case["x"][n].to("cpu").pin_memory() for n in ("q", "k", "v"))
    ho = torch.empty(o.shape, dtype=o.dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv))
    d2h = ho.numel() * ho.element_size()
    B, H, T = case["B"], case["H"], case["T"]
    dq, dk, dv = torch.empty_like(g["q"]), torch.empty_like(g["k"]), torch.empty_like(g["v"])

    def run_serial():
        dq.copy_(hq, non_blocking=True)
        dk.copy_(hk, non_blocking=True)
        dv.copy_(hv, non_blocking=True)
        S.sanatan_chunk_fwd(dq, dk, dv, g["gamma"], g["omega"], g["phi"], out=o, D_out=D,
                            workspace=ws)
        ho.copy_(o, non_blocking=True)

    def timed(run):
        for _ in range(3):
            run()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(steps):
            run()
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / steps

    ms_serial = timed(run_serial)
    o_ref = o.to("cpu")
    best = None
    by_slices = {}
    for n in E2E_SLICES:
        m = B * H // n
        if (B * H) % n or not (m % H == 0 or H % m == 0):
            continue
        hf = S.HostForward(B, H, T, slices=n, device=dev)
        hf.capture(hq, hk, hv, g["gamma"], g["omega"], g["phi"], ho)
        ms_n = timed(hf.replay)
        # the slices split the sequences differently: equal up to the bf16 bar
        ok = bool((ho - o_ref).abs().max().item() <= 5e-3)
        by_slices[n] = ms_n
        if best is None or ms_n < best[0]:
            best = (ms_n, n, ok)
        del hf
    ms, slices, ok = best
    return dict(ms=ms, h2d=h2d, d2h=d2h, ms_serial=ms_serial, slices=slices, matches=ok,
                by_slices=by_slices)


DECODE_STEPS = 1024   # the decode workload's steps after the prefill


def timed_decode(case, n_cold, flush, stream):
    """Device time of decode steps.  Cold: each step right after a 256 MiB
    L2-flush write, eager launches bracketed by events (the flush kernel hides
    the host's launch of the step, so the interval is the step's kernel, its
    state read from HBM).  Warm: one CUDA graph of all DECODE_STEPS steps back
    to back (a state that fits L2 stays there: the effective figure)."""
    step = case["step"]
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(n_cold)]
    for i in range(n_cold):
        flush.zero_()
        ev[i][0].record(stream)
        step(i)
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    cold = [a.elapsed_time(b) for a, b in ev]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in range(DECODE_STEPS):
            step(i)
    g.replay()  # upload (and one pass over the steps)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    flush.zero_()
    a.record(stream)
    g.replay()
    b.record(stream)
    torch.cuda.synchronize()
    return cold, a.elapsed_time(b) / DECODE_STEPS


def decode_case(batch, dev, flush, steps, warmup, stream):
    """Decode workload: 12 layers x 12 heads = 144 state slots per sequence,
    state built by a bf16 chunked prefill of 4096 N(0,1) tokens, then
    single-token steps with fresh f32 N(0,1) q, k, v at positions 4096, ..."""
    from constant_state_recurrence_gb300 import sanatan as S
    w = W.DECODE
    G = 144
    x = W.make(w, device=dev, B=batch, shard=SHARD)
    _, _, Sx, zx = S.sanatan_chunk_fwd(x["q"], x["k"], x["v"], x["gamma"], x["omega"], x["phi"],
                                       want_D=False, want_state=True)
    del x["q"], x["k"], x["v"]
    N = batch * G
    Sd = Sx.reshape(N, 384, 64)
    zd = zx.reshape(N, 384)
    gen = W.generator(w.seed + 100 * batch, dev)
    nsteps = max(steps, DECODE_STEPS) + warmup
    q, k, v = W.decode_tokens(N, 64, 64, nsteps, gen)
    pos = [torch.full((N,), 4096 + i, dtype=torch.int64, device=dev) for i in range(nsteps)]
    o = torch.empty(N, 64, dtype=torch.float32, device=dev)

    def step(i):
        S.sanatan_decode_step(Sd, zd, q[i], k[i], v[i], x["gamma"], x["omega"], x["phi"], pos[i],
                              out=o)

    for i in range(warmup):
        flush.zero_()
        step(i)
    torch.cuda.synchronize()
    return dict(step=lambda i: step(warmup + i), N=N)


def train_case(dev, flush, steps, warmup, stream):
    """Training step of the B=8, H=12, T=4096 workload: the chunked forward
    (keeping o and D) then the backward to dq, dk, dv, dgamma, domega, dphi
    (reusing the forward's per-segment state sums from its workspace)."""
    from constant_state_recurrence_gb300 import sanatan as S
    x = W.make(W.TRAIN, device=dev, with_grad_out=True, shard=SHARD)
    g = {n: x[n] for n in ("q", "k", "v", "gamma", "omega", "phi", "dO")}
    B, H, T = x["B"], x["H"], x["T"]
    o = torch.empty(B, H, T, 64, dtype=torch.float32, device=dev)
    D = torch.empty(B, H, T, dtype=torch.float32, device=dev)
    ws = torch.empty(max(S.chunk_fwd_workspace_size(B, H, T), 16), dtype=torch.uint8, device=dev)
    bws_n = S.chunk_bwd_workspace_size(B, H, T)
    bws = torch.empty(max(bws_n, 16), dtype=torch.uint8, device=dev) if bws_n else None
    _, fwd_launches = S.chunk_fwd_plan(B, H, T)

    def step(_i):
        S.sanatan_chunk_fwd(g["q"], g["k"], g["v"], g["gamma"], g["omega"], g["phi"], out=o,
                            D_out=D, workspace=ws)
        S.sanatan_chunk_bwd(g["q"], g["k"], g["v"], g["gamma"], g["omega"], g["phi"], o, D,
                            g["dO"], want_dphi=True, workspace=bws, fwd_workspace=ws)

    for _ in range(warmup):
        flush.zero_()
        step(0)
    torch.cuda.synchronize()
    S.device_status()
    return dict(step=step, B=B, H=H, T=T, fwd_launches=fwd_launches)


def power_case(p, dev, flush, steps, warmup, stream):
    """Power-sharpened attention (eq. (8) at integer p) over the layer-forward
    workload: feature preparation plus the quadratic tensor-core kernel."""
    from constant_state_recurrence_gb300 import sanatan as S
    x = W.make(W.LAYER, device=dev, shard=SHARD)
    g = {n: x[n] for n in ("q", "k", "v", "gamma", "omega", "phi")}
    B, H, T = x["B"], x["H"], x["T"]
    o = torch.empty(B, H, T, 64, dtype=torch.float32, device=dev)
    D = torch.empty(B, H, T, dtype=torch.float32, device=dev)
    ws = torch.empty(S.power_fwd_workspace_size(B, H, T), dtype=torch.uint8, device=dev)

    def step(_i):
        S.sanatan_power_fwd(g["q"], g["k"], g["v"], g["gamma"], g["omega"], g["phi"], p, out=o,
                            D_out=D, workspace=ws)

    for _ in range(warmup):
        flush.zero_()
        step(0)
    torch.cuda.synchronize()
    S.device_status()
    return dict(step=step, B=B, H=H, T=T, p=p)


def power_train_case(p, dev, flush, steps, warmup, stream):
    """Power-sharpened attention training step on the layer workload: the
    forward (keeping o and D) then the backward."""
    from constant_state_recurrence_gb300 import sanatan as S
    x = W.make(W.LAYER, device=dev, with_grad_out=True, shard=SHARD)
    g = {n: x[n] for n in ("q", "k", "v", "gamma", "omega", "phi", "dO")}
    B, H, T = x["B"], x["H"], x["T"]
    o = torch.empty(B, H, T, 64, dtype=torch.float32, device=dev)
    D = torch.empty(B, H, T, dtype=torch.float32, device=dev)
    ws = torch.empty(S.power_fwd_workspace_size(B, H, T), dtype=torch.uint8, device=dev)
    bws = torch.empty(S.power_bwd_workspace_size(B, H, T), dtype=torch.uint8, device=dev)

    def step(_i):
        S.sanatan_power_fwd(g["q"], g["k"], g["v"], g["gamma"], g["omega"], g["phi"], p, out=o,
                            D_out=D, workspace=ws)
        S.sanatan_power_bwd(g["q"], g["k"], g["v"], g["gamma"], g["omega"], g["phi"], p, o, D,
                            g["dO"], workspace=bws)

    for _ in range(warmup):
        flush.zero_()
        step(0)
    torch.cuda.synchronize()
    S.device_status()
    return dict(step=step, B=B, H=H, T=T, p=p)


def ablation_case(dev, flush, steps, warmup, stream):
    """The ablation maps on the layer-forward workload at p = 2: the four-channel
    map (clipped scores) and the three-channel map with the printed +d shift;
    feature preparation plus the quadratic tensor-core kernel, as the power leg."""
    from constant_state_recurrence_gb300 import sanatan as S
    x = W.make(W.LAYER, device=dev, shard=SHARD)
    g = {n: x[n] for n in ("q", "k", "v", "gamma", "omega", "phi")}
    B, H, T = x["B"], x["H"], x["T"]
    o = torch.empty(B, H, T, 64, dtype=torch.float32, device=dev)
    D = torch.empty(B, H, T, dtype=torch.float32, device=dev)
    ws = torch.empty(S.power_fwd_workspace_size(B, H, T), dtype=torch.uint8, device=dev)
    cases = {}
    for ch, shift in ((4, 0.0), (3, 64.0)):
        def step(_i, ch=ch, shift=shift):
            S.sanatan_ablation_fwd(g["q"], g["k"], g["v"], g["gamma"], g["omega"], g["phi"],
                                   ABLATION_P, ch, shift=shift, out=o, D_out=D, workspace=ws)
        for _ in range(warmup):
            flush.zero_()
            step(0)
        cases[ch] = dict(step=step, shift=shift)
    torch.cuda.synchronize()
    S.device_status()
    return dict(cases=cases, B=B, H=H, T=T)


def harmonic_case(dev, flush, steps, warmup, stream):
    """The harmonic map (N = 2) on the CUDA cores: the chunked forward over the
    layer-forward workload and one decode step of 144 slots (batch 1) from a
    state of that size."""
    from constant_state_recurrence_gb300 import sanatan as S
    x = W.make(W.LAYER, device=dev, shard=SHARD)
    g = {n: x[n] for n in ("q", "k", "v", "gamma", "omega", "phi")}
    B, H, T = x["B"], x["H"], x["T"]
    N = HARMONICS
    F = S.harmonic_features(N)

    def fwd(_i):
        S.sanatan_chunk_fwd_harmonic(g["q"], g["k"], g["v"], g["gamma"], g["omega"], g["phi"], N)

    def fwd3(_i):
        S.sanatan_chunk_fwd_harmonic(g["q"], g["k"], g["v"], g["gamma"], g["omega"], g["phi"], 3)

    dO = torch.randn(B, H, T, 64, generator=W.generator(W.LAYER.seed + 5, dev),
                     device=dev).to(torch.bfloat16)
    ws_b = torch.empty(max(int(S.lib().sanatan_chunk_bwd_harmonic_workspace_size(B, H, T, 64, 64,
                                                                                 N)), 16),
                       dtype=torch.uint8, device=dev)

    def train(_i):
        o, D, _, _ = S.sanatan_chunk_fwd_harmonic(g["q"], g["k"], g["v"], g["gamma"], g["omega"],
                                                  g["phi"], N)
        S.sanatan_chunk_bwd_harmonic(g["q"], g["k"], g["v"], g["gamma"], g["omega"], g["phi"], N,
                                     o, D, dO, want_dphi=True, workspace=ws_b)

    G = 144
    gen = W.generator(W.DECODE.seed + 11, dev)
    gd, od, pd = W.params(G, 64, "geometric", gen, device=dev)
    Sx = torch.randn(G, F, 64, generator=gen, device=dev) * 0.1
    zx = torch.rand(G, F, generator=gen, device=dev) + 1.0
    q, k, v = (t[0] for t in W.decode_tokens(G, 64, 64, 1, gen))
    pos = torch.full((G,), 4096, dtype=torch.int64, device=dev)

    def dec(_i):
        S.sanatan_decode_step_harmonic(Sx, zx, q, k, v, gd, od, pd, pos, N)

    for _ in range(warmup):
        flush.zero_()
        fwd(0)
        fwd3(0)
        train(0)
        dec(0)
    torch.cuda.synchronize()
    S.device_status()
    return dict(fwd=fwd, fwd3=fwd3, train=train, dec=dec, B=B, H=H, T=T, F=F,
                F3=S.harmonic_features(3), slots=G)


STACK_LAYERS, STACK_HEADS = 12, 12   # the 184M model's attention stack (12 layers x 12 heads)
STACK_STEPS_PER_GRAPH = 64


def stack_case(dev, flush):
    """One decode token through the 12-layer, 12-head attention stack with
    synthetic float32 projections (N(0,1)/sqrt(768)), batch 1; the states
    start from a 64-token run of the same stack."""
    from constant_state_recurrence_gb300 import sanatan as S
    L, heads, Dm = STACK_LAYERS, STACK_HEADS, STACK_HEADS * 64
    gen = W.generator(W.DECODE.seed + 7, dev)
    Wqkv = torch.randn(L, Dm, 3 * Dm, generator=gen, device=dev) / math.sqrt(Dm)
    Wo = torch.randn(L, Dm, Dm, generator=gen, device=dev) / math.sqrt(Dm)
    gamma = torch.full((L, heads), 4.0, device=dev)
    omega = torch.rand(L, heads, 64, generator=gen, device=dev) * (2 * math.pi) - math.pi
    phi = W.rates(heads, 64, "geometric").to(dev).unsqueeze(0).repeat(L, 1, 1).contiguous()
    Sx = torch.zeros(L, heads, 384, 64, device=dev)
    zx = torch.zeros(L, heads, 384, device=dev)
    n = 64 + STACK_STEPS_PER_GRAPH
    xs0 = torch.randn(n, 1, Dm, generator=gen, device=dev)
    xs = xs0.clone()   # the step writes each token's output over its input
    pos = [torch.full((heads,), i, dtype=torch.int64, device=dev) for i in range(n)]
    ws = torch.empty(max(S.lib().sanatan_stack_decode_workspace_size(1, heads, 64), 16),
                     dtype=torch.uint8, device=dev)

    def step(i):
        S.sanatan_stack_decode_step(xs[i], Wqkv, Wo, Sx, zx, gamma, omega, phi, pos[i],
                                    workspace=ws)

    for i in range(64):
        step(i)
    torch.cuda.synchronize()
    S.device_status()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        # every replay starts from the same token inputs (one copy per 64 tokens)
        xs[64:].copy_(xs0[64:])
        for i in range(STACK_STEPS_PER_GRAPH):
            step(64 + i)
    g.replay()
    torch.cuda.synchronize()
    bytes_per_token = (L * (Dm * 3 * Dm + Dm * Dm) * 4
                       + L * heads * 2 * (384 * 64 + 384) * 4)
    return dict(graph=g, bytes=bytes_per_token, launches=1)


def timed_stack(case, reps, stream):
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(reps):
        case["graph"].replay()
    b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / (reps * STACK_STEPS_PER_GRAPH)


def power_flops(B, H, T, F=384, dv=64):
    """Algorithmic flops of the causal quadratic form: every pair j <= t takes
    one F-long score and one dv-long weighted sum."""
    return B * H * (T * (T + 1) // 2) * (2 * F + 2 * dv)


def oracle_prefill_sample(batch=4, T=2048):
    """The float64 oracle's recurrent form on B x 12 heads x T tokens of the
    layer-forward workload; returns (tokens/s, seconds, threads)."""
    import numpy as np
    import oracle.sanatan_oracle as O
    x = W.make(W.LAYER, device="cpu", B=batch, T=T)
    f = W.to_f64
    args = [f(x[n]) for n in ("q", "k", "v", "gamma", "omega", "phi")]
    t0 = time.perf_counter()
    O.attn_recurrent(*args)
    dt = time.perf_counter() - t0
    threads = None
    try:
        from threadpoolctl import threadpool_info
        threads = max((i.get("num_threads") or 0) for i in threadpool_info()) or None
    except Exception:
        pass
    del np
    return batch * T / dt, dt, threads or os.cpu_count()


def dist_setup(args):
    from constant_state_recurrence_gb300 import replicas
    r = replicas.setup(use_cuda=torch.cuda.is_available() and args.impl != "reference")
    return r.world, r.rank, r.local


def barrier(world):
    from constant_state_recurrence_gb300 import replicas
    if world > 1:
        replicas.barrier(replicas.Replica(world, 0, 0))


def max_over_ranks(x, world, dev):
    from constant_state_recurrence_gb300 import replicas
    return replicas.max_over_ranks(x, replicas.Replica(world, 0, 0), dev)


def run_reference(args, world, rank):
    if rank != 0:
        return
    T_sample = 256
    vals = []
    for _ in range(args.warmup):
        oracle_prefill_sample(batch=1, T=T_sample)
    secs = 0.0
    threads = os.cpu_count()
    for _ in range(args.steps):
        tps, dt, threads = oracle_prefill_sample(batch=1, T=T_sample)
        vals.append(tps)
        secs += dt
    value = args.steps * T_sample / secs
    line = {
        "impl": "reference", "metric": METRIC, "value": value,
        "unit": "tokens/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * secs / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": W.LAYER.name, "B": 4, "H": 12, "T": 2048,
                   "sample_per_step": f"batch element 0, all 12 heads, first {T_sample} tokens"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                         "sample": f"recurrent float64 form, 1 x 12 heads x {T_sample} tokens "
                                   "per step"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--only", choices=["layer", "long", "decode", "train", "power", "stack",
                                       "ablation", "harmonic"],
                    default=None,
                    help="run one workload only (profiling); the JSON line keeps its keys")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    world, rank, local = dist_setup(args)
    global SHARD
    SHARD = rank
    if args.impl == "reference":
        run_reference(args, world, rank)
        return

    from constant_state_recurrence_gb300 import sanatan as S
    S.lib()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    pk = peaks()
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    steps, warm = args.steps, args.warmup

    want = (lambda name: args.only is None or args.only == name)
    lp_steps = max(4, steps // 5)
    d64_steps = max(4, steps // 5)
    layer = prefill_case(W.LAYER, dev, flush, steps, warm, stream) if want("layer") else None
    longp = prefill_case(W.LONG, dev, flush, lp_steps, warm, stream) if want("long") else None
    dec1 = decode_case(1, dev, flush, steps, warm, stream) if want("decode") else None
    dec64 = decode_case(64, dev, flush, d64_steps, warm, stream) if want("decode") else None
    tr_steps = max(3, steps // 10)
    train = train_case(dev, flush, tr_steps, warm, stream) if want("train") else None
    pw_steps = max(4, steps // 5)
    power = power_case(POWER_P, dev, flush, pw_steps, warm, stream) if want("power") else None
    ptrain = power_train_case(POWER_P, dev, flush, pw_steps, warm, stream) if want("power") else None
    stack = stack_case(dev, flush) if want("stack") else None
    abl = ablation_case(dev, flush, pw_steps, warm, stream) if want("ablation") else None
    hs_steps = max(3, steps // 10)
    harm = harmonic_case(dev, flush, hs_steps, warm, stream) if want("harmonic") else None

    gpu_idx = local
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        try:
            gpu_idx = int(vis.split(",")[local])
        except ValueError:
            pass
    barrier(world)
    torch.cuda.synchronize()
    nan = float("nan")
    l_whole = l_kern = lp_whole = lp_kern = d1_whole = d64_whole = [nan]
    d1_warm = d64_warm = nan
    with ClockSampler(gpu_idx) as clk:
        t_wall0 = time.perf_counter()
        if layer:
            l_whole, l_kern = timed_steps(layer["step"], steps, flush, stream, profile=True)
        if longp:
            lp_whole, lp_kern = timed_steps(longp["step"], lp_steps, flush, stream, profile=True)
        if dec1:
            d1_whole, d1_warm = timed_decode(dec1, steps, flush, stream)
            d64_whole, d64_warm = timed_decode(dec64, d64_steps, flush, stream)
        tr_whole, tr_kern = [nan], [nan]
        if train:
            tr_whole, tr_kern = timed_steps(train["step"], tr_steps, flush, stream, profile=True)
        pw_whole, pw_kern = [nan], [nan]
        pt_whole, pt_kern = [nan], [nan]
        if power:
            pw_whole, pw_kern = timed_steps(power["step"], pw_steps, flush, stream, profile=True)
            pt_whole, pt_kern = timed_steps(ptrain["step"], pw_steps, flush, stream, profile=True)
        st_ms = timed_stack(stack, 16, stream) if stack else nan
        abl_t = {}
        if abl:
            for ch, c in abl["cases"].items():
                abl_t[ch] = timed_steps(c["step"], pw_steps, flush, stream, profile=True)
        hf_whole = hf3_whole = ht_whole = hd_whole = [nan]
        if harm:
            hf_whole, _ = timed_steps(harm["fwd"], hs_steps, flush, stream)
            hf3_whole, _ = timed_steps(harm["fwd3"], hs_steps, flush, stream)
            ht_whole, _ = timed_steps(harm["train"], hs_steps, flush, stream)
            hd_whole, _ = timed_steps(harm["dec"], steps, flush, stream)
        torch.cuda.synchronize()
        t_wall = time.perf_counter() - t_wall0
    barrier(world)
    S.device_status()

    L = layer or dict(B=4, H=12, T=2048, segs=None, launches=0)
    LP = longp or dict(B=1, H=12, T=32768, segs=None)
    D1 = dec1 or dict(N=144)
    D64 = dec64 or dict(N=9216)
    ms = statistics.mean(l_whole)
    ms = max_over_ranks(ms, world, dev)
    tokens_per_step = L["B"] * L["T"]
    value = world * tokens_per_step / (ms * 1e-3)
    kern_ms = statistics.mean(l_kern)
    th_layer = L["B"] * L["H"] * L["T"]
    achieved_tf = FWD_FLOPS_PER_TOKEN_HEAD * th_layer / (kern_ms * 1e-3) / 1e12
    achieved_gbs = FWD_BYTES_PER_TOKEN_HEAD * th_layer / (kern_ms * 1e-3) / 1e9
    traffic = traffic_for("sanatan_tc_kernel", W.LAYER.name)

    lp_ms = statistics.mean(lp_whole)
    lp_kms = statistics.mean(lp_kern)
    th_long = LP["B"] * LP["H"] * LP["T"]
    d1_us = 1e3 * statistics.mean(d1_whole)
    d64_us = 1e3 * statistics.mean(d64_whole)

    e2e = e2e_prefill(layer, dev, steps, stream) if layer else dict(ms=nan, h2d=0, d2h=0)
    layer, longp, dec1, dec64 = L, LP, D1, D64

    line = {
        "metric": METRIC,
        "value": value,
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": steps,
        "warmup": warm,
        "ms_per_step": ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16 q/k/v; gamma=4; omega~U(-pi,pi); "
                "phi_a=10000^(-a/64))",
        "config": {"workload": W.LAYER.name, "B": 4, "H": 12, "T": 2048, "d": 64, "dv": 64,
                   "chunk": 128,
                   "chunk_note": "128-token tensor-core chunk (the M of a full-rate tcgen05.mma); "
                                 "the config's 64-token chunking gives the same sums up to "
                                 "rounding order",
                   "segments_per_sequence": layer["segs"],
                   "parallelism": f"{world} independent replica(s), sequences sharded by rank",
                   "l2": "256 MiB flush write before every timed step",
                   "launch": "each timed step replays a CUDA graph of one library call; "
                             "e2e replays the host pipeline's CUDA graph"},
        "gpu_launches": steps * layer["launches"],
        "roofline": {"bound": "tensor", "kernel": "sanatan_tc_kernel (main pass)",
                     "achieved": achieved_tf, "peak": pk["bf16"], "unit": "TFLOP/s",
                     "frac": achieved_tf / pk["bf16"],
                     "peak_source": f"{pk['source']} bf16 burst",
                     "flops_per_token_head": FWD_FLOPS_PER_TOKEN_HEAD,
                     "kernel_ms": kern_ms,
                     "traffic": traffic},
        "roofline_hbm": {"bound": "hbm", "achieved": achieved_gbs, "peak": pk["hbm"],
                         "unit": "GB/s", "frac": achieved_gbs / pk["hbm"],
                         "bytes_per_token_head": FWD_BYTES_PER_TOKEN_HEAD},
        "e2e": {"value": world * tokens_per_step / (e2e["ms"] * 1e-3), "unit": "tokens/s",
                "h2d_bytes_per_step": e2e["h2d"], "d2h_bytes_per_step": e2e["d2h"],
                "ms_per_step": e2e["ms"], "pipeline_slices": e2e.get("slices"),
                "ms_per_step_unpipelined": e2e.get("ms_serial"),
                "ms_per_step_by_slices": e2e.get("by_slices"),
                "output_matches_device_call": e2e.get("matches")},
        "long_prefill": {
            "workload": W.LONG.name, "tokens_per_s": longp["B"] * longp["T"] / (lp_ms * 1e-3),
            "ms_per_step": lp_ms, "kernel_ms": lp_kms,
            "tc_frac": FWD_FLOPS_PER_TOKEN_HEAD * th_long / (lp_kms * 1e-3) / 1e12 / pk["bf16"],
            "hbm_frac": FWD_BYTES_PER_TOKEN_HEAD * th_long / (lp_kms * 1e-3) / 1e9 / pk["hbm"],
            "segments_per_sequence": longp["segs"], "steps": lp_steps},
        "decode": {
            "B1": {"slots": dec1["N"], "us_per_step": d1_us,
                   "achieved_gbs": DECODE_BYTES_PER_SLOT * dec1["N"] / (d1_us * 1e-6) / 1e9,
                   "hbm_frac": DECODE_BYTES_PER_SLOT * dec1["N"] / (d1_us * 1e-6) / 1e9 / pk["hbm"],
                   "steps": steps,
                   "note": "14.4 MB state (28.9 MB per step read + written); L2 flushed before "
                           "each step; device time of the step's kernel",
                   "warm_us_per_step": 1e3 * d1_warm, "warm_steps": DECODE_STEPS,
                   "warm_effective_gbs": DECODE_BYTES_PER_SLOT * dec1["N"] / (d1_warm * 1e-3) / 1e9,
                   "warm_note": "the 1024 steps of the workload back to back in one CUDA graph, "
                                "no flush: the state stays in the 129 MB L2 (effective bandwidth)"},
            "B64": {"slots": dec64["N"], "us_per_step": d64_us,
                    "achieved_gbs": DECODE_BYTES_PER_SLOT * dec64["N"] / (d64_us * 1e-6) / 1e9,
                    "hbm_frac": DECODE_BYTES_PER_SLOT * dec64["N"] / (d64_us * 1e-6) / 1e9 / pk["hbm"],
                    "steps": d64_steps,
                    "warm_us_per_step": 1e3 * d64_warm, "warm_steps": DECODE_STEPS,
                    "warm_hbm_frac": DECODE_BYTES_PER_SLOT * dec64["N"] / (d64_warm * 1e-3) / 1e9
                                     / pk["hbm"]},
            "bytes_per_slot": DECODE_BYTES_PER_SLOT},
        "train": {
            "workload": W.TRAIN.name, "steps": tr_steps,
            "tokens_per_s": 8 * 4096 / (statistics.mean(tr_whole) * 1e-3),
            "ms_per_step": statistics.mean(tr_whole),
            "bwd_kernel_ms": statistics.mean(tr_kern),
            "tc_frac_step": (FWD_FLOPS_PER_TOKEN_HEAD + BWD_FLOPS_PER_TOKEN_HEAD) * 8 * 12 * 4096
                            / (statistics.mean(tr_whole) * 1e-3) / 1e12 / pk["bf16"],
            "flops_per_token_head": FWD_FLOPS_PER_TOKEN_HEAD + BWD_FLOPS_PER_TOKEN_HEAD,
            "note": "forward + backward per step; bwd_kernel_ms times the backward's dominant kernel"},
        "power": {
            "workload": W.LAYER.name, "p": POWER_P, "steps": pw_steps,
            "tokens_per_s": 4 * 2048 / (statistics.mean(pw_whole) * 1e-3),
            "ms_per_step": statistics.mean(pw_whole),
            "kernel_ms": statistics.mean(pw_kern),
            "flops_per_step": power_flops(4, 12, 2048),
            "tc_frac_kernel": power_flops(4, 12, 2048) / (statistics.mean(pw_kern) * 1e-3)
                              / 1e12 / pk["bf16"],
            "tc_frac_step": power_flops(4, 12, 2048) / (statistics.mean(pw_whole) * 1e-3)
                            / 1e12 / pk["bf16"],
            "traffic": traffic_for("pow_attn_kernel", W.LAYER.name),
            "note": "causal quadratic power attention; flops = pairs j<=t x (2*384 + 2*64); "
                    "step = feature preparation + attention kernel (kernel_ms)"},
        "power_train": {
            "workload": W.LAYER.name, "p": POWER_P, "steps": pw_steps,
            "tokens_per_s": 4 * 2048 / (statistics.mean(pt_whole) * 1e-3),
            "ms_per_step": statistics.mean(pt_whole),
            "bwd_key_pass_ms": statistics.mean(pt_kern),
            "note": "forward + backward of the power-sharpened attention per step"},
        "stack_decode": {
            "workload": f"{STACK_LAYERS} layers x {STACK_HEADS} heads x 64, batch 1, synthetic f32 "
                        "projections", "tokens": 16 * STACK_STEPS_PER_GRAPH,
            "us_per_token": 1e3 * st_ms,
            "bytes_per_token": stack["bytes"] if stack else None,
            "effective_gbs": (stack["bytes"] / (st_ms * 1e-3) / 1e9) if stack else None,
            "launches_per_token": stack["launches"] if stack else None,
            "note": "attention path only (q,k,v projections, p=1 decode of every head, output "
                    "projection + residual) in one cooperative kernel per token; steps replayed "
                    "from CUDA graphs of 64 tokens; the pages' 0.153 ms/token is on unnamed "
                    "hardware (context)"},
        "timed_region_wall_s": t_wall,
    }
    if abl:
        ab = {}
        for ch, (whole, kern) in abl_t.items():
            fl = power_flops(4, 12, 2048, F=ch * 64)
            ab[f"{ch}ch"] = {
                "p": ABLATION_P, "shift": abl["cases"][ch]["shift"],
                "tokens_per_s": 4 * 2048 / (statistics.mean(whole) * 1e-3),
                "ms_per_step": statistics.mean(whole), "kernel_ms": statistics.mean(kern),
                "flops_per_step": fl,
                "tc_frac_kernel": fl / (statistics.mean(kern) * 1e-3) / 1e12 / pk["bf16"]}
        line["ablation"] = dict(workload=W.LAYER.name, steps=pw_steps, **ab,
                                note="ablation maps of the notes at p = 2 (four channels: clipped "
                                     "scores, scale 3d; three channels: +d shift, scale 3d); "
                                     "flops = pairs j<=t x (2 F + 2 dv), F = channels x 64")
    if harm:
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        alu_peak = sms * FP32_LANES_PER_SM * 2 * pk.get("sm_max_mhz", 2070.0) * 1e6 / 1e12
        F = harm["F"]
        th = harm["B"] * harm["H"] * harm["T"]
        hd_ms = statistics.mean(hd_whole)
        dec_bytes = harm["slots"] * (2 * (F * 64 + F) * 4 + 4 * 64 * 4)

        def harm_fwd(whole, nf):
            ms = statistics.mean(whole)
            fl = 4 * nf * (64 + 1)   # state update + readout per token-head (recurrent minimum)
            ach = fl * th / (ms * 1e-3) / 1e12
            return {"workload": W.LAYER.name, "features": nf, "steps": hs_steps,
                    "ms_per_step": ms, "tokens_per_s": harm["B"] * harm["T"] / (ms * 1e-3),
                    "roofline": {"bound": "alu", "achieved": ach, "peak": alu_peak,
                                 "unit": "TFLOP/s", "frac": ach / alu_peak,
                                 "flops_per_token_head": fl,
                                 "peak_source": f"{sms} SMs x {FP32_LANES_PER_SM} FP32 FMA "
                                                "lanes x 2 flops x max SM clock"}}

        line["harmonic"] = {
            "harmonics": HARMONICS, "features": F,
            "forward": harm_fwd(hf_whole, F),
            "forward_N3": harm_fwd(hf3_whole, harm["F3"]),
            "train": {"workload": W.LAYER.name, "steps": hs_steps,
                      "ms_per_step": statistics.mean(ht_whole),
                      "tokens_per_s": harm["B"] * harm["T"] / (statistics.mean(ht_whole) * 1e-3),
                      "note": "forward + backward (dq, dk, dv, dgamma, domega, dphi) per step"},
            "decode": {"slots": harm["slots"], "steps": steps, "us_per_step": 1e3 * hd_ms,
                       "achieved_gbs": dec_bytes / (hd_ms * 1e-3) / 1e9,
                       "hbm_frac": dec_bytes / (hd_ms * 1e-3) / 1e9 / pk["hbm"],
                       "bytes_per_step": dec_bytes},
            "note": "float32 on the CUDA cores (the tensor-core path keeps 320 + 1 features); "
                    "L2 flushed before each step"}
    clocks = clk.summary()
    if clocks:
        line["clocks"] = clocks
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        tps, dt, threads = oracle_prefill_sample(batch=4, T=2048)
        line["cpu_baseline"] = {"value": tps, "unit": "tokens/s", "cores": threads,
                                "kind": "oracle",
                                "sample": f"recurrent float64 oracle on the full layer-forward "
                                          f"workload (4 x 12 heads x 2048 tokens), {dt:.1f} s"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
