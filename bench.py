#!/usr/bin/env python3
"""Benchmark of the Gated DeltaNet recurrence on GB300: prefill tokens/s and decode steps/s at
32 value heads of dimension 128, with the roofline fraction of the dominant kernel.

One timed step = one chunked prefill (gdn_chunk_fwd) of the 8k GQA workload: B=2 sequences of
T=8192 tokens, 16 query/key heads shared by 32 value heads, dk=dv=128, chunk 64, bf16 inputs,
fp32 state (random initial state).  The same line carries two more measurements:
  long_prefill: 4 packed sequences (65536/32768/24576/8192 tokens) with state reset, same heads;
  decode:       512 consecutive single-token steps for 256 sequences x 32 value heads, with the
                512 MiB fp32 state resident on the device (captured in one CUDA graph).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gdn|reference]

N > 1 (launched by torch.distributed.run) runs one independent replica per GPU (the recurrence
does not shard across GPUs: there is no exchange step); value is the sum over ranks divided by
the slowest rank's time.  --impl reference times the fp64 CPU oracle on the host cores instead.
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import gdn_inputs as gi  # noqa: E402

METRIC = "GDN prefill tokens/s & decode steps/s at H=32,d=128; % tensor/HBM roofline"
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}

# DRAM bytes per launch from ncu captures, valid only for the kernel source they were taken on
# (sha256 prefix of the file); None once the source has changed.
NCU_TRAFFIC = {
    # kernel: (source file, sha256 prefix of that file at capture, dram read + write bytes per launch)
    "gdn_tc_prep": ("gated_deltanet_recurrence_03_gb300/csrc/gdn_tc.cu", "0a60363b567a42dd", 139313920 + 343793920),
    "gdn_tc_chain": ("gated_deltanet_recurrence_03_gb300/csrc/gdn_tc.cu", "0a60363b567a42dd", 612444416 + 117266688),
    "decode_step_kernel": ("gated_deltanet_recurrence_03_gb300/csrc/gdn_decode.cu", "0a3ae9abf76d8679", 541133568 + 480455680),
}

PREFILL = gi.WORKLOADS["prefill_gqa_8k"]
LONG = gi.WORKLOADS["prefill_varlen_128k"]
DECODE = gi.WORKLOADS["decode_256x512"]


def rank_info():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


# ---------------------------------------------------------------- replicas (one process per GPU)
def max_over_ranks(dist, x, device="cpu"):
    """The largest of every rank's x (each rank's own time; the job takes as long as its slowest
    replica).  dist is torch.distributed, or None for a single process."""
    if dist is None:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(world, units_per_rank, ms_max):
    """Whole-job throughput: the units all ranks processed divided by the slowest rank's time."""
    return world * units_per_rank / (ms_max / 1e3)


def load_peaks():
    try:
        with open(PEAKS_FILE) as f:
            p = json.load(f)
        return {k: float(p[k]) for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained")}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def source_sha(path):
    with open(os.path.join(ROOT, path), "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def traffic_for(kernel):
    if kernel not in NCU_TRAFFIC:
        return None
    path, sha, nbytes = NCU_TRAFFIC[kernel]
    return nbytes if source_sha(path) == sha else None


# ---------------------------------------------------------------- algorithmic work per launch
def prefill_flops(tokens, w):
    """Canonical MMA flops of one chunked prefill, split by kernel (chunk C):
    prep  : Hqk (K K^T, Q K^T) 4 C dk + Hv (T diag(beta gamma) K) 2 C dk        per token
    chain : Hv ((T diag(beta)) V + (masked Q K^T) U) 4 C dv + Hv (W S, Q S, K^T U) 6 dk dv   per token
    (163,840 flop per token and value head at C = 64, d = 128)."""
    C = w.chunk
    prep = tokens * (w.Hqk * 4 * C * w.dk + w.Hv * 2 * C * w.dk)
    chain = tokens * w.Hv * (4 * C * w.dv + 6 * w.dk * w.dv)
    return prep, chain


def prefill_bytes(tokens, nseq, w, e=2):
    """Algorithmic HBM bytes: q, k, v, g, beta read, out written, S0 read and S_final written."""
    io = tokens * (2 * w.Hqk * w.dk + 2 * w.Hv * w.dv + 2 * w.Hv) * e
    state = 2 * nseq * w.Hv * w.dk * w.dv * 4
    return io + state


def decode_bytes(w, e=2):
    """One decode step: the fp32 state read and written once, plus q, k, v, g, beta, out."""
    state = 2 * w.B * w.Hv * w.dk * w.dv * 4
    io = w.B * (2 * w.Hqk * w.dk + 2 * w.Hv * w.dv + 2 * w.Hv) * e
    return state + io


# ---------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the timed regions run."""
    FIELDS = "clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown," \
             "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown," \
             "clocks_event_reasons.sw_power_cap"

    def __init__(self, index):
        self.index = index
        self.samples = []
        self.active = False
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            if self.active:
                self.samples.append([x.strip() for x in line.split(",")])

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm = [float(s[0]) for s in self.samples if s and s[0].replace(".", "").isdigit()]
        mx = [float(s[1]) for s in self.samples if len(s) > 1 and s[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for s in self.samples for i in range(4) if len(s) > 3 + i and s[3 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(self.samples)}


# ---------------------------------------------------------------- GPU arm
def device_inputs_from_generator(torch, dev, w, copies):
    x = gi.make_prefill_inputs(w)
    sets = []
    for _ in range(copies):
        sets.append({n: torch.from_numpy(np.ascontiguousarray(x[n])).to(dev).to(torch.bfloat16)
                     for n in ("q", "k", "v", "g", "beta")})
    S0 = None if x["S0"] is None else torch.from_numpy(x["S0"]).to(dev)
    return x, sets, S0


def device_inputs_random(torch, dev, w, steps=None, seed=1):
    """Same distributions as the shared generator, drawn on the device (for the large workloads)."""
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed)
    lead = (steps, w.B) if steps else (w.B, w.T)
    unit = lambda s: torch.nn.functional.normalize(torch.randn(*s, generator=gen, device=dev), dim=-1).bfloat16()
    q, k = unit((*lead, w.Hqk, w.dk)), unit((*lead, w.Hqk, w.dk))
    v = torch.randn(*lead, w.Hv, w.dv, generator=gen, device=dev).bfloat16()
    g = torch.nn.functional.logsigmoid(torch.randn(*lead, w.Hv, generator=gen, device=dev) + 3.0).bfloat16()
    beta = torch.sigmoid(torch.randn(*lead, w.Hv, generator=gen, device=dev)).bfloat16()
    return dict(q=q, k=k, v=v, g=g, beta=beta)


def run_gpu(args):
    import torch
    import gated_deltanet_recurrence_03_gb300 as gdn

    rank, world, local = rank_info()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    peaks, peak_src = load_peaks()
    stream = torch.cuda.current_stream(dev)
    clocks = ClockSampler(local)
    clocks.start()

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    def max_ms(x):
        return max_over_ranks(dist, x, dev)

    # ---- headline: chunked prefill of the 8k GQA workload, inputs rotated across 3 copies (> L2 each)
    w = PREFILL
    x, sets, S0 = device_inputs_from_generator(torch, dev, w, copies=3)
    tokens = w.B * w.T
    out = torch.empty_like(sets[0]["v"])
    S_final = torch.empty((w.B, w.Hv, w.dk, w.dv), dtype=torch.float32, device=dev)
    ws = torch.empty(max(1, gdn.workspace_size(w.B, w.T, w.Hqk, w.Hv, w.dk, w.dv)), dtype=torch.uint8, device=dev)
    n_ev = 3
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(n_ev)] for _ in range(args.steps)]
    for row in evs:
        for e in row:
            e.record(stream)

    def prefill_step(i, events=None):
        s = sets[i % len(sets)]
        gdn.gdn_chunk_fwd(s["q"], s["k"], s["v"], s["g"], s["beta"], S0, out=out, S_final=S_final, workspace=ws,
                          chunk=w.chunk, events=None if events is None else [e.cuda_event for e in events])

    for i in range(args.warmup):
        prefill_step(i)
    barrier()
    clocks.active = True
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for i in range(args.steps):
        prefill_step(i)
    t1.record(stream)
    barrier()
    # Kernel durations: a second pass of the same steps with an event recorded between the two kernels
    # (the chain then starts after the prep has finished, without the programmatic overlap of the steps
    # timed above).
    for i in range(args.steps):
        prefill_step(i, evs[i])
    barrier()
    clocks.active = False
    ms_total = max_ms(t0.elapsed_time(t1))
    ms_step = ms_total / args.steps
    k_prep = statistics.mean(r[0].elapsed_time(r[1]) for r in evs)
    k_chain = statistics.mean(r[1].elapsed_time(r[2]) for r in evs)
    gdn.check_device_status()
    f_prep, f_chain = prefill_flops(tokens, w)
    kernels = {"gdn_tc_prep": {"ms": k_prep, "tflops": f_prep / (k_prep * 1e9), "flop": f_prep},
               "gdn_tc_chain": {"ms": k_chain, "tflops": f_chain / (k_chain * 1e9), "flop": f_chain}}
    dominant = max(kernels, key=lambda kname: kernels[kname]["ms"])
    peak_tf = peaks["bf16_tflops"]
    dom = kernels[dominant]
    roofline = {"bound": "tensor", "kernel": dominant, "achieved": round(dom["tflops"], 2), "peak": peak_tf,
                "unit": "TFLOP/s", "frac": round(dom["tflops"] / peak_tf, 4), "traffic": traffic_for(dominant),
                "peak_source": f"{peak_src} burst bf16"}
    whole = (f_prep + f_chain) / (ms_step * 1e9)

    # ---- e2e through the public API with host buffers (pinned), copies inside the timed region.
    # Every step copies its inputs host -> device, runs the prefill and reads out and S_final back.
    # As a serving loop would, the copies of neighbouring steps overlap the compute: host -> device on
    # one stream, the kernels on another, device -> host on a third, double-buffered and ordered by
    # events.  The time is from the first copy in to the last copy out.
    host = {n: torch.from_numpy(np.ascontiguousarray(x[n])).to(torch.bfloat16).pin_memory()
            for n in ("q", "k", "v", "g", "beta")}
    host["S0"] = torch.from_numpy(x["S0"]).pin_memory()
    host_out = [torch.empty(out.shape, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    host_Sf = [torch.empty(S_final.shape, dtype=torch.float32).pin_memory() for _ in range(2)]
    dbuf = [{n: torch.empty(t.shape, dtype=t.dtype, device=dev) for n, t in host.items()} for _ in range(2)]
    dout_e = [torch.empty_like(out) for _ in range(2)]
    dSf_e = [torch.empty_like(S_final) for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = host_out[0].numel() * 2 + host_Sf[0].numel() * 4
    s_in, s_cmp, s_out = (torch.cuda.Stream(dev) for _ in range(3))
    e2e_steps = max(3, min(args.steps, 50))
    n_e = e2e_steps + 2
    ev_in = [torch.cuda.Event() for _ in range(n_e)]
    ev_cmp = [torch.cuda.Event() for _ in range(n_e)]
    ev_out = [torch.cuda.Event() for _ in range(n_e)]

    def e2e_run(steps, t_start=None, t_end=None):
        if t_start is not None:
            t_start.record(s_in)
        for i in range(steps):
            j = i % 2
            with torch.cuda.stream(s_in):   # inputs of step i (buffer set j is free once step i-2 ran)
                if i >= 2:
                    s_in.wait_event(ev_cmp[i - 2])
                for n in host:
                    dbuf[j][n].copy_(host[n], non_blocking=True)
                ev_in[i].record(s_in)
            with torch.cuda.stream(s_cmp):
                s_cmp.wait_event(ev_in[i])
                if i >= 2:
                    s_cmp.wait_event(ev_out[i - 2])   # outputs of step i-2 copied out
                b = dbuf[j]
                gdn.gdn_chunk_fwd(b["q"], b["k"], b["v"], b["g"], b["beta"], b["S0"], out=dout_e[j],
                                  S_final=dSf_e[j], workspace=ws, chunk=w.chunk, stream=s_cmp)
                ev_cmp[i].record(s_cmp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_cmp[i])
                host_out[j].copy_(dout_e[j], non_blocking=True)
                host_Sf[j].copy_(dSf_e[j], non_blocking=True)
                ev_out[i].record(s_out)
        if t_end is not None:
            t_end.record(s_out)

    e2e_run(2)
    barrier()
    te0, te1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e_run(e2e_steps, te0, te1)
    barrier()
    e2e_ms = max_ms(te0.elapsed_time(te1)) / e2e_steps

    # ---- long-context packed prefill (state reset at each boundary)
    wl = LONG
    xl = device_inputs_random(torch, dev, wl)
    cu = torch.tensor(wl.cu_seqlens, dtype=torch.int32, device=dev)
    out_l = torch.empty_like(xl["v"])
    Sf_l = torch.empty((wl.num_seqs, wl.Hv, wl.dk, wl.dv), dtype=torch.float32, device=dev)
    ws_l = torch.empty(max(1, gdn.workspace_size(1, wl.T, wl.Hqk, wl.Hv, wl.dk, wl.dv, num_seqs=wl.num_seqs)),
                       dtype=torch.uint8, device=dev)
    long_steps = max(3, min(10, args.steps))
    ev_l = [[torch.cuda.Event(enable_timing=True) for _ in range(n_ev)] for _ in range(long_steps)]
    for row in ev_l:
        for e in row:
            e.record(stream)

    def long_step(events=None):
        gdn.gdn_chunk_fwd(xl["q"], xl["k"], xl["v"], xl["g"], xl["beta"], None, cu_seqlens=cu, out=out_l,
                          S_final=Sf_l, workspace=ws_l, chunk=wl.chunk,
                          events=None if events is None else [e.cuda_event for e in events])

    for _ in range(3):
        long_step()
    barrier()
    clocks.active = True
    t0.record(stream)
    for i in range(long_steps):
        long_step(ev_l[i])
    t1.record(stream)
    barrier()
    clocks.active = False
    long_ms = max_ms(t0.elapsed_time(t1)) / long_steps
    lp = statistics.mean(r[0].elapsed_time(r[1]) for r in ev_l)
    lc = statistics.mean(r[1].elapsed_time(r[2]) for r in ev_l)
    lf_prep, lf_chain = prefill_flops(wl.T, wl)
    del xl, out_l, ws_l

    # ---- the recurrent core of one layer on the same workload: short causal conv of the packed q/k/v
    #      projection (one launch, q, k and v written as the dense tensors the recurrence takes), gates
    #      from the raw a/b projections, l2 norm of q and k, chunked recurrence, gated RMS norm with
    #      silu(z); prefill inputs larger than L2
    Cq, Cv = w.Hqk * w.dk, w.Hv * w.dv
    Cc = 2 * Cq + Cv
    bf = torch.bfloat16
    gen = torch.Generator(device=dev).manual_seed(5)
    proj = torch.randn(w.B, w.T, Cc, device=dev, generator=gen).to(bf)
    conv_w = 0.5 * torch.randn(Cc, 4, device=dev, generator=gen)
    qc = torch.empty(w.B, w.T, w.Hqk, w.dk, dtype=bf, device=dev)
    kc, vc = torch.empty_like(qc), torch.empty(w.B, w.T, w.Hv, w.dv, dtype=bf, device=dev)
    conv_cache = torch.empty(w.B, 3, Cc, dtype=bf, device=dev)
    a_raw = torch.randn(w.B, w.T, w.Hv, device=dev, generator=gen).to(bf)
    b_raw = torch.randn(w.B, w.T, w.Hv, device=dev, generator=gen).to(bf)
    A_log = -0.5 + 0.5 * torch.randn(w.Hv, device=dev, generator=gen)
    dt_bias = 0.5 * torch.randn(w.Hv, device=dev, generator=gen)
    z = torch.randn(w.B, w.T, w.Hv, w.dv, device=dev, generator=gen).to(bf)
    norm_w = 1.0 + 0.1 * torch.randn(w.dv, device=dev, generator=gen)
    layer_steps = max(3, min(10, args.steps))
    ev_c = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(layer_steps)]
    ev_p = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(layer_steps)]
    for row in ev_c + ev_p:
        for e in row:
            e.record(stream)

    def layer_step(i=None):
        if i is not None:
            ev_c[i][0].record(stream)
        gdn.gdn_causal_conv1d_fwd_qkv(proj, conv_w, (Cq, Cq, Cv), None, cache_out=conv_cache,
                                      out=(qc.view(w.B, w.T, Cq), kc.view(w.B, w.T, Cq), vc.view(w.B, w.T, Cv)))
        if i is not None:
            ev_c[i][1].record(stream)
        gdn.gdn_chunk_fwd(qc, kc, vc, a_raw, b_raw, S0, out=out, S_final=S_final, workspace=ws, chunk=w.chunk,
                          scale=w.dk ** -0.5, normalize_qk=True, raw_gates=(A_log, dt_bias),
                          output_gate=(z, norm_w, 1e-6),
                          events=None if i is None else [e.cuda_event for e in ev_p[i]])

    for _ in range(3):
        layer_step()
    barrier()
    clocks.active = True
    t0.record(stream)
    for i in range(layer_steps):
        layer_step(i)
    t1.record(stream)
    barrier()
    clocks.active = False
    layer_ms = max_ms(t0.elapsed_time(t1)) / layer_steps
    gdn.check_device_status()
    conv_ms = statistics.mean(r[0].elapsed_time(r[1]) for r in ev_c)
    gate_ms = statistics.mean(r[2].elapsed_time(r[3]) for r in ev_p)
    conv_bytes = 2 * (w.B * w.T * Cc * 2) + Cc * 4 * 4 + w.B * 3 * Cc * 2
    gate_bytes = 3 * (w.B * w.T * Cv * 2) + w.dv * 4
    del proj, qc, kc, vc, a_raw, b_raw, z

    # ---- backward pass of the same 8k workload (gradients w.r.t. q, k, v, g, beta, S0)
    xb = device_inputs_random(torch, dev, w, seed=3)
    dout = torch.randn(w.B, w.T, w.Hv, w.dv, device=dev).to(torch.bfloat16)
    dSf = 0.1 * torch.randn(w.B, w.Hv, w.dk, w.dv, device=dev)
    ws_b = torch.empty(gdn.backward_workspace_size(w.B, w.T, w.Hqk, w.Hv, w.dk, w.dv), dtype=torch.uint8, device=dev)
    bwd_steps = 3
    ev_b = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(bwd_steps)]   # around its 4 kernels

    def bwd_step(events=None):
        return gdn.gdn_recurrent_bwd(xb["q"], xb["k"], xb["v"], xb["g"], xb["beta"], S0, dout, dSf, workspace=ws_b,
                                     events=None if events is None else [e.cuda_event for e in events])

    for row in ev_b:
        for e in row:
            e.record(stream)
    for _ in range(3):
        bwd_step()
    barrier()
    clocks.active = True
    t0.record(stream)
    for i in range(bwd_steps):
        bwd_step(ev_b[i])
    t1.record(stream)
    barrier()
    clocks.active = False
    bwd_ms = max_ms(t0.elapsed_time(t1)) / bwd_steps
    gdn.check_device_status()
    bwd_flop = 20.0 * tokens * w.Hv * w.dk * w.dv   # one forward (4 dk dv) + the adjoint (16 dk dv) per token/head
    bwd_tf = bwd_flop / (bwd_ms * 1e9)
    alu_peak = 152 * 128 * 2 * 2.07e9 / 1e12      # fp32 FMA lanes x 2 flop x max SM clock
    bwd_kernels = {name: round(statistics.mean(r[i].elapsed_time(r[i + 1]) for r in ev_b), 4)
                   for i, name in enumerate(("bwd_wy", "bwd_state_fwd", "bwd_state_adj", "bwd_local"))}
    del xb, dout, ws_b

    # ---- backward of the layer's other pieces on the same 8k workload: the recurrence's backward through
    #      the fused front end (l2 norm of q, k; gates from raw a, b), the output gate's backward and the
    #      conv's backward over the packed q/k/v projection
    bf = torch.bfloat16
    gen = torch.Generator(device=dev).manual_seed(7)
    xb = device_inputs_random(torch, dev, w, seed=4)
    a_raw = torch.randn(w.B, w.T, w.Hv, device=dev, generator=gen).to(bf)
    b_raw = torch.randn(w.B, w.T, w.Hv, device=dev, generator=gen).to(bf)
    A_log = -0.5 + 0.5 * torch.randn(w.Hv, device=dev, generator=gen)
    dt_bias = 0.5 * torch.randn(w.Hv, device=dev, generator=gen)
    dout = torch.randn(w.B, w.T, w.Hv, w.dv, device=dev, generator=gen).to(bf)
    ws_f = torch.empty(int(gdn.backward_workspace_size(w.B, w.T, w.Hqk, w.Hv, w.dk, w.dv, front_end=True)),
                       dtype=torch.uint8, device=dev)

    def timed(fn, reps, warm=3):
        for _ in range(warm):
            fn()
        barrier()
        t0.record(stream)
        for _ in range(reps):
            fn()
        t1.record(stream)
        barrier()
        return max_ms(t0.elapsed_time(t1)) / reps

    clocks.active = True
    fe_ms = timed(lambda: gdn.gdn_recurrent_bwd(xb["q"], xb["k"], xb["v"], a_raw, b_raw, S0, dout, dSf, workspace=ws_f,
                                                normalize_qk=True, raw_gates=(A_log, dt_bias)), 2)
    del ws_f, xb, a_raw, b_raw
    o_g = torch.randn(w.B, w.T, w.Hv, w.dv, device=dev, generator=gen).to(bf)
    z_g = torch.randn(w.B, w.T, w.Hv, w.dv, device=dev, generator=gen).to(bf)
    nw = 1.0 + 0.1 * torch.randn(w.dv, device=dev, generator=gen)
    gate_bwd_ms = timed(lambda: gdn.gdn_output_gate_bwd(o_g, z_g, nw, dout), 10)
    gate_bwd_bytes = 3 * (w.B * w.T * Cv * 2) + 2 * (w.B * w.T * Cv * 4)   # o, z, dy in; do, dz out (fp32)
    del o_g, z_g
    proj = torch.randn(w.B, w.T, Cc, device=dev, generator=gen).to(bf)
    dy_c = torch.randn(w.B, w.T, Cc, device=dev, generator=gen).to(bf)
    conv_w = 0.5 * torch.randn(Cc, 4, device=dev, generator=gen)
    conv_bwd_ms = timed(lambda: gdn.gdn_causal_conv1d_bwd(proj, conv_w, dy_c, want_grad_cache_in=False), 10)
    slots_c = (w.B * w.T + 63) // 64 + w.B
    conv_bwd_bytes = 2 * (w.B * w.T * Cc * 2) + w.B * w.T * Cc * 4 + 2 * slots_c * Cc * 4 * 4   # x, dy in; dx, dw shares
    clocks.active = False
    gdn.check_device_status()
    del proj, dy_c, dout

    # ---- decode: 512 consecutive steps, state resident, one CUDA graph per pass
    wd = DECODE
    xd = device_inputs_random(torch, dev, wd, steps=wd.T, seed=2)
    S = (0.1 * torch.randn(wd.B, wd.Hv, wd.dk, wd.dv, device=dev))
    outs = torch.empty_like(xd["v"])

    def decode_pass():
        for t in range(wd.T):
            gdn.gdn_recurrent_step(xd["q"][t], xd["k"][t], xd["v"][t], xd["g"][t], xd["beta"][t], S, out=outs[t])

    for t in range(3):   # warm-up steps outside the graph
        gdn.gdn_recurrent_step(xd["q"][t], xd["k"][t], xd["v"][t], xd["g"][t], xd["beta"][t], S, out=outs[t])
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    cap = torch.cuda.Stream(dev)
    cap.wait_stream(stream)
    with torch.cuda.stream(cap):
        with torch.cuda.graph(graph, stream=cap):
            decode_pass()
    stream.wait_stream(cap)
    passes = 3
    graph.replay()   # warm-up pass
    barrier()
    clocks.active = True
    t0.record(stream)
    for _ in range(passes):
        graph.replay()
    t1.record(stream)
    barrier()
    clocks.active = False
    dec_ms = max_ms(t0.elapsed_time(t1)) / (passes * wd.T)
    gdn.check_device_status()
    dec_bytes = decode_bytes(wd)
    dec_gbs = dec_bytes / (dec_ms * 1e6)

    # ---- the recurrent core of a layer in decode, same sequences and heads: per step one conv step of the
    #      packed projection with its K-1 cache (q, k, v written as dense tensors), then the recurrent step
    #      with raw gates, l2 norm and the output gate; 128 steps in one CUDA graph
    dl_steps = 128
    bf = torch.bfloat16
    Cq, Cv = wd.Hqk * wd.dk, wd.Hv * wd.dv
    Cc = 2 * Cq + Cv
    genl = torch.Generator(device=dev).manual_seed(7)
    projd = torch.randn(dl_steps, wd.B, Cc, device=dev, generator=genl).to(bf)
    cwd = 0.5 * torch.randn(Cc, 4, device=dev, generator=genl)
    cached = torch.zeros(wd.B, 3, Cc, dtype=bf, device=dev)
    ad = torch.randn(dl_steps, wd.B, wd.Hv, device=dev, generator=genl).to(bf)
    bd = torch.randn(dl_steps, wd.B, wd.Hv, device=dev, generator=genl).to(bf)
    zd = torch.randn(dl_steps, wd.B, wd.Hv, wd.dv, device=dev, generator=genl).to(bf)
    A_logd = -0.5 + 0.5 * torch.randn(wd.Hv, device=dev, generator=genl)
    dt_biasd = 0.5 * torch.randn(wd.Hv, device=dev, generator=genl)
    nwd = 1.0 + 0.1 * torch.randn(wd.dv, device=dev, generator=genl)
    yq = torch.empty(wd.B, Cq, dtype=bf, device=dev)
    yk, yv = torch.empty_like(yq), torch.empty(wd.B, Cv, dtype=bf, device=dev)
    outd = torch.empty(dl_steps, wd.B, wd.Hv, wd.dv, dtype=bf, device=dev)

    def decode_layer_step(t):
        gdn.gdn_causal_conv1d_step_qkv(projd[t], cwd, cached, (Cq, Cq, Cv), out=(yq, yk, yv))
        gdn.gdn_recurrent_step(yq.view(wd.B, wd.Hqk, wd.dk), yk.view(wd.B, wd.Hqk, wd.dk),
                               yv.view(wd.B, wd.Hv, wd.dv), ad[t], bd[t], S, out=outd[t], scale=wd.dk ** -0.5,
                               normalize_qk=True, raw_gates=(A_logd, dt_biasd), output_gate=(zd[t], nwd, 1e-6))

    for t in range(3):
        decode_layer_step(t)
    torch.cuda.synchronize()
    graph_l = torch.cuda.CUDAGraph()
    cap_l = torch.cuda.Stream(dev)
    cap_l.wait_stream(stream)
    with torch.cuda.stream(cap_l):
        with torch.cuda.graph(graph_l, stream=cap_l):
            for t in range(dl_steps):
                decode_layer_step(t)
    stream.wait_stream(cap_l)
    graph_l.replay()
    barrier()
    clocks.active = True
    t0.record(stream)
    for _ in range(2):
        graph_l.replay()
    t1.record(stream)
    barrier()
    clocks.active = False
    dl_ms = max_ms(t0.elapsed_time(t1)) / (2 * dl_steps)
    gdn.check_device_status()
    # state read + written, projection, conv caches read + written, a, b, z, out
    dl_bytes = (2 * wd.B * wd.Hv * wd.dk * wd.dv * 4 + wd.B * Cc * 2 + 2 * wd.B * 3 * Cc * 2
                + 2 * wd.B * wd.Hv * 2 + 2 * wd.B * wd.Hv * wd.dv * 2)
    del projd, zd, outd

    # ---- the small character-LM workload (4 x 512 tokens, 4 / 4 heads, d = 32, bf16, S0 = 0, S_final
    # returned): a latency-bound call, timed over many back-to-back calls
    wc = gi.WORKLOADS["charlm_bf16"]
    xc = device_inputs_random(torch, dev, wc, seed=5)
    wsc = torch.empty(max(1, gdn.workspace_size(wc.B, wc.T, wc.Hqk, wc.Hv, wc.dk, wc.dv)), dtype=torch.uint8,
                      device=dev)
    outc = torch.empty_like(xc["v"])
    Sfc = torch.empty(wc.B, wc.Hv, wc.dk, wc.dv, device=dev)

    def charlm_call():
        gdn.gdn_chunk_fwd(xc["q"], xc["k"], xc["v"], xc["g"], xc["beta"], None, out=outc, S_final=Sfc,
                          workspace=wsc, chunk=wc.chunk)

    for _ in range(10):
        charlm_call()
    charlm_reps = 200
    barrier()
    t0.record(stream)
    for _ in range(charlm_reps):
        charlm_call()
    t1.record(stream)
    barrier()
    charlm_ms = max_ms(t0.elapsed_time(t1)) / charlm_reps
    gdn.check_device_status()
    clocks.stop()

    if rank != 0:
        return
    value = job_rate(world, tokens, ms_step)
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_step, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "prefill_gqa_8k: chunked prefill, B=2 x T=8192 tokens, Hqk=16 shared by Hv=32, "
                               "dk=dv=128, chunk 64, bf16 operands, fp32 accumulate and state, random S0",
                   "global_batch": w.B * world, "seq_len": w.T,
                   "parallelism": f"replicas x{world} (no cross-GPU exchange)",
                   "l2": "inputs larger than L2 (3 rotating input sets of 275 MB; L2 129 MB), no flush",
                   "inputs": "shared seeded generator (SplitMix64 + Box-Muller), resident in HBM"},
        "roofline": roofline,
        "kernels": {k: {"ms": round(v["ms"], 4), "tflops": round(v["tflops"], 2)} for k, v in kernels.items()},
        "kernels_timing": "CUDA events around each kernel in a second pass of the same steps (an event between "
                          "the kernels launches the chain after the prep instead of overlapping its set-up)",
        "step_tflops": round(whole, 2),
        "e2e": {"value": round(world * tokens / (e2e_ms / 1e3), 1), "unit": "tokens/s",
                "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "ms_per_step": round(e2e_ms, 4),
                "how": "pinned host buffers; per step q, k, v, g, beta, S0 in and out, S_final back; copies of "
                       "neighbouring steps overlap the kernels on separate streams (double-buffered)"},
        "gpu_launches": 2 * args.steps,
        "long_prefill": {"workload": "prefill_varlen_128k: 4 packed sequences 65536/32768/24576/8192, state reset",
                         "value": round(world * wl.T / (long_ms / 1e3), 1), "unit": "tokens/s",
                         "ms_per_step": round(long_ms, 4), "steps": long_steps,
                         "kernels": {"gdn_tc_prep": round(lp, 4), "gdn_tc_chain": round(lc, 4)},
                         "step_tflops": round((lf_prep + lf_chain) / (long_ms * 1e9), 2),
                         "roofline": {"bound": "tensor", "achieved": round((lf_prep + lf_chain) / (long_ms * 1e9), 2),
                                      "peak": peak_tf, "unit": "TFLOP/s",
                                      "frac": round((lf_prep + lf_chain) / (long_ms * 1e9) / peak_tf, 4)}},
        "layer": {"workload": "prefill_gqa_8k through the whole recurrent core: causal conv K=4 of the packed "
                              "q/k/v projection (one launch over its 8192 channels, q, k, v written as dense "
                              "tensors), gates from raw a/b, l2 norm, chunked recurrence, gated RMS norm x silu(z)",
                  "value": round(world * tokens / (layer_ms / 1e3), 1), "unit": "tokens/s",
                  "ms_per_step": round(layer_ms, 4), "steps": layer_steps, "gpu_launches": 4 * layer_steps,
                  "kernels_ms": {"conv_fwd_kernel": round(conv_ms, 4), "output_gate_kernel": round(gate_ms, 4)},
                  "conv_roofline": {"bound": "hbm", "achieved": round(conv_bytes / (conv_ms * 1e6), 1),
                                    "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                    "frac": round(conv_bytes / (conv_ms * 1e6) / peaks["hbm_gbs"], 4),
                                    "algorithmic_bytes": conv_bytes},
                  "gate_roofline": {"bound": "hbm", "achieved": round(gate_bytes / (gate_ms * 1e6), 1),
                                    "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                    "frac": round(gate_bytes / (gate_ms * 1e6) / peaks["hbm_gbs"], 4),
                                    "algorithmic_bytes": gate_bytes}},
        "backward": {"workload": "prefill_gqa_8k backward: gradients w.r.t. q, k, v, g, beta, S0 from dout and "
                                 "dS_final through the chunked form (64-token chunks: WY factors, forward and "
                                 "adjoint chunk chains, chunk-local gradients; fp32 accuracy: the chains on tcgen05 "
                                 "bf16 MMAs with three-part operand splits, the chunk-local kernel on split-tf32 "
                                 "mma.sync)",
                     "value": round(world * tokens / (bwd_ms / 1e3), 1), "unit": "tokens/s",
                     "ms_per_step": round(bwd_ms, 4), "steps": bwd_steps, "gpu_launches": 4 * bwd_steps,
                     "kernels_ms": bwd_kernels,
                     "roofline": {"bound": "tensor", "achieved": round(bwd_tf, 2),
                                  "peak": round(peaks["bf16_tflops"] / 3, 1), "unit": "TFLOP/s",
                                  "frac": round(bwd_tf / (peaks["bf16_tflops"] / 3), 4),
                                  "peak_source": "measured bf16 burst / 3: an fp32-accurate product from bf16 tensor "
                                                 "MMAs takes three part products when one operand is an exact bf16 "
                                                 "input (six when neither is)"},
                     "roofline_alu": {"bound": "alu", "achieved": round(bwd_tf, 2), "peak": round(alu_peak, 1),
                                      "unit": "TFLOP/s", "frac": round(bwd_tf / alu_peak, 4),
                                      "peak_source": "fp32 FMA lanes x 2 x 2070 MHz (unit counts)"}},
        "layer_backward": {"workload": "prefill_gqa_8k backward through the layer's other pieces: the recurrence's "
                                       "backward with the fused front end (l2 norm of q, k and gates from raw a, b: every "
                                       "kernel on the raw bf16 rows with in-kernel l2 scalars and gates, the chain rule "
                                       "back), the output gate's backward (bf16 in, fp32 gradients) and the causal conv's "
                                       "backward over the packed 8192-channel q/k/v projection (K=4)",
                           "front_end_backward_ms": round(fe_ms, 4),
                           "front_end_backward_tokens_per_s": round(world * tokens / (fe_ms / 1e3), 1),
                           "output_gate_backward": {"ms": round(gate_bwd_ms, 4), "roofline": {
                               "bound": "hbm", "achieved": round(gate_bwd_bytes / (gate_bwd_ms * 1e6), 1),
                               "peak": peaks["hbm_gbs"], "unit": "GB/s",
                               "frac": round(gate_bwd_bytes / (gate_bwd_ms * 1e6) / peaks["hbm_gbs"], 4),
                               "algorithmic_bytes": gate_bwd_bytes}},
                           "conv_backward": {"ms": round(conv_bwd_ms, 4), "roofline": {
                               "bound": "hbm", "achieved": round(conv_bwd_bytes / (conv_bwd_ms * 1e6), 1),
                               "peak": peaks["hbm_gbs"], "unit": "GB/s",
                               "frac": round(conv_bwd_bytes / (conv_bwd_ms * 1e6) / peaks["hbm_gbs"], 4),
                               "algorithmic_bytes": conv_bwd_bytes}}},
        "decode": {"workload": "decode_256x512: 256 sequences x 32 V heads (16 QK heads), d=128, 512 steps, "
                               "fp32 state 512 MiB resident, one CUDA graph per 512-step pass",
                   "value": round(world / (dec_ms / 1e3), 1), "unit": "steps/s",
                   "tokens_per_s": round(world * wd.B / (dec_ms / 1e3), 1), "us_per_step": round(dec_ms * 1e3, 2),
                   "gpu_launches": passes * wd.T,
                   "roofline": {"bound": "hbm", "kernel": "decode_step_kernel", "achieved": round(dec_gbs, 1),
                                "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": round(dec_gbs / peaks["hbm_gbs"], 4),
                                "traffic": traffic_for("decode_step_kernel"),
                                "algorithmic_bytes": dec_bytes, "peak_source": f"{peak_src} copy bandwidth"}},
        "charlm": {"workload": "charlm_bf16: B=4 x T=512 tokens, 4 / 4 heads, dk=dv=32, bf16, S0 = 0, final state "
                               "returned (chunked kernels on split-tf32 MMAs: d = 32 is off the tcgen05 tile)",
                   "value": round(world * wc.B * wc.T / (charlm_ms / 1e3), 1), "unit": "tokens/s",
                   "us_per_call": round(charlm_ms * 1e3, 2), "calls": charlm_reps, "bound": "latency"},
        "decode_layer": {"workload": "decode_256x512 heads through the layer's recurrent core: one conv step (K=4) "
                                     "of the packed 8192-channel projection with its cache (q, k, v written as dense "
                                     "tensors), then the recurrent step with raw gates, l2 norm and the output gate; "
                                     "128 steps per CUDA graph",
                         "value": round(world / (dl_ms / 1e3), 1), "unit": "steps/s",
                         "tokens_per_s": round(world * wd.B / (dl_ms / 1e3), 1), "us_per_step": round(dl_ms * 1e3, 2),
                         "gpu_launches": 2 * dl_steps * 2,
                         "roofline": {"bound": "hbm", "achieved": round(dl_bytes / (dl_ms * 1e6), 1),
                                      "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                      "frac": round(dl_bytes / (dl_ms * 1e6) / peaks["hbm_gbs"], 4),
                                      "algorithmic_bytes": dl_bytes}},
        "clocks": clocks.summary(),
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(budget_s=args.cpu_seconds)
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


# ---------------------------------------------------------------- CPU oracle (baseline / reference arm)
_ORACLE_INPUTS = {}


def oracle_rate(tokens_per_seq, threads=0):
    """Time the fp64 oracle on the first `tokens_per_seq` tokens of both sequences of the 8k GQA
    workload, all 32 value heads.  Returns (workload tokens per second, seconds, cores)."""
    from oracle import recurrence as orc
    if tokens_per_seq not in _ORACLE_INPUTS:
        _ORACLE_INPUTS.clear()
        _ORACLE_INPUTS[tokens_per_seq] = gi.make_prefill_inputs(gi.scaled(PREFILL, T=tokens_per_seq))
    w = gi.scaled(PREFILL, T=tokens_per_seq)
    x = _ORACLE_INPUTS[tokens_per_seq]
    t = time.perf_counter()
    orc.forward(x["q"], x["k"], x["v"], x["g"], x["beta"], S0=x["S0"], threads=threads)
    dt = time.perf_counter() - t
    return w.B * tokens_per_seq / dt, dt, orc.max_threads() if threads <= 0 else threads


def small_config_rates():
    """The oracle on the two small workloads (tiny_f32, charlm_bf16), on one core and on all cores:
    tokens/s of the whole workload, best of three runs."""
    from oracle import recurrence as orc
    res = {}
    for name in ("tiny_f32", "charlm_bf16"):
        w = gi.WORKLOADS[name]
        x = gi.make_prefill_inputs(w)
        for threads in (1, 0):
            best = None
            for _ in range(3):
                t = time.perf_counter()
                orc.forward(x["q"], x["k"], x["v"], x["g"], x["beta"], S0=x["S0"], threads=threads)
                dt = time.perf_counter() - t
                best = dt if best is None else min(best, dt)
            key = "1_core" if threads == 1 else f"{orc.max_threads()}_cores"
            res.setdefault(name, {})[key] = round(w.B * w.T / best, 1)
    return res


def cpu_baseline(budget_s=15.0):
    rate, dt, cores = oracle_rate(128)                      # calibration
    n = int(max(128, min(PREFILL.T, rate * budget_s / PREFILL.B)))
    # when the whole workload takes less than the budget, repeat it (at most 15 runs) and report the
    # aggregate rate over all runs
    runs, total = 0, 0.0
    while runs < 15 and (runs == 0 or total < budget_s):
        _, dt, cores = oracle_rate(n)
        runs, total = runs + 1, total + dt
    rate = runs * PREFILL.B * n / total
    what = "the whole workload" if n == PREFILL.T else f"the first {n} tokens of both sequences"
    return {"value": round(rate, 1), "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"{what} of prefill_gqa_8k, all 32 value heads, fp64 token loop, {runs} run(s) in "
                      f"{total:.1f} s",
            "small_workloads_tokens_per_s": small_config_rates()}


def run_reference(args):
    rank, world, _ = rank_info()
    if rank != 0:
        return
    rate, dt, cores = oracle_rate(128)
    per_step_s = max(0.2, 90.0 / max(1, args.steps + args.warmup))
    n = int(max(64, min(PREFILL.T, rate * per_step_s / PREFILL.B)))
    for _ in range(args.warmup):
        oracle_rate(n)
    times = []
    for _ in range(args.steps):
        r, dt, cores = oracle_rate(n)
        times.append(dt)
    ms = 1e3 * sum(times) / len(times)
    value = PREFILL.B * n / (ms / 1e3)
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "prefill_gqa_8k: chunked prefill, B=2 x T=8192 tokens, Hqk=16 shared by Hv=32, "
                               "dk=dv=128, chunk 64, bf16 operands, fp32 accumulate and state, random S0",
                   "global_batch": PREFILL.B, "seq_len": PREFILL.T, "parallelism": "host cores (OpenMP)"},
        "cpu_baseline": {"value": round(value, 1), "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"each step: first {n} tokens of both sequences, all 32 value heads, fp64 token loop"},
        "e2e": {"value": round(value, 1), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_profile_case(case):
    """One warm-up and one measured call of a single kernel family, for ncu captures."""
    import torch
    import gated_deltanet_recurrence_03_gb300 as gdn
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    if case == "prefill":
        w = PREFILL
        x = device_inputs_random(torch, dev, w)
        S0 = 0.1 * torch.randn(w.B, w.Hv, w.dk, w.dv, device=dev)
        ws = torch.empty(gdn.workspace_size(w.B, w.T, w.Hqk, w.Hv, w.dk, w.dv), dtype=torch.uint8, device=dev)
        for _ in range(2):
            gdn.gdn_chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], S0, workspace=ws)
    elif case == "backward":
        # the backward pass of the 8k GQA workload (about 2.6 GB of device memory with its workspace), twice
        w = PREFILL
        x = device_inputs_random(torch, dev, w)
        S0 = 0.1 * torch.randn(w.B, w.Hv, w.dk, w.dv, device=dev)
        dout = torch.randn_like(x["v"])
        dSf = 0.1 * torch.randn_like(S0)
        ws = torch.empty(gdn.backward_workspace_size(w.B, w.T, w.Hqk, w.Hv, w.dk, w.dv), dtype=torch.uint8, device=dev)
        for _ in range(2):
            gdn.gdn_recurrent_bwd(x["q"], x["k"], x["v"], x["g"], x["beta"], S0, dout, dSf, workspace=ws)
    elif case == "layer":
        # the conv of the packed q/k/v projection (one launch) and the prefill with the fused front end
        # and the output gate, twice
        w = PREFILL
        x = device_inputs_random(torch, dev, w)
        Cq, Cv = w.Hqk * w.dk, w.Hv * w.dv
        proj = torch.randn(w.B, w.T, 2 * Cq + Cv, device=dev).to(torch.bfloat16)
        cw = 0.5 * torch.randn(2 * Cq + Cv, 4, device=dev)
        S0 = 0.1 * torch.randn(w.B, w.Hv, w.dk, w.dv, device=dev)
        ws = torch.empty(gdn.workspace_size(w.B, w.T, w.Hqk, w.Hv, w.dk, w.dv), dtype=torch.uint8, device=dev)
        z = torch.randn_like(x["v"])
        A_log, dt_bias = -0.5 + 0.5 * torch.randn(w.Hv, device=dev), 0.5 * torch.randn(w.Hv, device=dev)
        nw = 1.0 + 0.1 * torch.randn(w.dv, device=dev)
        for _ in range(2):
            gdn.gdn_causal_conv1d_fwd_qkv(proj, cw, (Cq, Cq, Cv), None, return_cache=False,
                                          out=(x["q"].view(w.B, w.T, Cq), x["k"].view(w.B, w.T, Cq),
                                               x["v"].view(w.B, w.T, Cv)))
            gdn.gdn_chunk_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], S0, workspace=ws, normalize_qk=True,
                              raw_gates=(A_log, dt_bias), output_gate=(z, nw, 1e-6))
    else:
        w = DECODE
        x = device_inputs_random(torch, dev, w, steps=2, seed=2)
        S = 0.1 * torch.randn(w.B, w.Hv, w.dk, w.dv, device=dev)
        for t in range(2):
            gdn.gdn_recurrent_step(x["q"][t], x["k"][t], x["v"][t], x["g"][t], x["beta"][t], S)
    torch.cuda.synchronize()
    gdn.check_device_status()
    print(f"profile case {case} done")


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["gdn", "reference"], default="gdn")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--profile-case", choices=["prefill", "decode", "layer", "backward"], default=None,
                    help="run one warm-up and one measured call of one kernel family (for ncu) and exit")
    args = ap.parse_args(argv)
    if not args.profile_case and args.warmup < 3:
        ap.error("--warmup must be at least 3")
    return args


def main():
    args = parse_args()
    if args.profile_case:
        run_profile_case(args.profile_case)
        return
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
