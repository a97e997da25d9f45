#!/usr/bin/env python3
"""Benchmark of the selective-scan hot path on B300.

One step = one pass of the whole hot path over one batch of synthetic input:
the selective scan of a layer (chunk load, discretisation, in-register
recurrence, split-sequence carry when planned, fused epilogue) returning
last_state, followed by one decode step on that state for the next token.

Default workload: the long-sequence scan, B1 D5120 N16 L32768 bf16 (the
largest single-GPU configuration; it takes the split-sequence carry). The
Mamba-1.4B- and 130M-shaped layers (B16 D4096 and B8 D1536, N16 L2048 bf16) are
timed as well and reported under "layers". Other workloads (--workload
m1p4b|m130|tiny) can be made the headline for exploration.

Prints ONE JSON line on rank 0. ``--impl reference`` times the fp64 CPU oracle
instead (bounded samples of the same workload on the host cores).
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from selective_state_space_125_b300.workloads import (SCAN_CONFIGS, bf16_bits,  # noqa: E402
                                                      make_config_inputs, make_decode_inputs)

METRIC = "selective-scan channel-steps/s"
L2_BYTES = 126 * 2**20
FP32_LANES_PER_SM = 128          # FP32 lanes per SM (B300): one FMUL/FADD/FFMA lane-op each per clock
# FP32 lane-ops per (channel, step, state) that the bf16 scan needs: dt*A,
# the input product, the two FMAs of the state update and the two of the
# readout (C / A times the scaled state, accumulated); exp runs on MUFU.
ALG_OPS_PER_STATE_STEP = 6
# FP32 lane-ops per (channel, step, state) that the backward needs given the
# forward states: one forward update to recompute h (4: dt*A, B*u, the add and
# the FMA of the scaled update) and the adjoint step (16: lambda, h_t and its
# dC product, dt*A, (abar-1)/A (2), B*u, A h_{t-1} + B u, abar*lambda, the dt
# term and its sum, the two dA_log FMAs, lambda*q, its dB and du products).
ALG_BWD_OPS_PER_STATE_STEP = 20
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "scan_traffic.json")


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default="long", choices=sorted(SCAN_CONFIGS))
    p.add_argument("--seqlen", type=int, default=0,
                   help="override the workload's sequence length (smaller profiling cases of the same kernel)")
    p.add_argument("--no-layers", action="store_true", help="skip timing the extra layer workloads")
    p.add_argument("--layers", default="m1p4b,m130", help="extra scan workloads timed beside the headline")
    p.add_argument("--seed", type=int, default=0)
    p.add_argument("--e2e-steps", type=int, default=100)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-seconds", type=float, default=12.0, help="budget of the CPU baseline sample")
    p.add_argument("--cpu-threads", type=int, default=0, help="--impl reference: host threads (0: all cores)")
    p.add_argument("--lanes", type=int, default=0, help="plan override: lanes per channel")
    p.add_argument("--segments", type=int, default=0, help="plan override: time segments")
    p.add_argument("--no-decode", action="store_true", help="skip the full-size decode measurement")
    p.add_argument("--no-variants", action="store_true", help="skip the simplified-discretisation scan timing")
    p.add_argument("--no-bwd", action="store_true", help="skip the backward-scan timing")
    p.add_argument("--decode-only", action="store_true",
                   help="time only the decode step on the full decode workloads and print their JSON")
    p.add_argument("--decode-workload", default="both", choices=["both", "decode", "decode128"])
    p.add_argument("--decode-calls", type=int, default=200)
    return p.parse_args()


def read_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return dict(hbm_gbs=d.get("hbm_gbs", 6400.0), sm_max_mhz=d.get("sm_max_mhz", 2032.0), source="measured")
    return dict(hbm_gbs=6400.0, sm_max_mhz=2032.0, source="fallback")


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()

    def summary(self, t0, t1):
        rows = []
        for ts, line in self.lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            rows.append((ts, parts))
        inside = [r for ts, r in rows if t0 <= ts <= t1]
        use = inside if inside else [r for ts, r in rows][-3:]
        if not use:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        sm = [float(r[1]) for r in use if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in use if r[2].replace(".", "").isdigit()]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in use:
            for name, val in zip(names, r[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(inside)}


SCAN_KERNEL_SOURCES = ("device_common.cuh", "scan_args.h", "scan_kernel.cuh", "scan_bf16.cu", "scan_f32.cu")


def decode_names(args):
    return ("decode", "decode128") if args.decode_workload == "both" else (args.decode_workload,)


def max_over_ranks(x: float, world: int, device) -> float:
    """The slowest rank's figure: every rank's timed region ends at a barrier,
    so the job's step time is the max over ranks."""
    if world <= 1:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_rate(units_per_rank: float, world: int, ms_per_step: float) -> float:
    """Units all ranks processed per second (weak scaling: every rank runs the same workload)."""
    return world * units_per_rank / (ms_per_step / 1e3)


def kernel_source_sha():
    """Hash of the scan kernel's sources, so that stored ncu figures are used only for the kernel they measured."""
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "selective_state_space_125_b300", "csrc")
    for name in SCAN_KERNEL_SOURCES:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def stored_traffic(workload, chosen):
    """DRAM bytes per scan call from the committed ncu summary of this workload,
    if it was taken on the same plan and the current kernel sources."""
    if workload is None or not os.path.exists(TRAFFIC_FILE):
        return None, "no ncu summary for this workload and plan"
    with open(TRAFFIC_FILE) as f:
        tr = json.load(f).get(workload)
    if not tr or getattr(chosen, "time_lanes", 0) > 1:
        return None, "no ncu summary for this workload and plan"
    if tr.get("plan") == [chosen.lanes_per_channel, chosen.segments] and \
            tr.get("kernel_source_sha") == kernel_source_sha():
        return tr.get("dram_bytes_per_call"), tr.get("source")
    return None, "ncu summary is for another plan or an older kernel"


def measure_decode(device, stream, peaks, calls=200, which=("decode", "decode128")):
    """Decode step on the full decode workloads (B128 D5120, N = 16 and 128): us per call and GB/s.

    Each call reads and writes the resident fp32 state and reads one token's
    bf16 activations; 16 distinct tokens are cycled. Calls rotate over enough
    independent state buffers (one per layer of a model, say) that together
    exceed three times L2, so every call streams its state from HBM."""
    import torch
    from selective_state_space_125_b300 import binding
    from selective_state_space_125_b300.workloads import DECODE_CONFIGS, make_decode_config_inputs
    out = {}
    for name in which:
        cfg = DECODE_CONFIGS[name]
        inp = make_decode_config_inputs(cfg, seed=0)
        B, Dm, N = cfg.batch, cfg.dim, cfg.dstate
        bf = lambda a: torch.from_numpy(bf16_bits(a).view(np.int16)).to(device).view(torch.bfloat16)
        f32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(device)
        state0 = f32(inp["state0"])
        nbuf = max(1, int(np.ceil(3 * L2_BYTES / (state0.numel() * 4))))
        states = [state0] + [state0.clone() for _ in range(nbuf - 1)]
        toks = [{k: bf(inp[k][p]) for k in ("u", "delta", "z", "B", "C")} for p in range(cfg.pool)]
        A_log, Dv, bias = f32(inp["A_log"]), f32(inp["D"]), f32(inp["delta_bias"])
        y = torch.empty((B, Dm), dtype=torch.bfloat16, device=device)

        # Raw C-ABI calls with the pointers marshalled once: a call then costs the host
        # about a microsecond, well under the kernel's time, so launches stay queued.
        lib = binding.library()
        sh = stream.cuda_stream
        argv = [[(B, Dm, N, binding.MAMBA_BF16, st.data_ptr(), t["u"].data_ptr(), t["delta"].data_ptr(),
                  A_log.data_ptr(), t["B"].data_ptr(), t["C"].data_ptr(), Dv.data_ptr(), t["z"].data_ptr(),
                  bias.data_ptr(), y.data_ptr(), sh) for t in toks] for st in states]
        binding.mamba_selective_state_update(state0, toks[0]["u"], toks[0]["delta"], A_log, toks[0]["B"],
                                             toks[0]["C"], Dv, toks[0]["z"], bias, y)  # checked once

        def call(i):
            if lib.mamba_selective_state_update(*argv[i % nbuf][(i // nbuf) % cfg.pool]) != 0:
                raise RuntimeError("decode step failed")
        for i in range(10):
            call(i)
        torch.cuda.synchronize(device)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(calls):
            call(i)
        e1.record(stream)
        torch.cuda.synchronize(device)
        us = e0.elapsed_time(e1) / calls * 1e3
        alg = B * Dm * N * 4 * 2 + 4 * B * Dm * 2 + 2 * B * N * 2 + Dm * N * 4 + 2 * Dm * 4
        gbs = alg / (us * 1e-6) / 1e9
        out[name] = {"workload": cfg.description, "us_per_call": us, "channel_steps_per_s": B * Dm / (us * 1e-6),
                     "bytes_per_call": alg, "GB/s": gbs, "hbm_frac": gbs / peaks["hbm_gbs"], "calls": calls,
                     "state_buffers": nbuf}
        del states, state0, toks
        torch.cuda.empty_cache()
    return out


def scan_figures(cfg, ms, sms, peaks):
    """Algorithmic bytes and FP32 lane-ops of one scan call of ``cfg`` and the
    rates ``ms`` per call gives, against the HBM and FP32 peaks."""
    B, Dm, N, L = cfg.batch, cfg.dim, cfg.dstate, cfg.seqlen
    es = 2 if cfg.dtype == "bf16" else 4
    alg_bytes = (4 * es * B * L * Dm + 2 * N * es * B * L + Dm * N * 4 + 2 * Dm * 4
                 + (B * Dm * N * 4 if cfg.last_state else 0))
    alg_ops = ALG_OPS_PER_STATE_STEP * N * B * L * Dm
    peak_tops = FP32_LANES_PER_SM * sms * peaks["sm_max_mhz"] * 1e6 / 1e12
    tops = alg_ops / (ms / 1e3) / 1e12
    gbs = alg_bytes / (ms / 1e3) / 1e9
    return dict(alg_bytes=alg_bytes, alg_ops=alg_ops, peak_tops=peak_tops, tops=tops, gbs=gbs,
                alu_frac=tops / peak_tops, hbm_frac=gbs / peaks["hbm_gbs"])


def measure_layer(name, device, stream, peaks, sms, calls=50, seed=0, time_lanes=0):
    """The scan alone on another workload (inputs resident, last_state
    returned): CUDA events around ``calls`` graph-replayed calls that rotate
    over input sets larger than L2 together. ``time_lanes`` > 1 times the
    time-parallel chunk scan in place of the automatic plan."""
    import torch
    from selective_state_space_125_b300 import binding
    cfg = SCAN_CONFIGS[name]
    B, Dm, N, L = cfg.batch, cfg.dim, cfg.dstate, cfg.seqlen
    inp = make_config_inputs(cfg, seed=seed)
    dev_x = lambda a: torch.from_numpy(bf16_bits(a).view(np.int16)).to(device).view(torch.bfloat16)
    f32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(device)
    base = {k: dev_x(inp[k]) for k in ("u", "delta", "z", "B", "C")}
    A_log, Dv, bias = f32(inp["A_log"]), f32(inp["D"]), f32(inp["delta_bias"])
    del inp
    set_bytes = sum(t.numel() * t.element_size() for t in base.values()) + B * L * Dm * 2
    nsets = max(2, int(np.ceil(3 * L2_BYTES / set_bytes)) + 1)
    sets = []
    for i in range(nsets):
        st = {k: (v if i == 0 else v.clone()) for k, v in base.items()}
        st["out"] = torch.empty((B, L, Dm), dtype=torch.bfloat16, device=device)
        st["last"] = torch.empty((B, Dm, N), dtype=torch.float32, device=device)
        sets.append(st)
    plan = binding.ScanPlan(0, 0, 0, 0, time_lanes) if time_lanes > 1 else None
    chosen, launches = binding.mamba_selective_scan_plan(B, Dm, N, L, cfg.dtype, plan)

    def scan(st):
        binding.mamba_selective_scan_fwd(st["u"], st["delta"], A_log, st["B"], st["C"], Dv, st["z"], bias,
                                         st["out"], st["last"], plan=plan)
    for i in range(3):
        scan(sets[i % nsets])
    torch.cuda.synchronize(device)
    graphs = []
    for st in sets:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            scan(st)
        graphs.append(g)
    for i in range(nsets):
        graphs[i].replay()
    torch.cuda.synchronize(device)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(calls):
        graphs[i % nsets].replay()
    e1.record(stream)
    torch.cuda.synchronize(device)
    assert binding.mamba_device_status() == 0, "a kernel reported a timeout"
    ms = e0.elapsed_time(e1) / calls
    f = scan_figures(cfg, ms, sms, peaks)
    traffic, traffic_note = stored_traffic(name, chosen)
    del sets, graphs, base
    torch.cuda.empty_cache()
    return {"workload": cfg.description, "kernel_ms": ms, "channel_steps_per_s": B * Dm * L / (ms / 1e3),
            "hbm": {"achieved": f["gbs"], "unit": "GB/s", "frac": f["hbm_frac"], "bytes_per_call": f["alg_bytes"],
                    "traffic": traffic, "traffic_source": traffic_note},
            "alu": {"achieved": f["tops"], "unit": "T FP32 lane-op/s", "frac": f["alu_frac"],
                    "ops_per_call": f["alg_ops"]},
            "plan": {"lanes_per_channel": chosen.lanes_per_channel, "segments": chosen.segments,
                     "time_lanes": chosen.time_lanes, "launches": launches},
            "calls": calls, "l2": f"{nsets} rotating input sets of {set_bytes / 2**20:.0f} MiB"}


def measure_bwd_layer(name, device, stream, peaks, sms, calls=20, seed=0):
    """The backward scan on a layer workload (random dout; the call's memsets
    included): ms per call, against the FP32 peak at the backward's lane-op count."""
    import torch
    from selective_state_space_125_b300 import binding
    cfg = SCAN_CONFIGS[name]
    B, Dm, N, L = cfg.batch, cfg.dim, cfg.dstate, cfg.seqlen
    inp = make_config_inputs(cfg, seed=seed)
    dev_x = lambda a: torch.from_numpy(bf16_bits(a).view(np.int16)).to(device).view(torch.bfloat16)
    f32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(device)
    t = {k: dev_x(inp[k]) for k in ("u", "delta", "z", "B", "C")}
    A_log, Dv, bias = f32(inp["A_log"]), f32(inp["D"]), f32(inp["delta_bias"])
    del inp
    dout = torch.randn((B, L, Dm), device=device, generator=torch.Generator(device).manual_seed(11)).to(torch.bfloat16)

    def call():
        return binding.mamba_selective_scan_bwd(t["u"], t["delta"], A_log, t["B"], t["C"], dout, D=Dv, z=t["z"],
                                                delta_bias=bias)
    for _ in range(3):
        call()
    torch.cuda.synchronize(device)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(calls):
        call()
    e1.record(stream)
    torch.cuda.synchronize(device)
    assert binding.mamba_device_status() == 0, "a kernel reported a timeout"
    ms = e0.elapsed_time(e1) / calls
    ops = ALG_BWD_OPS_PER_STATE_STEP * N * B * L * Dm
    peak = FP32_LANES_PER_SM * sms * peaks["sm_max_mhz"] * 1e6 / 1e12
    del t, dout
    torch.cuda.empty_cache()
    return {"workload": cfg.description + ", backward", "ms_per_call": ms,
            "channel_steps_per_s": B * L * Dm / (ms / 1e3), "achieved": ops / (ms / 1e3) / 1e12,
            "unit": "T FP32 lane-op/s", "frac": ops / (ms / 1e3) / 1e12 / peak, "calls": calls}


# ------------------------------------------------------------- our arm
def workload_config(args):
    """The headline workload, with its sequence length overridden by --seqlen."""
    import dataclasses
    cfg = SCAN_CONFIGS[args.workload]
    if args.seqlen > 0:
        cfg = dataclasses.replace(cfg, seqlen=args.seqlen,
                                  description=f"{cfg.description} with L = {args.seqlen}")
    return cfg


def run_ours(args, rank, world, device):
    import torch
    from selective_state_space_125_b300 import binding

    cfg = workload_config(args)
    B, Dm, N, L = cfg.batch, cfg.dim, cfg.dstate, cfg.seqlen
    tdt = torch.bfloat16 if cfg.dtype == "bf16" else torch.float32
    es = 2 if cfg.dtype == "bf16" else 4
    inp = make_config_inputs(cfg, seed=args.seed + rank)
    tok = make_decode_inputs(B, Dm, N, cfg.dtype, seed=args.seed + 1000 + rank, pool=1)

    def dev_x(a):
        if cfg.dtype == "bf16":
            return torch.from_numpy(bf16_bits(a).view(np.int16)).to(device).view(torch.bfloat16)
        return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(device)

    f32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(device)
    base = {k: dev_x(inp[k]) for k in ("u", "delta", "z", "B", "C")}
    A_log, Dv, bias = f32(inp["A_log"]), f32(inp["D"]), f32(inp["delta_bias"])
    base_tok = {k: dev_x(tok[k][0]) for k in ("u", "delta", "z", "B", "C")}
    set_bytes = sum(t.numel() * t.element_size() for t in base.values()) + B * L * Dm * es
    nsets = max(2, int(np.ceil(3 * L2_BYTES / set_bytes)) + 1)
    sets = []
    for i in range(nsets):
        s = {k: (v if i == 0 else v.clone()) for k, v in base.items()}
        s["out"] = torch.empty((B, L, Dm), dtype=tdt, device=device)
        s["last"] = torch.empty((B, Dm, N), dtype=torch.float32, device=device)
        s["tok"] = {k: (v if i == 0 else v.clone()) for k, v in base_tok.items()}
        s["tok_out"] = torch.empty((B, Dm), dtype=tdt, device=device)
        sets.append(s)
    plan = None
    if args.lanes or args.segments:
        plan = binding.ScanPlan(args.lanes, args.segments, 0)
    chosen, scan_launches = binding.mamba_selective_scan_plan(B, Dm, N, L, cfg.dtype, plan)
    stream = torch.cuda.current_stream(device)

    def scan(s):
        binding.mamba_selective_scan_fwd(s["u"], s["delta"], A_log, s["B"], s["C"], Dv, s["z"], bias,
                                         s["out"], s["last"], plan=plan)

    def decode(s):
        t = s["tok"]
        binding.mamba_selective_state_update(s["last"], t["u"], t["delta"], A_log, t["B"], t["C"], Dv, t["z"],
                                             bias, s["tok_out"])

    for i in range(args.warmup):
        scan(sets[i % nsets])
        decode(sets[i % nsets])
    torch.cuda.synchronize(device)

    # One CUDA graph per input set holds a whole step (scan + decode step): the
    # timed region replays them, so the host's per-call marshalling is not on
    # the device's critical path. A second set of graphs holds the scan alone,
    # for the scan kernel's own time.
    step_graphs, scan_graphs = [], []
    for s in sets:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            scan(s)
            decode(s)
        step_graphs.append(g)
        g2 = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g2):
            scan(s)
        scan_graphs.append(g2)
    for i in range(max(3, nsets)):
        step_graphs[i % nsets].replay()
    torch.cuda.synchronize(device)

    K = args.steps
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(device.index if device.index is not None else 0)
    sampler.start()
    time.sleep(0.3)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(device)
    t_wall0 = time.time()
    ev0.record(stream)
    for i in range(K):
        step_graphs[i % nsets].replay()
    ev1.record(stream)
    torch.cuda.synchronize(device)
    t_wall1 = time.time()
    if world > 1:
        torch.distributed.barrier()
    # the scan kernel alone, back to back, for the roofline's per-launch time
    Ks = max(20, min(K, 500))
    es0, es1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    es0.record(stream)
    for i in range(Ks):
        scan_graphs[i % nsets].replay()
    es1.record(stream)
    torch.cuda.synchronize(device)
    time.sleep(0.2)
    sampler.stop()
    assert binding.mamba_device_status() == 0, "a kernel reported a timeout"
    ms_total = ev0.elapsed_time(ev1)
    scan_ms = [es0.elapsed_time(es1) / Ks]
    ms_per_step = max_over_ranks(ms_total / K, world, device)
    chsteps = B * Dm * (L + 1)
    value = job_rate(chsteps, world, ms_per_step)

    # ---- e2e through the public API with pinned host buffers. Every step copies its
    # inputs host -> device, runs the scan and the decode step, and copies the outputs
    # back. The three stages run on their own streams over the rotating input sets, so
    # step i's compute overlaps step i+1's upload and step i-1's download.
    pin = {k: v.cpu().pin_memory() for k, v in base.items()}
    pin_tok = {k: v.cpu().pin_memory() for k, v in base_tok.items()}
    host_out = [torch.empty((B, L, Dm), dtype=tdt).pin_memory() for _ in range(nsets)]
    host_tok_out = [torch.empty((B, Dm), dtype=tdt).pin_memory() for _ in range(nsets)]
    h2d = sum(v.numel() * v.element_size() for v in pin.values()) + sum(
        v.numel() * v.element_size() for v in pin_tok.values())
    d2h = host_out[0].numel() * host_out[0].element_size() + host_tok_out[0].numel() * host_tok_out[0].element_size()
    Ke = max(1, min(args.e2e_steps, K))
    up, down = torch.cuda.Stream(device), torch.cuda.Stream(device)
    inputs_ready = [torch.cuda.Event() for _ in range(nsets)]
    computed = [torch.cuda.Event() for _ in range(nsets)]
    downloaded = [torch.cuda.Event() for _ in range(nsets)]
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(device)
    e0.record(up)
    for i in range(Ke):
        j = i % nsets
        s = sets[j]
        with torch.cuda.stream(up):
            if i >= nsets:
                up.wait_event(computed[j])  # the set's inputs were consumed
            for k in pin:
                s[k].copy_(pin[k], non_blocking=True)
            for k in pin_tok:
                s["tok"][k].copy_(pin_tok[k], non_blocking=True)
            inputs_ready[j].record(up)
        stream.wait_event(inputs_ready[j])
        if i >= nsets:
            stream.wait_event(downloaded[j])  # the set's outputs were read back
        scan(s)
        decode(s)
        computed[j].record(stream)
        with torch.cuda.stream(down):
            down.wait_event(computed[j])
            host_out[j].copy_(s["out"], non_blocking=True)
            host_tok_out[j].copy_(s["tok_out"], non_blocking=True)
            downloaded[j].record(down)
    down.wait_event(computed[(Ke - 1) % nsets])
    e1.record(down)
    torch.cuda.synchronize(device)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / Ke, world, device)

    peaks = read_peaks()
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    scan_avg_ms = float(np.mean(scan_ms))
    fig = scan_figures(cfg, scan_avg_ms, sms, peaks)
    alg_bytes, alg_ops, peak_tops = fig["alg_bytes"], fig["alg_ops"], fig["peak_tops"]
    achieved_tops, achieved_gbs = fig["tops"], fig["gbs"]
    clocks = sampler.summary(t_wall0, t_wall1)
    traffic, traffic_note = stored_traffic(args.workload if args.seqlen == 0 else None, chosen)
    decode = None if args.no_decode else measure_decode(device, stream, peaks, args.decode_calls, decode_names(args))
    # The same scan with the simplified discretisation (Bbar = dt B): 4 FP32 lane-ops per state.
    simple = None
    if not args.no_variants:
        v0, v1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        nv = 50
        splan = binding.ScanPlan(chosen.lanes_per_channel, chosen.segments, 0, binding.MAMBA_SIMPLIFIED)
        for i in range(3):
            s = sets[i % nsets]
            binding.mamba_selective_scan_fwd(s["u"], s["delta"], A_log, s["B"], s["C"], Dv, s["z"], bias,
                                             s["out"], s["last"], plan=splan)
        torch.cuda.synchronize(device)
        v0.record(stream)
        for i in range(nv):
            s = sets[i % nsets]
            binding.mamba_selective_scan_fwd(s["u"], s["delta"], A_log, s["B"], s["C"], Dv, s["z"], bias,
                                             s["out"], s["last"], plan=splan)
        v1.record(stream)
        torch.cuda.synchronize(device)
        sms_ = v0.elapsed_time(v1) / nv
        sops = 4 * N * B * L * Dm
        # The scan with the causal conv1d (width 4) + SiLU fused in front of it, on the same inputs.
        cw = torch.randn((Dm, 4), device=device, generator=torch.Generator(device).manual_seed(7)) * 0.5
        cbias = torch.zeros((Dm,), device=device)
        cplan = binding.ScanPlan(chosen.lanes_per_channel, chosen.segments, 0, 0)
        for i in range(3):
            s = sets[i % nsets]
            binding.mamba_conv1d_selective_scan_fwd(s["u"], cw, cbias, s["delta"], A_log, s["B"], s["C"], Dv,
                                                    s["z"], bias, s["out"], s["last"], plan=cplan)
        torch.cuda.synchronize(device)
        v0.record(stream)
        for i in range(nv):
            s = sets[i % nsets]
            binding.mamba_conv1d_selective_scan_fwd(s["u"], cw, cbias, s["delta"], A_log, s["B"], s["C"], Dv,
                                                    s["z"], bias, s["out"], s["last"], plan=cplan)
        v1.record(stream)
        torch.cuda.synchronize(device)
        cms = v0.elapsed_time(v1) / nv
        conv = {"step": "causal conv1d (width 4) + SiLU fused in front of the scan", "kernel_ms": cms,
                "achieved": alg_ops / (cms / 1e3) / 1e12, "unit": "T FP32 lane-op/s",
                "frac": alg_ops / (cms / 1e3) / 1e12 / peak_tops, "calls": nv,
                "hbm_frac": alg_bytes / (cms / 1e3) / 1e9 / peaks["hbm_gbs"]}
        simple = {"discretization": "simplified (Bbar = dt B)", "kernel_ms": sms_,
                  "achieved": sops / (sms_ / 1e3) / 1e12, "unit": "T FP32 lane-op/s",
                  "frac": sops / (sms_ / 1e3) / 1e12 / peak_tops, "ops_per_launch": sops,
                  "hbm_frac": alg_bytes / (sms_ / 1e3) / 1e9 / peaks["hbm_gbs"], "calls": nv}
    # The backward scan on the same inputs: gradients of every input for a random dout.
    bwd = None
    if not args.no_bwd:
        gen = torch.Generator(device).manual_seed(11)
        douts = [torch.randn((B, L, Dm), device=device, generator=gen).to(tdt) for _ in range(nsets)]

        def bwd_call(i):
            s = sets[i % nsets]
            return binding.mamba_selective_scan_bwd(s["u"], s["delta"], A_log, s["B"], s["C"], douts[i % nsets],
                                                    D=Dv, z=s["z"], delta_bias=bias)
        for i in range(3):
            bwd_call(i)
        torch.cuda.synchronize(device)
        nb = 20
        b0, b1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        b0.record(stream)
        for i in range(nb):
            bwd_call(i)
        b1.record(stream)
        torch.cuda.synchronize(device)
        bms = b0.elapsed_time(b1) / nb
        bops = ALG_BWD_OPS_PER_STATE_STEP * N * B * L * Dm
        bbytes = (7 * es * B * L * Dm + 2 * N * es * B * L + 2 * N * 4 * B * L + 2 * Dm * N * 4 + 4 * Dm * 4)
        bwd = {"step": "backward scan: du, ddelta, dz, dA_log, dB, dC, dD, ddelta_bias for a random dout "
                       "(5 memsets + 1 kernel launch per call)",
               "ms_per_call": bms, "channel_steps_per_s": B * L * Dm / (bms / 1e3),
               "achieved": bops / (bms / 1e3) / 1e12, "unit": "T FP32 lane-op/s",
               "frac": bops / (bms / 1e3) / 1e12 / peak_tops, "ops_per_call": bops,
               "hbm_bytes_per_call": bbytes, "hbm_frac": bbytes / (bms / 1e3) / 1e9 / peaks["hbm_gbs"],
               "calls": nb}
        del douts
    result = {
        "metric": METRIC, "value": value, "unit": "channel-steps/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic (seeded numpy draws of the workload's shapes and distributions)",
        "config": {"workload": cfg.description, "batch": B, "d_inner": Dm, "d_state": N, "seqlen": L,
                   "input_dtype": cfg.dtype, "state_dtype": "f32",
                   "step": "scan(L tokens, last_state) + 1 decode step", "channel_steps_per_step": chsteps,
                   "l2": f"{nsets} rotating input/output sets of {set_bytes / 2**20:.0f} MiB (> L2)",
                   "plan": {"lanes_per_channel": chosen.lanes_per_channel, "segments": chosen.segments,
                            "tma": chosen.use_tma == 1}},
        "roofline": {"bound": "alu", "achieved": achieved_tops, "peak": peak_tops, "unit": "T FP32 lane-op/s",
                     "frac": achieved_tops / peak_tops, "traffic": traffic, "traffic_source": traffic_note,
                     "kernel": f"selective scan call ({scan_launches} launch(es))", "kernel_ms": scan_avg_ms,
                     "ops_per_launch": alg_ops,
                     "peak_basis": f"{FP32_LANES_PER_SM} FP32 lanes x {sms} SMs x {peaks['sm_max_mhz']:.0f} MHz "
                                   "(recipe unit counts and maximum SM clock)"},
        "hbm": {"achieved": achieved_gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved_gbs / peaks["hbm_gbs"], "bytes_per_launch": alg_bytes,
                "peak_source": f"MEASURED_PEAKS.json ({peaks['source']})"},
        "e2e": {"value": job_rate(chsteps, world, e2e_ms), "unit": "channel-steps/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": Ke,
                "pipelining": "upload, compute and download on three streams over the rotating input sets"},
        "gpu_launches": K * (scan_launches + 1),
        "timing": "CUDA-graph replay of the step (scan + decode) per input set; scan kernel time from a graph "
                  "of back-to-back scans",
        "clocks": clocks,
    }
    if decode is not None:
        result["decode"] = decode
    if simple is not None:
        result["scan_simplified"] = simple
        result["scan_conv1d_fused"] = conv
    if bwd is not None:
        result["scan_bwd"] = bwd
    if not args.no_layers:
        del sets
        torch.cuda.empty_cache()
        result["layers"] = {name: measure_layer(name, device, stream, peaks, sms)
                            for name in args.layers.split(",") if name and name != args.workload}
        # The time-parallel chunk scan (plan knob time_lanes) on the 130M-shaped
        # layer, whose 12,288 channels leave the sequential plan short of warps.
        for tl in (2, 4):
            result["layers"][f"m130_time_lanes_{tl}"] = measure_layer("m130", device, stream, peaks, sms,
                                                                     time_lanes=tl)
        result["layers"]["m130_bwd"] = measure_bwd_layer("m130", device, stream, peaks, sms)
    return result


# ------------------------------------------------- CPU oracle (baseline)
def oracle_sample_rate(cfg, inp, seconds, threads):
    """Oracle scan over the first k channels (all steps) of batch row 0, sized to ~seconds."""
    import oracle
    L, Dm = cfg.seqlen, cfg.dim

    def run(k):
        sl = slice(0, k)
        t0 = time.perf_counter()
        oracle.selective_scan(inp["u"][:1, :, sl], inp["delta"][:1, :, sl], inp["A_log"][sl], inp["B"][:1],
                              inp["C"][:1], inp["D"][sl], inp["z"][:1, :, sl], inp["delta_bias"][sl],
                              nthreads=threads)
        return time.perf_counter() - t0

    k = max(1, min(Dm, threads))
    dt = run(k)
    while dt < 0.5 and k < Dm:
        k = min(Dm, k * 4)
        dt = run(k)
    per_ch = dt / k
    k_final = max(1, min(Dm, int(seconds / per_ch)))
    total, reps = 0.0, 0
    while total < seconds:  # whole calls until the time budget is spent
        total += run(k_final)
        reps += 1
    rate = reps * k_final * L / total
    return rate, f"oracle scan of {k_final} channels x {L} steps (batch row 0) x {reps}, {total:.1f} s"


def cpu_baseline(args, cfg):
    """The fp64 oracle on all host cores (the value) and on one core, each on a
    bounded sample of the workload."""
    threads = os.cpu_count() or 1
    inp = make_config_inputs(cfg, seed=args.seed)
    rate, sample = oracle_sample_rate(cfg, inp, args.cpu_seconds, threads)
    rate1, sample1 = oracle_sample_rate(cfg, inp, args.cpu_seconds / 2, 1)
    return {"value": rate, "unit": "channel-steps/s", "cores": threads, "kind": "oracle", "sample": sample,
            "single_core": {"value": rate1, "unit": "channel-steps/s", "cores": 1, "sample": sample1}}


def run_reference(args, rank, world):
    """--impl reference: the fp64 oracle on host cores, K timed steps of bounded samples."""
    import oracle
    cfg = workload_config(args)
    threads = args.cpu_threads if args.cpu_threads > 0 else (os.cpu_count() or 1)
    inp = make_config_inputs(cfg, seed=args.seed)
    L, Dm = cfg.seqlen, cfg.dim
    budget = min(args.cpu_seconds, 120.0 / max(1, args.steps + args.warmup))   # seconds per step
    rate, _ = oracle_sample_rate(cfg, inp, min(2.0, budget), threads)
    k = max(1, min(Dm, int(budget * rate / L)))
    sl = slice(0, k)

    def step():
        oracle.selective_scan(inp["u"][:1, :, sl], inp["delta"][:1, :, sl], inp["A_log"][sl], inp["B"][:1],
                              inp["C"][:1], inp["D"][sl], inp["z"][:1, :, sl], inp["delta_bias"][sl],
                              nthreads=threads)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = (time.perf_counter() - t0) / args.steps
    value = k * L / dt
    sample = f"oracle scan of {k} channels x {L} steps (batch row 0 of the {cfg.name} workload) per step"
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "channel-steps/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded numpy)",
        "config": {"workload": cfg.description, "sample": sample},
        "cpu_baseline": {"value": value, "unit": "channel-steps/s", "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "channel-steps/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args, rank, world)), flush=True)
        return
    import torch
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=device)
    from selective_state_space_125_b300 import build
    if rank == 0 or world == 1:
        build.build()
    if world > 1:
        torch.distributed.barrier()
    if args.decode_only:
        out = measure_decode(device, torch.cuda.current_stream(device), read_peaks(), args.decode_calls,
                             decode_names(args))
        if rank == 0:
            print(json.dumps({"decode": out}), flush=True)
        return
    result = run_ours(args, rank, world, device)
    if rank == 0:
        if not args.no_cpu_baseline and world == 1:
            result["cpu_baseline"] = cpu_baseline(args, workload_config(args))
        print(json.dumps(result), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
