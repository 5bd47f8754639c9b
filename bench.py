#!/usr/bin/env python3
"""Benchmark of the gated linear-recurrence scans on one node.

One step = one pass of the whole hot path over one batch of synthetic input:
the RG-LRU scan at B=8, L=4096, D=2560 (bf16 I/O), the selective SSM scan at
B=4, L=16384, d_inner=4096, N=16 (bf16 I/O) and the HGRN2 recurrence at
B=4, L=4096, 16 heads x 128 (bf16 I/O).  The metric is
token-channel steps per second over the step (B*L*channels summed over the
scans, HGRN2 counting its output channels), with per-scan GB/s, % of the
measured HBM peak and, for HGRN2, TFLOP/s and tensor utilisation.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

With N > 1 the script runs under torch.distributed.run, one rank per GPU;
every rank runs the same per-rank workload (independent replicas, weak
scaling) and rank 0 prints one JSON line with the whole-job throughput
(the units all ranks processed over the slowest rank's time).

``--impl reference`` times the float64 CPU oracle (the correctness
reference, never tuned) on the host cores on a bounded sample of the same
workload and prints the same JSON line with "impl": "reference".
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from selective_state_space_chunked_gb300 import workloads as wl  # noqa: E402

METRIC = "scan tok·ch/s"
UNIT = "tok·ch/s"


# ----------------------------------------------------------------------------
# workload bookkeeping (algorithmic bytes / flops per launch)
# ----------------------------------------------------------------------------
def algorithmic(cfg: wl.Config) -> dict:
    """Bytes a launch must move (inputs read once, outputs written once) and
    the tensor-core flops of HGRN2's chunked form."""
    es = 2 if cfg.io == "bf16" else 4
    B, L, D = cfg.B, cfg.L, cfg.D
    if cfg.form == "rglru":
        by = 4 * es * B * L * D + 4 * D + (2 * 4 * B * D if cfg.with_h0 else 4 * B * D)
        return {"bytes": by, "flops": 0, "units": B * L * D}
    if cfg.form == "selective":
        N = cfg.N
        by = (4 * es * B * L * D + 2 * es * B * L * N + 4 * D * N + 4 * D
              + (2 if cfg.with_h0 else 1) * 4 * B * D * N)
        return {"bytes": by, "flops": 0, "units": B * L * D}
    d = cfg.head_dim
    by = 5 * es * B * L * cfg.H * d + 4 * B * cfg.H * d * d
    # per token and head: QK^T and P V over the chunk (2*C*d each), Q S^T and
    # the state update (2*d*d each)
    fl = B * L * cfg.H * (4 * cfg.chunk * d + 4 * d * d)
    return {"bytes": by, "flops": fl, "units": B * L * cfg.H * d}


# The scans one step runs (the workloads the pages' layers are sized for).
STEP_WORKLOADS = ("rglru_bf16", "selective_bf16", "hgrn2_bf16")


def step_configs(only=None, seq_len=None, io=None):
    """The step's workloads; ``only`` keeps one form, ``seq_len`` shortens
    the sequences and ``io`` changes the I/O dtype (profiling cases: a launch
    of a kernel on another input, never a benchmark number)."""
    import dataclasses
    cfgs = [wl.WORKLOADS[k] for k in STEP_WORKLOADS]
    if only:
        cfgs = [c for c in cfgs if c.form == only]
    if seq_len:
        cfgs = [dataclasses.replace(c, L=seq_len) for c in cfgs]
    if io:
        cfgs = [dataclasses.replace(c, io=io) for c in cfgs]
    return cfgs


# ALU roofline of the selective scan.  Every (token, channel, state) element
# costs one exp2 on the MUFU pipe (the discretised decay) and four fp32 ops on
# the FMA pipe (the decay argument, the input product, the state FMA, the
# readout FMA).  At 128 fp32 lanes and 32 exp2 results per clock per SM the
# two pipes cap the update at min(128/4, 32/1) = 32 elements per clock per SM.
# The powers form of the decays (A_log on the multi-scale lattice) moves most
# exp2s off the MUFU pipe but keeps four fp32 ops per element (a power-chain
# multiply replaces the decay argument), so the same 32 per clock bound it.
# The SM count is the device's; the clock is the maximum SM clock that
# nvidia-smi reports during the timed region (2070 MHz on a GB300 when no
# record could be taken).
ALU_ELEMS_PER_CLK_SM = 32
FALLBACK_MAX_MHZ = 2070


def alu_peak(sms: int, max_mhz) -> tuple:
    mhz = float(max_mhz) if max_mhz else float(FALLBACK_MAX_MHZ)
    src = (f"derived: {sms} SMs (device attribute) x {mhz:.0f} MHz "
           f"({'nvidia-smi clocks.max.sm' if max_mhz else 'GB300 maximum, no clock record'}) "
           f"x {ALU_ELEMS_PER_CLK_SM} state updates/clk/SM")
    return sms * mhz * 1e6 * ALU_ELEMS_PER_CLK_SM / 1e9, src


def kernel_roofline(cfg: wl.Config, a: dict, ms: float, peaks: dict, alu=None) -> dict:
    """Roofline entry of one scan's kernel for one launch of ``ms``: HBM
    bandwidth of its algorithmic bytes against the measured copy peak, and
    for the selective scan also its state updates against the ALU peak
    ``alu`` = (Gelem/s, how it was derived), the bound it really meets."""
    sec = ms * 1e-3
    gbs = a["bytes"] / sec / 1e9
    e = {"kernel": cfg.name, "bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"],
         "unit": "GB/s", "frac": gbs / peaks["hbm_gbs"], "traffic": traffic_for(cfg),
         "peak_source": peaks["source"] + " (MEASURED_PEAKS.json hbm_gbs)"}
    if cfg.form == "selective" and alu is not None:
        ach = a["units"] * cfg.N / sec / 1e9
        e["alu"] = {"bound": "alu", "achieved": ach, "peak": alu[0], "unit": "Gelem/s",
                    "frac": ach / alu[0], "peak_source": alu[1]}
        e["limited_by"] = "alu (issue-bound state updates; HBM is not the binding limit)"
        e["decay_form"] = ("powers: the workload's A_log is on the multi-scale lattice, "
                           "checked per warp in the kernel")
    if cfg.form == "hgrn2" and a["flops"]:
        tf = a["flops"] / sec / 1e12
        e["tensor"] = {"bound": "tensor", "achieved": tf, "peak": peaks["bf16_tflops_sustained"],
                       "unit": "TFLOP/s", "frac": tf / peaks["bf16_tflops_sustained"],
                       "peak_source": peaks["source"] + " (bf16_tflops_sustained)"}
    return e


# ----------------------------------------------------------------------------
# clocks sampling (nvidia-smi during the timed region)
# ----------------------------------------------------------------------------
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (FileNotFoundError, OSError):
            self.proc = None
        time.sleep(0.3)

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for r in rows for k in range(4) if r[5 + k] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


# ----------------------------------------------------------------------------
# distributed helpers
# ----------------------------------------------------------------------------
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world: int, backend: str):
    if world > 1 and not torch.distributed.is_initialized():
        torch.distributed.init_process_group(backend=backend)


def barrier(world: int):
    if world > 1:
        torch.distributed.barrier()


def job_throughput(world: int, units_per_rank_step: int, steps: int, max_ms: float) -> float:
    """Whole-job rate: the units every rank processed over the slowest rank's
    time (each rank runs the same per-rank workload: weak scaling)."""
    return world * units_per_rank_step * steps / (max_ms * 1e-3)


def max_over_ranks(v: float, world: int, device) -> float:
    if world == 1:
        return v
    t = torch.tensor([v], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------
# CPU oracle baseline (bounded samples of the same workloads)
# ----------------------------------------------------------------------------
def oracle_sample(cfg: wl.Config):
    """A bounded slice of a workload for the CPU oracle: whole sequences of a
    subset of channels (RG-LRU, selective) or heads (HGRN2) of batch row 0."""
    if cfg.form == "rglru":
        p = wl.make_inputs(cfg, B=1)
        ch = 1024
        return ("rglru", dict(x=p["x"][:, :, :ch], r=p["r"][:, :, :ch], i=p["i"][:, :, :ch],
                              a_log=p["a_log"][:ch], c=p["c"],
                              h0=None if p["h0"] is None else p["h0"][:, :ch]),
                cfg.L * ch)
    if cfg.form == "selective":
        p = wl.make_inputs(cfg, B=1)
        ch = 256
        return ("selective", dict(x=p["x"][:, :, :ch], dt=p["dt"][:, :, :ch],
                                  z=p["z"][:, :, :ch], Bm=p["Bm"], Cm=p["Cm"],
                                  A_log=p["A_log"][:ch], Dskip=p["Dskip"][:ch],
                                  h0=None if p["h0"] is None else p["h0"][:, :ch]),
                cfg.L * ch)
    p = wl.make_inputs(cfg, B=1)
    heads = cfg.H
    hd = cfg.head_dim
    sl = slice(0, heads * hd)
    return ("hgrn2", dict(q=p["q"][:, :, sl], k=p["k"][:, :, sl], v=p["v"][:, :, sl],
                          g=p["g"][:, :, sl], H=heads), cfg.L * heads * hd)


def run_oracle(kind, args, threads=0):
    import oracle
    if kind == "rglru":
        return oracle.rglru_scan(**args, threads=threads)
    if kind == "selective":
        return oracle.selective_scan(**args, threads=threads)
    return oracle.hgrn2(**args, threads=threads)


def cpu_baseline(cfgs, repeats=1, samples=None, single_thread=False) -> dict:
    """Times the oracle on each workload's sample; the step-equivalent rate is
    total units / sum over scans of (units / sampled rate)."""
    import oracle
    cores = oracle.max_threads()
    if samples is None:
        samples = [(cfg, *oracle_sample(cfg)) for cfg in cfgs]
    rates = {}
    sample_s = 0.0
    for cfg, kind, args, units in samples:
        run_oracle(kind, args)  # warm (page-in, thread pool)
        t0 = time.perf_counter()
        for _ in range(repeats):
            run_oracle(kind, args)
        dt = (time.perf_counter() - t0) / repeats
        rates[cfg.name] = units / dt
        sample_s += dt
    total_units = sum(algorithmic(c)["units"] for c in cfgs)
    step_time = sum(algorithmic(c)["units"] / rates[c.name] for c in cfgs)
    desc = "; ".join(f"{c.name}: {u} of {algorithmic(c)['units']} units"
                     for c, _, _, u in samples)
    out = {"value": total_units / step_time, "unit": UNIT, "cores": cores, "kind": "oracle",
           "sample": "whole sequences of a channel/head subset of batch row 0 -- " + desc,
           "per_scan_units_per_s": rates, "sample_ms": sample_s * 1e3}
    if single_thread:
        # the same samples on one host thread (one timed run each)
        rates1 = {}
        for cfg, kind, args, units in samples:
            t0 = time.perf_counter()
            run_oracle(kind, args, threads=1)
            rates1[cfg.name] = units / (time.perf_counter() - t0)
        out["single_thread"] = {
            "value": total_units / sum(algorithmic(c)["units"] / rates1[c.name] for c in cfgs),
            "unit": UNIT, "cores": 1, "per_scan_units_per_s": rates1}
    return out


# ----------------------------------------------------------------------------
# GPU arm
# ----------------------------------------------------------------------------
def make_call(lr, cfg, p, out=None, ws=None, sync_host=True):
    """One call of a workload's scan through the public torch API; ``ws``: the
    workspace tensor it keeps using (its first bytes hold each call's device
    status); ``sync_host=False``: a host-buffer call returns once queued."""
    if cfg.form == "rglru":
        return lambda: lr.rglru_scan(p["x"], p["r"], p["i"], p["a_log"], p["c"], h0=p["h0"],
                                     out=out, workspace=ws, sync_host=sync_host)
    if cfg.form == "selective":
        return lambda: lr.selective_scan(p["x"], p["dt"], p["Bm"], p["Cm"], p["A_log"],
                                         z=p["z"], Dskip=p["Dskip"], h0=p["h0"], out=out,
                                         workspace=ws, sync_host=sync_host)
    return lambda: lr.hgrn2(p["q"], p["k"], p["v"], p["g"], H=p["H"], out=out, workspace=ws,
                            sync_host=sync_host)


def host_workspace_for(lr, cfg, dev):
    """The device staging workspace of one workload's host-buffer call."""
    io = lr.LR_BF16 if cfg.io == "bf16" else lr.LR_F32
    if cfg.form == "rglru":
        n = lr.lr_rglru_scan_fwd_host_workspace_size(cfg.B, cfg.L, cfg.D, io)
    elif cfg.form == "selective":
        n = lr.lr_selective_scan_fwd_host_workspace_size(cfg.B, cfg.L, cfg.D, cfg.N, io)
    else:
        n = lr.lr_hgrn2_fwd_host_workspace_size(cfg.B, cfg.L, cfg.H, cfg.head_dim, cfg.head_dim, io)
    return torch.empty(max(int(n), 256), dtype=torch.uint8, device=dev)


def workspace_for(lr, cfg, dev):
    """The device workspace of one workload's device call."""
    io = lr.LR_BF16 if cfg.io == "bf16" else lr.LR_F32
    if cfg.form == "rglru":
        n = lr.lr_rglru_scan_workspace_size(cfg.B, cfg.L, cfg.D, io)
    elif cfg.form == "selective":
        n = lr.lr_selective_scan_workspace_size(cfg.B, cfg.L, cfg.D, cfg.N, io)
    else:
        n = lr.lr_hgrn2_workspace_size(cfg.B, cfg.L, cfg.H, cfg.head_dim, cfg.head_dim, io)
    return torch.empty(max(int(n), 256), dtype=torch.uint8, device=dev)


def check_calls(lr, wss, stream, when):
    """Raises if any workload's latest call recorded a device-side error."""
    for ws in wss:
        code = lr.status(ws, stream)
        if code != 0:
            raise RuntimeError(f"device status {lr.lr_status_string(code)} {when}")


def decode_timings(lr, cfgs, dev, steps: int = 20, reps: int = 20) -> list:
    """Single-token decode: `steps` in-place steps of each form at the
    workload's batch and width, captured in one CUDA graph and replayed;
    per-step device time and the bytes a step must move (state read and
    written, inputs read, output written)."""
    res = []
    for cfg in cfgs:
        p = wl.make_inputs(cfg, device=dev, L=1)
        es = 2 if cfg.io == "bf16" else 4
        if cfg.form == "rglru":
            h = torch.zeros(cfg.B, cfg.D, device=dev)
            args = [p[n][:, 0].contiguous() for n in ("x", "r", "i")]
            fn = lambda: lr.rglru_scan_step(*args, p["a_log"], p["c"], h=h, h_out=h)
            by = 8 * cfg.B * cfg.D + 4 * es * cfg.B * cfg.D + 4 * cfg.D
        elif cfg.form == "selective":
            h = torch.zeros(cfg.B, cfg.D, cfg.N, device=dev)
            args = [p[n][:, 0].contiguous() for n in ("x", "dt", "Bm", "Cm")]
            zt = p["z"][:, 0].contiguous()
            fn = lambda: lr.selective_scan_step(*args, p["A_log"], z=zt, Dskip=p["Dskip"], h=h, h_out=h)
            by = (8 * cfg.B * cfg.D * cfg.N + 4 * es * cfg.B * cfg.D + 2 * es * cfg.B * cfg.N
                  + 4 * cfg.D * (cfg.N + 1))
        else:
            d = cfg.head_dim
            h = torch.zeros(cfg.B, cfg.H, d, d, device=dev)
            args = [p[n][:, 0].contiguous() for n in ("q", "k", "v", "g")]
            fn = lambda: lr.hgrn2_step(*args, cfg.H, S=h, S_out=h)
            by = 8 * cfg.B * cfg.H * d * d + 5 * es * cfg.B * cfg.H * d
        fn()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        st = torch.cuda.Stream(dev)
        with torch.cuda.stream(st):
            fn()
            st.synchronize()
            with torch.cuda.graph(g, stream=st):
                for _ in range(steps):
                    fn()
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            g.replay()
        e1.record()
        torch.cuda.synchronize()
        us = e0.elapsed_time(e1) * 1e3 / (reps * steps)
        res.append({"workload": f"{cfg.form} step B={cfg.B}" +
                    (f" H={cfg.H} d={cfg.head_dim}" if cfg.form == "hgrn2" else f" D={cfg.D}"),
                    "us_per_step": us, "bytes_per_step": by, "gb_per_s": by / (us * 1e-6) / 1e9})
    return res


def off_lattice_A_log(A_log: torch.Tensor) -> torch.Tensor:
    """A_log moved off the multi-scale initialisation lattice (seeded noise of
    0.05), as training moves it: the selective kernel then takes its general
    one-exp-per-state decays."""
    g = torch.Generator(device=A_log.device).manual_seed(12)
    return A_log + 0.05 * torch.randn(A_log.shape, device=A_log.device, generator=g)


def extra_timings(lr, dev, peaks, alu, reps: int = 20) -> list:
    """Scans outside the step, timed the same way (CUDA events on the
    launching stream, median of ``reps`` launches): the two oracle-sized
    workloads (fp32 RG-LRU B2 L128 D64 and fp32 selective B2 L1024 D1536,
    whose inputs fit in L2: timed with the 129 MB L2 flushed before every
    launch, and the selective one also hot, launched back to back), the
    selective workload with general (off-lattice) decays, the MinMax
    recurrence at the RG-LRU workload's shape, the pre-activation gate forms
    and fp32 HGRN2 (inputs larger than L2)."""
    flush_buf = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def timed(fn, flush=False):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(reps)]
        for a, b in ev:
            if flush:
                flush_buf.zero_()   # evicts the previous launch's lines from L2
            a.record()
            fn()
            b.record()
        torch.cuda.synchronize()
        return statistics.median(a.elapsed_time(b) for a, b in ev)

    def entry(name, ms, units, by, l2=None):
        gbs = by / (ms * 1e-3) / 1e9
        d = {"workload": name, "ms": ms, "tok_ch_per_s": units / (ms * 1e-3), "gb_per_s": gbs,
             "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                          "frac": gbs / peaks["hbm_gbs"], "peak_source": peaks["source"]}}
        if l2:
            d["l2"] = l2
        return d

    res = []
    # the two small workloads (their inputs fit in L2)
    for key in ("rglru_f32_small", "selective_f32"):
        cfg = wl.WORKLOADS[key]
        p = wl.make_inputs(cfg, device=dev)
        ws = workspace_for(lr, cfg, dev)
        fn = make_call(lr, cfg, p, ws=ws)
        a = algorithmic(cfg)
        modes = (("flushed", True), ("hot", False)) if cfg.form == "selective" else (("flushed", True),)
        for mode, fl in modes:
            ms = timed(fn, flush=fl)
            e = entry(f"{cfg.name} ({mode} L2)", ms, a["units"], a["bytes"],
                      l2="129 MB L2 flushed before every launch" if fl else
                      "hot: inputs resident in L2 (launched back to back, no flush)")
            if cfg.form == "selective":
                e["roofline"] = kernel_roofline(cfg, a, ms, peaks, alu)
                e["roofline"]["traffic"] = None
            res.append(e)
        check_calls(lr, [ws], torch.cuda.current_stream(dev), f"in the {cfg.name} timing")
        del p, ws, fn
    del flush_buf
    # the selective workload with A_log moved off the initialisation lattice
    # (as training moves it): the general one-exp-per-state decays
    cfg = wl.WORKLOADS["selective_bf16"]
    p = wl.make_inputs(cfg, device=dev)
    A_off = off_lattice_A_log(p["A_log"])
    ms = timed(lambda: lr.selective_scan(p["x"], p["dt"], p["Bm"], p["Cm"], A_off, z=p["z"],
                                         Dskip=p["Dskip"], h0=p["h0"]))
    rl = kernel_roofline(cfg, algorithmic(cfg), ms, peaks, alu)
    rl["decay_form"] = "general: one exp2 per state (A_log off the lattice)"
    rl["traffic"] = None
    res.append({"workload": cfg.name + " A_log off the lattice", "ms": ms,
                "tok_ch_per_s": cfg.B * cfg.L * cfg.D / (ms * 1e-3),
                "gb_per_s": algorithmic(cfg)["bytes"] / (ms * 1e-3) / 1e9, "roofline": rl})
    del p, A_off
    B, L, D = 8, 4096, 2560
    g = torch.Generator(device=dev).manual_seed(11)
    r = torch.randn(B, L, D, device=dev, generator=g).to(torch.bfloat16)
    s_ = (torch.randn(B, L, D, device=dev, generator=g) - 1.0).to(torch.bfloat16)
    x0 = torch.randn(B, D, device=dev, generator=g)
    res.append(entry(f"minmax_bf16_B{B}_L{L}_D{D}", timed(lambda: lr.minmax_scan(r, s_, x0)),
                     B * L * D, 3 * 2 * B * L * D + 2 * 4 * B * D))
    del r, s_
    # the RG-LRU and HGRN2 workloads with their gates before the activation
    # (sigmoid / lower-bounded sigmoid applied in the kernel)
    cfg = wl.WORKLOADS["rglru_bf16"]
    p = wl.make_inputs(cfg, device=dev)
    res.append(entry(cfg.name + " gates_preact", timed(lambda: lr.rglru_scan(
        p["x"], p["r"], p["i"], p["a_log"], p["c"], h0=p["h0"], gates_preact=True)),
        cfg.B * cfg.L * cfg.D, algorithmic(cfg)["bytes"]))
    del p
    cfg = wl.WORKLOADS["hgrn2_bf16"]
    p = wl.make_inputs(cfg, device=dev)
    res.append(entry(cfg.name + " gate_lb=0.2", timed(lambda: lr.hgrn2(
        p["q"], p["k"], p["v"], p["g"], H=p["H"], gate_lb=0.2)),
        algorithmic(cfg)["units"], algorithmic(cfg)["bytes"]))
    # fp32 I/O at the same shape: the split-bf16 tensor-core kernel
    pf = {n: p[n].float() for n in ("q", "k", "v", "g")}
    del p
    res.append(entry(f"hgrn2_f32_B{cfg.B}_L{cfg.L}_H{cfg.H}_d{cfg.head_dim} split-bf16 tensor-core kernel",
                     timed(lambda: lr.hgrn2(pf["q"], pf["k"], pf["v"], pf["g"], H=cfg.H)),
                     algorithmic(cfg)["units"], 2 * algorithmic(cfg)["bytes"]))
    return res


def launches_per_call(cfg: wl.Config) -> int:
    """Kernels one call of a workload's scan launches (the library's rules):
    the RG-LRU scan one; the selective scan two with warm-ups (the default for
    bf16 outputs: the stealing launch and the launch for deferred shares), one
    without; HGRN2 with 128 x 128 heads two (the tensor-core pass and the pass
    that re-runs marked heads: a redo pass of the same kernel for bf16, the
    step-by-step kernel for fp32), other head dims one.  The ncu launch list
    in profiles/ confirms the count for the step."""
    if cfg.form == "rglru":
        return 1
    if cfg.form == "selective":
        return 2 if cfg.io == "bf16" else 1
    return 2 if cfg.head_dim == 128 else 1


def input_bytes(p) -> int:
    return sum(t.numel() * t.element_size() for t in p.values() if torch.is_tensor(t))


def gpu_arm(args):
    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    init_dist(world, "nccl")
    from selective_state_space_chunked_gb300 import binding as lr
    cfgs = step_configs(args.only, args.seq_len, args.io)
    inputs = [wl.make_inputs(c, device=dev) for c in cfgs]
    if args.a_log_off_lattice:
        for c, p in zip(cfgs, inputs):
            if c.form == "selective":
                p["A_log"] = off_lattice_A_log(p["A_log"])
    wss = [workspace_for(lr, c, dev) for c in cfgs]
    calls = [make_call(lr, c, p, ws=w) for c, p, w in zip(cfgs, inputs, wss)]
    alg = [algorithmic(c) for c in cfgs]
    stream = torch.cuda.current_stream(dev)

    for _ in range(args.warmup):
        for fn in calls:
            fn()
    torch.cuda.synchronize()
    check_calls(lr, wss, stream, "during warm-up")

    clocks = ClockSampler(local)
    if rank == 0:
        clocks.start()
    ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in cfgs] for _ in range(args.steps)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    t_start.record(stream)
    for k in range(args.steps):
        for j, fn in enumerate(calls):
            ev[k][j][0].record(stream)
            fn()
            ev[k][j][1].record(stream)
    t_end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop() if rank == 0 else None
    total_ms = t_start.elapsed_time(t_end)
    total_ms = max_over_ranks(total_ms, world, dev)
    check_calls(lr, wss, stream, "in the timed region")

    per_scan = []
    for j, c in enumerate(cfgs):
        ms = statistics.mean(ev[k][j][0].elapsed_time(ev[k][j][1]) for k in range(args.steps))
        a = alg[j]
        d = {"workload": c.name, "ms": ms, "tok_ch_per_s": a["units"] / (ms * 1e-3),
             "gb_per_s": a["bytes"] / (ms * 1e-3) / 1e9}
        if a["flops"]:
            d["tflop_per_s"] = a["flops"] / (ms * 1e-3) / 1e12
        per_scan.append(d)

    # end-to-end through the public API with host buffers: pinned host inputs,
    # the library copies them in, runs, copies outputs back and synchronises
    host_inputs = [{k: (v.cpu().pin_memory() if torch.is_tensor(v) else v) for k, v in p.items()}
                   for p in inputs]
    # the caller's result buffers: pinned host tensors, allocated once; each
    # scan has its own staging workspace, so its queued calls can overlap
    host_outs = [make_call(lr, c, p)() for c, p in zip(cfgs, host_inputs)]
    host_wss = [host_workspace_for(lr, c, dev) for c in cfgs]
    host_calls = [make_call(lr, c, p, out=o, ws=w, sync_host=False)
                  for c, p, o, w in zip(cfgs, host_inputs, host_outs, host_wss)]
    h2d = sum(input_bytes(p) for p in host_inputs)
    for _ in range(max(1, args.warmup)):   # the same W warm-up steps as the device leg
        for fn in host_calls:
            fn()
        lr.host_sync()
    torch.cuda.synchronize()
    # every step queues the three scans' host-buffer calls (each returns once
    # its work is queued, so one call's inputs go in while the previous one's
    # last chunks run) and returns when lr.host_sync() has every output in the
    # caller's host buffers; timed over up to 50 steps, per-step times kept
    e2e_steps = max(3, min(args.steps, 50))
    barrier(world)
    d2h = 0
    e2e_ms = []
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        ts = time.perf_counter()
        d2h = 0
        for fn in host_calls:
            outs = fn()
            d2h += sum(t.numel() * t.element_size() for t in outs)
        lr.host_sync()
        e2e_ms.append((time.perf_counter() - ts) * 1e3)
    torch.cuda.synchronize()
    e2e_s = max_over_ranks(time.perf_counter() - t0, world, dev) / e2e_steps
    check_calls(lr, host_wss, stream, "in the end-to-end leg")
    del host_inputs, host_calls, host_outs, host_wss

    units_step = sum(a["units"] for a in alg)
    value = job_throughput(world, units_step, args.steps, total_ms)
    peaks = load_peaks()
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    alu = alu_peak(sms, clk.get("sm_max_mhz") if clk else None)
    dom = max(range(len(cfgs)), key=lambda j: per_scan[j]["ms"])
    rooflines = [kernel_roofline(c, a, d["ms"], peaks, alu) for c, a, d in zip(cfgs, alg, per_scan)]
    if args.a_log_off_lattice:
        for r in rooflines:
            if "decay_form" in r:
                r["decay_form"] = "general: one exp2 per state (A_log off the lattice)"
                r["traffic"] = None
    roof = dict(rooflines[dom])
    for d in per_scan:
        d["hbm_frac"] = d["gb_per_s"] / peaks["hbm_gbs"]
        if "tflop_per_s" in d:
            d["tensor_frac"] = d["tflop_per_s"] / peaks["bf16_tflops_sustained"]
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": total_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "io_dtype": args.io or "bf16",
        "data": "synthetic (seeded generators with the pages' layer distributions)",
        "config": {"workload": " + ".join(c.name for c in cfgs),
                   "l2": "inputs larger than L2 (129 MB) on every launch, no flush",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "per_scan": per_scan,
        "roofline": roof,
        "rooflines": rooflines,
        "e2e": {"value": world * units_step / e2e_s, "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "steps": e2e_steps, "ms_per_step": e2e_s * 1e3,
                "ms_per_step_median": statistics.median(e2e_ms),
                "ms_per_step_min": min(e2e_ms), "ms_per_step_max": max(e2e_ms),
                "slowest_step": e2e_ms.index(max(e2e_ms)),
                "path": "lr_*_fwd_host_async on pinned host buffers, one lr_host_sync per step: the "
                        "library copies each chunk in, scans it and copies the outputs back, the "
                        "three calls overlapping (wall clock, host timer)"},
        "gpu_launches": sum(launches_per_call(c) for c in cfgs) * args.steps,
        "clocks": clk,
    }
    if args.a_log_off_lattice:
        line["config"]["selective_A_log"] = "moved off the initialisation lattice (profiling case)"
    if args.io:
        line["config"]["io_override"] = f"{args.io} I/O (profiling case)"
    if not args.seq_len and not args.only and not args.io and not args.no_extras:
        line["decode"] = decode_timings(lr, cfgs, dev)
        line["extra"] = extra_timings(lr, dev, peaks, alu)
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(cfgs, single_thread=True)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def load_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "source": "fallback"}


# CUDA sources each scan's kernel is compiled from.
KERNEL_SOURCES = {"rglru": ("lr_diag_scan.cu", "lr_device.cuh"),
                  "selective": ("lr_selective.cuh", "lr_selective.cu", "lr_device.cuh"),
                  "hgrn2": ("lr_hgrn2.cu", "lr_device.cuh")}


def kernel_source_digest(form: str) -> str:
    """Digest of the sources of one scan's kernel: a stored ncu traffic figure
    is used only while the kernel it was taken from is unchanged."""
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "selective_state_space_chunked_gb300", "csrc")
    for f in KERNEL_SOURCES[form]:
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def traffic_for(cfg: wl.Config):
    """DRAM read+write bytes per full-size launch from the committed ncu
    summary (profiles/traffic.json), or None when it is missing or was taken
    from a kernel that has changed since."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    e = d.get(cfg.form)
    if not e or e.get("source_digest") != kernel_source_digest(cfg.form) or e.get("L") != cfg.L:
        return None
    return e.get("per_launch_bytes")


# ----------------------------------------------------------------------------
# reference arm: the oracle on host cores
# ----------------------------------------------------------------------------
def reference_arm(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    cfgs = step_configs(args.only, args.seq_len)
    samples = [(cfg, *oracle_sample(cfg)) for cfg in cfgs]
    cb = None
    vals, sample_ms = [], []
    for _ in range(args.warmup):
        cpu_baseline(cfgs, samples=samples)
    for _ in range(args.steps):
        cb = cpu_baseline(cfgs, samples=samples)
        vals.append(cb["value"])
        sample_ms.append(cb["sample_ms"])
    value = statistics.mean(vals)
    cb["value"] = value
    full_units = sum(algorithmic(c)["units"] for c in cfgs)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        # one step is the bounded sample of every scan: this is its measured
        # wall time; the rate is that of the sample
        "ms_per_step": statistics.mean(sample_ms),
        "ms_per_step_kind": "measured: one step = the bounded sample of each scan (cpu_baseline.sample)",
        "full_workload_ms_per_step_extrapolated": full_units / value * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded generators with the pages' layer distributions)",
        "config": {"workload": " + ".join(c.name for c in cfgs),
                   "l2": "n/a (host cores)", "parallelism": "host threads",
                   "sample": "whole sequences of a channel/head subset of batch row 0 of each scan"},
        "cpu_baseline": cb,
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--no-cpu-baseline", action="store_true",
                    help="skip timing the CPU oracle beside the GPU arm")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the decode-step and extra-scan timings after the step")
    ap.add_argument("--only", choices=["rglru", "selective", "hgrn2"], default=None,
                    help="run one scan of the step (profiling case)")
    ap.add_argument("--seq-len", type=int, default=None,
                    help="shorter sequences for a profiling case (not a benchmark number)")
    ap.add_argument("--io", choices=["bf16", "f32"], default=None,
                    help="I/O dtype of the step's scans (a profiling case, not the workload)")
    ap.add_argument("--a-log-off-lattice", action="store_true",
                    help="selective A_log moved off the initialisation lattice (the general "
                         "decay form; a profiling case, not the workload)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        reference_arm(args)
    else:
        gpu_arm(args)


if __name__ == "__main__":
    main()
