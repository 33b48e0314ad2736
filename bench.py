#!/usr/bin/env python
"""Benchmark of exact attention (forward + backward) on B300.

One step = forward and backward of every point of the long-context causal
sequence sweep (N = 4096, 8192, 16384; B * N = 32768; H = 16; d = 128; bf16;
Q and K scaled by 2), through the library's C ABI. Prints one JSON line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Multi-GPU (torchrun): every rank runs the same per-rank workload on its own
GPU (independent problems, no collective on the data path; weak scaling);
the timing is the max over ranks.
"""
from __future__ import annotations

import argparse
import datetime
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "attention fwd/bwd TFLOP/s and % of B300 fp16/bf16 tensor peak vs seq len"
SWEEP = [
    "long_b8_h16_n4096_d128_bf16_causal",
    "long_b4_h16_n8192_d128_bf16_causal",
    "long_b2_h16_n16384_d128_bf16_causal",
]
WORKLOAD_NAME = ("long-context causal attention sweep N in {4096, 8192, 16384}, B*N = 32768, "
                 "H = 16, d = 128, bf16, Q and K scaled by 2; one step = fwd + bwd of all three")

# DRAM traffic of one bwd_main_kernel launch per sweep point, from an ncu capture
# (dram__bytes_read.sum + dram__bytes_write.sum), valid only for the kernel
# sources hashed in "source_sha256". Measured on B/4 of each sweep point (one
# launch) and scaled by 4: the DRAM bytes grow with the number of heads.
TRAFFIC = {
    "source_sha256": "7c0999cac1f02e345deb6c00d195d43119fd12cc38f94597115772a1b78d15fb",
    "bytes_per_launch": {"4096": 4 * (205226496 + 85993216), "8192": 4 * (256429824 + 119474432),
                         "16384": 4 * (257691904 + 123221504)},
}
KERNEL_SOURCES = ["exact_io_aware_108_b300/csrc/bwd_kernel.cuh",
                  "exact_io_aware_108_b300/csrc/common.cuh",
                  "exact_io_aware_108_b300/csrc/ptx.cuh",
                  "exact_io_aware_108_b300/csrc/schedule.cuh",
                  "exact_io_aware_108_b300/csrc/sdesc.cuh"]


def kernel_sha():
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def flops_fwd(w, density=1.0):
    return 4.0 * w.B * w.H * w.N * w.N * w.d * (0.5 if w.causal else 1.0) * density


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as fh:
            d = json.load(fh)
        return {"bf16_tflops": d["bf16_tflops"], "bf16_tflops_sustained": d["bf16_tflops_sustained"],
                "hbm_gbs": d["hbm_gbs"], "source": "measured"}
    return {"bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0, "hbm_gbs": 6400.0,
            "source": "fallback"}


# ------------------------------------------------------------------ clocks

REASONS = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]


class ClockSampler:
    """nvidia-smi samples of the SM clock and the throttle reasons every 50 ms;
    the summary keeps the samples whose timestamps fall between mark_start()
    and mark_end() (the timed region), so the idle GPU before and after it
    does not enter the median."""

    def __init__(self, gpu_id, interval_ms=50):
        self.gpu_id = gpu_id
        self.interval_ms = interval_ms
        self.proc = None
        self.lines = []
        self.t_start = self.t_end = None

    def __enter__(self):
        q = ("timestamp,clocks.sm,clocks.max.sm,power.draw," +
             ",".join("clocks_event_reasons." + r for r in REASONS))
        cmd = ["nvidia-smi", f"--query-gpu={q}", "--format=csv,noheader,nounits", "-lms",
               str(self.interval_ms)]
        if self.gpu_id is not None:
            cmd += ["-i", str(self.gpu_id)]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def mark_start(self):
        self.t_start = time.time()

    def mark_end(self):
        self.t_end = time.time()

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            out, _ = self.proc.communicate(timeout=10)
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    @staticmethod
    def parse(line):
        """(unix time, sm MHz, max sm MHz, set of active reasons) or None."""
        parts = [p.strip() for p in line.split(",")]
        if len(parts) < 4 + len(REASONS):
            return None
        try:
            ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
            sm, mx = float(parts[1]), float(parts[2])
        except ValueError:
            return None
        reasons = {r for r, v in zip(REASONS, parts[4:]) if v.lower() == "active"}
        return ts, sm, mx, reasons

    def summary(self):
        samples = [x for x in (self.parse(ln) for ln in self.lines) if x is not None]
        inside = samples
        if self.t_start is not None and self.t_end is not None:
            inside = [x for x in samples if self.t_start <= x[0] <= self.t_end]
        in_window = bool(inside)
        if not inside:  # a region shorter than the sampling interval
            inside = samples
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        reasons = set()
        for x in inside:
            reasons |= x[3]
        return {"sm_mhz": statistics.median(x[1] for x in inside), "sm_max_mhz": max(x[2] for x in inside),
                "reasons": sorted(reasons), "samples": len(inside),
                "window": "timed region" if in_window else "whole sampling period"}


# ------------------------------------------------------------------ ranks

def max_over_ranks(x, dist=None, device="cpu"):
    """Max of a per-rank float over all ranks (the slowest rank sets the time)."""
    if dist is None:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(flops_per_rank_step, ms_per_step_max, world):
    """Weak scaling: every rank runs the same per-rank workload; the job's rate
    is all ranks' flops divided by the slowest rank's time (TFLOP/s)."""
    return world * flops_per_rank_step / (ms_per_step_max * 1e-3) / 1e12


def rank_seed_offset(rank):
    """Each rank draws its own independent problem (a different seed)."""
    return int(rank)


# ------------------------------------------------------------------ GPU arm

class Problem:
    """Device buffers of one sweep point; step() = fwd + bwd through the C ABI."""

    def __init__(self, w, seed_offset, device):
        import torch
        from exact_io_aware_108_b300 import inputs
        import exact_io_aware_108_b300 as fa
        self.w = w
        self.fa = fa
        host = inputs.make_qkv(w.B, w.H, w.N, w.d, w.dtype, seed=w.seed + seed_offset,
                               qk_mult=w.qk_mult, with_dout=True)
        self.host = {n: host[n].pin_memory() for n in ("q", "k", "v", "dout")}
        self.dev = {n: t.to(device) for n, t in self.host.items()}
        q = self.dev["q"]
        self.o = torch.empty_like(q)
        self.o_res = torch.empty_like(q)
        self.lse = torch.empty(q.shape[:-1], dtype=torch.float32, device=device)
        self.dq = torch.empty_like(q)
        self.dk = torch.empty_like(q)
        self.dv = torch.empty_like(q)
        self.ws = torch.empty(fa.fa_bwd_workspace_size(w.B, w.H, w.N, w.d), dtype=torch.uint8,
                              device=device)
        self.out_host = {n: torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
                         for n, t in (("o", self.o), ("lse", self.lse), ("dq", self.dq),
                                      ("dk", self.dk), ("dv", self.dv))}
        self.flops_fwd = flops_fwd(w)
        self.flops_bwd = 2.5 * self.flops_fwd

    def step(self, stream, main_events=None, fwd_events=None):
        fa, w, d = self.fa, self.w, self.dev
        if fwd_events is not None:
            fwd_events[0].record(stream)
        fa.fa_fwd_ex(d["q"], d["k"], d["v"], self.o, self.lse, w.scale, w.causal, None,
                     o_res=self.o_res, stream=stream)
        if fwd_events is not None:
            fwd_events[1].record(stream)
        fa.fa_bwd_prepare(d["q"], d["v"], self.o, self.o_res, self.lse, d["dout"], self.ws, stream=stream)
        if main_events is not None:
            main_events[0].record(stream)
        fa.fa_bwd_main(d["q"], d["k"], d["v"], d["dout"], self.dk, self.dv, w.scale, w.causal,
                       workspace=self.ws, stream=stream)
        if main_events is not None:
            main_events[1].record(stream)
        fa.fa_bwd_finish(self.dq, self.ws, stream=stream)

    def fwd_plain(self, stream):
        """The forward alone: O and LSE, no residual."""
        fa, w, d = self.fa, self.w, self.dev
        fa.fa_fwd(d["q"], d["k"], d["v"], self.o, self.lse, w.scale, w.causal, stream=stream)

    def copy_in(self, stream):
        for n in ("q", "k", "v", "dout"):
            self.dev[n].copy_(self.host[n], non_blocking=True)

    def copy_out(self, stream):
        for n, t in (("o", self.o), ("lse", self.lse), ("dq", self.dq), ("dk", self.dk),
                     ("dv", self.dv)):
            self.out_host[n].copy_(t, non_blocking=True)

    def h2d_bytes(self):
        return sum(t.numel() * t.element_size() for t in self.host.values())

    def d2h_bytes(self):
        return sum(t.numel() * t.element_size() for t in self.out_host.values())


def run_ours(args, rank, world, local_rank):
    import torch
    import exact_io_aware_108_b300 as fa
    from exact_io_aware_108_b300 import inputs
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    torch.cuda.set_device(local_rank)
    device = torch.device("cuda", local_rank)
    fa.load_library()
    peaks = load_peaks()
    probs = [Problem(inputs.WORKLOADS[n], rank_seed_offset(rank), device) for n in SWEEP]
    stream = torch.cuda.Stream(device)
    torch.cuda.synchronize()

    def barrier():
        torch.cuda.synchronize()
        if dist is not None:
            dist.barrier()

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            for p in probs:
                p.step(stream)
    barrier()
    assert fa.fa_get_device_error(stream) == 0, "device error during warm-up"

    gpu_uuid = None
    try:
        gpu_uuid = "GPU-" + str(torch.cuda.get_device_properties(device).uuid)
    except Exception:
        gpu_uuid = None
    K = args.steps
    main_ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                for _ in probs] for _ in range(K)]
    fwd_ev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in probs] for _ in range(K)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    with ClockSampler(gpu_uuid) as clocks:
        clocks.mark_start()
        with torch.cuda.stream(stream):
            t0.record(stream)
            for s in range(K):
                for i, p in enumerate(probs):
                    p.step(stream, main_events=main_ev[s][i], fwd_events=fwd_ev[s][i])
            t1.record(stream)
        barrier()
        clocks.mark_end()
    ms_total = t0.elapsed_time(t1)
    assert fa.fa_get_device_error(stream) == 0, "device error in the timed region"
    ms_max = max_over_ranks(ms_total, dist, device)
    ms_step = ms_max / K
    flops_step = sum(p.flops_fwd + p.flops_bwd for p in probs)
    value = whole_job_rate(flops_step, ms_step, world)

    # per-sweep-point breakdown and the dominant kernel (bwd_main) roofline
    sweep = []
    main_ms_total = 0.0
    main_flops_total = 0.0
    for i, p in enumerate(probs):
        f_ms = sum(fwd_ev[s][i][0].elapsed_time(fwd_ev[s][i][1]) for s in range(K)) / K
        m_ms = sum(main_ev[s][i][0].elapsed_time(main_ev[s][i][1]) for s in range(K)) / K
        main_ms_total += m_ms
        main_flops_total += p.flops_bwd
        sweep.append({
            "N": p.w.N, "B": p.w.B,
            "fwd_ms": round(f_ms, 4),
            "fwd_tflops": round(p.flops_fwd / (f_ms * 1e-3) / 1e12, 1),
            "fwd_frac_of_measured_burst": round(p.flops_fwd / (f_ms * 1e-3) / 1e12 / peaks["bf16_tflops"], 4),
            "bwd_main_ms": round(m_ms, 4),
            "bwd_main_tflops": round(p.flops_bwd / (m_ms * 1e-3) / 1e12, 1),
            "bwd_main_frac_of_measured_burst": round(p.flops_bwd / (m_ms * 1e-3) / 1e12 / peaks["bf16_tflops"], 4),
        })
    achieved = main_flops_total / (main_ms_total * 1e-3) / 1e12
    traffic = None
    if TRAFFIC["source_sha256"] == kernel_sha() and TRAFFIC["bytes_per_launch"]:
        vals = [TRAFFIC["bytes_per_launch"].get(str(p.w.N)) for p in probs]
        if all(v is not None for v in vals):
            traffic = sum(vals) / len(vals)
    # The denominator is the measured peak at the clock this run saw: the
    # burst figure (measured at the maximum SM clock) while the sampled median
    # SM clock is within 5 % of the maximum, else the burst figure scaled by
    # median / maximum clock. The sustained figure (measured under the power
    # cap at a lower clock) is reported beside it.
    csum = clocks.summary()
    peak = peaks["bf16_tflops"]
    peak_kind = f"{peaks['source']} bf16 burst (the run's median SM clock is at its maximum)"
    if csum.get("sm_mhz") and csum.get("sm_max_mhz") and csum["sm_mhz"] < 0.95 * csum["sm_max_mhz"]:
        peak = peaks["bf16_tflops"] * csum["sm_mhz"] / csum["sm_max_mhz"]
        peak_kind = (f"{peaks['source']} bf16 burst scaled to the run's median SM clock "
                     f"({csum['sm_mhz']:.0f} of {csum['sm_max_mhz']:.0f} MHz)")
    roofline = {"bound": "tensor", "achieved": round(achieved, 1), "peak": round(peak, 1),
                "unit": "TFLOP/s", "frac": round(achieved / peak, 4), "traffic": traffic,
                "kernel": "bwd_main_kernel<d=128,bf16 in,causal> (3 launches per step)",
                "peak_kind": peak_kind,
                "frac_of_measured_sustained": round(achieved / peaks["bf16_tflops_sustained"], 4)}

    # the forward alone (O and LSE, no residual) per sweep point
    fwd_plain_ms = []
    with torch.cuda.stream(stream):
        for p in probs:
            for _ in range(args.warmup):
                p.fwd_plain(stream)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(K):
                p.fwd_plain(stream)
            e1.record(stream)
            e1.synchronize()
            fwd_plain_ms.append(e0.elapsed_time(e1) / K)
    assert fa.fa_get_device_error(stream) == 0, "device error in the forward timing"
    for row, p, ms in zip(sweep, probs, fwd_plain_ms):
        tf = p.flops_fwd / (ms * 1e-3) / 1e12
        row.update(fwd_plain_ms=round(ms, 4), fwd_plain_tflops=round(tf, 1),
                   fwd_plain_frac_of_measured_burst=round(tf / peaks["bf16_tflops"], 4))

    # end to end: pinned host inputs -> device -> fwd+bwd -> host outputs,
    # through the public API. The copies of one sweep point overlap the
    # compute of the others: inputs go up on one stream, results come down on
    # another, and the compute stream orders each point's buffers.
    e2e_k = max(1, K // 2)
    h2d = torch.cuda.Stream(device)
    d2h = torch.cuda.Stream(device)
    n = len(probs)

    def e2e_step(prev):
        """One step; prev = per-point (compute done, copy-out done) events of
        the step before, or None. Returns this step's events."""
        cur = []
        for i, p in enumerate(probs):
            if prev is not None:
                h2d.wait_event(prev[i][0])        # inputs still read by the previous step
            with torch.cuda.stream(h2d):
                p.copy_in(h2d)
            ready = torch.cuda.Event()
            ready.record(h2d)
            stream.wait_event(ready)
            if prev is not None:
                stream.wait_event(prev[i][1])     # outputs still being copied out
            with torch.cuda.stream(stream):
                p.step(stream)
            done = torch.cuda.Event()
            done.record(stream)
            d2h.wait_event(done)
            with torch.cuda.stream(d2h):
                p.copy_out(d2h)
            out = torch.cuda.Event()
            out.record(d2h)
            cur.append((done, out))
        return cur

    for p in probs:  # the tensors are used on the copy streams too
        for t in list(p.dev.values()) + [p.o, p.lse, p.dq, p.dk, p.dv]:
            t.record_stream(h2d)
            t.record_stream(d2h)
    prev = e2e_step(None)
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    h2d.wait_event(e0)
    d2h.wait_event(e0)
    prev = None
    for _ in range(e2e_k):
        prev = e2e_step(prev)
    for i in range(n):
        stream.wait_event(prev[i][1])
    e1.record(stream)
    barrier()
    assert fa.fa_get_device_error(stream) == 0, "device error in the end-to-end timing"
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_k, dist, device)
    # the copies alone (same bytes, same two copy streams, no compute): the
    # floor the end-to-end step is held to by the host link
    c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    c0.record(stream)
    h2d.wait_event(c0)
    d2h.wait_event(c0)
    for _ in range(e2e_k):
        for p in probs:
            with torch.cuda.stream(h2d):
                p.copy_in(h2d)
            with torch.cuda.stream(d2h):
                p.copy_out(d2h)
    for cs in (h2d, d2h):
        ev = torch.cuda.Event()
        ev.record(cs)
        stream.wait_event(ev)
    c1.record(stream)
    barrier()
    copy_ms = max_over_ranks(c0.elapsed_time(c1) / e2e_k, dist, device)
    e2e = {"value": round(whole_job_rate(flops_step, e2e_ms, world), 1), "unit": "TFLOP/s",
           "h2d_bytes_per_step": sum(p.h2d_bytes() for p in probs),
           "d2h_bytes_per_step": sum(p.d2h_bytes() for p in probs),
           "ms_per_step": round(e2e_ms, 3),
           "copies_alone_ms_per_step": round(copy_ms, 3),
           "overlap": "h2d, compute and d2h on three streams; one sweep point's copies "
                      "overlap the others' compute"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(args)

    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "TFLOP/s", "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": round(ms_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1), Q and K x2)",
        "config": {
            "workload": WORKLOAD_NAME, "H": 16, "d": 128, "causal": True,
            "flops_per_step_per_gpu": flops_step,
            "flop_count": "fwd 4*B*H*N^2*d/2 (causal), bwd 2.5x fwd",
            "l2": "no flush: every input tensor (134 MB) is larger than the 126 MB L2",
            "frac_of_measured_burst": round(value / world / peaks["bf16_tflops"], 4),
            "frac_of_measured_sustained": round(value / world / peaks["bf16_tflops_sustained"], 4),
            "sweep": sweep, "parallelism": f"{world} independent replica(s)" if world > 1 else "1 GPU",
        },
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": e2e,
        # per sweep point: forward, bwd prepare, bwd conversion (bf16), bwd main, bwd finish
        "gpu_launches": K * len(probs) * 5,
        "clocks": csum,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


# ------------------------------------------------------------------ CPU (oracle)

def _oracle_head_inputs(n_heads):
    """The first n_heads heads (b = 0) of the N = 4096 sweep point, on the CPU."""
    from exact_io_aware_108_b300 import inputs
    w = inputs.WORKLOADS[SWEEP[0]]
    t = inputs.make_qkv(w.B, w.H, w.N, w.d, w.dtype, seed=w.seed, qk_mult=w.qk_mult)
    sl = slice(0, n_heads)
    return w, {n: t[n][0:1, sl].contiguous() for n in ("q", "k", "v", "dout")}


def _oracle_step(w, t, nthreads):
    from oracle import ref
    ref.attn_fwd(t["q"], t["k"], t["v"], w.scale, w.causal, nthreads=nthreads)
    ref.attn_bwd(t["q"], t["k"], t["v"], t["dout"], w.scale, w.causal, rows_per_task=256,
                 nthreads=nthreads)


def cpu_baseline(args, n_heads=16):
    """The fp64 oracle, as it stands, on this host's cores: fwd + bwd of
    n_heads full heads (all 4096 rows each) of the N = 4096 sweep point."""
    from oracle import ref
    ref.load()
    nthreads = os.cpu_count() or 1
    w, t = _oracle_head_inputs(n_heads)
    t0 = time.perf_counter()
    _oracle_step(w, t, nthreads)
    sec = time.perf_counter() - t0
    flops = 3.5 * 4.0 * n_heads * w.N * w.N * w.d * 0.5
    return {"value": round(flops / sec / 1e12, 6), "unit": "TFLOP/s", "cores": nthreads,
            "kind": "oracle",
            "sample": f"fwd+bwd of {n_heads} heads (b=0, h=0..{n_heads - 1}) of the N=4096 point, "
                      f"all rows, fp64; {sec:.1f} s"}


def run_reference(args, rank, world):
    """The oracle as the reference arm: every step is fwd + bwd of one full head
    of the N = 4096 sweep point on the host cores."""
    if rank != 0:
        return
    from oracle import ref
    ref.load()
    nthreads = os.cpu_count() or 1
    w, t = _oracle_head_inputs(1)
    for _ in range(args.warmup):
        _oracle_step(w, t, nthreads)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        _oracle_step(w, t, nthreads)
    sec = (time.perf_counter() - t0) / args.steps
    flops = 3.5 * 4.0 * w.N * w.N * w.d * 0.5
    value = round(flops / sec / 1e12, 6)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(sec * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded N(0,1), Q and K x2)",
        "config": {"workload": WORKLOAD_NAME,
                   "sample_per_step": "fwd+bwd of one full head (b=0, h=0) of the N=4096 point"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": nthreads, "kind": "oracle",
                         "sample": "fwd+bwd of one full head of the N=4096 point per step"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_configs(args):
    """Per-workload forward / backward timings (one JSON line per workload).

    Every workload of inputs.WORKLOADS, inputs resident on the device, CUDA
    events around `args.steps` launches after `args.warmup`; no L2 flush (the
    small workloads fit in L2). Forward with and without O's residual; the
    backward is the whole fa_bwd (prepare, main, finish) with the residual.
    """
    import torch
    import exact_io_aware_108_b300 as fa
    from exact_io_aware_108_b300 import inputs
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream()
    peaks = load_peaks()

    def timed(fn):
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        if fa.fa_get_device_error() != 0:
            raise RuntimeError("device error during the timed launches")
        return e0.elapsed_time(e1) / args.steps

    for name, w in inputs.WORKLOADS.items():
        if w.nq is not None:
            # paged decode: HBM-bound; algorithmic bytes = the K and V rows of
            # every sequence's context once, q and o once, lse
            t = {k: (v.to(dev) if torch.is_tensor(v) else v) for k, v in inputs.make_workload(w).items()}
            o = torch.empty_like(t["q"])
            lse = torch.empty(t["q"].shape[:-1], dtype=torch.float32, device=dev)
            hkv = w.hkv or w.H
            pps = t["block_table"].shape[1]
            n_splits = fa.fa_decode_paged_num_splits(w.B, w.H, hkv, w.nq, w.d, w.page_size, pps, w.num_splits)
            wsd = torch.empty(max(1, fa.fa_decode_paged_workspace_size(w.B, w.H, hkv, w.nq, w.d, w.page_size,
                                                                       pps, w.num_splits)),
                              dtype=torch.uint8, device=dev)

            def dec():
                fa.fa_decode_paged(t["q"], t["k_cache"], t["v_cache"], t["block_table"], t["seq_len"], o, lse,
                                   w.scale, num_splits=w.num_splits, workspace=wsd, stream=stream)
            ctx = int(t["seq_len"].to(torch.int64).sum())
            nbytes = (ctx * hkv * w.d * 2 * 2 + 2 * t["q"].numel() * 2 + lse.numel() * 4
                      + t["block_table"].numel() * 4)
            flops = 4.0 * ctx * w.H * w.nq * w.d
            ms = timed(dec)
            line = {"config": name, "num_splits": n_splits, "context_tokens": ctx,
                    "algorithmic_bytes": nbytes, "decode_ms": round(ms, 4),
                    "decode_gbs": round(nbytes / ms / 1e6, 1),
                    "decode_frac_of_measured_hbm": round(nbytes / ms / 1e6 / peaks["hbm_gbs"], 4),
                    "decode_tflops": round(flops / ms / 1e9, 2)}
            print(json.dumps(line), flush=True)
            continue
        if w.dtype == "e4m3":
            # 8-bit q, k, v: forward only, against the fp8 tensor rate (the
            # measured bf16 burst x 2, the nominal fp8 / bf16 ratio)
            t = {k: (v.to(dev) if torch.is_tensor(v) else v) for k, v in inputs.make_workload(w).items()}
            o = torch.empty(t["q"].shape, dtype=torch.bfloat16, device=dev)
            lse = torch.empty(t["q"].shape[:-1], dtype=torch.float32, device=dev)
            hkv = w.hkv or w.H
            ws8 = torch.empty(fa.fa_fwd_fp8_workspace_size(w.B, hkv, w.N, w.d), dtype=torch.uint8, device=dev)
            kl = t["kv_len"].to(torch.int32) if "kv_len" in t else None

            def fwd8():
                fa.fa_fwd_fp8(t["q"], t["k"], t["v"], o, lse, w.scale, t["q_descale"], t["k_descale"],
                              t["v_descale"], w.causal, kl, workspace=ws8, stream=stream)
            ff = flops_fwd(w)
            ms = timed(fwd8)
            line = {"config": name, "density": 1.0, "fwd_gflop": round(ff / 1e9, 3), "fwd_ms": round(ms, 4),
                    "fwd_tflops": round(ff / ms / 1e9, 1),
                    "fwd_frac_of_fp8_peak": round(ff / ms / 1e9 / (2 * peaks["bf16_tflops"]), 4),
                    "fp8_peak_tflops": 2 * peaks["bf16_tflops"]}
            print(json.dumps(line), flush=True)
            continue
        t = {k: v.to(dev) for k, v in inputs.make_workload(w, with_dout=True).items()}
        q, k, v, dout = t["q"], t["k"], t["v"], t["dout"]
        kl = t["kv_len"].to(torch.int32) if "kv_len" in t else None
        bm = t.get("block_mask")
        density = 1.0 if bm is None else float(bm.float().mean())
        o, o_res = torch.empty_like(q), torch.empty_like(q)
        lse = torch.empty(q.shape[:-1], dtype=torch.float32, device=dev)
        dq, dk, dvv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        gqa = w.hkv is not None and w.hkv != w.H
        ws = torch.empty(fa.fa_bwd_workspace_size(w.B, w.H, w.N, w.d), dtype=torch.uint8, device=dev)
        split = w.num_splits is not None
        if split:
            n_splits = fa.fa_fwd_splitkv_num_splits(w.B, w.H, w.N, w.d, w.causal, w.num_splits)
            ws_split = torch.empty(max(1, fa.fa_fwd_splitkv_workspace_size(
                w.B, w.H, w.N, w.d, w.causal, w.num_splits)), dtype=torch.uint8, device=dev)

        def fwd_unsplit(res):
            fa.fa_fwd_gqa(q, k, v, o, lse, w.scale, w.causal, kl, o_res=res, stream=stream)

        def fwd(res):
            if split:
                fa.fa_fwd_splitkv(q, k, v, o, lse, w.scale, w.causal, kl, o_res=res,
                                  num_splits=w.num_splits, workspace=ws_split, stream=stream)
            elif bm is not None:
                fa.fa_fwd_blocksparse(q, k, v, o, lse, w.scale, bm, o_res=res, stream=stream)
            elif gqa:
                fa.fa_fwd_gqa(q, k, v, o, lse, w.scale, w.causal, kl, o_res=res, stream=stream)
            else:
                fa.fa_fwd_ex(q, k, v, o, lse, w.scale, w.causal, kl, o_res=res, stream=stream)

        def bwd():
            if bm is not None:
                fa.fa_bwd_blocksparse(q, k, v, o, lse, dout, dq, dk, dvv, w.scale, bm, o_res, ws,
                                      stream=stream)
            elif gqa:
                fa.fa_bwd_gqa(q, k, v, o, lse, dout, dq, dk, dvv, w.scale, w.causal, kl, o_res, ws,
                              stream=stream)
            else:
                fa.fa_bwd(q, k, v, o, lse, dout, dq, dk, dvv, w.scale, w.causal, kl, o_res, ws,
                          stream=stream)

        ff = flops_fwd(w, density)
        line = {"config": name, "density": round(density, 5), "fwd_gflop": round(ff / 1e9, 3)}
        ms = timed(lambda: fwd(None))
        line.update(fwd_ms=round(ms, 4), fwd_tflops=round(ff / ms / 1e9, 1))
        ms = timed(lambda: fwd(o_res))
        line.update(fwd_res_ms=round(ms, 4), fwd_res_tflops=round(ff / ms / 1e9, 1))
        if split:
            ms = timed(lambda: fwd_unsplit(None))
            line.update(num_splits=n_splits, unsplit_fwd_ms=round(ms, 4),
                        unsplit_fwd_tflops=round(ff / ms / 1e9, 1))
        if w.backward:
            fwd(o_res)
            ms = timed(bwd)
            line.update(bwd_ms=round(ms, 4), bwd_tflops=round(2.5 * ff / ms / 1e9, 1))
        for key in ("fwd_tflops", "fwd_res_tflops", "bwd_tflops"):
            if key in line:
                line[key.replace("tflops", "frac_of_measured_burst")] = round(
                    line[key] / peaks["bf16_tflops"], 4)
        print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--configs", action="store_true",
                    help="time forward and backward of every workload (one JSON line each)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.configs:
        run_configs(args)
    elif args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_ours(args, rank, world, local_rank)


if __name__ == "__main__":
    main()
