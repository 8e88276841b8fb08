#!/usr/bin/env python3
"""Benchmark of the GQA attention forward hot path on GB300.

One step = one causal prefill over S=32768 tokens plus one decode of a single
token against a KV cache of L=65536 positions (the largest prefill and decode
sizes of the chowfi/kernels README "Result" table), batch 1, 32 query / 8 KV
heads, head dim 128, bf16 in/out, fp32 accumulate, synthetic seeded N(0,1)
inputs.  Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the fp64 CPU oracle (the only reference this path
has) on the host cores, on a bounded sample of the same workload.
For N > 1 (torchrun, one rank per GPU) every rank runs an independent replica
of the step ("replicas only": the path needs no exchange between GPUs).
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

# CUDA feeds each stream to the GPU through one of a few hardware work queues
# (8 by default), assigned round-robin as streams are created; two streams
# that share a queue run strictly in submission order.  The end-to-end leg
# overlaps copies on two streams with kernels on a third, so it asks for the
# maximum number of queues (read when the CUDA context is created).
os.environ.setdefault("CUDA_DEVICE_MAX_CONNECTIONS", "32")

S_PREFILL = 32768
L_DECODE = 65536
HQ, HKV, D = 32, 8, 128
METRIC = "GQA attn fwd: prefill TFLOP/s, decode HBM GB/s, % of GB300 roofline"
WORKLOAD = ("causal prefill S=32768 + decode L=65536, batch 1, 32 q / 8 KV heads, "
            "D=128, bf16, N(0,1) seeds q=1 k=2 v=3")

# The pages' RTX 5090 numbers for the two halves of the step (context only).
PAGES_PREFILL_32K_MS = 38.816
PAGES_DECODE_64K_MS = 0.176
# ... and the step throughput derived from them with this file's FLOP count,
# 2*S^2*H*D + 4*H*D*L over 38.992 ms: another machine's number.
PAGES_STEP_TFLOPS = 225.6

FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# GB300's nominal HBM3e bandwidth, the figure the decode target is quoted against
NOMINAL_HBM_GBS = 8000.0


def prefill_flops(S: int) -> float:
    """Causal prefill FLOPs as the target metric counts them: 2*S^2*H*D."""
    return 2.0 * S * S * HQ * D


def decode_flops(L: int) -> float:
    return 4.0 * HQ * D * L


def decode_bytes(L: int) -> float:
    """K and V caches once, plus q and out: 2*L*8*128*2 + 2*(32*128*2)."""
    return 2.0 * L * HKV * D * 2 + 2 * HQ * D * 2


def step_flops() -> float:
    return prefill_flops(S_PREFILL) + decode_flops(L_DECODE)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {k: float(p[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


KERNEL_SOURCES = {"prefill": ("prefill.cu", "ptx.cuh", "internal.h"),
                  "decode": ("decode.cu", "ptx.cuh", "internal.h")}


def _code_only(text: str) -> str:
    """C/C++ source without comments and with whitespace collapsed, so that a
    comment-only edit does not count as a kernel change."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_source_hash(kernel: str) -> str:
    """Hash of the code (comments ignored) of the source files that define
    `kernel` (prefill or decode)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "gqa_flash_attention_causal_gb300", "csrc")
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(csrc, name), encoding="utf-8") as f:
            h.update(name.encode() + _code_only(f.read()).encode())
    return h.hexdigest()[:16]


def profiled_traffic(kernel: str):
    """DRAM bytes per launch recorded from an ncu capture in
    profiles/traffic.json, or None if absent or taken on other sources."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            rec = json.load(f)[kernel]
    except Exception:
        return None
    if rec.get("source_hash") != kernel_source_hash(kernel):
        return None
    return rec.get("bytes_per_launch")


# ----------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples (every 50 ms) of SM clock, power and throttle
    reasons; `mark_start`/`mark_stop` bracket the timed region and only the
    samples taken inside it are summarised."""

    # power.draw is a one-second average on this part; the timed region is
    # shorter, so the instantaneous reading is the one that means something
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw.instant,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.file = None
        self.t0 = self.t1 = None

    def __enter__(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=self.file, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def mark_start(self):
        self.t0 = time.time()

    def mark_stop(self):
        self.t1 = time.time()

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.12)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if self.proc is None or self.file is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        import datetime
        self.file.flush()
        rows = []
        with open(self.file.name) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) == 9:
                    rows.append(parts)
        os.unlink(self.file.name)

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        def stamp(x):
            try:
                return datetime.datetime.strptime(x, "%Y/%m/%d %H:%M:%S.%f").timestamp()
            except ValueError:
                return None
        inside = [r for r in rows
                  if self.t0 is not None and stamp(r[0]) is not None
                  and self.t0 - 0.05 <= stamp(r[0]) <= (self.t1 or 1e30) + 0.05]
        use = inside or rows
        if not use:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [num(r[1]) for r in use if num(r[1]) is not None]
        smax = [num(r[2]) for r in use if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in use for i in range(4) if r[5 + i] == "Active"})
        power = [num(r[3]) for r in use if num(r[3]) is not None]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(use),
                "samples_in_timed_region": len(inside),
                "power_w_max": max(power) if power else None}


# ----------------------------------------------------------------- oracle
class OracleSample:
    """Times the fp64 CPU oracle on a bounded sample of the step.

    Every query row i of the S=32768 causal prefill costs 4*H*D*(i+1) flops;
    rows are taken evenly over the sequence until about `seconds` of work,
    and the decode at L=65536 is computed in full.  The rate is those flops
    over the wall time, in TFLOP/s (the GPU metric's unit)."""

    def __init__(self):
        import oracle
        from gqa_flash_attention_causal_gb300.inputs import decode_inputs, prefill_inputs
        self.oracle = oracle
        self.q, self.k, self.v = prefill_inputs(S_PREFILL)
        self.dq, self.kc, self.vc = decode_inputs(L_DECODE)
        self.cores = oracle.max_threads()
        self.rate = None
        self.last = None  # (rows, oracle prefill rows, oracle decode) of the last run

    @staticmethod
    def row_flops(rows):
        return sum(4.0 * HQ * D * (int(r) + 1) for r in rows)

    def _rows(self, n):
        import numpy as np
        return [int(x) for x in np.linspace(0, S_PREFILL - 1, n).astype(int)]

    def calibrate(self):
        rows = self._rows(2 * self.cores)
        t0 = time.perf_counter()
        self.oracle.prefill_rows(self.q, self.k, self.v, rows, causal=True)
        self.rate = self.row_flops(rows) / max(time.perf_counter() - t0, 1e-6)

    def run(self, seconds: float):
        if self.rate is None:
            self.calibrate()
        t0 = time.perf_counter()
        want_dec = self.oracle.decode(self.dq, self.kc, self.vc)
        t_dec = time.perf_counter() - t0
        mean_row = 4.0 * HQ * D * S_PREFILL / 2
        n = int(min(S_PREFILL, max(self.cores, (seconds - t_dec) * self.rate / mean_row)))
        rows = self._rows(n)
        t0 = time.perf_counter()
        want_pre = self.oracle.prefill_rows(self.q, self.k, self.v, rows, causal=True)
        t_pre = time.perf_counter() - t0
        flops = self.row_flops(rows) + decode_flops(L_DECODE)
        desc = (f"{n} of {S_PREFILL} causal prefill query rows (all 32 heads, evenly spaced) "
                f"+ one full decode at L={L_DECODE}; fp64 C oracle, OpenMP over (row, head); "
                f"prefill {t_pre:.2f} s, decode {t_dec:.2f} s")
        self.last = (rows, want_pre, want_dec)
        return flops / (t_pre + t_dec) / 1e12, desc, t_pre + t_dec


# ----------------------------------------------------------------- distributed
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def aggregate(local_ms: float, local_units: float, world: int):
    """Whole-job time = max over ranks, work = sum over ranks (torch.distributed
    must be initialised when world > 1)."""
    if world == 1:
        return local_ms, local_units
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([local_ms], dtype=torch.float64, device=dev)
    u = torch.tensor([local_units], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ----------------------------------------------------------------- arms
def run_reference(args, n_world):
    """The oracle as it stands, on the host cores: W warm-up and K timed
    steps, each a bounded sample of the step sized so the whole run takes
    about --ref-total seconds."""
    sample = OracleSample()
    secs = min(args.ref_seconds, max(1.0, args.ref_total / (args.steps + args.warmup)))
    for _ in range(args.warmup):
        sample.run(secs)
    rates, times, desc = [], [], ""
    for _ in range(args.steps):
        tf, desc, t = sample.run(secs)
        rates.append(tf)
        times.append(t)
    value = statistics.median(rates)
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": n_world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * statistics.median(times), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "sample": desc},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": sample.cores,
                         "kind": "oracle", "sample": desc},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def run_ours(args, world, rank, local):
    import torch
    import gqa_flash_attention_causal_gb300 as gqa
    from gqa_flash_attention_causal_gb300.inputs import decode_inputs, prefill_inputs

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    gqa.lib()
    peaks, peaks_src = load_peaks()

    q, k, v = prefill_inputs(S_PREFILL)
    dq, kc, vc = decode_inputs(L_DECODE)
    d_q, d_k, d_v = q.to(dev), k.to(dev), v.to(dev)
    d_dq, d_kc, d_vc = dq.to(dev), kc.to(dev), vc.to(dev)
    out = torch.empty_like(d_q)
    dout = torch.empty_like(d_dq)
    stream = torch.cuda.current_stream()

    ws = torch.empty(gqa.decode_workspace_bytes(L_DECODE), dtype=torch.uint8, device=dev)

    def run_prefill():
        gqa.prefill(d_q, d_k, d_v, causal=True, out=out)

    def run_decode():
        gqa.decode(d_dq, d_kc, d_vc, out=dout, workspace=ws)

    for _ in range(max(3, args.warmup)):
        run_prefill()
        run_decode()
    torch.cuda.synchronize()
    if gqa.device_error() != 0:
        raise RuntimeError("device-side wait timed out during warm-up")

    # Each half of the step is captured once as a CUDA graph and replayed, so
    # the timed region holds no host launch gaps between kernels.
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        g_pre, g_dec = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_pre, stream=side):
            run_prefill()
        with torch.cuda.graph(g_dec, stream=side):
            run_decode()
    stream.wait_stream(side)
    g_pre.replay()
    g_dec.replay()
    torch.cuda.synchronize()

    # ------------------------------------------------ timed region (device)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(torch.cuda.current_device()) as clocks:
        clocks.mark_start()
        start.record(stream)
        for i in range(args.steps):
            ev[i][0].record(stream)
            g_pre.replay()
            ev[i][1].record(stream)
            g_dec.replay()
            ev[i][2].record(stream)
        stop.record(stream)
        torch.cuda.synchronize()
        clocks.mark_stop()
    barrier(world)
    total_ms = start.elapsed_time(stop)
    pre_ms = [e[0].elapsed_time(e[1]) for e in ev]
    dec_ms = [e[1].elapsed_time(e[2]) for e in ev]
    if gqa.device_error() != 0:
        raise RuntimeError("device-side wait timed out in the timed region")
    launches = args.steps * (gqa.launches_per_call(False) + gqa.launches_per_call(True))
    # the outputs of the timed region's last step, for the parity check below
    timed_out, timed_dout = out.cpu(), dout.cpu()

    ms_step_local = total_ms / args.steps
    ms_step, flops_all = aggregate(ms_step_local, step_flops() * args.steps, world)
    value = flops_all / (ms_step * args.steps * 1e-3) / 1e12

    pre_avg = statistics.mean(pre_ms)
    dec_avg = statistics.mean(dec_ms)
    pre_tflops = prefill_flops(S_PREFILL) / (pre_avg * 1e-3) / 1e12
    dec_gbs = decode_bytes(L_DECODE) / (dec_avg * 1e-3) / 1e9
    # the timed region is ~0.1 s right after warm-up: the burst peak applies
    peak_tc = peaks["bf16_tflops"]

    # ------------------------------------------------ sustained (seconds-long)
    # The timed region above is ~0.1 s right after warm-up, i.e. a burst.  Here
    # the same graphs run back to back for --sustain-s seconds; the last
    # third is timed (CUDA events per kernel) with its own clock record and
    # compared with the sustained bf16 peak.
    sustained = None
    if args.sustain_s > 0:
        chunk = 10
        t_end = time.time() + args.sustain_s * 2 / 3
        while time.time() < t_end:
            for _ in range(chunk):
                g_pre.replay()
                g_dec.replay()
            torch.cuda.synchronize()
        n_sus = max(chunk, int(args.sustain_s / 3 / (ms_step_local * 1e-3)))
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(n_sus)]
        with ClockSampler(torch.cuda.current_device()) as sclk:
            sclk.mark_start()
            for i in range(n_sus):
                evs[i][0].record(stream)
                g_pre.replay()
                evs[i][1].record(stream)
                g_dec.replay()
                evs[i][2].record(stream)
                if i % chunk == chunk - 1:
                    torch.cuda.synchronize()
            torch.cuda.synchronize()
            sclk.mark_stop()
        s_total = evs[0][0].elapsed_time(evs[-1][2])
        s_pre = statistics.mean(e[0].elapsed_time(e[1]) for e in evs)
        s_pre_tf = prefill_flops(S_PREFILL) / (s_pre * 1e-3) / 1e12
        sustained = {
            "seconds_before_timing": round(args.sustain_s * 2 / 3, 2), "steps": n_sus,
            "value": step_flops() * n_sus / (s_total * 1e-3) / 1e12, "unit": "TFLOP/s",
            "ms_per_step": s_total / n_sus, "prefill_tflops": s_pre_tf,
            "peak": peaks["bf16_tflops_sustained"], "peak_kind": f"bf16 sustained ({peaks_src})",
            "frac": s_pre_tf / peaks["bf16_tflops_sustained"],
            "decode_gbs": decode_bytes(L_DECODE) / (statistics.mean(
                e[1].elapsed_time(e[2]) for e in evs) * 1e-3) / 1e9,
            "clocks": sclk.summary(),
        }
        if gqa.device_error() != 0:
            raise RuntimeError("device-side wait timed out in the sustained run")

    # ------------------------------------------------ end to end (host buffers)
    # Every step copies its own inputs from pinned host memory, runs the
    # prefill and the decode through the public API and copies both results
    # back.  Pipelined: two buffer sets, copies on their own streams, so the
    # copies of step i+1 and of step i-1's results overlap step i's kernels.
    h_in = [tuple(t.pin_memory() for t in (q, k, v, dq, kc, vc)) for _ in range(2)]
    h_out = [(torch.empty(out.shape, dtype=out.dtype).pin_memory(),
              torch.empty(dout.shape, dtype=dout.dtype).pin_memory()) for _ in range(2)]
    d_in = [(d_q, d_k, d_v, d_dq, d_kc, d_vc),
            tuple(torch.empty_like(t) for t in (d_q, d_k, d_v, d_dq, d_kc, d_vc))]
    d_out = [(out, dout), (torch.empty_like(out), torch.empty_like(dout))]
    h2d = sum(t.numel() * t.element_size() for t in h_in[0])
    d2h = sum(t.numel() * t.element_size() for t in h_out[0])
    # kernels and both copy directions on three streams created back to back,
    # so that round-robin queue assignment gives each its own hardware queue
    s_cmp, s_h2d, s_d2h = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    s_cmp.wait_stream(stream)

    def e2e_run(steps, pipelined, timeline=None):
        """ms per step; with `timeline` (a list), also the start and end of
        every step's host-to-device copies, kernels and device-to-host
        copies (ms from the start, CUDA events on their own streams) for the
        first few steps."""
        done_compute = [None, None]
        done_d2h = [None, None]
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        marks = []

        def mark(strm, i):
            if timeline is None:
                return None
            e = torch.cuda.Event(enable_timing=True)
            e.record(strm)
            return e

        e0.record(s_cmp)
        s_h2d.wait_stream(s_cmp)
        s_d2h.wait_stream(s_cmp)
        for i in range(steps):
            b = i % 2 if pipelined else 0
            with torch.cuda.stream(s_h2d):
                if done_compute[b] is not None:
                    s_h2d.wait_event(done_compute[b])  # buffers of step i-2 are free
                m = [mark(s_h2d, i)]
                # the prefill's inputs first, so that it can start before the
                # decode's caches have arrived
                ready = []
                for first, last in ((0, 3), (3, 6)):
                    for dst, src in zip(d_in[b][first:last], h_in[b][first:last]):
                        dst.copy_(src, non_blocking=True)
                    ready.append(torch.cuda.Event())
                    ready[-1].record(s_h2d)
                m.append(mark(s_h2d, i))
            s_cmp.wait_event(ready[0])
            if done_d2h[b] is not None:
                s_cmp.wait_event(done_d2h[b])  # outputs of step i-2 are copied out
            m.append(mark(s_cmp, i))
            with torch.cuda.stream(s_cmp):
                gqa.prefill(d_in[b][0], d_in[b][1], d_in[b][2], causal=True, out=d_out[b][0])
                s_cmp.wait_event(ready[1])
                gqa.decode(d_in[b][3], d_in[b][4], d_in[b][5], out=d_out[b][1])
            m.append(mark(s_cmp, i))
            done_compute[b] = torch.cuda.Event()
            done_compute[b].record(s_cmp)
            with torch.cuda.stream(s_d2h):
                s_d2h.wait_event(done_compute[b])
                m.append(mark(s_d2h, i))
                h_out[b][0].copy_(d_out[b][0], non_blocking=True)
                h_out[b][1].copy_(d_out[b][1], non_blocking=True)
                m.append(mark(s_d2h, i))
                done_d2h[b] = torch.cuda.Event()
                done_d2h[b].record(s_d2h)
            if m[0] is not None:
                marks.append(m)
            if not pipelined:
                s_cmp.wait_event(done_d2h[b])
        s_cmp.wait_stream(s_d2h)
        e1.record(s_cmp)
        torch.cuda.synchronize()
        if timeline is not None:
            for m in marks:
                t = [round(e0.elapsed_time(e), 3) for e in m]
                timeline.append({"h2d": t[0:2], "kernels": t[2:4], "d2h": t[4:6]})
        return e0.elapsed_time(e1) / steps

    e2e_run(2, True)
    # as many steps as the device-timed region, so the one-off pipeline fill
    # (the first step's upload) and drain (the last step's download) weigh the same
    e2e_steps = max(2, args.steps)
    barrier(world)
    # Three pipelined runs, the median reported: the host link of this part
    # occasionally drops to about a tenth of its rate for 50-100 ms (seen
    # in per-copy event timelines: 640 MiB host-to-device taking 25-45 ms
    # instead of 3.5), which a single run may or may not catch.
    runs = []
    for _ in range(3):
        tl = []
        runs.append((e2e_run(e2e_steps, True, tl), tl))
    e2e_ms_local, timeline = sorted(runs, key=lambda r: r[0])[1]
    serial_ms_local = e2e_run(e2e_steps, False)
    e2e_ms, e2e_flops = aggregate(e2e_ms_local, step_flops(), world)
    e2e_value = e2e_flops / (e2e_ms * 1e-3) / 1e12
    serial_value = step_flops() / (serial_ms_local * 1e-3) / 1e12
    if gqa.device_error() != 0:
        raise RuntimeError("device-side wait timed out in the end-to-end run")

    if rank != 0:
        return None

    cpu = None
    parity = None
    if world == 1 and not args.no_cpu_baseline:
        sample = OracleSample()
        tf, desc, _ = sample.run(args.ref_seconds)
        cpu = {"value": tf, "unit": "TFLOP/s", "cores": sample.cores, "kind": "oracle",
               "sample": desc}
        parity = timed_parity(sample.last, timed_out, timed_dout)

    clk = clocks.summary()
    traffic = profiled_traffic("prefill")
    line = {
        "metric": METRIC,
        "value": value,
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": value / PAGES_STEP_TFLOPS,
        "baseline_note": "RTX 5090 Triton kernel of the pages (38.816 + 0.176 ms per step)",
        "dtype": "bf16",
        "data": "synthetic",
        "config": {
            "workload": WORKLOAD,
            "global_batch": 1 * world,
            "seq_len": S_PREFILL,
            "kv_len": L_DECODE,
            "parallelism": f"replicas{world}",
            "l2": "inputs larger than L2 (prefill q 256 MiB + k,v 128 MiB; decode KV 256 MiB)",
            "launch": "each step replays a CUDA graph of the prefill and one of the decode",
        },
        "sustained": sustained,
        "roofline": {
            "kernel": "prefill_kernel",
            "bound": "tensor",
            "achieved": pre_tflops,
            "peak": peak_tc,
            "unit": "TFLOP/s",
            "frac": pre_tflops / peak_tc,
            "traffic": traffic,
            "peak_kind": (f"bf16 burst ({peaks_src}): the timed region lasts "
                          f"{total_ms / 1e3:.2f} s, a burst, not a seconds-long sustained load"),
            "frac_of_sustained": pre_tflops / peaks["bf16_tflops_sustained"],
        },
        "prefill": {
            "S": S_PREFILL, "ms": pre_avg, "ms_min": min(pre_ms), "tflops": pre_tflops,
            "frac_of_burst": pre_tflops / peaks["bf16_tflops"],
            "frac_of_sustained": pre_tflops / peaks["bf16_tflops_sustained"],
            "pages_rtx5090_ms": PAGES_PREFILL_32K_MS,
        },
        "decode": {
            "L": L_DECODE, "ms": dec_avg, "ms_min": min(dec_ms), "gbs": dec_gbs,
            "bound": "hbm", "frac_of_measured_hbm": dec_gbs / peaks["hbm_gbs"],
            "frac_of_8tbs": dec_gbs / NOMINAL_HBM_GBS,
            "n_split": gqa.decode_num_splits(L_DECODE),
            "pages_rtx5090_ms": PAGES_DECODE_64K_MS,
        },
        "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms, "steps": e2e_steps,
                "how": "public API from pinned host buffers; copies of neighbouring steps "
                       "overlap the kernels (two buffer sets, separate copy streams); median "
                       "of three runs of as many steps as the device-timed region",
                "runs_ms_per_step": [round(r[0], 4) for r in runs],
                "serialized": {"value": serial_value, "ms_per_step": serial_ms_local},
                "timeline": timeline_summary(timeline)},
        "gpu_launches": launches,
        "clocks": clk,
        "cpu_baseline": cpu,
        "parity": parity,
    }
    return line


def timeline_summary(tl):
    """Where the pipelined end-to-end steps spend their time: per stage
    (host-to-device copies, kernels, device-to-host copies) the mean span,
    the kernels' idle time between consecutive steps, and the first steps'
    start/end stamps (ms from the start of the run)."""
    import statistics as st
    if not tl:
        return None
    span = {k: st.mean(t[k][1] - t[k][0] for t in tl) for k in ("h2d", "kernels", "d2h")}
    gaps = [b["kernels"][0] - a["kernels"][1] for a, b in zip(tl, tl[1:])]
    late = [b["kernels"][0] - b["h2d"][1] for b in tl]  # >0: kernels started after the copy
    return {"mean_span_ms": {k: round(v, 3) for k, v in span.items()},
            "kernel_idle_between_steps_ms": {"mean": round(st.mean(gaps), 3) if gaps else None,
                                             "max": round(max(gaps), 3) if gaps else None},
            "kernels_start_after_h2d_end_ms_mean": round(st.mean(late), 3),
            "steps": len(tl), "first_steps": tl[:3], "last_steps": tl[-2:]}


def bf16_rne_bits(x):
    """bf16 bit patterns of float64 values rounded to nearest, ties to even,
    directly from float64 (no intermediate float32 rounding).  Normal range
    only, which covers attention outputs of N(0,1) inputs; zeros stay zero."""
    import numpy as np
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)                       # x = m * 2^e, 0.5 <= |m| < 1
    r = np.ldexp(np.rint(np.ldexp(m, 8)), e - 8)   # 8 significant bits, half to even
    return (r.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)


def bf16_ulp_distance(a_bits, b_bits):
    """Distance in bf16 units in the last place between two arrays of bf16
    bit patterns (adjacent representable values are 1 apart; +0 and -0 are
    the same point)."""
    import numpy as np
    def order(b):
        b = np.asarray(b, dtype=np.uint16).astype(np.int64)
        mag = b & 0x7FFF
        return np.where(b & 0x8000, -mag, mag)
    return np.abs(order(a_bits) - order(b_bits))


def ulp_summary(got_bits, want):
    """How far bf16 outputs are from the correctly rounded bf16 of the fp64
    reference values: the fractions at 0, within 1 and within 4 ulp.  (No
    maximum: an output near zero has a tiny ulp, so an absolute error well
    inside the tolerance can be thousands of ulps there.)"""
    d = bf16_ulp_distance(got_bits, bf16_rne_bits(want))
    return {"exact": float((d == 0).mean()), "within_1": float((d <= 1).mean()),
            "within_4": float((d <= 4).mean())}


def timed_parity(oracle_last, out, dout):
    """Error of the timed region's outputs against the oracle rows the CPU
    baseline computed (evenly spaced prefill rows, all heads; the whole
    decode), with the tolerance of the parity tests: max-abs <= 2e-2 and
    mean-abs <= 2e-3 for these N(0,1) inputs."""
    import numpy as np
    import torch
    rows, want_pre, want_dec = oracle_last
    got_pre = out[0, rows].double().numpy()
    got_dec = dout.double().numpy().reshape(want_dec.shape)
    pre_bits = out[0, rows].contiguous().view(torch.int16).numpy().view(np.uint16)
    dec_bits = dout.contiguous().view(torch.int16).numpy().view(np.uint16).reshape(want_dec.shape)
    e_pre, e_dec = np.abs(got_pre - want_pre), np.abs(got_dec - want_dec)
    finite = bool(np.isfinite(got_pre).all() and np.isfinite(got_dec).all())
    ok = (finite and e_pre.max() <= 2e-2 and e_pre.mean() <= 2e-3
          and e_dec.max() <= 2e-2 and e_dec.mean() <= 2e-3)
    return {"ok": bool(ok), "tolerance": {"max_abs": 2e-2, "mean_abs": 2e-3},
            "prefill": {"rows": len(rows), "tiles_covered": len({r // 128 for r in rows}),
                        "tiles": S_PREFILL // 128, "heads": HQ,
                        "max_abs": float(e_pre.max()), "mean_abs": float(e_pre.mean())},
            "decode": {"max_abs": float(e_dec.max()), "mean_abs": float(e_dec.mean())},
            "ulp": {"prefill": ulp_summary(pre_bits, want_pre),
                    "decode": ulp_summary(dec_bits, want_dec),
                    "what": "distance of each bf16 output from the correctly rounded bf16 "
                            "of the fp64 oracle value"},
            "what": "outputs of the timed region's last step vs the fp64 oracle rows of the "
                    "CPU baseline"}


def rotation_copies(l2_bytes: int, cache_bytes: int) -> int:
    """KV-cache copies a decode timing loop rotates through so that every
    call reads its cache from DRAM.  Between two reads of one copy the other
    copies stream at least 6x the L2 size: with only 2x (as first used), an
    ncu capture of the rotation found launches at L=32768 and 65536 that
    read 23 % and 10 % of their cache from L2, whose replacement is not
    strict LRU; from 5 copies at L=65536 every launch read the full
    algorithmic bytes from DRAM."""
    return max(1, -(-6 * l2_bytes // cache_bytes) + 1)


def sweep_time(fn, calls=1, burn_in=50, rounds=8):
    """Per-call GPU time of `fn` (which makes `calls` calls): at least
    `burn_in` calls first, then `rounds` timed rounds (CUDA events on the
    current stream).  Returns (median, p05, p95) over rounds, ms per call."""
    import numpy as np
    import torch
    for _ in range(max(1, -(-burn_in // calls))):
        fn()
    torch.cuda.synchronize()
    ts = []
    for _ in range(rounds):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        fn()
        b.record()
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b) / calls)
    return (float(np.median(ts)), float(np.percentile(ts, 5)), float(np.percentile(ts, 95)))


def _graph(calls):
    """A CUDA graph replaying `calls` (callables) once each, captured on a
    side stream after one eager round."""
    import torch
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for c in calls:
            c()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=side):
            for c in calls:
                c()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    return g


def sweep_heads(kind, hq, hkv, n, dev, peaks, src):
    """Throughput and parity of the runtime head-count entries
    (gqa_attn_prefill_heads / gqa_attn_decode_heads) for one layout."""
    import numpy as np
    import torch
    import gqa_flash_attention_causal_gb300 as gqa
    import oracle
    from gqa_flash_attention_causal_gb300.inputs import normal_bf16
    if kind == "prefill":
        q = normal_bf16((1, n, hq, D), 1)
        k = normal_bf16((1, n, hkv, D), 2)
        v = normal_bf16((1, n, hkv, D), 3)
        dq, dk, dv = q.to(dev), k.to(dev), v.to(dev)
        out = torch.empty_like(dq)
        call = lambda: gqa.prefill_heads(dq, dk, dv, out=out)  # noqa: E731
        ms_eager = sweep_time(call)[0]
        reps = max(1, min(200, int(2.0 / max(ms_eager, 1e-3))))
        ms, p05, p95 = sweep_time(_graph([call] * reps).replay, calls=reps)
        call()
        torch.cuda.synchronize()
        rows = sorted({0, 1, n // 2, n - 1})
        err = np.abs(out[0, rows].double().cpu().numpy() - oracle.prefill_rows(q, k, v, rows))
        tput = 2.0 * n * n * hq * D / (ms * 1e-3) / 1e12
        line = {"workload": "prefill_heads", "hq": hq, "hkv": hkv, "S": n, "ms": ms,
                "ms_p05": p05, "ms_p95": p95, "tflops": tput,
                "frac_of_burst": tput / peaks["bf16_tflops"]}
    else:
        q = normal_bf16((1, hq, D), 1)
        kc = normal_bf16((1, n, hkv, D), 2)
        vc = normal_bf16((1, n, hkv, D), 3)
        dq = q.to(dev)
        nbytes = 2 * n * hkv * D * 2 + 2 * hq * D * 2
        l2 = torch.cuda.get_device_properties(dev).L2_cache_size
        copies = rotation_copies(l2, nbytes - 2 * hq * D * 2)
        caches = [(kc.to(dev), vc.to(dev)) for _ in range(copies)]
        out = torch.empty_like(dq)
        calls = [lambda c=c: gqa.decode_heads(dq, c[0], c[1], out=out) for c in caches]
        ms, p05, p95 = sweep_time(_graph(calls).replay, calls=copies)
        calls[0]()
        torch.cuda.synchronize()
        err = np.abs(out[0].double().cpu().numpy() - oracle.decode(q[0], kc[0], vc[0]))
        tput = nbytes / (ms * 1e-3) / 1e9
        line = {"workload": "decode_heads", "hq": hq, "hkv": hkv, "L": n, "ms": ms,
                "ms_p05": p05, "ms_p95": p95, "gbs": tput,
                "frac_of_measured_hbm": tput / peaks["hbm_gbs"], "cache_copies": copies}
        del caches
    line.update({"max_abs_err": float(err.max()), "mean_abs_err": float(err.mean()),
                 "parity_ok": bool(err.max() <= 2e-2 and err.mean() <= 2e-3), "peaks": src})
    if gqa.device_error() != 0:
        raise RuntimeError("device-side wait timed out")
    return line


def sweep_batch(kind, shape, dev, peaks, src):
    """Throughput and parity of a packed prefill batch or a batched decode."""
    import numpy as np
    import torch
    import gqa_flash_attention_causal_gb300 as gqa
    import oracle
    from gqa_flash_attention_causal_gb300.inputs import normal_bf16

    def med_time(fn):
        t = sweep_time(fn)
        stats.update({"ms_p05": t[1], "ms_p95": t[2]})
        return t[0]

    stats = {}

    if kind == "varlen":
        lens = list(shape)
        total = sum(lens)
        q = normal_bf16((total, HQ, D), 1)
        k = normal_bf16((total, HKV, D), 2)
        v = normal_bf16((total, HKV, D), 3)
        cu = torch.tensor([0] + np.cumsum(lens).tolist(), dtype=torch.int32, device=dev)
        dq, dk, dv = q.to(dev), k.to(dev), v.to(dev)
        out = torch.empty_like(dq)
        ms = med_time(lambda: gqa.prefill_varlen(dq, dk, dv, cu, max(lens), out=out))
        errs = []
        for s_, n in enumerate(lens):
            a = int(cu[s_])
            rows = sorted({0, n - 1, n // 2})
            want = oracle.prefill_rows(q[a:a + n], k[a:a + n], v[a:a + n], rows)
            errs.append(np.abs(out[a:a + n][rows].double().cpu().numpy() - want))
        err = np.concatenate([e.ravel() for e in errs])
        flops = sum(prefill_flops(n) for n in lens)
        tput = flops / (ms * 1e-3) / 1e12
        line = {"workload": "prefill_varlen", "lengths": lens, "ms": ms, "tflops": tput,
                "frac_of_burst": tput / peaks["bf16_tflops"]}
    else:
        B, Lmax = shape
        q = normal_bf16((B, HQ, D), 1)
        kc = normal_bf16((B, Lmax, HKV, D), 2)
        vc = normal_bf16((B, Lmax, HKV, D), 3)
        dq, dk, dv = q.to(dev), kc.to(dev), vc.to(dev)
        sl = torch.full((B,), Lmax, dtype=torch.int32, device=dev)
        out = torch.empty_like(dq)
        ms = med_time(lambda: gqa.decode_batched(dq, dk, dv, sl, out=out))
        errs = [np.abs(out[b].double().cpu().numpy() - oracle.decode(q[b], kc[b], vc[b]))
                for b in (0, B - 1)]
        err = np.concatenate([e.ravel() for e in errs])
        nbytes = B * decode_bytes(Lmax)
        tput = nbytes / (ms * 1e-3) / 1e9
        line = {"workload": "decode_batched", "batch": B, "L": Lmax, "ms": ms, "gbs": tput,
                "frac_of_measured_hbm": tput / peaks["hbm_gbs"],
                "frac_of_8tbs": tput / NOMINAL_HBM_GBS,
                "note": "eager calls; the batch's caches exceed L2"}
    line.update(stats)
    line.update({"max_abs_err": float(err.max()), "mean_abs_err": float(err.mean()),
                 "parity_ok": bool(err.max() <= 2e-2 and err.mean() <= 2e-3), "peaks": src})
    if gqa.device_error() != 0:
        raise RuntimeError("device-side wait timed out")
    return line


def run_sweep(args):
    """One JSON line per configuration of the pages' Result table (plus the
    S=512 and stress cases): GPU time, throughput, fraction of roofline,
    error against the fp64 oracle on sampled rows, and the oracle's own time
    on this host (measured on the sampled rows, scaled by FLOPs)."""
    import numpy as np
    import torch
    import gqa_flash_attention_causal_gb300 as gqa
    import oracle
    from gqa_flash_attention_causal_gb300.inputs import decode_inputs, prefill_inputs
    peaks, src = load_peaks()
    dev = torch.device("cuda")
    gqa.lib()
    rng = np.random.default_rng(0)

    cases = [("prefill", S, False) for S in (512, 2048, 4096, 8192, 16384, 32768)]
    cases += [("prefill", 4096, True)]
    cases += [("prefill_full", S, False) for S in (4096, 16384)]
    cases += [("prefill_pair", S, False) for S in (4096, 16384, 32768)]
    cases += [("decode", L, False) for L in (2048, 4096, 8192, 16384, 32768, 65536)]
    cases += [("decode", 32768, True)]
    cases += [("varlen", (4096,) * 8, False), ("varlen", (8192, 4096, 2048, 1024, 512, 256), False)]
    cases += [("batched", (8, 8192), False), ("batched", (32, 4096), False),
              ("batched", (128, 2048), False)]
    cases += [("heads", ("prefill", 64, 8, 8192), False), ("heads", ("prefill", 32, 32, 8192), False),
              ("heads", ("decode", 64, 8, 32768), False), ("heads", ("decode", 32, 32, 16384), False),
              ("heads", ("decode", 128, 8, 32768), False)]
    # ragged sizes (a partial last 128-row tile / 64-key stage): tails at full speed?
    cases += [("prefill", 12345, False), ("decode", 50001, False)]
    for kind, n, stress in cases:
        if kind == "heads":
            print(json.dumps(sweep_heads(*n, dev, peaks, src)), flush=True)
            continue
        if kind in ("varlen", "batched"):
            print(json.dumps(sweep_batch(kind, n, dev, peaks, src)), flush=True)
            continue
        if kind.startswith("prefill"):
            causal = kind != "prefill_full"
            fn = gqa.prefill_pair if kind == "prefill_pair" else gqa.prefill
            q, k, v = prefill_inputs(n, stress=stress)
            dq, dk, dv = q.to(dev), k.to(dev), v.to(dev)
            out = torch.empty_like(dq)
            call = lambda: fn(dq, dk, dv, causal=causal, out=out)  # noqa: E731
            ms_eager = sweep_time(call)[0]
            # GPU time per call: a CUDA graph of back-to-back calls (at small
            # S a single eager call is dominated by the host-side launch path)
            reps = max(1, min(200, int(2.0 / max(ms_eager, 1e-3))))
            side = torch.cuda.Stream()
            side.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(side):
                call()
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=side):
                    for _ in range(reps):
                        call()
            torch.cuda.current_stream().wait_stream(side)
            ms, p05, p95 = sweep_time(g.replay, calls=reps)
            call()
            rows = sorted({0, 1, n - 1, n // 2} | set(rng.integers(0, n, 30).tolist()))
            t0 = time.perf_counter()
            want = oracle.prefill_rows(q, k, v, rows, causal=causal)
            t_or = time.perf_counter() - t0
            got = out[0, rows].double().cpu().numpy()
            got_bits = out[0, rows].cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
            if causal:
                sample_flops = sum(4.0 * HQ * D * (r + 1) for r in rows)
                oracle_ms = 1e3 * t_or * (2.0 * HQ * D * n * (n + 1)) / sample_flops
                tput = prefill_flops(n) / (ms * 1e-3) / 1e12
            else:
                oracle_ms = 1e3 * t_or * n / len(rows)
                tput = 2.0 * prefill_flops(n) / (ms * 1e-3) / 1e12  # 4*S^2*H*D
            line = {"workload": kind, "S": n, "stress": stress, "ms": ms, "ms_p05": p05,
                    "ms_p95": p95, "ms_eager_call": ms_eager, "graph_reps": reps, "tflops": tput,
                    "frac_of_burst": tput / peaks["bf16_tflops"],
                    "frac_of_sustained": tput / peaks["bf16_tflops_sustained"]}
        else:
            q, kc, vc = decode_inputs(n, stress=stress)
            dq = q.to(dev)
            l2 = torch.cuda.get_device_properties(dev).L2_cache_size
            copies = rotation_copies(l2, 4 * kc.numel())
            caches = [(kc.to(dev), vc.to(dev)) for _ in range(copies)]
            ws = torch.empty(gqa.decode_workspace_bytes(n), dtype=torch.uint8, device=dev)
            out = torch.empty_like(dq)
            side = torch.cuda.Stream()
            side.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(side):
                gqa.decode(dq, *caches[0], out=out, workspace=ws)
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=side):
                    for c in caches:
                        gqa.decode(dq, *c, out=out, workspace=ws)
            torch.cuda.current_stream().wait_stream(side)
            ms, p05, p95 = sweep_time(g.replay, calls=copies)
            gqa.decode(dq, *caches[0], out=out, workspace=ws)
            t0 = time.perf_counter()
            want = oracle.decode(q, kc, vc)
            oracle_ms = 1e3 * (time.perf_counter() - t0)
            got = out.double().cpu().numpy().reshape(want.shape)
            got_bits = out.cpu().contiguous().view(torch.int16).numpy().view(
                np.uint16).reshape(want.shape)
            tput = decode_bytes(n) / (ms * 1e-3) / 1e9
            line = {"workload": "decode", "L": n, "stress": stress, "ms": ms, "ms_p05": p05,
                    "ms_p95": p95, "gbs": tput,
                    "frac_of_measured_hbm": tput / peaks["hbm_gbs"],
                    "frac_of_8tbs": tput / NOMINAL_HBM_GBS, "cache_copies": copies}
            del caches
        torch.cuda.synchronize()
        err = np.abs(got - want)
        scale = float(v.float().abs().max()) if kind.startswith("prefill") and stress else (
            float(vc.float().abs().max()) if stress else 1.0)
        if (kind == "prefill" and n % 128) or (kind == "decode" and n % 64):
            line["workload"] += "_tail"
        line.update({"max_abs_err": float(err.max()), "mean_abs_err": float(err.mean()),
                     "tolerance_scale": scale,
                     "parity_ok": bool(err.max() <= 2e-2 * scale and err.mean() <= 2e-3 * scale),
                     "ulp": ulp_summary(got_bits, want),
                     "oracle_ms_est": oracle_ms, "oracle_cores": oracle.max_threads(),
                     "peaks": src})
        print(json.dumps(line), flush=True)
        if gqa.device_error() != 0:
            raise RuntimeError("device-side wait timed out")
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__,
                                 formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--ref-seconds", type=float, default=12.0,
                    help="CPU seconds of oracle work for the baseline (at most, per step)")
    ap.add_argument("--ref-total", type=float, default=150.0,
                    help="CPU seconds the whole reference arm should take")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--sustain-s", type=float, default=3.0,
                    help="seconds of back-to-back steps for the sustained figure (0: skip)")
    ap.add_argument("--sweep", action="store_true",
                    help="instead of the step, print one line per configuration of the "
                         "pages' Result table (time, throughput, roofline, parity)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    world, rank, local = dist_env()
    if args.sweep:
        return run_sweep(args)
    if args.impl == "reference":
        # rank 0 alone times the oracle; other ranks exit without work
        if rank != 0:
            return 0
        print(json.dumps(run_reference(args, world)))
        return 0
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    try:
        line = run_ours(args, world, rank, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            if dist.is_initialized():
                dist.destroy_process_group()
    if line is not None:
        print(json.dumps(line))
    return 0


if __name__ == "__main__":
    sys.exit(main())
