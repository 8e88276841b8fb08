"""Run the library once on synthetic inputs and report CUDA-event times.

    python -m gqa_flash_attention_causal_gb300.run --prefill 16384 --decode 65536 --iters 3

Each requested call runs `--iters` times back to back on the current stream
(the first is a warm-up); the median of the rest is printed together with
TFLOP/s (prefill, causal FLOPs 2*S^2*H*D) or GB/s (decode, 2*L*8*128*2 bytes
plus q and out).  Handy as the target of a profiler run.
"""
from __future__ import annotations

import argparse
import statistics

import torch

from . import decode, decode_workspace_bytes, prefill, prefill_pair
from .inputs import decode_inputs, prefill_inputs


def _time(fn, iters):
    times = []
    for _ in range(iters):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        fn()
        b.record()
        torch.cuda.synchronize()
        times.append(a.elapsed_time(b))
    return statistics.median(times[1:] if len(times) > 1 else times)


def _time_graph(fn, reps, iters):
    """Median time of one call, from a CUDA graph of `reps` back-to-back calls
    (removes host launch gaps)."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()  # warm-up outside capture (first-call set-up)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for _ in range(reps):
                fn()
    torch.cuda.current_stream().wait_stream(s)
    times = []
    for _ in range(iters):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        g.replay()
        b.record()
        torch.cuda.synchronize()
        times.append(a.elapsed_time(b) / reps)
    return statistics.median(times[1:] if len(times) > 1 else times)


def _host_us(fn, n=200):
    """Host time of one call (enqueue only), microseconds."""
    import time
    fn()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(n):
        fn()
    t1 = time.perf_counter()
    torch.cuda.synchronize()
    return (t1 - t0) / n * 1e6


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--prefill", type=int, default=0, help="prompt length S (0 = skip)")
    ap.add_argument("--non-causal", action="store_true")
    ap.add_argument("--pair", action="store_true",
                    help="prefill with the paired-CTA kernel (gqa_attn_prefill_pair)")
    ap.add_argument("--decode", type=int, default=0, help="KV cache length L (0 = skip)")
    ap.add_argument("--iters", type=int, default=3)
    ap.add_argument("--graph", type=int, default=0,
                    help="also time decode as a CUDA graph of this many back-to-back calls")
    ap.add_argument("--host", action="store_true", help="also report host time per call")
    args = ap.parse_args(argv)
    dev = torch.device("cuda")
    if args.prefill:
        S = args.prefill
        q, k, v = (t.to(dev) for t in prefill_inputs(S))
        out = torch.empty_like(q)
        fn = prefill_pair if args.pair else prefill
        ms = _time(lambda: fn(q, k, v, causal=not args.non_causal, out=out), args.iters)
        flops = (2.0 if not args.non_causal else 4.0) * S * S * 32 * 128
        print(f"prefill{'_pair' if args.pair else ''} S={S} causal={not args.non_causal}: {ms:.4f} ms, "
              f"{flops / ms / 1e9:.1f} TFLOP/s")
    if args.decode:
        L = args.decode
        q, kc, vc = (t.to(dev) for t in decode_inputs(L))
        out = torch.empty_like(q)
        ms = _time(lambda: decode(q, kc, vc, out=out), args.iters)
        nbytes = 2.0 * L * 8 * 128 * 2 + 2 * 32 * 128 * 2
        line = f"decode L={L}: {ms * 1e3:.2f} us, {nbytes / ms / 1e6:.1f} GB/s"
        if args.graph:
            # rotate through enough cache copies that they cannot stay in L2:
            # the other copies stream 6x the L2 size between two reads of one
            # (2x still left some launches reading part of their cache from L2)
            l2 = torch.cuda.get_device_properties(dev).L2_cache_size
            copies = max(1, -(-6 * l2 // (kc.numel() * 4)) + 1)
            caches = [(kc, vc)] + [(kc.clone(), vc.clone()) for _ in range(copies - 1)]
            ws = torch.empty(decode_workspace_bytes(L), dtype=torch.uint8, device=dev)
            calls = [lambda c=c: decode(q, c[0], c[1], out=out, workspace=ws) for c in caches]
            reps = max(args.graph, copies)
            gms = _time_graph(lambda: [calls[i % copies]() for i in range(reps)], 1,
                              max(args.iters, 3)) / reps
            line += (f"; graph ({copies} cache copies) {gms * 1e3:.2f} us, "
                     f"{nbytes / gms / 1e6:.1f} GB/s")
        if args.host:
            line += f"; host {_host_us(lambda: decode(q, kc, vc, out=out)):.1f} us/call"
        print(line)


if __name__ == "__main__":
    main()
