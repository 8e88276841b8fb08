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

from . import decode, prefill
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


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--prefill", type=int, default=0, help="prompt length S (0 = skip)")
    ap.add_argument("--non-causal", action="store_true")
    ap.add_argument("--decode", type=int, default=0, help="KV cache length L (0 = skip)")
    ap.add_argument("--iters", type=int, default=3)
    args = ap.parse_args(argv)
    dev = torch.device("cuda")
    if args.prefill:
        S = args.prefill
        q, k, v = (t.to(dev) for t in prefill_inputs(S))
        out = torch.empty_like(q)
        ms = _time(lambda: prefill(q, k, v, causal=not args.non_causal, out=out), args.iters)
        flops = (2.0 if not args.non_causal else 4.0) * S * S * 32 * 128
        print(f"prefill S={S} causal={not args.non_causal}: {ms:.4f} ms, "
              f"{flops / ms / 1e9:.1f} TFLOP/s")
    if args.decode:
        L = args.decode
        q, kc, vc = (t.to(dev) for t in decode_inputs(L))
        out = torch.empty_like(q)
        ms = _time(lambda: decode(q, kc, vc, out=out), args.iters)
        nbytes = 2.0 * L * 8 * 128 * 2 + 2 * 32 * 128 * 2
        print(f"decode L={L}: {ms * 1e3:.2f} us, {nbytes / ms / 1e6:.1f} GB/s")


if __name__ == "__main__":
    main()
