"""Host-side helpers of bench.py (CPU): the parity check of the timed
outputs, the end-to-end timeline summary and the decode rotation size."""
import numpy as np
import torch

import bench
import oracle
from gqa_flash_attention_causal_gb300.inputs import normal_bf16


def _oracle_rows(S=256, L=64):
    """A small prefill and decode with their oracle results, shaped like the
    CPU baseline's (rows, prefill rows, decode) record."""
    q = normal_bf16((1, S, 32, 128), 1)
    k = normal_bf16((1, S, 8, 128), 2)
    v = normal_bf16((1, S, 8, 128), 3)
    dq = normal_bf16((1, 1, 32, 128), 4)
    kc = normal_bf16((1, L, 8, 128), 5)
    vc = normal_bf16((1, L, 8, 128), 6)
    rows = [0, 1, 127, 128, 200, S - 1]
    want_pre = oracle.prefill_rows(q, k, v, rows, causal=True)
    want_dec = oracle.decode(dq, kc, vc)
    out = torch.zeros((1, S, 32, 128), dtype=torch.bfloat16)
    out[0, rows] = torch.from_numpy(want_pre).to(torch.bfloat16)
    dout = torch.from_numpy(want_dec).to(torch.bfloat16).reshape(1, 1, 32, 128)
    return (rows, want_pre, want_dec), out, dout


def test_timed_parity_accepts_rounded_oracle(monkeypatch):
    monkeypatch.setattr(bench, "S_PREFILL", 256)
    last, out, dout = _oracle_rows()
    p = bench.timed_parity(last, out, dout)
    assert p["ok"], p
    assert p["prefill"]["rows"] == 6 and p["prefill"]["tiles_covered"] == 2
    assert p["prefill"]["max_abs"] <= 2e-2 and p["decode"]["max_abs"] <= 2e-2


def test_timed_parity_flags_a_wrong_row_and_a_nan(monkeypatch):
    monkeypatch.setattr(bench, "S_PREFILL", 256)
    last, out, dout = _oracle_rows()
    bad = out.clone()
    bad[0, 128, 5] += 0.5  # one element of one sampled row, one head
    assert not bench.timed_parity(last, bad, dout)["ok"]
    bad = dout.clone()
    bad[0, 0, 31, 127] = float("nan")
    assert not bench.timed_parity(last, out, bad)["ok"]


def test_timeline_summary():
    tl = [{"h2d": [0.0, 3.0], "kernels": [3.0, 8.0], "d2h": [8.0, 9.5]},
          {"h2d": [3.0, 6.0], "kernels": [8.1, 13.1], "d2h": [13.1, 14.6]},
          {"h2d": [8.0, 11.0], "kernels": [13.1, 18.1], "d2h": [18.1, 19.6]}]
    s = bench.timeline_summary(tl)
    assert s["steps"] == 3
    assert abs(s["mean_span_ms"]["kernels"] - 5.0) < 1e-9
    assert abs(s["kernel_idle_between_steps_ms"]["max"] - 0.1) < 1e-9
    assert s["first_steps"] == tl[:3] and s["last_steps"] == tl[-2:]
    assert bench.timeline_summary([]) is None


def test_rotation_copies_stream_six_l2_between_reuses():
    l2 = 135528448
    for L in (2048, 16384, 32768, 65536):
        cache = 4096 * L
        n = bench.rotation_copies(l2, cache)
        assert (n - 1) * cache >= 6 * l2 > (n - 2) * cache
    assert bench.rotation_copies(l2, 10 * l2) == 2


def test_bf16_rounding_from_float64_is_nearest_even():
    """bf16_rne_bits against the definition: representable values map to
    themselves, a value between two neighbours goes to the nearer, and an
    exact midpoint goes to the neighbour whose last mantissa bit is 0."""
    bits = np.arange(0x3F00, 0x4100, dtype=np.uint16)  # [0.5, 8), both parities
    a = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    nxt = ((bits.astype(np.uint32) + 1) << 16).view(np.float32).astype(np.float64)
    ulp = nxt - a
    assert np.array_equal(bench.bf16_rne_bits(a), bits)
    assert np.array_equal(bench.bf16_rne_bits(a + 0.3 * ulp), bits)
    assert np.array_equal(bench.bf16_rne_bits(a + 0.7 * ulp), bits + 1)
    even = np.where(bits % 2 == 0, bits, bits + 1).astype(np.uint16)
    assert np.array_equal(bench.bf16_rne_bits(a + 0.5 * ulp), even)
    assert np.array_equal(bench.bf16_rne_bits(-(a + 0.7 * ulp)), (bits + 1) | 0x8000)
    assert bench.bf16_rne_bits(np.array([0.0]))[0] == 0


def test_bf16_ulp_distance_orders_across_zero():
    d = bench.bf16_ulp_distance
    assert d(np.array([0x3F80]), np.array([0x3F81]))[0] == 1      # 1.0 and its neighbour
    assert d(np.array([0x0000]), np.array([0x8000]))[0] == 0      # +0 and -0
    assert d(np.array([0x0001]), np.array([0x8001]))[0] == 2      # +/- smallest step
    assert d(np.array([0xBF80]), np.array([0xBF82]))[0] == 2      # -1.0 side


def test_timed_parity_ulp_of_rounded_oracle(monkeypatch):
    """Outputs that are the oracle rounded to bf16 sit at 0 ulp (torch rounds
    through float32, which can differ from direct rounding only at ties)."""
    monkeypatch.setattr(bench, "S_PREFILL", 256)
    last, out, dout = _oracle_rows()
    u = bench.timed_parity(last, out, dout)["ulp"]
    for part in ("prefill", "decode"):
        assert u[part]["within_1"] == 1.0 and u[part]["exact"] >= 0.999, u


def test_reference_arm_line_keeps_the_contract():
    """`bench.py --impl reference` (the fp64 oracle on the host cores, a short
    bounded sample here) prints one JSON line with the reference arm's keys:
    its own cpu_baseline and an e2e object with no host<->device bytes, both
    carrying the line's value."""
    import json
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3", "--ref-seconds", "0.2",
                        "--ref-total", "2"], capture_output=True, text=True, timeout=300,
                       cwd=root)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 1 and d["steps"] == 1
    assert d["value"] > 0 and d["unit"] == "TFLOP/s" and d["higher_is_better"] is True
    assert d["metric"] and d["config"]["workload"] and d["vs_baseline"] is None
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["sample"] and cb["value"] == d["value"]
    e = d["e2e"]
    assert e["value"] == d["value"] and e["unit"] == d["unit"]
    assert e["h2d_bytes_per_step"] == 0 and e["d2h_bytes_per_step"] == 0
