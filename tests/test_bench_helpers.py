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
