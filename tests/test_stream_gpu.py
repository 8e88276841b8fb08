"""Calls without a stream argument run on torch's current stream: captured
inside torch.cuda.graph (whose capture stream is then current), they must be
recorded into the graph and reproduce the eager result on replay."""
import pytest
import torch

import gqa_flash_attention_causal_gb300 as gqa
from gqa_flash_attention_causal_gb300.inputs import decode_inputs, prefill_inputs

pytestmark = pytest.mark.gpu


def _capture_and_compare(call, out):
    call()
    torch.cuda.synchronize()
    want = out.clone()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    out.fill_(float("nan"))
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    assert gqa.device_error() == 0
    assert torch.equal(out, want)


def test_prefill_uses_current_stream():
    q, k, v = (t.cuda() for t in prefill_inputs(1000))
    out = torch.empty_like(q)
    _capture_and_compare(lambda: gqa.prefill(q, k, v, out=out), out)


def test_decode_uses_current_stream():
    q, kc, vc = (t.cuda() for t in decode_inputs(5000))
    out = torch.empty_like(q)
    ws = torch.empty(gqa.decode_workspace_bytes(5000), dtype=torch.uint8, device="cuda")
    _capture_and_compare(lambda: gqa.decode(q, kc, vc, out=out, workspace=ws), out)


def test_explicit_stream_is_used():
    q, kc, vc = (t.cuda() for t in decode_inputs(3000))
    out = torch.empty_like(q)
    ws = torch.empty(gqa.decode_workspace_bytes(3000), dtype=torch.uint8, device="cuda")
    gqa.decode(q, kc, vc, out=out, workspace=ws)
    torch.cuda.synchronize()
    want = out.clone()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    # capture on `side` while it is current, but pass it explicitly too
    with torch.cuda.graph(g, stream=side):
        gqa.decode(q, kc, vc, out=out, workspace=ws, stream=side)
    out.fill_(float("nan"))
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, want)


def test_prefill_pair_uses_current_stream():
    """The paired-CTA prefill (a cluster launch) captures into a graph too;
    its first call, which sets up the per-device launch attributes, runs
    before the capture."""
    q, k, v = (t.cuda() for t in prefill_inputs(1000))
    out = torch.empty_like(q)
    _capture_and_compare(lambda: gqa.prefill_pair(q, k, v, out=out), out)


def test_prefill_pair_then_prefill_on_one_stream():
    """A paired prefill followed by a single-CTA prefill on the same stream
    (each a programmatic dependent of the one before): both outputs equal."""
    q, k, v = (t.cuda() for t in prefill_inputs(2500))
    a, b = torch.empty_like(q), torch.empty_like(q)
    for _ in range(3):
        gqa.prefill_pair(q, k, v, out=a)
        gqa.prefill(q, k, v, out=b)
    torch.cuda.synchronize()
    assert gqa.device_error() == 0
    assert torch.equal(a, b)


_TWO_THREADS = r"""
import sys, threading
sys.path.insert(0, sys.argv[1])
import torch
import gqa_flash_attention_causal_gb300 as gqa
from gqa_flash_attention_causal_gb300.inputs import decode_inputs, prefill_inputs
q, k, v = (t.cuda() for t in prefill_inputs(1500))
dq, kc, vc = (t.cuda() for t in decode_inputs(3000))
torch.cuda.synchronize()
results, errors = {}, []
start = threading.Barrier(2)

def worker(i):
    try:
        s = torch.cuda.Stream()
        ws = torch.empty(gqa.decode_workspace_bytes(3000), dtype=torch.uint8, device="cuda")
        with torch.cuda.stream(s):
            start.wait()  # both threads make the process's first library calls together
            outs = [(gqa.prefill(q, k, v), gqa.decode(dq, kc, vc, workspace=ws),
                     gqa.prefill_pair(q, k, v)) for _ in range(3)]
        s.synchronize()
        results[i] = outs
    except Exception as e:
        errors.append(repr(e))

threads = [threading.Thread(target=worker, args=(i,)) for i in range(2)]
for t in threads:
    t.start()
for t in threads:
    t.join(timeout=120)
assert not errors, errors
assert gqa.device_error() == 0
want_p, want_d = gqa.prefill(q, k, v), gqa.decode(dq, kc, vc)
torch.cuda.synchronize()
for outs in results.values():
    for p, d, pp in outs:
        assert torch.equal(p, want_p) and torch.equal(d, want_d) and torch.equal(pp, want_p)
print("two-thread first calls ok")
"""


def test_first_calls_from_two_host_threads():
    """Two host threads of a fresh process make its first library calls at
    the same moment, each on its own stream (prefill needs no workspace; each
    decode passes its own): the per-device launch set-up (kernel attributes,
    cluster occupancy) runs once, and every result is right."""
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", _TWO_THREADS, root], capture_output=True,
                       text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "two-thread first calls ok" in r.stdout
