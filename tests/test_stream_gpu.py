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
