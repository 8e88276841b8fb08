"""Failure detection on the GPU without a fault: a bounded device wait that
is made to run out must report GQA_ERR_TIMEOUT through the device error
word and leave the context usable for the next call."""
import ctypes

import pytest
import torch

import gqa_flash_attention_causal_gb300 as gqa
import oracle
from gqa_flash_attention_causal_gb300.inputs import decode_inputs
from tests.parity import assert_close

pytestmark = pytest.mark.gpu


def test_expired_wait_is_reported_and_context_survives():
    flags = ctypes.c_uint(0)
    st = gqa.lib().gqa_attn_selftest_wait_timeout(ctypes.byref(flags))
    assert st == 6, gqa.STATUS.get(st)
    assert flags.value == 1 << 31
    assert gqa.device_error() == 0          # cleared by the self-test
    q, kc, vc = decode_inputs(3000)
    out = gqa.decode(q.cuda(), kc.cuda(), vc.cuda())
    torch.cuda.synchronize()
    assert gqa.device_error() == 0
    assert_close(out, oracle.decode(q, kc, vc), what="decode after an expired wait")


def test_decode_ws_captures_in_a_cuda_graph():
    L = 20000
    q, kc, vc = (t.cuda() for t in decode_inputs(L))
    ws = torch.empty(gqa.decode_workspace_bytes(L), dtype=torch.uint8, device="cuda")
    eager = gqa.decode(q, kc, vc, workspace=ws)
    out = torch.empty_like(eager)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            gqa.decode(q, kc, vc, out=out, workspace=ws)
    torch.cuda.current_stream().wait_stream(s)
    out.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, eager)
