"""Parity at the bench's full sizes, in the launch configuration bench.py
times: one CUDA graph replaying the causal prefill at S=32768, one replaying
the decode at L=65536 with a caller workspace.  The prefill is compared with
the oracle on the first, the last and a random row of every 128-row query
tile (768 rows, all heads), the decode in full."""
import numpy as np
import pytest
import torch

import gqa_flash_attention_causal_gb300 as gqa
import oracle
from gqa_flash_attention_causal_gb300.inputs import decode_inputs, prefill_inputs
from tests.parity import assert_close, covered_tiles, sample_rows, tile_rows

pytestmark = pytest.mark.gpu


def test_bench_step_graph_replay_matches_oracle():
    S, L = 32768, 65536
    q, k, v = prefill_inputs(S)
    dq, kc, vc = decode_inputs(L)
    d_q, d_k, d_v, d_dq, d_kc, d_vc = (t.cuda() for t in (q, k, v, dq, kc, vc))
    out = torch.full_like(d_q, float("nan"))
    dout = torch.full_like(d_dq, float("nan"))
    ws = torch.empty(gqa.decode_workspace_bytes(L), dtype=torch.uint8, device="cuda")
    gqa.prefill(d_q, d_k, d_v, out=out)
    gqa.decode(d_dq, d_kc, d_vc, out=dout, workspace=ws)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        g_pre, g_dec = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_pre, stream=side):
            gqa.prefill(d_q, d_k, d_v, out=out)
        with torch.cuda.graph(g_dec, stream=side):
            gqa.decode(d_dq, d_kc, d_vc, out=dout, workspace=ws)
    torch.cuda.current_stream().wait_stream(side)
    out.fill_(float("nan"))
    dout.fill_(float("nan"))
    for _ in range(2):
        g_pre.replay()
        g_dec.replay()
    torch.cuda.synchronize()
    assert gqa.device_error() == 0
    assert bool(torch.isfinite(out.float()).all())
    rows = sorted(set(sample_rows(S, n_random=16, seed=3)) | set(tile_rows(S, seed=3)))
    assert covered_tiles(rows, S) == S // 128
    assert_close(out[0, rows], oracle.prefill_rows(q, k, v, rows), what="bench prefill")
    assert_close(dout, oracle.decode(dq, kc, vc), what="bench decode")
