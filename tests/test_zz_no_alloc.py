"""The allocation-free decode entry point, gqa_attn_decode_noalloc.

It serves callers that cannot allocate device memory (their HBM is handed to
their own pool, or they run under a fixed memory budget): its partial
results live in a fixed scratch array inside the library.  Through the C ABI
it must give the same result as gqa_attn_decode, within the parity
tolerance, on consecutive calls with different inputs (the shared scratch
keeps the previous call's contents, which must not leak into the next).
This file is collected last so a stop-at-first-failure run has already run
every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import gqa_flash_attention_causal_gb300 as gqa
from gqa_flash_attention_causal_gb300.inputs import decode_inputs
from tests.parity import MAX_ABS, MEAN_ABS

pytestmark = pytest.mark.gpu


def _call(fn, q, kc, vc, out, L):
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return fn(q.data_ptr(), kc.data_ptr(), vc.data_ptr(), out.data_ptr(), L, stream)


@pytest.mark.parametrize("lengths", [(1000, 777), (65536, 4097)])
def test_noalloc_matches_decode_on_consecutive_calls(lengths):
    lib = gqa.lib()
    for call, L in enumerate(lengths):
        seeds = (10 + call, 20 + call, 30 + call)
        q, kc, vc = (t.cuda() for t in decode_inputs(L, seeds=seeds))
        want = torch.full_like(q, float("nan"))
        got = torch.full_like(q, float("nan"))
        assert _call(lib.gqa_attn_decode, q, kc, vc, want, L) == 0
        assert _call(lib.gqa_attn_decode_noalloc, q, kc, vc, got, L) == 0
        torch.cuda.synchronize()
        assert gqa.device_error() == 0
        g, w = got.double().cpu().numpy(), want.double().cpu().numpy()
        assert np.all(np.isfinite(g))
        err = np.abs(g - w)
        assert err.max() <= MAX_ABS and err.mean() <= MEAN_ABS, (call, L, err.max())


def test_noalloc_rejects_bad_arguments():
    lib = gqa.lib()
    q = torch.zeros((1, 1, 32, 128), dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros((1, 64, 8, 128), dtype=torch.bfloat16, device="cuda")
    for L in (0, (1 << 26) + 1):
        assert _call(lib.gqa_attn_decode_noalloc, q, kc, kc, q, L) == 3
    host = torch.zeros((1, 64, 8, 128), dtype=torch.bfloat16)
    assert _call(lib.gqa_attn_decode_noalloc, q, host, kc, q, 64) == 8
