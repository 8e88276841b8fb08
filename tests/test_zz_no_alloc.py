"""The allocation-free decode entry point, gqa_attn_decode_noalloc.

It serves callers that cannot allocate device memory (their HBM is handed to
their own pool, or they run under a fixed memory budget): its partial
results live in a fixed scratch array inside the library.  It runs the same
split plan and the same kernels as gqa_attn_decode, so through the C ABI its
output must be bit-identical to that entry point's, on consecutive calls
with different inputs and lengths (the shared scratch keeps the previous
call's partials, and none of them may leak into the next call).  One call is
also checked against the fp64 oracle.  This file is collected last so a
stop-at-first-failure run has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import gqa_flash_attention_causal_gb300 as gqa
import oracle
from gqa_flash_attention_causal_gb300.inputs import decode_inputs
from tests.parity import assert_close

pytestmark = pytest.mark.gpu


def _call(fn, q, kc, vc, out, L):
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return fn(q.data_ptr(), kc.data_ptr(), vc.data_ptr(), out.data_ptr(), L, stream)


# a long call (many chunks) followed by shorter ones, so stale partials of an
# earlier call sit in the scratch slots a later call's combine must not read
@pytest.mark.parametrize("lengths", [(1000, 777), (65536, 4097, 64)])
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
        assert bool(torch.isfinite(got.float()).all()), (call, L)
        assert torch.equal(got, want), (call, L, (got.float() - want.float()).abs().max())


def test_noalloc_matches_oracle():
    lib = gqa.lib()
    L = 3000
    q, kc, vc = decode_inputs(L, seeds=(41, 42, 43))
    got = torch.full((1, 1, 32, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    assert _call(lib.gqa_attn_decode_noalloc, q.cuda(), kc.cuda(), vc.cuda(), got, L) == 0
    torch.cuda.synchronize()
    assert gqa.device_error() == 0
    assert_close(got, oracle.decode(q, kc, vc), what=f"noalloc decode L={L}")


def test_noalloc_rejects_bad_arguments():
    lib = gqa.lib()
    q = torch.zeros((1, 1, 32, 128), dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros((1, 64, 8, 128), dtype=torch.bfloat16, device="cuda")
    for L in (0, (1 << 26) + 1):
        assert _call(lib.gqa_attn_decode_noalloc, q, kc, kc, q, L) == 3
    host = torch.zeros((1, 64, 8, 128), dtype=torch.bfloat16)
    assert _call(lib.gqa_attn_decode_noalloc, q, host, kc, q, 64) == 8
