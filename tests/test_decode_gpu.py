"""Decode (split-KV + log-sum-exp combine) against the fp64 oracle."""
import numpy as np
import pytest
import torch

import gqa_flash_attention_causal_gb300 as gqa
import oracle
from gqa_flash_attention_causal_gb300.inputs import decode_inputs
from tests.parity import assert_close, poisoned, tolerance_scale

pytestmark = pytest.mark.gpu

# the pages' decode sizes (2K..64K), tails around the 64-key stage and the
# chunk boundaries, and the degenerate L=1
LENGTHS = [1, 2, 7, 63, 64, 65, 127, 255, 1000, 2048, 4096, 4097, 8192,
           16384, 32768, 65535, 65536]


def run(L, stress=False, ws=False):
    q, kc, vc = decode_inputs(L, stress=stress)
    dq, dk, dv = q.cuda(), kc.cuda(), vc.cuda()
    out = poisoned((1, 1, 32, 128))
    workspace = None
    if ws:
        workspace = torch.empty(gqa.decode_workspace_bytes(L), dtype=torch.uint8, device="cuda")
    gqa.decode(dq, dk, dv, out=out, workspace=workspace)
    torch.cuda.synchronize()
    assert gqa.device_error() == 0
    return (q, kc, vc), out


@pytest.mark.parametrize("L", LENGTHS)
def test_decode_matches_oracle(L):
    (q, kc, vc), out = run(L)
    want = oracle.decode(q, kc, vc)
    assert_close(out, want, what=f"decode L={L}")


def test_decode_stress_l32768():
    (q, kc, vc), out = run(32768, stress=True)
    want = oracle.decode(q, kc, vc)
    assert_close(out, want, scale=tolerance_scale(vc, True), what="decode stress")


@pytest.mark.parametrize("L", [100, 8192])
def test_decode_caller_workspace(L):
    (q, kc, vc), out = run(L, ws=True)
    assert_close(out, oracle.decode(q, kc, vc), what=f"decode ws L={L}")


def test_split_plan_uses_every_sm():
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for L in (2048, 16384, 65536):
        n = gqa.decode_num_splits(L)
        assert 1 <= n <= (L + 63) // 64
        if L >= 16384:
            assert n * 8 >= sms, (L, n)


def test_decode_permutation_invariance():
    L = 4097
    q, kc, vc = decode_inputs(L)
    perm = torch.randperm(L, generator=torch.Generator().manual_seed(5))
    a = gqa.decode(q.cuda(), kc.cuda(), vc.cuda())
    b = gqa.decode(q.cuda(), kc[:, perm].contiguous().cuda(), vc[:, perm].contiguous().cuda())
    torch.cuda.synchronize()
    d = (a.double() - b.double()).abs()
    assert float(d.max()) <= 2e-2 and float(d.mean()) <= 2e-3


def test_decode_gqa_packing_identical_heads():
    """All 4 query heads of a group given the same q must give identical bits."""
    L = 3000
    q, kc, vc = decode_inputs(L)
    q = q.view(1, 1, 8, 4, 128)[:, :, :, :1].expand(1, 1, 8, 4, 128).reshape(1, 1, 32, 128)
    out = gqa.decode(q.contiguous().cuda(), kc.cuda(), vc.cuda()).view(8, 4, 128)
    torch.cuda.synchronize()
    for j in range(1, 4):
        assert torch.equal(out[:, 0], out[:, j])


def test_decode_constant_v():
    L = 5000
    q, kc, _ = decode_inputs(L, stress=True)
    const = torch.randn(1, 1, 8, 128).to(torch.bfloat16)
    vc = const.expand(1, L, 8, 128).contiguous()
    out = gqa.decode(q.cuda(), kc.cuda(), vc.cuda())
    torch.cuda.synchronize()
    want = const.repeat_interleave(4, dim=2).view(1, 1, 32, 128)
    d = (out.cpu().double() - want.double()).abs()
    assert float(d.max()) <= 2e-2 * float(const.abs().max())


def test_decode_deterministic():
    L = 20000
    q, kc, vc = decode_inputs(L)
    dq, dk, dv = q.cuda(), kc.cuda(), vc.cuda()
    a = gqa.decode(dq, dk, dv)
    b = gqa.decode(dq, dk, dv)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_decode_large_cache():
    """L = 2^20: each cache spans 2 GiB, so chunk offsets past 2^31 bytes
    must be computed in 64 bits."""
    (q, kc, vc), out = run(1 << 20)
    assert_close(out, oracle.decode(q, kc, vc), what="L=2^20")
