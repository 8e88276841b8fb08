"""Decode (split-KV + log-sum-exp combine) against the fp64 oracle."""
import numpy as np
import pytest
import torch

import gqa_flash_attention_causal_gb300 as gqa
import oracle
from gqa_flash_attention_causal_gb300.inputs import decode_inputs
from tests.parity import assert_close, bf16_ulp_distance, poisoned, tolerance_scale

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
    """Every cached V row equal to c: each chunk's normalised partial is c
    times sum(bf16(p)) / sum(p), within 2^-9 of c in relative terms, and the
    log-sum-exp merge of such partials stays there, so every output element
    is c or a bf16 neighbour of c."""
    L = 5000
    q, kc, _ = decode_inputs(L, stress=True)
    const = torch.randn(1, 1, 8, 128, generator=torch.Generator().manual_seed(9)).to(
        torch.bfloat16)
    vc = const.expand(1, L, 8, 128).contiguous()
    out = gqa.decode(q.cuda(), kc.cuda(), vc.cuda())
    torch.cuda.synchronize()
    want = const.repeat_interleave(4, dim=2).view(1, 1, 32, 128)
    assert int(bf16_ulp_distance(out.cpu(), want).max()) <= 1


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


def test_decode_one_hot_at_l_2_25():
    """L = 2^25: each cache spans 64 GiB (the entry accepts up to 2^26, whose
    two caches alone would take 256 GiB of the device), too large for a host
    copy for the oracle, so the check is a property that holds at any size.
    Every key is zero except key j, which every query head matches with score
    128 * 2.125^2 / sqrt(128) ~ 51, against ln L ~ 17: all but ~1e-15 of each
    head's softmax weight falls on j, so each output head equals v[j] of its KV
    head (query head h reads KV head h // 4) exactly in bf16.  V differs by
    position, KV head and dimension, and every value is at least 2^-7 in
    magnitude (an odd multiple of 1/128 before rounding), so reading a wrong
    position or head, or truncating a 64-bit offset, changes the result.
    j is tried near the start, past the 2^31-byte offset and in the last split."""
    L = 1 << 25
    torch.cuda.empty_cache()
    kc = torch.zeros((1, L, 8, 128), dtype=torch.bfloat16, device="cuda")
    vc = torch.empty_like(kc)
    g = torch.arange(8, device="cuda", dtype=torch.float32).view(1, 8, 1)
    d = torch.arange(128, device="cuda", dtype=torch.float32).view(1, 1, 128)
    step = 1 << 20
    for r0 in range(0, L, step):
        j = torch.arange(r0, r0 + step, device="cuda", dtype=torch.int64)
        pos = ((j * 37) % 101 - 50).to(torch.float32).view(-1, 1, 1)
        vc[0, r0:r0 + step] = ((8 * pos + 32 * g + 2 * d + 1) / 128).to(torch.bfloat16)
    q = torch.full((1, 1, 32, 128), 2.125, dtype=torch.bfloat16, device="cuda")
    try:
        for jstar in (5, (1 << 24) + 12345, L - 3):
            kc[0, jstar] = 2.125
            out = gqa.decode(q, kc, vc)
            torch.cuda.synchronize()
            assert gqa.device_error() == 0
            want = vc[0, jstar].repeat_interleave(4, dim=0)
            assert torch.equal(out[0, 0], want), f"one-hot key {jstar}"
            kc[0, jstar] = 0
    finally:
        del kc, vc
        torch.cuda.empty_cache()
