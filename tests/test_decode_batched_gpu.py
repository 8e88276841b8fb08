"""Batched decode (per-sequence cache lengths) against the fp64 oracle."""
import numpy as np
import pytest
import torch

import gqa_flash_attention_causal_gb300 as gqa
import oracle
from gqa_flash_attention_causal_gb300.inputs import decode_inputs, normal_bf16
from tests.parity import assert_close, poisoned

pytestmark = pytest.mark.gpu


def batch_inputs(B, Lmax, seed=3, stress=False):
    mq, mv = (8.0, 100.0) if stress else (1.0, 1.0)
    q = normal_bf16((B, 32, 128), seed, mq)
    kc = normal_bf16((B, Lmax, 8, 128), seed + 1, mq)
    vc = normal_bf16((B, Lmax, 8, 128), seed + 2, mv)
    return q, kc, vc


def run(q, kc, vc, lens, lse=False):
    out = poisoned(tuple(q.shape))
    sl = None if lens is None else torch.tensor(lens, dtype=torch.int32, device="cuda")
    res = gqa.decode_batched(q.cuda(), kc.cuda(), vc.cuda(), sl, out=out, return_lse=lse)
    torch.cuda.synchronize()
    return res


@pytest.mark.parametrize("B,Lmax,lens", [
    (4, 5000, [1, 777, 5000, 4097]),
    (64, 2048, "random"),
    (3, 65536, [65536, 100, 32768]),
])
def test_batched_matches_oracle(B, Lmax, lens):
    if lens == "random":
        lens = np.random.default_rng(1).integers(1, Lmax + 1, B).tolist()
    q, kc, vc = batch_inputs(B, Lmax)
    out, lse = run(q, kc, vc, lens, lse=True)
    assert gqa.device_error() == 0
    for b, L in enumerate(lens):
        want, want_lse = oracle.decode(q[b], kc[b, :L], vc[b, :L], with_lse=True)
        assert_close(out[b].cpu(), want, what=f"seq {b} L={L}")
        assert np.all(np.abs(lse[b].cpu().numpy() - want_lse) <= 1e-3 + 1e-5 * np.abs(want_lse))


def test_batched_full_length_and_stress():
    B, Lmax = 2, 3000
    q, kc, vc = batch_inputs(B, Lmax, stress=True)
    out = run(q, kc, vc, None)
    for b in range(B):
        scale = float(vc[b].float().abs().max())
        assert_close(out[b].cpu(), oracle.decode(q[b], kc[b], vc[b]), scale=scale,
                     what=f"stress seq {b}")


def test_batch_of_one_equals_decode():
    L = 9000
    q, kc, vc = decode_inputs(L)
    single = gqa.decode(q.cuda(), kc.cuda(), vc.cuda())
    batched = run(q[0], kc, vc, [L])
    assert torch.equal(single[0], batched)


def test_bad_length_is_flagged_and_left_untouched():
    B, Lmax = 3, 1000
    q, kc, vc = batch_inputs(B, Lmax, seed=9)
    out = run(q, kc, vc, [500, 0, 1001])
    assert gqa.device_error() & (1 << 5)
    assert_close(out[0].cpu(), oracle.decode(q[0], kc[0, :500], vc[0, :500]), what="seq 0")
    assert bool(torch.isnan(out[1:].float()).all())
