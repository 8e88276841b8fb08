"""Paired-CTA prefill (gqa_attn_prefill_pair: cta_group::2 MMAs over a
cluster of two CTAs, each staging half of every K/V tile) against the fp64
oracle, and against the single-CTA kernel it must agree with."""
import pytest
import torch

import gqa_flash_attention_causal_gb300 as gqa
import oracle
from gqa_flash_attention_causal_gb300.inputs import prefill_inputs
from tests.parity import assert_close, covered_tiles, poisoned, sample_rows, tile_rows

pytestmark = pytest.mark.gpu

# around the 128-row tile and the 256-row item, ragged tails, and the
# degenerate S=1
FULL = [1, 2, 127, 128, 129, 255, 256, 257, 300, 511, 512, 513, 1000]


def run(S, causal=True, stress=False, lse=False):
    q, k, v = prefill_inputs(S, stress=stress)
    out = poisoned((1, S, 32, 128))
    res = gqa.prefill_pair(q.cuda(), k.cuda(), v.cuda(), causal=causal, out=out, return_lse=lse)
    torch.cuda.synchronize()
    assert gqa.device_error() == 0
    return (q, k, v), res


@pytest.mark.parametrize("S", FULL)
def test_pair_causal_full(S):
    (q, k, v), out = run(S)
    assert_close(out, oracle.prefill(q, k, v, causal=True)[None], what=f"pair causal S={S}")


@pytest.mark.parametrize("S", [1, 300, 700])
def test_pair_noncausal_full(S):
    (q, k, v), out = run(S, causal=False)
    assert_close(out, oracle.prefill(q, k, v, causal=False)[None], what=f"pair full S={S}")


@pytest.mark.parametrize("S", [4096, 16384])
def test_pair_causal_every_tile(S):
    """The first, last and a random row of every 128-row tile, all heads:
    both CTAs (both heads of a pair) of every item."""
    (q, k, v), out = run(S)
    rows = sorted(set(sample_rows(S)) | set(tile_rows(S, seed=S + 1)))
    assert covered_tiles(rows, S) == S // 128
    assert_close(out[0, rows], oracle.prefill_rows(q, k, v, rows, causal=True),
                 what=f"pair causal S={S}")
    assert bool(torch.isfinite(out.float()).all()), "unwritten output rows"


@pytest.mark.parametrize("S,causal", [(1000, True), (3001, True), (2048, False)])
def test_pair_matches_single_cta_kernel(S, causal):
    """Each CTA of a pair computes one head of the single-CTA kernel's item:
    same rows, same KV tiles in the same order, same fp32 accumulation per
    row, so the paired kernel reproduces gqa_attn_prefill exactly."""
    q, k, v = (t.cuda() for t in prefill_inputs(S))
    a = gqa.prefill(q, k, v, causal=causal)
    b = gqa.prefill_pair(q, k, v, causal=causal)
    torch.cuda.synchronize()
    assert gqa.device_error() == 0
    assert torch.equal(a, b)


def test_pair_lse_and_stress():
    S = 2048
    (q, k, v), (out, lse) = run(S, stress=True, lse=True)
    rows = sorted(set(tile_rows(S, seed=5)))
    want, want_lse = oracle.prefill_rows(q, k, v, rows, causal=True, with_lse=True)
    assert_close(out[0, rows], want, scale=float(v.float().abs().max()), what="pair stress")
    got_lse = lse[0].cpu().double().numpy().T[rows]
    err = abs(got_lse - want_lse)
    assert (err <= 1e-3 + 1e-5 * abs(want_lse)).all(), float(err.max())


def test_pair_rejects_bad_arguments():
    q = torch.zeros((1, 128, 32, 128), dtype=torch.bfloat16, device="cuda")
    k = torch.zeros((1, 128, 8, 128), dtype=torch.bfloat16, device="cuda")
    lib = gqa.lib()
    assert lib.gqa_attn_prefill_pair(q.data_ptr(), k.data_ptr(), k.data_ptr(), q.data_ptr(),
                                     None, 0, 1, None) == 3
    assert lib.gqa_attn_prefill_pair(None, k.data_ptr(), k.data_ptr(), q.data_ptr(),
                                     None, 128, 1, None) == 1
    assert lib.gqa_attn_prefill_pair(q.data_ptr() + 2, k.data_ptr(), k.data_ptr(), q.data_ptr(),
                                     None, 128, 1, None) == 2
