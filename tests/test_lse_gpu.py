"""Log-sum-exp export (prefill and decode) against the fp64 oracle's lse."""
import numpy as np
import pytest
import torch

import gqa_flash_attention_causal_gb300 as gqa
import oracle
from gqa_flash_attention_causal_gb300.inputs import decode_inputs, prefill_inputs
from tests.parity import assert_close, sample_rows, tile_rows

pytestmark = pytest.mark.gpu


def _lse_close(got, want, what):
    # fp32 score sums from exact bf16 products: ~1e-6 relative
    err = np.abs(got - want)
    bound = 1e-3 + 1e-5 * np.abs(want)
    assert np.all(np.isfinite(got)), what
    assert np.all(err <= bound), f"{what}: max lse err {err.max():.3e}"


@pytest.mark.parametrize("S,causal,stress", [(1, True, False), (129, True, False),
                                             (1000, True, False), (700, False, False),
                                             (2048, True, True)])
def test_prefill_lse_full(S, causal, stress):
    q, k, v = prefill_inputs(S, stress=stress)
    out, lse = gqa.prefill(q.cuda(), k.cuda(), v.cuda(), causal=causal, return_lse=True)
    torch.cuda.synchronize()
    assert gqa.device_error() == 0
    want, want_lse = oracle.prefill(q, k, v, causal=causal, with_lse=True)
    scale = float(v.float().abs().max()) if stress else 1.0
    assert_close(out, want[None], scale=scale, what="out with lse")
    _lse_close(lse[0].cpu().numpy().T, want_lse, f"prefill lse S={S}")


def test_prefill_lse_sampled_16k():
    S = 16384
    q, k, v = prefill_inputs(S)
    _, lse = gqa.prefill(q.cuda(), k.cuda(), v.cuda(), return_lse=True)
    torch.cuda.synchronize()
    rows = sorted(set(sample_rows(S)) | set(tile_rows(S, seed=9)))  # every 128-row tile
    _, want_lse = oracle.prefill_rows(q, k, v, rows, with_lse=True)
    _lse_close(lse[0].cpu().numpy().T[rows], want_lse, "prefill lse sampled")


@pytest.mark.parametrize("L,stress", [(1, False), (1000, False), (65536, False), (32768, True)])
def test_decode_lse(L, stress):
    q, kc, vc = decode_inputs(L, stress=stress)
    out, lse = gqa.decode(q.cuda(), kc.cuda(), vc.cuda(), return_lse=True)
    torch.cuda.synchronize()
    want, want_lse = oracle.decode(q, kc, vc, with_lse=True)
    scale = float(vc.float().abs().max()) if stress else 1.0
    assert_close(out, want, scale=scale, what="decode out with lse")
    _lse_close(lse[0].cpu().numpy(), want_lse, f"decode lse L={L}")


def test_lse_merge_of_two_key_ranges():
    """The exported lse lets two decodes over disjoint halves of the cache be
    merged into the decode over the whole cache (the use it exists for)."""
    L = 6000
    q, kc, vc = (t.cuda() for t in decode_inputs(L))
    full = gqa.decode(q, kc, vc).double()
    o1, l1 = gqa.decode(q, kc[:, :2500].contiguous(), vc[:, :2500].contiguous(), return_lse=True)
    o2, l2 = gqa.decode(q, kc[:, 2500:].contiguous(), vc[:, 2500:].contiguous(), return_lse=True)
    m = torch.maximum(l1, l2)
    w1, w2 = torch.exp(l1 - m), torch.exp(l2 - m)
    merged = (o1.double()[0, 0] * w1[0, :, None] + o2.double()[0, 0] * w2[0, :, None]) / \
        (w1 + w2)[0, :, None]
    assert float((merged - full[0, 0]).abs().max()) <= 2e-2
