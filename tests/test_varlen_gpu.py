"""Packed variable-length prefill (batch > 1) against the fp64 oracle, one
sequence at a time."""
import numpy as np
import pytest
import torch

import gqa_flash_attention_causal_gb300 as gqa
import oracle
from gqa_flash_attention_causal_gb300.inputs import normal_bf16, prefill_inputs
from tests.parity import assert_close, sample_rows, tile_rows

pytestmark = pytest.mark.gpu


def packed(lengths, seed=7, stress=False):
    total = sum(lengths)
    mq, mv = (8.0, 100.0) if stress else (1.0, 1.0)
    q = normal_bf16((total, 32, 128), seed, mq)
    k = normal_bf16((total, 8, 128), seed + 1, mq)
    v = normal_bf16((total, 8, 128), seed + 2, mv)
    cu = torch.tensor([0] + list(np.cumsum(lengths)), dtype=torch.int32)
    return q, k, v, cu


def run(q, k, v, cu, max_len, causal=True, lse=False):
    out = torch.full((q.shape[0], 32, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    res = gqa.prefill_varlen(q.cuda(), k.cuda(), v.cuda(), cu.cuda(), max_len, causal=causal,
                             out=out, return_lse=lse)
    torch.cuda.synchronize()
    return res


@pytest.mark.parametrize("causal", [True, False])
def test_varlen_matches_oracle_per_sequence(causal):
    lengths = [1, 129, 700, 1000, 3, 256, 0, 300]
    q, k, v, cu = packed(lengths)
    out, lse = run(q, k, v, cu, max(lengths), causal=causal, lse=True)
    assert gqa.device_error() == 0
    for s, n in enumerate(lengths):
        a, b = int(cu[s]), int(cu[s + 1])
        if n == 0:
            continue
        want, want_lse = oracle.prefill(q[a:b], k[a:b], v[a:b], causal=causal, with_lse=True)
        assert_close(out[a:b].cpu(), want, what=f"seq {s} (len {n})")
        got_lse = lse[:, a:b].cpu().numpy().T
        assert np.all(np.abs(got_lse - want_lse) <= 1e-3 + 1e-5 * np.abs(want_lse))


def test_varlen_single_sequence_equals_dense_prefill():
    S = 3001
    q, k, v = prefill_inputs(S)
    dense = gqa.prefill(q.cuda(), k.cuda(), v.cuda())
    cu = torch.tensor([0, S], dtype=torch.int32)
    var = run(q[0], k[0], v[0], cu, S)
    assert torch.equal(dense[0], var)


def test_varlen_long_mixed_batch_sampled():
    lengths = [4096, 300, 2048, 17, 5000]
    q, k, v, cu = packed(lengths, seed=21, stress=True)
    out = run(q, k, v, cu, max(lengths))
    assert gqa.device_error() == 0
    for s, n in enumerate(lengths):
        a = int(cu[s])
        # every 128-row tile of every sequence (compact item order)
        rows = sorted(set(sample_rows(n, n_random=8, seed=s)) | set(tile_rows(n, seed=s)))
        want = oracle.prefill_rows(q[a:a + n], k[a:a + n], v[a:a + n], rows)
        scale = float(v[a:a + n].float().abs().max())
        assert_close(out[a:a + n][rows].cpu(), want, scale=scale, what=f"seq {s}")


def test_varlen_sequence_longer_than_max_is_flagged_not_computed():
    lengths = [100, 2000, 100]
    q, k, v, cu = packed(lengths, seed=31)
    out = run(q, k, v, cu, 1000)   # the middle sequence exceeds max_seqlen's blocks
    flags = gqa.device_error()
    assert flags & (1 << 5)
    for s in (0, 2):
        a, b = int(cu[s]), int(cu[s + 1])
        assert_close(out[a:b].cpu(), oracle.prefill(q[a:b], k[a:b], v[a:b]), what=f"seq {s}")
    assert bool(torch.isnan(out[100:2100].float()).all())  # untouched


def test_varlen_rejects_bad_host_arguments():
    q, k, v, cu = packed([10, 20])
    with pytest.raises(TypeError):
        gqa.prefill_varlen(q.cuda(), k.cuda(), v.cuda(), cu.cuda().long(), 20)
    with pytest.raises(gqa.GqaError):
        gqa.prefill_varlen(q.cuda(), k.cuda(), v.cuda(), cu.cuda(), 0)


def _check_sequences(q, k, v, cu, lengths, out, which, n_rows=3):
    for s in which:
        n = lengths[s]
        if n == 0:
            continue
        a = int(cu[s])
        rows = sorted({0, n - 1, n // 2} | set(range(min(n, n_rows))))
        want = oracle.prefill_rows(q[a:a + n], k[a:a + n], v[a:a + n], rows)
        assert_close(out[a:a + n][rows].cpu(), want, what=f"seq {s} (len {n})")


def test_varlen_uniform_batch_plain_order():
    """Every sequence at max_seqlen: the plain item order (no empty blocks)."""
    lengths = [700] * 5
    q, k, v, cu = packed(lengths, seed=41)
    out = run(q, k, v, cu, 700)
    assert gqa.device_error() == 0
    _check_sequences(q, k, v, cu, lengths, out, range(5))


@pytest.mark.parametrize("n_seq", [64, 70])
def test_varlen_many_mixed_sequences(n_seq):
    """64 mixed-length sequences use the compact item order (the largest batch
    it takes), 70 the plain order with empty items."""
    rng = np.random.default_rng(n_seq)
    lengths = [int(x) for x in rng.integers(1, 700, n_seq)]
    lengths[n_seq // 2] = 1500  # one long sequence: many blocks empty for the rest
    q, k, v, cu = packed(lengths, seed=n_seq)
    out = run(q, k, v, cu, max(lengths))
    assert gqa.device_error() == 0
    assert bool(torch.isfinite(out.float()).all())
    _check_sequences(q, k, v, cu, lengths, out, [0, 1, n_seq // 2, n_seq - 2, n_seq - 1])


@pytest.mark.parametrize("seed", range(6))
def test_varlen_random_batches(seed):
    """Random mixed batches (2-64 sequences, lengths 0-1000, causal or not,
    max_seqlen sometimes above the longest sequence): every sequence's
    sampled rows against the oracle, and no row left unwritten."""
    rng = np.random.default_rng(100 + seed)
    n_seq = int(rng.integers(2, 65))
    lengths = [int(x) for x in rng.integers(0, 1001, n_seq)]
    if sum(lengths) == 0:
        lengths[0] = 5
    causal = bool(seed % 2 == 0)
    max_len = max(lengths) + (int(rng.integers(1, 400)) if seed % 3 == 0 else 0)
    q, k, v, cu = packed(lengths, seed=200 + seed)
    out = run(q, k, v, cu, max_len, causal=causal)
    assert gqa.device_error() == 0
    assert bool(torch.isfinite(out.float()).all())
    for s, n in enumerate(lengths):
        if n == 0:
            continue
        a = int(cu[s])
        rows = sorted({0, n - 1, int(rng.integers(0, n))})
        want = oracle.prefill_rows(q[a:a + n], k[a:a + n], v[a:a + n], rows, causal=causal)
        assert_close(out[a:a + n][rows].cpu(), want, what=f"seq {s} (len {n})")
