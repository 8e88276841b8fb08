"""Pins of the fp64 oracle to facts outside itself.

Each ``pin_*`` function takes an ``oracle.OracleLib`` and raises
``AssertionError`` if the oracle disagrees with brute force, a closed form or
an invariant of softmax attention.  ``test_oracle.py`` runs them on the real
oracle; ``test_oracle_mutants.py`` runs them on builds with planted mistakes
and requires each mistake to trip at least one pin.

The attention being pinned is the one the chowfi/kernels README describes
("Result" section): grouped-query attention forward, query head h reading KV
head h // (Hq/Hkv), softmax scale 1/sqrt(D), causal prefill (query i sees keys
0..i) and decode of one query against every cached position.
"""
from __future__ import annotations

import math

import numpy as np
import torch

from gqa_flash_attention_causal_gb300.inputs import normal_bf16

TOL = 1e-12


def _qkv(S, hq, hkv, d, seed=11, mag_qk=1.0, mag_v=1.0):
    q = normal_bf16((S, hq, d), seed, mag_qk)
    k = normal_bf16((S, hkv, d), seed + 1, mag_qk)
    v = normal_bf16((S, hkv, d), seed + 2, mag_v)
    return q, k, v


def _bf(x) -> torch.Tensor:
    return torch.as_tensor(x, dtype=torch.float32).to(torch.bfloat16)


def brute_force(q, k, v, causal):
    """Independent pure-Python fp64 attention with math.fsum, tiny shapes only.

    Values come from torch's own bf16->float conversion, not the oracle's.
    """
    qf, kf, vf = (t.float().tolist() for t in (q, k, v))
    n_q, hq, d = len(qf), len(qf[0]), len(qf[0][0])
    n_kv, hkv = len(kf), len(kf[0])
    group = hq // hkv
    out = np.zeros((n_q, hq, d))
    lse = np.zeros((n_q, hq))
    for i in range(n_q):
        keys = list(range(i + 1)) if causal else list(range(n_kv))
        for h in range(hq):
            g = h // group
            s = [math.fsum(qf[i][h][c] * kf[j][g][c] for c in range(d)) / math.sqrt(d)
                 for j in keys]
            top = max(s)
            e = [math.exp(x - top) for x in s]
            z = math.fsum(e)
            lse[i, h] = top + math.log(z)
            for c in range(d):
                out[i, h, c] = math.fsum(e[t] * vf[j][g][c] for t, j in enumerate(keys)) / z
    return out, lse


def _close(a, b, tol=TOL, what=""):
    a, b = np.asarray(a), np.asarray(b)
    assert a.shape == b.shape, f"{what}: shape {a.shape} != {b.shape}"
    assert np.all(np.isfinite(a)), f"{what}: non-finite values"
    err = float(np.max(np.abs(a - b))) if a.size else 0.0
    assert err <= tol, f"{what}: max abs diff {err:.3e} > {tol:.1e}"


def pin_brute_force(orc):
    for (S, hq, hkv, d) in ((6, 32, 8, 128), (9, 4, 1, 16), (5, 8, 8, 8)):
        q, k, v = _qkv(S, hq, hkv, d, seed=100 + S)
        for causal in (True, False):
            want, want_lse = brute_force(q, k, v, causal)
            got, got_lse = orc.prefill(q, k, v, causal=causal, with_lse=True)
            _close(got, want, what=f"prefill S={S} hq={hq} causal={causal}")
            _close(got_lse, want_lse, what="lse")
    L = 11
    q = normal_bf16((1, 32, 128), 7)
    kc = normal_bf16((L, 8, 128), 8)
    vc = normal_bf16((L, 8, 128), 9)
    want, want_lse = brute_force(q, kc, vc, causal=False)
    got, got_lse = orc.decode(q, kc, vc, with_lse=True)
    _close(got, want[0], what="decode L=11")
    _close(got_lse, want_lse[0], what="decode lse")


def pin_weights_are_probabilities(orc):
    S, hq, hkv, d = 40, 32, 8, 128
    q, k, v = _qkv(S, hq, hkv, d, seed=21, mag_qk=3.0)
    for causal in (True, False):
        for (i, h) in ((0, 0), (1, 5), (17, 31), (39, 12)):
            w, _ = orc.weights(q, k, v, i, h, causal=causal)
            assert w.size == (i + 1 if causal else S)
            assert np.all(w >= 0.0), "negative softmax weight"
            assert abs(math.fsum(w.tolist()) - 1.0) <= TOL, "weights do not sum to 1"


def pin_gqa_equals_repeated_mha(orc):
    """Grouped heads == plain multi-head attention with K/V repeated per group
    (Llama-style repeat_interleave along the head dim): identical bits."""
    S, hq, hkv, d = 33, 32, 8, 128
    q, k, v = _qkv(S, hq, hkv, d, seed=31)
    rk = k.repeat_interleave(hq // hkv, dim=1)
    rv = v.repeat_interleave(hq // hkv, dim=1)
    for causal in (True, False):
        a = orc.prefill(q, k, v, causal=causal)
        b = orc.prefill(q, rk, rv, causal=causal)
        assert np.array_equal(a, b), "GQA differs from MHA with repeated K/V"
    qd = normal_bf16((1, hq, d), 35)
    a = orc.decode(qd, k, v)
    b = orc.decode(qd, rk, rv)
    assert np.array_equal(a, b), "decode GQA differs from repeated MHA"


def pin_constant_v(orc):
    S, hq, hkv, d = 29, 32, 8, 128
    q, k, _ = _qkv(S, hq, hkv, d, seed=41, mag_qk=4.0)
    const = normal_bf16((1, hkv, d), 44)
    v = const.expand(S, hkv, d).contiguous()
    want = const.double().repeat_interleave(hq // hkv, dim=1).numpy()
    for causal in (True, False):
        out = orc.prefill(q, k, v, causal=causal)
        _close(out, np.broadcast_to(want, out.shape), tol=1e-13 * 8,
               what="constant V")


def pin_decode_permutation_invariance(orc):
    L, hq, hkv, d = 300, 32, 8, 128
    q = normal_bf16((1, hq, d), 51)
    kc = normal_bf16((L, hkv, d), 52)
    vc = normal_bf16((L, hkv, d), 53)
    perm = torch.randperm(L, generator=torch.Generator().manual_seed(54))
    a = orc.decode(q, kc, vc)
    b = orc.decode(q, kc[perm].contiguous(), vc[perm].contiguous())
    _close(a, b, what="decode under a joint KV permutation")


def pin_causal_row0_is_v0(orc):
    S, hq, hkv, d = 17, 32, 8, 128
    q, k, v = _qkv(S, hq, hkv, d, seed=61, mag_qk=8.0, mag_v=100.0)
    out = orc.prefill(q, k, v, causal=True)
    want = v[0].double().repeat_interleave(hq // hkv, dim=0).numpy()
    assert np.array_equal(out[0], want), "causal row 0 is not v[0]"


def pin_zero_query_means(orc):
    """q = 0 makes every score 0: row i is the plain mean of the visible v rows."""
    S, hq, hkv, d = 23, 32, 8, 128
    _, k, v = _qkv(S, hq, hkv, d, seed=71)
    q = torch.zeros((S, hq, d), dtype=torch.bfloat16)
    vv = v.double().numpy()
    causal = orc.prefill(q, k, v, causal=True)
    full = orc.prefill(q, k, v, causal=False)
    for i in range(S):
        for h in range(hq):
            g = h // (hq // hkv)
            _close(causal[i, h], vv[: i + 1, g].mean(axis=0), what="causal mean")
            _close(full[i, h], vv[:, g].mean(axis=0), what="full mean")


def pin_two_key_sigmoid(orc):
    """Two keys with scores 0 and a*b/sqrt(128): the second key's weight is the
    logistic function of the score gap, which fixes the softmax scale."""
    d, hq, hkv = 128, 4, 1
    a = [1.0, 2.0, -3.0, 0.5]
    b = 4.0
    q = torch.zeros((2, hq, d))
    for h in range(hq):
        q[1, h, 0] = a[h]
    k = torch.zeros((2, hkv, d))
    k[1, 0, 0] = b
    v = torch.zeros((2, hkv, d))
    v[0, 0, :] = -1.0
    v[1, 0, :] = 3.0
    out = orc.prefill(_bf(q), _bf(k), _bf(v), causal=True)
    for h in range(hq):
        p = 1.0 / (1.0 + math.exp(-a[h] * b / math.sqrt(128.0)))
        _close(out[1, h], np.full(d, -1.0 + 4.0 * p), tol=1e-14, what="sigmoid")
        _close(out[0, h], np.full(d, -1.0), tol=0.0, what="row 0")


def pin_prefill_rows_match_decode(orc):
    """Causal prefill row i == decode of q[i] against the first i+1 positions;
    non-causal row i == decode against all S; S=1 prefill == decode at L=1."""
    S, hq, hkv, d = 37, 32, 8, 128
    q, k, v = _qkv(S, hq, hkv, d, seed=81, mag_qk=2.0)
    causal = orc.prefill(q, k, v, causal=True)
    full = orc.prefill(q, k, v, causal=False)
    for i in (0, 1, 18, 36):
        dec = orc.decode(q[i], k[: i + 1].contiguous(), v[: i + 1].contiguous())
        _close(causal[i], dec, what=f"causal row {i} vs decode")
        _close(full[i], orc.decode(q[i], k, v), what=f"full row {i} vs decode")
    one = orc.prefill(q[:1], k[:1], v[:1], causal=True)
    _close(one[0], orc.decode(q[0], k[:1], v[:1]), tol=0.0, what="S=1")


def pin_rows_subset(orc):
    S, hq, hkv, d = 31, 32, 8, 128
    q, k, v = _qkv(S, hq, hkv, d, seed=91)
    rows = [30, 0, 7, 7, 15]
    for causal in (True, False):
        full = orc.prefill(q, k, v, causal=causal)
        part = orc.prefill_rows(q, k, v, rows, causal=causal)
        assert np.array_equal(part, full[rows]), "row subset differs"


def pin_extreme_scores_one_hot(orc):
    """Scores far apart (q.k of order 2^40) make the softmax one-hot: the
    output is exactly the V row of the largest score, with no overflow."""
    S, hq, hkv, d = 6, 4, 1, 128
    big = 2.0 ** 20
    q = torch.zeros((S, hq, d))
    k = torch.zeros((S, hkv, d))
    q[:, :, 0] = big
    for j in range(S):
        k[j, 0, 0] = big * (1.0 if j != 3 else 2.0) * (j + 1) / 8.0
    v = normal_bf16((S, hkv, d), 95)
    out = orc.prefill(_bf(q), _bf(k), v, causal=False)
    # the score of key j grows with (j+1), key 3 doubled: key 5 (6/8) < key 3 (8/8)
    want = v[3, 0].double().numpy()
    for i in range(S):
        for h in range(hq):
            assert np.array_equal(out[i, h], want), "not one-hot at key 3"


def pin_stress_convex_hull(orc):
    """Attention output is a convex combination of visible V rows: it lies in
    their per-coordinate range, also at stress magnitudes (q,k x8, v x100)."""
    S, hq, hkv, d = 64, 32, 8, 128
    q, k, v = _qkv(S, hq, hkv, d, seed=97, mag_qk=8.0, mag_v=100.0)
    out = orc.prefill(q, k, v, causal=True)
    vv = v.double().numpy()
    for i in (0, 5, 63):
        for h in range(hq):
            g = h // (hq // hkv)
            lo = vv[: i + 1, g].min(axis=0) - 1e-9
            hi = vv[: i + 1, g].max(axis=0) + 1e-9
            assert np.all((out[i, h] >= lo) & (out[i, h] <= hi)), "outside hull"


ALL_PINS = [
    pin_brute_force,
    pin_weights_are_probabilities,
    pin_gqa_equals_repeated_mha,
    pin_constant_v,
    pin_decode_permutation_invariance,
    pin_causal_row0_is_v0,
    pin_zero_query_means,
    pin_two_key_sigmoid,
    pin_prefill_rows_match_decode,
    pin_rows_subset,
    pin_extreme_scores_one_hot,
    pin_stress_convex_hull,
]
