"""Other head layouts (query heads a multiple of KV heads) against the fp64
oracle: multi-head (Hkv = Hq), multi-query (Hkv = 1), every decode
group from 1 to 8 plus 9, 12 and 16, single sequences and packed batches."""
import numpy as np
import pytest
import torch

import gqa_flash_attention_causal_gb300 as gqa
import oracle
from gqa_flash_attention_causal_gb300.inputs import normal_bf16
from tests.parity import assert_close, poisoned, tile_rows

pytestmark = pytest.mark.gpu

# (query heads, KV heads)
PREFILL_LAYOUTS = [(32, 8), (64, 8), (32, 32), (16, 1), (28, 4), (14, 2), (7, 7), (40, 5)]
DECODE_LAYOUTS = [(32, 8), (64, 8), (32, 32), (8, 1), (28, 4), (16, 8), (12, 4), (48, 8),
                  (10, 2), (16, 4), (64, 16), (128, 8), (16, 1), (36, 3), (9, 1)]


def qkv(S, hq, hkv, seed=21):
    return (normal_bf16((1, S, hq, 128), seed), normal_bf16((1, S, hkv, 128), seed + 1),
            normal_bf16((1, S, hkv, 128), seed + 2))


@pytest.mark.parametrize("hq,hkv", PREFILL_LAYOUTS)
@pytest.mark.parametrize("causal", [True, False])
def test_prefill_heads_full(hq, hkv, causal):
    S = 300
    q, k, v = qkv(S, hq, hkv)
    out = poisoned((1, S, hq, 128))
    _, lse = gqa.prefill_heads(q.cuda(), k.cuda(), v.cuda(), causal=causal, out=out,
                               return_lse=True)
    torch.cuda.synchronize()
    assert gqa.device_error() == 0
    want, want_lse = oracle.prefill(q, k, v, causal=causal, with_lse=True)
    assert_close(out, want[None], what=f"prefill {hq}/{hkv} causal={causal}")
    got_lse = lse.cpu().numpy().T  # [S, hq]
    assert np.all(np.abs(got_lse - want_lse) <= 1e-3 + 1e-5 * np.abs(want_lse))


def test_prefill_heads_32_8_is_the_default_path():
    S = 777
    q, k, v = qkv(S, 32, 8, seed=5)
    dq, dk, dv = q.cuda(), k.cuda(), v.cuda()
    a = gqa.prefill(dq, dk, dv)
    b = gqa.prefill_heads(dq, dk, dv)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


@pytest.mark.parametrize("hq,hkv", [(64, 8), (16, 1), (28, 4)])
def test_prefill_heads_packed_sampled(hq, hkv):
    lens = [1500, 1, 700, 2049]
    total = sum(lens)
    q = normal_bf16((total, hq, 128), 31)
    k = normal_bf16((total, hkv, 128), 32)
    v = normal_bf16((total, hkv, 128), 33)
    cu = torch.tensor([0] + np.cumsum(lens).tolist(), dtype=torch.int32, device="cuda")
    out = poisoned((total, hq, 128))
    gqa.prefill_heads(q.cuda(), k.cuda(), v.cuda(), cu, max(lens), out=out)
    torch.cuda.synchronize()
    assert gqa.device_error() == 0
    for s, n in enumerate(lens):
        a = int(cu[s])
        # every 128-row tile of every sequence, all heads
        rows = sorted({0, n - 1, n // 2, min(n - 1, 127), min(n - 1, 256)} | set(tile_rows(n, s)))
        want = oracle.prefill_rows(q[a:a + n], k[a:a + n], v[a:a + n], rows, causal=True)
        assert_close(out[a:a + n][rows], want, what=f"packed {hq}/{hkv} seq {s}")


@pytest.mark.parametrize("hq,hkv", DECODE_LAYOUTS)
def test_decode_heads(hq, hkv):
    B, Lmax = 3, 5000
    lens = [5000, 1, 2345]
    q = normal_bf16((B, hq, 128), 41)
    kc = normal_bf16((B, Lmax, hkv, 128), 42)
    vc = normal_bf16((B, Lmax, hkv, 128), 43)
    sl = torch.tensor(lens, dtype=torch.int32, device="cuda")
    out = poisoned((B, hq, 128))
    _, lse = gqa.decode_heads(q.cuda(), kc.cuda(), vc.cuda(), sl, out=out, return_lse=True)
    torch.cuda.synchronize()
    assert gqa.device_error() == 0
    for b, L in enumerate(lens):
        want, want_lse = oracle.decode(q[b], kc[b, :L], vc[b, :L], with_lse=True)
        assert_close(out[b].cpu(), want, what=f"decode {hq}/{hkv} seq {b} L={L}")
        got = lse[b].cpu().numpy()
        assert np.all(np.abs(got - want_lse) <= 1e-3 + 1e-5 * np.abs(want_lse))


def test_decode_heads_32_8_is_the_default_path():
    L = 9000
    q = normal_bf16((1, 32, 128), 51)
    kc = normal_bf16((1, L, 8, 128), 52)
    vc = normal_bf16((1, L, 8, 128), 53)
    a = gqa.decode(q.view(1, 1, 32, 128).cuda(), kc.view(1, L, 8, 128).cuda(),
                   vc.view(1, L, 8, 128).cuda())
    b = gqa.decode_heads(q.cuda(), kc.cuda(), vc.cuda())
    torch.cuda.synchronize()
    assert torch.equal(a.view(1, 32, 128), b)


def test_heads_rejects_unsupported_layouts():
    q = torch.zeros((1, 8, 32, 128), dtype=torch.bfloat16, device="cuda")
    k = torch.zeros((1, 8, 5, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(gqa.GqaError) as e:  # 32 is not a multiple of 5
        gqa.prefill_heads(q, k, k)
    assert e.value.code == 3
    qd = torch.zeros((1, 32, 128), dtype=torch.bfloat16, device="cuda")
    kd = torch.zeros((1, 64, 1, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(gqa.GqaError) as e:  # 32 query heads per KV head: decode holds 16
        gqa.decode_heads(qd, kd, kd)
    assert e.value.code == 3


@pytest.mark.parametrize("hq,hkv,S", [(256, 8, 200), (256, 256, 130)])
def test_prefill_heads_at_the_head_limit(hq, hkv, S):
    """256 query heads, the most the entry point takes (groups of 32 and 1)."""
    q, k, v = qkv(S, hq, hkv, seed=61)
    out = poisoned((1, S, hq, 128))
    gqa.prefill_heads(q.cuda(), k.cuda(), v.cuda(), out=out)
    torch.cuda.synchronize()
    assert gqa.device_error() == 0
    rows = sorted({0, S // 2, S - 1} | set(tile_rows(S)))
    assert_close(out[0, rows], oracle.prefill_rows(q, k, v, rows), what=f"prefill {hq}/{hkv}")


def test_decode_heads_at_the_head_limit():
    """256 query heads over 32 KV heads: the largest layout with groups of 8."""
    hq, hkv, L = 256, 32, 3000
    q = normal_bf16((2, hq, 128), 71)
    kc = normal_bf16((2, L, hkv, 128), 72)
    vc = normal_bf16((2, L, hkv, 128), 73)
    sl = torch.tensor([L, 1234], dtype=torch.int32, device="cuda")
    out = poisoned((2, hq, 128))
    gqa.decode_heads(q.cuda(), kc.cuda(), vc.cuda(), sl, out=out)
    torch.cuda.synchronize()
    assert gqa.device_error() == 0
    for b, n in enumerate((L, 1234)):
        assert_close(out[b].cpu(), oracle.decode(q[b], kc[b, :n], vc[b, :n]), what=f"seq {b}")
