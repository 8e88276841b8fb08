"""The C-ABI library: exports and host-side argument validation (CPU), and
validation errors that need a device (GPU)."""
import ctypes
import os
import re

import pytest

import gqa_flash_attention_causal_gb300 as gqa

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "gqa_attn.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gqa_attn_\w+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    from gqa_flash_attention_causal_gb300 import _build
    _build.build()
    return gqa.lib()


def test_header_matches_binding():
    assert declared_functions() == sorted(gqa.SIGNATURES)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for code in gqa.STATUS:
        assert lib.gqa_attn_status_string(code)
    assert lib.gqa_attn_status_string(99) == b"unknown status"


def test_null_pointers_rejected_without_device(lib):
    p = ctypes.c_void_p(4096)
    assert lib.gqa_attn_prefill(None, p, p, p, 16, 1, None) == 1
    assert lib.gqa_attn_prefill(p, p, p, None, 16, 1, None) == 1
    assert lib.gqa_attn_decode(p, None, p, p, 16, None) == 1


def test_misaligned_pointers_rejected_without_device(lib):
    p, bad = ctypes.c_void_p(4096), ctypes.c_void_p(4096 + 2)
    assert lib.gqa_attn_prefill(p, bad, p, p, 16, 1, None) == 2
    assert lib.gqa_attn_decode(p, p, p, bad, 16, None) == 2


def test_bad_lengths_rejected_without_device(lib):
    p = ctypes.c_void_p(4096)
    for S in (0, -5, (1 << 20) + 1):
        assert lib.gqa_attn_prefill(p, p, p, p, S, 1, None) == 3
    for L in (0, -1, (1 << 26) + 1):
        assert lib.gqa_attn_decode(p, p, p, p, L, None) == 3
    assert lib.gqa_attn_decode_workspace_bytes(0) == 0
    assert lib.gqa_attn_decode_num_splits(-3) == 0


def test_bad_head_counts_rejected_without_device(lib):
    p = ctypes.c_void_p(4096)
    # (query heads, KV heads): not a multiple, zero, more KV than query heads, > 256
    for hq, hkv in ((32, 5), (32, 0), (8, 16), (512, 8), (0, 0), (-8, -4)):
        assert lib.gqa_attn_prefill_heads(p, p, p, p, None, None, 1, 64, 64, hq, hkv, 1,
                                          None) == 3, (hq, hkv)
        assert lib.gqa_attn_decode_heads(p, p, p, p, None, None, 1, 64, hq, hkv,
                                         None) == 3, (hq, hkv)
    # decode holds at most 16 query heads per KV head
    for hq, hkv in ((64, 2), (32, 1), (136, 8)):
        assert lib.gqa_attn_decode_heads(p, p, p, p, None, None, 1, 64, hq, hkv, None) == 3
    # a single sequence (no cu_seqlens) must have batch 1 and max_seqlen == total
    assert lib.gqa_attn_prefill_heads(p, p, p, p, None, None, 2, 64, 128, 32, 8, 1, None) == 3
    assert lib.gqa_attn_prefill_heads(p, p, p, p, None, None, 1, 64, 65, 32, 8, 1, None) == 3


def test_launch_counts(lib):
    assert lib.gqa_attn_launches_per_call(0) == 1
    assert lib.gqa_attn_launches_per_call(1) == 2


@pytest.mark.gpu
def test_host_memory_rejected(lib):
    import torch
    dev = torch.zeros((1, 16, 32, 128), dtype=torch.bfloat16, device="cuda")
    kv = torch.zeros((1, 16, 8, 128), dtype=torch.bfloat16, device="cuda")
    host = torch.zeros((1, 16, 8, 128), dtype=torch.bfloat16)
    st = lib.gqa_attn_prefill(dev.data_ptr(), host.data_ptr(), kv.data_ptr(),
                              dev.data_ptr(), 16, 1, None)
    assert st == 8


@pytest.mark.gpu
def test_python_wrapper_checks():
    import torch
    q = torch.zeros((1, 16, 32, 128), dtype=torch.bfloat16, device="cuda")
    kv = torch.zeros((1, 16, 8, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ValueError):
        gqa.prefill(q, kv[:, :8], kv)
    with pytest.raises(TypeError):
        gqa.prefill(q.float(), kv, kv)
    with pytest.raises(ValueError):
        gqa.prefill(q, kv.transpose(1, 2).contiguous().transpose(1, 2), kv)


@pytest.mark.gpu
def test_workspace_too_small(lib):
    import torch
    q = torch.zeros((1, 1, 32, 128), dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros((1, 4096, 8, 128), dtype=torch.bfloat16, device="cuda")
    need = gqa.decode_workspace_bytes(4096)
    assert need > 0
    ws = torch.empty(need // 2, dtype=torch.uint8, device="cuda")
    with pytest.raises(gqa.GqaError) as e:
        gqa.decode(q, kc, kc, workspace=ws)
    assert e.value.code == 5


@pytest.mark.parametrize("sms", [152, 148, 132, 8, 1])
def test_decode_plan_invariants(lib, sms):
    """The split plan covers every key exactly once, in 64-key multiples,
    and uses at most one wave of (split, KV head, sequence) CTAs."""
    for batch in (1, 2, 7, 19, 64, 1000):
        for L in (1, 2, 63, 64, 65, 1000, 2048, 4097, 16384, 65535, 65536, 1 << 20):
            n, chunk = gqa.decode_plan(L, batch, sms)
            assert chunk % 64 == 0 and chunk >= 64
            assert n >= 1 and (n - 1) * chunk < L <= n * chunk
            assert n <= (L + 63) // 64
            if sms * 1 >= 8 * batch:
                assert n * 8 * batch <= sms or n == 1
            else:
                assert n == 1
    assert gqa.decode_plan(65536, 1, 152) == (19, 3456)


def test_decode_plan_rejects_bad_arguments(lib):
    with pytest.raises(ValueError):
        gqa.decode_plan(0)
    with pytest.raises(ValueError):
        gqa.decode_plan(100, 0)
