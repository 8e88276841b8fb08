"""GB300 (sm_103a) grouped-query attention forward: Python binding.

The compute lives entirely in ``libgqa_attn.so`` (hand-written CUDA behind
the C ABI of ``include/gqa_attn.h``); this module only checks and marshals
torch tensors (device pointers, the current CUDA stream) and turns status
codes into exceptions.  There is no fallback: if the library is missing or
the device is not a GB300, every call raises.

Geometry (chowfi/kernels README, "Result" section): batch 1, 32 query heads
sharing 8 KV heads, head dim 128, bf16, sequence-major BSHD tensors.
"""
from __future__ import annotations

import ctypes
import os

from .inputs import HEAD_DIM, HKV, HQ

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libgqa_attn.so")

STATUS = {
    0: "GQA_OK", 1: "GQA_ERR_NULL", 2: "GQA_ERR_ALIGN", 3: "GQA_ERR_SHAPE",
    4: "GQA_ERR_DEVICE", 5: "GQA_ERR_WORKSPACE", 6: "GQA_ERR_TIMEOUT",
    7: "GQA_ERR_CUDA", 8: "GQA_ERR_POINTER",
}

# Every symbol include/gqa_attn.h declares, with its ctypes signature.
_P, _I, _S = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
SIGNATURES = {
    "gqa_attn_prefill": (_I, [_P, _P, _P, _P, _I, _I, _P]),
    "gqa_attn_prefill_lse": (_I, [_P, _P, _P, _P, _P, _I, _I, _P]),
    "gqa_attn_decode_lse": (_I, [_P, _P, _P, _P, _P, _I, _P]),
    "gqa_attn_prefill_varlen": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _P]),
    "gqa_attn_decode_batched": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _P]),
    "gqa_attn_prefill_heads": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P]),
    "gqa_attn_decode_heads": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _P]),
    "gqa_attn_prefill_pair": (_I, [_P, _P, _P, _P, _P, _I, _I, _P]),
    "gqa_attn_decode": (_I, [_P, _P, _P, _P, _I, _P]),
    "gqa_attn_decode_workspace_bytes": (_S, [_I]),
    "gqa_attn_decode_ws": (_I, [_P, _P, _P, _P, _I, _P, _S, _P]),
    "gqa_attn_decode_noalloc": (_I, [_P, _P, _P, _P, _I, _P]),
    "gqa_attn_decode_num_splits": (_I, [_I]),
    "gqa_attn_decode_plan": (_I, [_I, _I, _I, ctypes.POINTER(_I), ctypes.POINTER(_I)]),
    "gqa_attn_launches_per_call": (_I, [_I]),
    "gqa_attn_device_error": (_I, [ctypes.POINTER(ctypes.c_uint), _I]),
    "gqa_attn_status_string": (ctypes.c_char_p, [_I]),
    "gqa_attn_last_error_string": (ctypes.c_char_p, []),
    "gqa_attn_selftest_wait_timeout": (_I, [ctypes.POINTER(ctypes.c_uint)]),
}

_lib = None


class GqaError(RuntimeError):
    """A non-OK status from the C ABI."""

    def __init__(self, fn: str, code: int):
        self.code = code
        msg = lib().gqa_attn_status_string(code).decode()
        if code == 7:
            detail = lib().gqa_attn_last_error_string().decode()
            if detail:
                msg += f"; {detail}"
        super().__init__(f"{fn}: {STATUS.get(code, code)} ({msg})")


def lib():
    """The loaded C-ABI library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with "
                "`python -c 'import __graft_entry__ as g; g.build()'`")
        l = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            f = getattr(l, name)
            f.restype, f.argtypes = res, args
        _lib = l
    return _lib


def _check(fn: str, code: int):
    if code != 0:
        raise GqaError(fn, code)


_torch_refs = None


def _refs():
    """(torch, torch.bfloat16, raw current-stream getter, current-device
    getter), looked up once: every call goes through here."""
    global _torch_refs
    if _torch_refs is None:
        import torch
        _torch_refs = (torch, torch.bfloat16,
                       getattr(torch._C, "_cuda_getCurrentRawStream", None),
                       getattr(torch._C, "_cuda_getDevice", None))
    return _torch_refs


def _stream(stream):
    """cudaStream_t (as an int) of `stream`, default torch's current stream
    on the current device."""
    if stream is not None:
        return stream.cuda_stream
    torch, _, raw_stream, cur_dev = _refs()
    if raw_stream is not None and cur_dev is not None:
        return raw_stream(cur_dev())
    return torch.cuda.current_stream().cuda_stream


def _expect(t, shape, name):
    torch, bf16 = _refs()[:2]
    try:  # the common case in one expression; the checks below name the failure
        if t.dtype is bf16 and t.is_cuda and t.shape == shape and t.is_contiguous():
            return
    except AttributeError:
        pass
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != torch.bfloat16:
        raise TypeError(f"{name} must be bf16, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def prefill(q, k, v, causal: bool = True, out=None, stream=None, return_lse: bool = False):
    """Attention over a whole prompt: q [1,S,32,128], k/v [1,S,8,128] bf16.

    Returns ``out`` [1,S,32,128] bf16 (allocated if not given), enqueued on
    ``stream`` (default: torch's current stream).  With ``return_lse`` it
    returns ``(out, lse)``, lse [1,32,S] fp32 = ln sum_j exp(score_ij).
    """
    import torch
    S = q.shape[1]
    _expect(q, (1, S, HQ, HEAD_DIM), "q")
    _expect(k, (1, S, HKV, HEAD_DIM), "k")
    _expect(v, (1, S, HKV, HEAD_DIM), "v")
    if out is None:
        out = torch.empty_like(q)
    _expect(out, (1, S, HQ, HEAD_DIM), "out")
    if return_lse:
        lse = torch.empty((1, HQ, S), dtype=torch.float32, device=q.device)
        _check("gqa_attn_prefill_lse", lib().gqa_attn_prefill_lse(
            q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(), S,
            1 if causal else 0, _stream(stream)))
        return out, lse
    _check("gqa_attn_prefill", lib().gqa_attn_prefill(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), S,
        1 if causal else 0, _stream(stream)))
    return out


def prefill_pair(q, k, v, causal: bool = True, out=None, stream=None,
                 return_lse: bool = False):
    """``prefill`` computed by the paired-CTA kernel (two CTAs per TPC share
    every K/V tile through cta_group::2 MMAs).  Same arguments and result."""
    import torch
    S = q.shape[1]
    _expect(q, (1, S, HQ, HEAD_DIM), "q")
    _expect(k, (1, S, HKV, HEAD_DIM), "k")
    _expect(v, (1, S, HKV, HEAD_DIM), "v")
    if out is None:
        out = torch.empty_like(q)
    _expect(out, (1, S, HQ, HEAD_DIM), "out")
    lse = torch.empty((1, HQ, S), dtype=torch.float32, device=q.device) if return_lse else None
    _check("gqa_attn_prefill_pair", lib().gqa_attn_prefill_pair(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
        lse.data_ptr() if lse is not None else None, S, 1 if causal else 0, _stream(stream)))
    return (out, lse) if return_lse else out


def prefill_varlen(q, k, v, cu_seqlens, max_seqlen: int, causal: bool = True, out=None,
                   stream=None, return_lse: bool = False):
    """Prefill of sequences packed along dim 0: q [total,32,128], k/v
    [total,8,128] bf16; sequence s is rows cu_seqlens[s]:cu_seqlens[s+1]
    (int32 CUDA tensor of batch+1 offsets).  Returns out [total,32,128] (and
    lse [32,total] fp32 with ``return_lse``)."""
    import torch
    total = q.shape[0]
    _expect(q, (total, HQ, HEAD_DIM), "q")
    _expect(k, (total, HKV, HEAD_DIM), "k")
    _expect(v, (total, HKV, HEAD_DIM), "v")
    if cu_seqlens.dtype != torch.int32 or not cu_seqlens.is_cuda or cu_seqlens.dim() != 1:
        raise TypeError("cu_seqlens must be a 1-D int32 CUDA tensor")
    batch = cu_seqlens.numel() - 1
    if out is None:
        out = torch.empty_like(q)
    _expect(out, (total, HQ, HEAD_DIM), "out")
    lse = torch.empty((HQ, total), dtype=torch.float32, device=q.device) if return_lse else None
    _check("gqa_attn_prefill_varlen", lib().gqa_attn_prefill_varlen(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
        lse.data_ptr() if lse is not None else None, cu_seqlens.data_ptr(), batch,
        int(max_seqlen), total, 1 if causal else 0, _stream(stream)))
    return (out, lse) if return_lse else out


def decode(q, kcache, vcache, out=None, workspace=None, stream=None, return_lse: bool = False):
    """One query token q [1,1,32,128] against kcache/vcache [1,L,8,128] bf16.

    With ``workspace`` (a CUDA tensor of at least ``decode_workspace_bytes(L)``
    bytes) the caller-workspace entry point is used; otherwise the library's
    own per-device workspace.
    """
    import torch
    L = kcache.shape[1]
    _expect(q, (1, 1, HQ, HEAD_DIM), "q")
    _expect(kcache, (1, L, HKV, HEAD_DIM), "kcache")
    _expect(vcache, (1, L, HKV, HEAD_DIM), "vcache")
    if out is None:
        out = torch.empty_like(q)
    _expect(out, (1, 1, HQ, HEAD_DIM), "out")
    s = _stream(stream)
    if return_lse:
        if workspace is not None:
            raise ValueError("return_lse uses the library workspace")
        lse = torch.empty((1, HQ), dtype=torch.float32, device=q.device)
        _check("gqa_attn_decode_lse", lib().gqa_attn_decode_lse(
            q.data_ptr(), kcache.data_ptr(), vcache.data_ptr(), out.data_ptr(),
            lse.data_ptr(), L, s))
        return out, lse
    if workspace is None:
        _check("gqa_attn_decode", lib().gqa_attn_decode(
            q.data_ptr(), kcache.data_ptr(), vcache.data_ptr(), out.data_ptr(), L, s))
    else:
        nbytes = workspace.numel() * workspace.element_size()
        _check("gqa_attn_decode_ws", lib().gqa_attn_decode_ws(
            q.data_ptr(), kcache.data_ptr(), vcache.data_ptr(), out.data_ptr(), L,
            workspace.data_ptr(), nbytes, s))
    return out


def decode_batched(q, kcache, vcache, seqlens=None, out=None, stream=None,
                   return_lse: bool = False):
    """Decode of a batch: q [B,32,128] against caches [B,Lmax,8,128] bf16;
    sequence b attends to its first seqlens[b] rows (int32 CUDA tensor [B];
    None = all Lmax).  Returns out [B,32,128] (and lse [B,32] fp32)."""
    import torch
    B, Lmax = kcache.shape[0], kcache.shape[1]
    _expect(q, (B, HQ, HEAD_DIM), "q")
    _expect(kcache, (B, Lmax, HKV, HEAD_DIM), "kcache")
    _expect(vcache, (B, Lmax, HKV, HEAD_DIM), "vcache")
    if seqlens is not None and (seqlens.dtype != torch.int32 or not seqlens.is_cuda
                                or tuple(seqlens.shape) != (B,)):
        raise TypeError("seqlens must be an int32 CUDA tensor of shape [B]")
    if out is None:
        out = torch.empty_like(q)
    _expect(out, (B, HQ, HEAD_DIM), "out")
    lse = torch.empty((B, HQ), dtype=torch.float32, device=q.device) if return_lse else None
    _check("gqa_attn_decode_batched", lib().gqa_attn_decode_batched(
        q.data_ptr(), kcache.data_ptr(), vcache.data_ptr(), out.data_ptr(),
        lse.data_ptr() if lse is not None else None,
        seqlens.data_ptr() if seqlens is not None else None, B, Lmax, _stream(stream)))
    return (out, lse) if return_lse else out


def prefill_heads(q, k, v, cu_seqlens=None, max_seqlen=None, causal: bool = True, out=None,
                  stream=None, return_lse: bool = False):
    """Prefill for any head layout (query heads a multiple of KV heads):
    q [1,S,Hq,128] with k/v [1,S,Hkv,128], or packed q [total,Hq,128] with
    k/v [total,Hkv,128] and ``cu_seqlens`` (int32 CUDA tensor of batch+1
    offsets) plus ``max_seqlen``.  Returns out shaped like q (and lse
    [Hq,total] fp32 with ``return_lse``)."""
    import torch
    if q.dim() == 4:
        if cu_seqlens is not None:
            raise ValueError("4-D tensors are one sequence; pass packed 3-D tensors with cu_seqlens")
        total, hq, hkv = q.shape[1], q.shape[2], k.shape[2]
        _expect(q, (1, total, hq, HEAD_DIM), "q")
        _expect(k, (1, total, hkv, HEAD_DIM), "k")
        _expect(v, (1, total, hkv, HEAD_DIM), "v")
        batch, max_seqlen = 1, total
    else:
        total, hq, hkv = q.shape[0], q.shape[1], k.shape[1]
        _expect(q, (total, hq, HEAD_DIM), "q")
        _expect(k, (total, hkv, HEAD_DIM), "k")
        _expect(v, (total, hkv, HEAD_DIM), "v")
        if cu_seqlens is None:
            batch, max_seqlen = 1, total
        else:
            if cu_seqlens.dtype != torch.int32 or not cu_seqlens.is_cuda or cu_seqlens.dim() != 1:
                raise TypeError("cu_seqlens must be a 1-D int32 CUDA tensor")
            if max_seqlen is None:
                raise ValueError("max_seqlen is required with cu_seqlens")
            batch = cu_seqlens.numel() - 1
    if out is None:
        out = torch.empty_like(q)
    _expect(out, tuple(q.shape), "out")
    lse = torch.empty((hq, total), dtype=torch.float32, device=q.device) if return_lse else None
    _check("gqa_attn_prefill_heads", lib().gqa_attn_prefill_heads(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
        lse.data_ptr() if lse is not None else None,
        cu_seqlens.data_ptr() if cu_seqlens is not None else None, batch, int(max_seqlen),
        total, hq, hkv, 1 if causal else 0, _stream(stream)))
    return (out, lse) if return_lse else out


def decode_heads(q, kcache, vcache, seqlens=None, out=None, stream=None,
                 return_lse: bool = False):
    """Decode for any head layout with at most 16 query heads per KV head:
    q [B,Hq,128] against caches [B,Lmax,Hkv,128] bf16; sequence b attends to
    its first seqlens[b] rows (int32 CUDA tensor [B]; None = all Lmax).
    Returns out [B,Hq,128] (and lse [B,Hq] fp32)."""
    import torch
    B, hq = q.shape[0], q.shape[1]
    Lmax, hkv = kcache.shape[1], kcache.shape[2]
    _expect(q, (B, hq, HEAD_DIM), "q")
    _expect(kcache, (B, Lmax, hkv, HEAD_DIM), "kcache")
    _expect(vcache, (B, Lmax, hkv, HEAD_DIM), "vcache")
    if seqlens is not None and (seqlens.dtype != torch.int32 or not seqlens.is_cuda
                                or tuple(seqlens.shape) != (B,)):
        raise TypeError("seqlens must be an int32 CUDA tensor of shape [B]")
    if out is None:
        out = torch.empty_like(q)
    _expect(out, (B, hq, HEAD_DIM), "out")
    lse = torch.empty((B, hq), dtype=torch.float32, device=q.device) if return_lse else None
    _check("gqa_attn_decode_heads", lib().gqa_attn_decode_heads(
        q.data_ptr(), kcache.data_ptr(), vcache.data_ptr(), out.data_ptr(),
        lse.data_ptr() if lse is not None else None,
        seqlens.data_ptr() if seqlens is not None else None, B, Lmax, hq, hkv,
        _stream(stream)))
    return (out, lse) if return_lse else out


def decode_noalloc(q, kcache, vcache, out, stream=None):
    """Decode through the entry point that allocates nothing (its partial
    results use the library's fixed 1 MiB scratch; calls on one device must
    not overlap in time).  ``out`` must be given: this call allocates no
    tensor either."""
    L = kcache.shape[1]
    _expect(q, (1, 1, HQ, HEAD_DIM), "q")
    _expect(kcache, (1, L, HKV, HEAD_DIM), "kcache")
    _expect(vcache, (1, L, HKV, HEAD_DIM), "vcache")
    _expect(out, (1, 1, HQ, HEAD_DIM), "out")
    _check("gqa_attn_decode_noalloc", lib().gqa_attn_decode_noalloc(
        q.data_ptr(), kcache.data_ptr(), vcache.data_ptr(), out.data_ptr(), L,
        _stream(stream)))
    return out


def decode_workspace_bytes(L: int) -> int:
    return int(lib().gqa_attn_decode_workspace_bytes(int(L)))


def decode_plan(L: int, batch: int = 1, num_sms: int = 152):
    """(n_split, chunk) of the decode for cache length L (host-side, no GPU)."""
    n, c = ctypes.c_int(0), ctypes.c_int(0)
    if not lib().gqa_attn_decode_plan(int(L), int(batch), int(num_sms), ctypes.byref(n),
                                      ctypes.byref(c)):
        raise ValueError("decode_plan: arguments out of range")
    return n.value, c.value


def decode_num_splits(L: int) -> int:
    return int(lib().gqa_attn_decode_num_splits(int(L)))


def launches_per_call(is_decode: bool) -> int:
    return int(lib().gqa_attn_launches_per_call(1 if is_decode else 0))


def device_error(clear: bool = True) -> int:
    """Synchronise the device and return its error word (0 = no error)."""
    word = ctypes.c_uint(0)
    code = lib().gqa_attn_device_error(ctypes.byref(word), 1 if clear else 0)
    if code not in (0, 6):
        raise GqaError("gqa_attn_device_error", code)
    return int(word.value)
