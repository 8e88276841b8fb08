"""fp64 CPU oracle for grouped-query attention forward -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
arm of ``bench.py`` may import this package.  The product library never links,
loads or calls it, and it shares no code with the CUDA path.

The arithmetic lives in ``gqa_oracle.c`` (plain C, fp64, OpenMP over
(row, head)); this module only marshals numpy/torch buffers through ctypes.
It follows the attention the chowfi/kernels README describes ("Result"
section: GQA forward, 32 query heads sharing 8 KV heads, head size 128, bf16,
causal prefill over the whole prompt and decode of one token against a KV
cache):

    out[i,h,:] = sum_j softmax_j(q[i,h,:] . k[j,h//G,:] / sqrt(D)) v[j,h//G,:]

Parity of every function here is pinned by ``tests/test_oracle.py`` against
brute force, closed forms and invariants of attention.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gqa_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libgqa_oracle.so")


_u16p = ctypes.POINTER(ctypes.c_uint16)
_f64p = ctypes.POINTER(ctypes.c_double)
_i64p = ctypes.POINTER(ctypes.c_int64)


def compile_source(src_path: str, lib_path: str) -> str:
    """gcc-compile one C oracle source file into a shared library."""
    tmp = lib_path + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
           "-Wall", "-Wextra", "-o", tmp, src_path, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, lib_path)
    return lib_path


def build(force: bool = False) -> str:
    """Compile the C oracle into ``oracle/libgqa_oracle.so`` with gcc."""
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        compile_source(_SRC, _LIB_PATH)
    return _LIB_PATH


def _bits(x) -> np.ndarray:
    """bf16 tensor (torch) or uint16 bit array (numpy) -> contiguous uint16."""
    if isinstance(x, np.ndarray):
        if x.dtype != np.uint16:
            raise TypeError("oracle inputs are bf16 bit patterns (uint16)")
        return np.ascontiguousarray(x)
    import torch
    if x.dtype != torch.bfloat16:
        raise TypeError("oracle inputs must be bf16")
    return x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def _squeeze(a: np.ndarray) -> np.ndarray:
    """Drop a leading batch dimension of 1 (BSHD with B=1)."""
    if a.ndim == 4:
        if a.shape[0] != 1:
            raise ValueError("the oracle covers batch 1")
        a = a[0]
    return np.ascontiguousarray(a)


def _ptr(a, typ):
    return None if a is None else a.ctypes.data_as(typ)


def _check(rc: int, what: str):
    if rc != 0:
        raise ValueError(f"{what}: oracle returned {rc}")


def _geometry(q: np.ndarray, k: np.ndarray):
    if q.ndim != 3 or k.ndim != 3 or q.shape[2] != k.shape[2]:
        raise ValueError("expected q [n,hq,d] and k/v [n,hkv,d]")
    return q.shape[1], k.shape[1], q.shape[2]


class OracleLib:
    """ctypes front of one build of the C oracle."""

    def __init__(self, lib_path: str):
        lib = ctypes.CDLL(lib_path)
        c_int, c_long = ctypes.c_int, ctypes.c_long
        lib.gqa_oracle_prefill_rows.argtypes = [
            _u16p, _u16p, _u16p, c_long, c_int, c_int, c_int, c_int, _i64p,
            c_long, _f64p, _f64p, c_int]
        lib.gqa_oracle_prefill.argtypes = [
            _u16p, _u16p, _u16p, c_long, c_int, c_int, c_int, c_int, _f64p,
            _f64p, c_int]
        lib.gqa_oracle_decode.argtypes = [
            _u16p, _u16p, _u16p, c_long, c_int, c_int, c_int, _f64p, _f64p,
            c_int]
        lib.gqa_oracle_weights.argtypes = [
            _u16p, _u16p, _u16p, c_long, c_int, c_int, c_int, c_int, c_long,
            c_int, _f64p, _f64p]
        lib.gqa_oracle_max_threads.argtypes = []
        for f in (lib.gqa_oracle_prefill_rows, lib.gqa_oracle_prefill,
                  lib.gqa_oracle_decode, lib.gqa_oracle_weights,
                  lib.gqa_oracle_max_threads):
            f.restype = c_int
        self.lib = lib
        self.path = lib_path

    def max_threads(self) -> int:
        return self.lib.gqa_oracle_max_threads()

    def prefill_rows(self, q, k, v, rows, causal: bool = True,
                     threads: int = 0, with_lse: bool = False):
        """fp64 attention output of the listed query rows of a prefill.

        q [S,hq,d], k/v [S,hkv,d] (bf16 or uint16 bits; a leading batch dim
        of 1 is dropped).  Returns out [len(rows),hq,d] float64 (and, with
        ``with_lse``, the natural-log log-sum-exp of the scores [len,hq]).
        """
        q, k, v = (_squeeze(_bits(t)) for t in (q, k, v))
        hq, hkv, d = _geometry(q, k)
        S = q.shape[0]
        if k.shape[0] != S or v.shape != k.shape:
            raise ValueError("prefill needs q, k, v of the same length")
        rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).ravel())
        out = np.empty((rows.size, hq, d), dtype=np.float64)
        lse = np.empty((rows.size, hq), dtype=np.float64) if with_lse else None
        rc = self.lib.gqa_oracle_prefill_rows(
            _ptr(q, _u16p), _ptr(k, _u16p), _ptr(v, _u16p), S, hq, hkv, d,
            int(bool(causal)), _ptr(rows, _i64p), rows.size, _ptr(out, _f64p),
            _ptr(lse, _f64p), threads)
        _check(rc, "prefill_rows")
        return (out, lse) if with_lse else out

    def prefill(self, q, k, v, causal: bool = True, threads: int = 0,
                with_lse: bool = False):
        """fp64 attention output of every row of a prefill: out [S,hq,d]."""
        q, k, v = (_squeeze(_bits(t)) for t in (q, k, v))
        hq, hkv, d = _geometry(q, k)
        S = q.shape[0]
        if k.shape[0] != S or v.shape != k.shape:
            raise ValueError("prefill needs q, k, v of the same length")
        out = np.empty((S, hq, d), dtype=np.float64)
        lse = np.empty((S, hq), dtype=np.float64) if with_lse else None
        rc = self.lib.gqa_oracle_prefill(
            _ptr(q, _u16p), _ptr(k, _u16p), _ptr(v, _u16p), S, hq, hkv, d,
            int(bool(causal)), _ptr(out, _f64p), _ptr(lse, _f64p), threads)
        _check(rc, "prefill")
        return (out, lse) if with_lse else out

    def decode(self, q, kcache, vcache, threads: int = 0,
               with_lse: bool = False):
        """fp64 decode of one query q [hq,d] against caches [L,hkv,d]."""
        q = _bits(q)
        q = np.ascontiguousarray(q.reshape(q.shape[-2], q.shape[-1]))
        kc, vc = (_squeeze(_bits(t)) for t in (kcache, vcache))
        hq, d = q.shape
        L, hkv, dk = kc.shape
        if dk != d or vc.shape != kc.shape:
            raise ValueError("decode needs q [hq,d] and caches [L,hkv,d]")
        out = np.empty((hq, d), dtype=np.float64)
        lse = np.empty((hq,), dtype=np.float64) if with_lse else None
        rc = self.lib.gqa_oracle_decode(
            _ptr(q, _u16p), _ptr(kc, _u16p), _ptr(vc, _u16p), L, hq, hkv, d,
            _ptr(out, _f64p), _ptr(lse, _f64p), threads)
        _check(rc, "decode")
        return (out, lse) if with_lse else out

    def weights(self, q, k, v, i: int, h: int, causal: bool = True):
        """Normalised softmax weights of query row i, head h, and its output."""
        q, k, v = (_squeeze(_bits(t)) for t in (q, k, v))
        hq, hkv, d = _geometry(q, k)
        S = q.shape[0]
        n_keys = i + 1 if causal else S
        w = np.empty((n_keys,), dtype=np.float64)
        row = np.empty((d,), dtype=np.float64)
        rc = self.lib.gqa_oracle_weights(
            _ptr(q, _u16p), _ptr(k, _u16p), _ptr(v, _u16p), S, hq, hkv, d,
            int(bool(causal)), i, h, _ptr(w, _f64p), _ptr(row, _f64p))
        _check(rc, "weights")
        return w, row


_default = None


def default() -> OracleLib:
    """The oracle built from ``oracle/gqa_oracle.c`` (compiled on first use)."""
    global _default
    if _default is None:
        _default = OracleLib(build())
    return _default


def max_threads() -> int:
    return default().max_threads()


def prefill_rows(*a, **kw):
    return default().prefill_rows(*a, **kw)


def prefill(*a, **kw):
    return default().prefill(*a, **kw)


def decode(*a, **kw):
    return default().decode(*a, **kw)


def weights(*a, **kw):
    return default().weights(*a, **kw)
