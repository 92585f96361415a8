"""Oracle for the fused grouped-query attention forward: a plain fp64 CPU
definition of O = softmax(Q K^T * scale) V and of the log-sum-exp.

TEST INFRASTRUCTURE ONLY. Nothing on the product path imports this package:
only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` use it. It shares no code with the CUDA library; the only thing
both sides share is the seeded input generator, which holds none of the
method's arithmetic.

The arithmetic lives in ``sdp_oracle.c`` (plain C, fp64, OpenMP over rows);
this module compiles it with gcc, loads it with ctypes and marshals numpy
arrays. Every function it exposes is pinned by ``tests/test_oracle.py``
against closed forms, invariants, an arbitrary-precision brute force and
PyTorch's float64 CPU attention; none is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sdp_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libsdp_oracle.so")

FP16 = 0
BF16 = 1

_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/libsdp_oracle.so`` (gcc + OpenMP)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-Wall", "-Wextra",
               "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        p = ctypes.c_void_p
        i = ctypes.c_int
        lib.oracle_sdp_fwd_rows.argtypes = [p, p, p, i, i, i, i, i, i, i, ctypes.c_double, i, p, i, p, p]
        lib.oracle_sdp_fwd_rows.restype = i
        lib.oracle_sdp_row_probs.argtypes = [p, p, p, i, i, i, i, i, i, i, ctypes.c_double, i,
                                             i, i, i, p, p, p]
        lib.oracle_sdp_row_probs.restype = i
        lib.oracle_sdp_fwd_varlen.argtypes = [p, p, p, i, i, i, i, i, ctypes.c_double, i, p, p,
                                              ctypes.c_long, ctypes.c_long, p, p]
        lib.oracle_sdp_fwd_varlen.restype = i
        lib.oracle_fp16_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_fp16_to_double.restype = ctypes.c_double
        lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_to_double.restype = ctypes.c_double
        lib.oracle_sdp_merge.argtypes = [p, p, i, ctypes.c_long, i, p, p]
        lib.oracle_sdp_merge.restype = i
        lib.oracle_num_threads.argtypes = []
        lib.oracle_num_threads.restype = i
        _lib = lib
    return _lib


def _bits(a) -> np.ndarray:
    """16-bit patterns of an fp16/bf16 torch tensor or a uint16/float16 numpy array."""
    if hasattr(a, "detach"):  # torch tensor; keep torch an optional dependency here
        import torch
        a = a.detach().cpu().contiguous().view(torch.int16).numpy()
    a = np.ascontiguousarray(a)
    if a.dtype == np.float16:
        a = a.view(np.uint16)
    return np.ascontiguousarray(a.view(np.uint16))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def num_threads() -> int:
    """Threads the oracle's parallel regions use on this host."""
    return int(_load().oracle_num_threads())


def fp16_to_double(bits: int) -> float:
    return float(_load().oracle_fp16_to_double(int(bits) & 0xFFFF))


def bf16_to_double(bits: int) -> float:
    return float(_load().oracle_bf16_to_double(int(bits) & 0xFFFF))


def sdp_fwd_rows(q, k, v, dtype: int, shape, scale: float, rows: np.ndarray, causal: bool = False):
    """O and LSE (fp64) of the query rows ``rows[b, h, :]`` of every (b, h).

    q: [B, Hq, Sq, D], k/v: [B, Hkv, Skv, D] 16-bit patterns (or fp16/bf16
    tensors). ``rows`` is int32 [B, Hq, n]. Returns (o [B, Hq, n, D], lse [B, Hq, n]).
    With ``causal``, row i sees keys 0..i.
    """
    B, Hq, Hkv, Sq, Skv, D = (int(x) for x in shape)
    qb, kb, vb = _bits(q), _bits(k), _bits(v)
    assert qb.size == B * Hq * Sq * D and kb.size == B * Hkv * Skv * D and vb.size == kb.size
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int32))
    assert rows.ndim == 3 and rows.shape[:2] == (B, Hq)
    n = rows.shape[2]
    o = np.empty((B, Hq, n, D), dtype=np.float64)
    lse = np.empty((B, Hq, n), dtype=np.float64)
    rc = _load().oracle_sdp_fwd_rows(_ptr(qb), _ptr(kb), _ptr(vb), int(dtype), B, Hq, Hkv, Sq, Skv, D,
                                     float(scale), int(bool(causal)), _ptr(rows), n, _ptr(o), _ptr(lse))
    if rc != 0:
        raise ValueError("oracle rejected the shape or row indices")
    return o, lse


def sdp_fwd(q, k, v, dtype: int, shape, scale: float, causal: bool = False):
    """O and LSE (fp64) of every query row."""
    B, Hq, _, Sq, _, _ = (int(x) for x in shape)
    rows = np.broadcast_to(np.arange(Sq, dtype=np.int32), (B, Hq, Sq))
    return sdp_fwd_rows(q, k, v, dtype, shape, scale, rows, causal)


def row_probs(q, k, v, dtype: int, shape, scale: float, b: int, h: int, i: int, causal: bool = False):
    """Softmax weights (fp64 [Skv]), O row and LSE of query row (b, h, i)."""
    B, Hq, Hkv, Sq, Skv, D = (int(x) for x in shape)
    qb, kb, vb = _bits(q), _bits(k), _bits(v)
    p = np.empty(Skv, dtype=np.float64)
    o = np.empty(D, dtype=np.float64)
    lse = np.empty(1, dtype=np.float64)
    rc = _load().oracle_sdp_row_probs(_ptr(qb), _ptr(kb), _ptr(vb), int(dtype), B, Hq, Hkv, Sq, Skv, D,
                                      float(scale), int(bool(causal)), int(b), int(h), int(i), _ptr(p), _ptr(o),
                                      _ptr(lse))
    if rc != 0:
        raise ValueError("oracle rejected the shape or row index")
    return p, o, float(lse[0])


def sdp_merge(o_parts, lse_parts):
    """Merge partial results over disjoint key sets (fp64).

    o_parts: [P, rows, D] (any real dtype: numpy, or a torch tensor, upcast
    exactly to float64); lse_parts: [P, rows]. Returns (o [rows, D], lse [rows]).
    """
    def f64(x):
        if hasattr(x, "detach"):
            x = x.detach().cpu().double().numpy()
        return np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    op, lp = f64(o_parts), f64(lse_parts)
    P, rows, D = op.shape
    assert lp.shape == (P, rows)
    o = np.empty((rows, D), dtype=np.float64)
    lse = np.empty(rows, dtype=np.float64)
    rc = _load().oracle_sdp_merge(_ptr(op), _ptr(lp), int(P), int(rows), int(D), _ptr(o), _ptr(lse))
    if rc != 0:
        raise ValueError("oracle rejected the merge sizes")
    return o, lse


def sdp_fwd_varlen(q, k, v, dtype: int, cu_q, cu_k, scale: float, causal: bool = False):
    """Attention over a variable-length batch packed back to back (fp64).

    q: [total_q, Hq, D], k/v: [total_k, Hkv, D] 16-bit patterns (or fp16/bf16
    tensors); cu_q, cu_k: int32 [nseq + 1] sequence offsets. Sequence b's query
    rows attend to its own keys only (causal: its keys 0..i). Returns
    (o [total_q, Hq, D], lse [Hq, total_q]); a row that sees no key has O = 0
    and LSE = -inf.
    """
    qb, kb, vb = _bits(q), _bits(k), _bits(v)
    total_q, Hq, D = (int(x) for x in q.shape)
    total_k, Hkv = int(k.shape[0]), int(k.shape[1])
    assert tuple(k.shape) == tuple(v.shape) and int(k.shape[2]) == D
    cq = np.ascontiguousarray(np.asarray(cu_q, dtype=np.int32))
    ck = np.ascontiguousarray(np.asarray(cu_k, dtype=np.int32))
    assert cq.ndim == 1 and cq.shape == ck.shape
    o = np.empty((total_q, Hq, D), dtype=np.float64)
    lse = np.empty((Hq, total_q), dtype=np.float64)
    rc = _load().oracle_sdp_fwd_varlen(_ptr(qb), _ptr(kb), _ptr(vb), int(dtype), int(cq.size - 1), Hq, Hkv, D,
                                       float(scale), int(bool(causal)), _ptr(cq), _ptr(ck), total_q, total_k,
                                       _ptr(o), _ptr(lse))
    if rc != 0:
        raise ValueError("oracle rejected the sizes or sequence offsets")
    return o, lse
