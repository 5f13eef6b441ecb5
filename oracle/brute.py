"""Plain-definition attention oracle (fp64), C core loaded through ctypes.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Every score row is materialised in double precision, softmax-normalised by its
exact log-sum-exp and multiplied by V; see ``attn_oracle.c`` for the formulas
and their sources.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD_DIR, "libattn_oracle.so")
_lock = threading.Lock()
_lib = None


def lib_path() -> str:
    return _LIB


def build(force: bool = False) -> str:
    """Compile attn_oracle.c into a shared library (gcc, OpenMP, -O2).

    Plain -O2 without fast-math keeps IEEE double semantics; no
    machine-specific flags, so the same source builds on x86_64 and aarch64.
    """
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
           "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            lib.attn_oracle_rows.restype = ctypes.c_int
            lib.attn_oracle_rows.argtypes = [
                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                ctypes.c_double, ctypes.c_int,
                ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p,
                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
            ]
            lib.attn_oracle_rows_qk.restype = ctypes.c_int
            lib.attn_oracle_rows_qk.argtypes = [
                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                ctypes.c_double, ctypes.c_int,
                ctypes.c_void_p, ctypes.c_int64,
                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
            ]
            lib.attn_oracle_max_threads.restype = ctypes.c_int
            lib.attn_oracle_max_threads.argtypes = []
            _lib = lib
    return _lib


def max_threads() -> int:
    return int(_load().attn_oracle_max_threads())


def _bf16_bits(x) -> np.ndarray:
    """Accept a numpy uint16 array of bf16 bit patterns or a torch bfloat16 tensor."""
    if isinstance(x, np.ndarray):
        if x.dtype != np.uint16:
            raise TypeError("numpy inputs must hold bf16 bit patterns as uint16")
        return np.ascontiguousarray(x)
    # torch tensor (duck-typed so this module does not need torch)
    if str(getattr(x, "dtype", "")) != "torch.bfloat16":
        raise TypeError("torch inputs must be bfloat16")
    import torch  # local: only when a tensor is passed
    return x.detach().to("cpu").contiguous().view(torch.int16).numpy().view(np.uint16)


def attention_rows(q, k, v, scale: float, causal: bool, rows=None,
                   shifts=None, nthreads: int = 0):
    """O and LSE (float64) for the requested rows of a [B, H, N, D] problem.

    q, k, v : bf16 bits, shape [..., N, D] (leading dims flattened to BH)
    rows    : flat row indices bh*N + i (None = all rows, in order)
    shifts  : optional per-row additive score shift (same length as rows)
    Returns (o [nrows, D], lse [nrows], threads_used).
    """
    qb, kb, vb = _bf16_bits(q), _bf16_bits(k), _bf16_bits(v)
    if not (qb.shape == kb.shape == vb.shape) or qb.ndim < 2:
        raise ValueError("q, k, v must share one [..., N, D] shape")
    N, D = int(qb.shape[-2]), int(qb.shape[-1])
    BH = int(qb.size // (N * D)) if N * D > 0 else 0
    if rows is None:
        nrows = BH * N
        rows_arr = None
    else:
        rows_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        nrows = int(rows_arr.size)
    sh = None
    if shifts is not None:
        sh = np.ascontiguousarray(np.asarray(shifts, dtype=np.float64))
        if sh.size != nrows:
            raise ValueError("shifts must have one entry per requested row")
    o = np.empty((nrows, D), dtype=np.float64)
    lse = np.empty((nrows,), dtype=np.float64)
    if nrows == 0:
        return o, lse, 0
    lib = _load()
    used = lib.attn_oracle_rows(
        qb.ctypes.data, kb.ctypes.data, vb.ctypes.data, BH, N, D,
        float(scale), int(bool(causal)),
        rows_arr.ctypes.data if rows_arr is not None else None, nrows,
        sh.ctypes.data if sh is not None else None,
        o.ctypes.data, lse.ctypes.data, int(nthreads))
    if used < 0:
        raise ValueError("attn_oracle_rows rejected its arguments")
    return o, lse, int(used)


def attention(q, k, v, scale: float, causal: bool, nthreads: int = 0):
    """Every row: returns (o [..., N, D] float64, lse [..., N] float64)."""
    qb = _bf16_bits(q)
    o, lse, _ = attention_rows(qb, k, v, scale, causal, None, None, nthreads)
    return o.reshape(qb.shape), lse.reshape(qb.shape[:-1])


def attention_qk_rows(q, k, v, scale: float, causal: bool, rows=None, nthreads: int = 0):
    """O and LSE (float64) for queries and keys of different lengths.

    q : bf16 bits [..., Nq, D];  k, v : bf16 bits [..., Nk, D] (same leading dims)
    causal: key j visible to query i iff j <= i + (Nk - Nq) (the queries are
    the last Nq positions of the sequence); requires Nq <= Nk.
    rows : flat query-row indices bh*Nq + i (None = all rows, in order)
    Returns (o [nrows, D], lse [nrows], threads_used).
    """
    qb, kb, vb = _bf16_bits(q), _bf16_bits(k), _bf16_bits(v)
    if kb.shape != vb.shape or qb.ndim < 2 or qb.shape[:-2] != kb.shape[:-2] or \
            qb.shape[-1] != kb.shape[-1]:
        raise ValueError("q [..., Nq, D] and k, v [..., Nk, D] must share leading dims and D")
    Nq, Nk, D = int(qb.shape[-2]), int(kb.shape[-2]), int(qb.shape[-1])
    BH = int(qb.size // (Nq * D)) if Nq * D > 0 else 0
    if rows is None:
        nrows = BH * Nq
        rows_arr = None
    else:
        rows_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        nrows = int(rows_arr.size)
    o = np.empty((nrows, D), dtype=np.float64)
    lse = np.empty((nrows,), dtype=np.float64)
    if nrows == 0:
        return o, lse, 0
    used = _load().attn_oracle_rows_qk(
        qb.ctypes.data, kb.ctypes.data, vb.ctypes.data, BH, Nq, Nk, D,
        float(scale), int(bool(causal)),
        rows_arr.ctypes.data if rows_arr is not None else None, nrows,
        o.ctypes.data, lse.ctypes.data, int(nthreads))
    if used < 0:
        raise ValueError("attn_oracle_rows_qk rejected its arguments")
    return o, lse, int(used)


def attention_qk(q, k, v, scale: float, causal: bool, nthreads: int = 0):
    """Every query row: returns (o [..., Nq, D] float64, lse [..., Nq] float64)."""
    qb = _bf16_bits(q)
    o, lse, _ = attention_qk_rows(qb, k, v, scale, causal, None, nthreads)
    return o.reshape(qb.shape), lse.reshape(qb.shape[:-1])
