"""CPU oracle for the hot path's contractions and IKBO attention (fp64).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the benchmark's CPU-baseline / reference legs may import this package.  The
product library never loads it and never falls back to it.

The arithmetic lives in ``oracle.c`` (plain C, built with gcc + OpenMP into
``liboracle.so`` beside this file).  This module only marshals numpy arrays:
bf16 inputs are passed as their raw uint16 bit patterns, outputs come back as
float64.  See ``oracle.c`` for which passage of the TLX write-ups each
routine follows.

Every routine is pinned by the ``-m "not gpu"`` tests in
``tests/test_oracle_pins.py`` against brute force, closed forms and exact
integer arithmetic.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so (gcc, -O2, OpenMP). Returns the path."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared",
           "-Wall", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            P = ctypes.c_void_p
            I = ctypes.c_int
            L = ctypes.c_long
            lib.oracle_gemm.argtypes = [I, I, I, I, P, L, L, P, L, L, P, L, I,
                                        P, L, L, P, I]
            lib.oracle_gemm.restype = None
            lib.oracle_gemm_rmsnorm.argtypes = [I, I, I, I, P, L, L, P, L, L,
                                                ctypes.c_double, P, L, I, P, L, L, P, I]
            lib.oracle_gemm_rmsnorm.restype = None
            lib.oracle_gemm_layernorm.argtypes = [I, I, I, I, P, L, L, P, L, L,
                                                  ctypes.c_double, P, L, I, P, L, L, P, I]
            lib.oracle_gemm_layernorm.restype = None
            lib.oracle_grouped.argtypes = [I, I, I, I, P, L, P, L, L, P, P, L,
                                           I, P, L]
            lib.oracle_grouped.restype = I
            lib.oracle_ikbo.argtypes = [I, I, I, I, I, I, P, P, P, P, P, P, I]
            lib.oracle_ikbo.restype = I
            lib.oracle_ikbo_decomposed.argtypes = [I, I, I, I, I, I, P, P, P,
                                                   P, P, P]
            lib.oracle_ikbo_decomposed.restype = I
            lib.oracle_ikbo_attention.argtypes = [I, I, I, I, I, I, P, P, P, P,
                                                  ctypes.c_double, P, P, I]
            lib.oracle_ikbo_attention.restype = I
            lib.oracle_ikbo_attention_grouped.argtypes = [I, I, I, I, I, I, P, P, P, P,
                                                          ctypes.c_double, P]
            lib.oracle_ikbo_attention_grouped.restype = I
            lib.oracle_num_threads.argtypes = []
            lib.oracle_num_threads.restype = I
            _lib = lib
    return _lib


def _u16(x) -> np.ndarray:
    """Raw bf16 bits as a C-contiguous uint16 array (torch bf16 or uint16 numpy)."""
    if hasattr(x, "dtype") and str(x.dtype) == "torch.bfloat16":
        import torch
        x = x.detach().to("cpu").contiguous().view(torch.int16).numpy()
    a = np.ascontiguousarray(x)
    if a.dtype == np.int16:
        a = a.view(np.uint16)
    if a.dtype != np.uint16:
        raise TypeError("oracle inputs are bf16 bit patterns (uint16), got %s" % a.dtype)
    return a


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def num_threads() -> int:
    return _load().oracle_num_threads()


EPI = {"none": 0, "bias": 1, "bias_silu": 2, "bias_gelu": 3}


def gemm(A, B, bias=None, epi: str = "none", rows=None) -> np.ndarray:
    """C[b,m,n] = epi(sum_k A[b,m,k] B[b,n,k]) in fp64.

    A: [batch,M,K] or [M,K] bf16; B: [batch,N,K] or [N,K] bf16 (a 2-D B with
    a 3-D A is shared by every batch); bias: [batch,N] or [N] bf16 (a 1-D
    bias is shared).  rows: optional list of m to compute (others are NaN).
    Returns float64 [batch,M,N] (or [M,N] for 2-D A).
    """
    lib = _load()
    a = _u16(A)
    b = _u16(B)
    squeeze = a.ndim == 2
    if squeeze:
        a = a[None]
    batch, M, K = a.shape
    if b.ndim == 2:
        b3, sB = b, 0
    else:
        b3, sB = b, b.shape[1] * b.shape[2]
    N = b.shape[-2]
    if b.shape[-1] != K:
        raise ValueError("K mismatch")
    code = EPI[epi]
    bias_a, sBias = None, 0
    if code:
        bias_a = _u16(bias)
        sBias = 0 if bias_a.ndim == 1 else bias_a.shape[-1]
    C = np.full((batch, M, N), np.nan, dtype=np.float64)
    rows_a = None
    nrows = 0
    if rows is not None:
        rows_a = np.ascontiguousarray(np.asarray(rows, dtype=np.int32))
        if rows_a.size and (rows_a.min() < 0 or rows_a.max() >= M):
            raise ValueError("row index out of range")
        nrows = rows_a.size
    lib.oracle_gemm(batch, M, N, K, _ptr(a), K, M * K, _ptr(b3), K, sB,
                    _ptr(bias_a), sBias, code, _ptr(C), N, M * N,
                    _ptr(rows_a), nrows)
    return C[0] if squeeze else C


def gemm_rmsnorm(A, B, eps: float = 1e-6, bias=None, epi: str = "none", rows=None) -> np.ndarray:
    """C[b,m,n] = epi(r[b,m] * sum_k A[b,m,k] B[b,n,k] (+ bias)), with
    r[b,m] = 1/sqrt(mean_k A[b,m,k]^2 + eps).  Conventions as gemm()."""
    lib = _load()
    a = _u16(A)
    b = _u16(B)
    squeeze = a.ndim == 2
    if squeeze:
        a = a[None]
    batch, M, K = a.shape
    sB = 0 if b.ndim == 2 else b.shape[1] * b.shape[2]
    N = b.shape[-2]
    if b.shape[-1] != K:
        raise ValueError("K mismatch")
    code = EPI[epi]
    bias_a, sBias = None, 0
    if code:
        bias_a = _u16(bias)
        sBias = 0 if bias_a.ndim == 1 else bias_a.shape[-1]
    C = np.full((batch, M, N), np.nan, dtype=np.float64)
    rows_a, nrows = None, 0
    if rows is not None:
        rows_a = np.ascontiguousarray(np.asarray(rows, dtype=np.int32))
        nrows = rows_a.size
    lib.oracle_gemm_rmsnorm(batch, M, N, K, _ptr(a), K, M * K, _ptr(b), K, sB, float(eps),
                            _ptr(bias_a), sBias, code, _ptr(C), N, M * N, _ptr(rows_a), nrows)
    return C[0] if squeeze else C


def gemm_layernorm(A, B, eps: float = 1e-5, bias=None, epi: str = "none", rows=None) -> np.ndarray:
    """C[b,m,n] = epi(sum_k xhat[b,m,k] B[b,n,k] (+ bias)), xhat the row's
    LayerNorm (mean and variance over k, two passes).  Conventions as gemm()."""
    lib = _load()
    a = _u16(A)
    b = _u16(B)
    squeeze = a.ndim == 2
    if squeeze:
        a = a[None]
    batch, M, K = a.shape
    sB = 0 if b.ndim == 2 else b.shape[1] * b.shape[2]
    N = b.shape[-2]
    if b.shape[-1] != K:
        raise ValueError("K mismatch")
    code = EPI[epi]
    bias_a, sBias = None, 0
    if code:
        bias_a = _u16(bias)
        sBias = 0 if bias_a.ndim == 1 else bias_a.shape[-1]
    C = np.full((batch, M, N), np.nan, dtype=np.float64)
    rows_a, nrows = None, 0
    if rows is not None:
        rows_a = np.ascontiguousarray(np.asarray(rows, dtype=np.int32))
        nrows = rows_a.size
    lib.oracle_gemm_layernorm(batch, M, N, K, _ptr(a), K, M * K, _ptr(b), K, sB, float(eps),
                              _ptr(bias_a), sBias, code, _ptr(C), N, M * N, _ptr(rows_a), nrows)
    return C[0] if squeeze else C


def grouped(A, B, offsets, bias=None, epi: str = "none") -> np.ndarray:
    """Grouped GEMM: rows [off[g], off[g+1]) of A times B[g]^T. fp64 [M_total,N]."""
    lib = _load()
    a = _u16(A)
    b = _u16(B)
    off = np.ascontiguousarray(np.asarray(offsets, dtype=np.int32))
    G = off.size - 1
    M_total, K = a.shape
    Gb, N, Kb = b.shape
    if Gb != G or Kb != K:
        raise ValueError("shape mismatch")
    code = EPI[epi]
    bias_a, sBias = None, 0
    if code:
        bias_a = _u16(bias)
        sBias = 0 if bias_a.ndim == 1 else bias_a.shape[-1]
    C = np.full((M_total, N), np.nan, dtype=np.float64)
    rc = lib.oracle_grouped(G, M_total, N, K, _ptr(a), K, _ptr(b), K, N * K,
                            _ptr(off), _ptr(bias_a), sBias, code, _ptr(C), N)
    if rc != 0:
        raise ValueError("bad group offsets")
    return C


def ikbo(U, Cf, W, user_offsets, cands=None) -> np.ndarray:
    """IKBO linear compression, materialised form: Y[c] = W . [U[user(c)]; Cf[c]].

    U [users,Du,D], Cf [cand,Dc,D], W [O,Du+Dc] bf16; returns fp64 [cand,O,D]
    (rows of candidates not in ``cands`` are NaN when ``cands`` is given).
    """
    lib = _load()
    u = _u16(U)
    c = _u16(Cf)
    w = _u16(W)
    off = np.ascontiguousarray(np.asarray(user_offsets, dtype=np.int32))
    nu, Du, D = u.shape
    nc, Dc, D2 = c.shape
    O, F = w.shape
    if D2 != D or F != Du + Dc or off.size != nu + 1:
        raise ValueError("shape mismatch")
    Y = np.full((nc, O, D), np.nan, dtype=np.float64)
    cands_a, ncands = None, 0
    if cands is not None:
        cands_a = np.ascontiguousarray(np.asarray(cands, dtype=np.int32))
        ncands = cands_a.size
    rc = lib.oracle_ikbo(nu, nc, Du, Dc, D, O, _ptr(u), _ptr(c), _ptr(w),
                         _ptr(off), _ptr(Y), _ptr(cands_a), ncands)
    if rc != 0:
        raise ValueError("bad user offsets or candidate index (rc=%d)" % rc)
    return Y


def ikbo_decomposed(U, Cf, W, user_offsets) -> np.ndarray:
    """IKBO by decomposition W_u.U[u] + W_c.Cf[c] (second coding, fp64)."""
    lib = _load()
    u = _u16(U)
    c = _u16(Cf)
    w = _u16(W)
    off = np.ascontiguousarray(np.asarray(user_offsets, dtype=np.int32))
    nu, Du, D = u.shape
    nc, Dc, _ = c.shape
    O = w.shape[0]
    Y = np.full((nc, O, D), np.nan, dtype=np.float64)
    P = np.zeros((max(nu, 1), O, D), dtype=np.float64)
    rc = lib.oracle_ikbo_decomposed(nu, nc, Du, Dc, D, O, _ptr(u), _ptr(c),
                                    _ptr(w), _ptr(off), _ptr(Y), _ptr(P))
    if rc != 0:
        raise ValueError("bad user offsets")
    return Y


def _attn_shapes(Q, K, V, user_offsets, Lq):
    q = _u16(Q)
    k = _u16(K)
    v = _u16(V)
    off = np.ascontiguousarray(np.asarray(user_offsets, dtype=np.int32))
    nu, Lkv, H, Dh = k.shape
    if v.shape != k.shape or off.size != nu + 1:
        raise ValueError("shape mismatch")
    nq, Hq, Dq = q.shape
    if Hq != H or Dq != Dh or nq % Lq:
        raise ValueError("query shape")
    return q, k, v, off, nu, nq // Lq, Lkv, H, Dh


def ikbo_attention(Q, K, V, user_offsets, Lq: int = 1, scale=None, cands=None) -> np.ndarray:
    """IKBO attention, materialised form: each query row of candidate c
    attends over its user's keys/values (one copy per candidate), per head.

    Q [num_cand*Lq, H, Dh], K/V [users, Lkv, H, Dh] bf16; scale defaults to
    1/sqrt(Dh).  Returns fp64 [num_cand*Lq, H, Dh] (rows of candidates not in
    ``cands`` are NaN when ``cands`` is given)."""
    lib = _load()
    q, k, v, off, nu, nc, Lkv, H, Dh = _attn_shapes(Q, K, V, user_offsets, Lq)
    if scale is None:
        scale = 1.0 / np.sqrt(Dh)
    O = np.full((nc * Lq, H, Dh), np.nan, dtype=np.float64)
    cands_a, ncands = None, 0
    if cands is not None:
        cands_a = np.ascontiguousarray(np.asarray(cands, dtype=np.int32))
        ncands = cands_a.size
    rc = lib.oracle_ikbo_attention(nu, nc, Lq, H, Dh, Lkv, _ptr(q), _ptr(k), _ptr(v), _ptr(off),
                                   float(scale), _ptr(O), _ptr(cands_a), ncands)
    if rc != 0:
        raise ValueError("bad user offsets or candidate index (rc=%d)" % rc)
    return O


def ikbo_attention_grouped(Q, K, V, user_offsets, Lq: int = 1, scale=None) -> np.ndarray:
    """IKBO attention, second coding (per user: stacked queries, S = QK^T,
    row softmax, O = PV).  Same conventions as ikbo_attention()."""
    lib = _load()
    q, k, v, off, nu, nc, Lkv, H, Dh = _attn_shapes(Q, K, V, user_offsets, Lq)
    if scale is None:
        scale = 1.0 / np.sqrt(Dh)
    O = np.full((nc * Lq, H, Dh), np.nan, dtype=np.float64)
    rc = lib.oracle_ikbo_attention_grouped(nu, nc, Lq, H, Dh, Lkv, _ptr(q), _ptr(k), _ptr(v),
                                           _ptr(off), float(scale), _ptr(O))
    if rc != 0:
        raise ValueError("bad user offsets (rc=%d)" % rc)
    return O
