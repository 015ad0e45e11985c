"""CPU oracle for exact attention (fp64).  TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg may
import this package.  The product path (the CUDA library and its Python binding) never
imports it, and this package imports nothing from the product path.

``attn_fwd`` / ``attn_bwd`` (and ``attn_fwd_kv``, queries after a longer key cache, and
``attn_fwd_varlen``, packed sequences of different lengths, built on it) wrap
the plain-C fp64 implementation in ``attn_oracle.c``
(materialised S and P, chain-rule gradients); ``tiled`` holds a step-by-step fp32
emulation of the tiled online softmax with the conditional rescale; ``fp8`` holds the
e4m3 encoding, the per-block quantiser and the fp64 forward of dequantised FP8 inputs.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``attn_oracle.c`` into ``liboracle.so`` (gcc, OpenMP, fp64)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", "-std=c11",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i, p, dbl = ctypes.c_int, ctypes.c_void_p, ctypes.c_double
            lib.oracle_attn_fwd.argtypes = [p, p, p, i, i, i, i, i, i, dbl, i, p, p, p]
            lib.oracle_attn_fwd.restype = i
            lib.oracle_attn_bwd.argtypes = [p, p, p, p, i, i, i, i, i, i, dbl, i, p, p, p, p]
            lib.oracle_attn_bwd.restype = i
            lib.oracle_attn_fwd_kv.argtypes = [p, p, p, i, i, i, i, i, i, i, dbl, i, p, p, p]
            lib.oracle_attn_fwd_kv.restype = i
            _lib = lib
    return _lib


def _bits(t) -> np.ndarray:
    """bf16 torch tensor (or uint16 numpy array of bf16 bit patterns) -> contiguous uint16."""
    if isinstance(t, np.ndarray):
        assert t.dtype == np.uint16
        return np.ascontiguousarray(t)
    import torch
    assert t.dtype == torch.bfloat16, t.dtype
    return np.ascontiguousarray(t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def attn_fwd(q, k, v, causal: bool, scale: float, heads=None):
    """fp64 forward.  ``q [B,Hq,N,d]``, ``k``/``v [B,Hkv,N,d]`` in bf16.

    ``heads``: list of (b, hq) to compute (default: all).  Returns (O, LSE) with shapes
    ``[len(heads), N, d]`` and ``[len(heads), N]`` (or ``[B,Hq,N,d]``/``[B,Hq,N]`` when
    ``heads`` is None)."""
    qb, kb, vb = _bits(q), _bits(k), _bits(v)
    B, Hq, N, d = qb.shape
    Hkv = kb.shape[1]
    if heads is None:
        sel = np.arange(B * Hq, dtype=np.int32)
    else:
        sel = np.asarray([b * Hq + h for b, h in heads], dtype=np.int32)
    O = np.zeros((len(sel), N, d), dtype=np.float64)
    L = np.zeros((len(sel), N), dtype=np.float64)
    rc = _load().oracle_attn_fwd(_ptr(qb), _ptr(kb), _ptr(vb), B, Hq, Hkv, N, d, int(bool(causal)),
                                 float(scale), len(sel), _ptr(sel), _ptr(O), _ptr(L))
    if rc != 0:
        raise RuntimeError(f"oracle_attn_fwd failed ({rc})")
    if heads is None:
        return O.reshape(B, Hq, N, d), L.reshape(B, Hq, N)
    return O, L


def attn_bwd(q, k, v, do, causal: bool, scale: float, kv_heads=None):
    """fp64 backward by the chain rule.

    ``kv_heads``: list of (b, hkv) to compute (default: all).  Returns (dQ, dK, dV) with
    shapes ``[S, g, N, d]``, ``[S, N, d]``, ``[S, N, d]`` for S selected key/value heads
    (or ``[B,Hq,N,d]``, ``[B,Hkv,N,d]``, ``[B,Hkv,N,d]`` when ``kv_heads`` is None)."""
    qb, kb, vb, db = _bits(q), _bits(k), _bits(v), _bits(do)
    B, Hq, N, d = qb.shape
    Hkv = kb.shape[1]
    g = Hq // Hkv
    if kv_heads is None:
        sel = np.arange(B * Hkv, dtype=np.int32)
    else:
        sel = np.asarray([b * Hkv + h for b, h in kv_heads], dtype=np.int32)
    dQ = np.zeros((len(sel), g, N, d), dtype=np.float64)
    dK = np.zeros((len(sel), N, d), dtype=np.float64)
    dV = np.zeros((len(sel), N, d), dtype=np.float64)
    rc = _load().oracle_attn_bwd(_ptr(qb), _ptr(kb), _ptr(vb), _ptr(db), B, Hq, Hkv, N, d,
                                 int(bool(causal)), float(scale), len(sel), _ptr(sel),
                                 _ptr(dQ), _ptr(dK), _ptr(dV))
    if rc != 0:
        raise RuntimeError(f"oracle_attn_bwd failed ({rc})")
    if kv_heads is None:
        return dQ.reshape(B, Hq, N, d), dK.reshape(B, Hkv, N, d), dV.reshape(B, Hkv, N, d)
    return dQ, dK, dV


def attn_fwd_kv(q, k, v, causal: bool, scale: float, heads=None):
    """fp64 forward with Nq queries after Nk >= Nq keys: ``q [B,Hq,Nq,d]``, ``k``/``v
    [B,Hkv,Nk,d]`` in bf16.  Causal: query i sees keys j <= i + Nk - Nq.  Returns (O, LSE)
    shaped like ``attn_fwd``'s with Nq rows."""
    qb, kb, vb = _bits(q), _bits(k), _bits(v)
    B, Hq, Nq, d = qb.shape
    Hkv, Nk = kb.shape[1], kb.shape[2]
    if heads is None:
        sel = np.arange(B * Hq, dtype=np.int32)
    else:
        sel = np.asarray([b * Hq + h for b, h in heads], dtype=np.int32)
    O = np.zeros((len(sel), Nq, d), dtype=np.float64)
    L = np.zeros((len(sel), Nq), dtype=np.float64)
    rc = _load().oracle_attn_fwd_kv(_ptr(qb), _ptr(kb), _ptr(vb), B, Hq, Hkv, Nq, Nk, d, int(bool(causal)),
                                    float(scale), len(sel), _ptr(sel), _ptr(O), _ptr(L))
    if rc != 0:
        raise ValueError(f"oracle_attn_fwd_kv failed ({rc})")
    if heads is None:
        return O.reshape(B, Hq, Nq, d), L.reshape(B, Hq, Nq)
    return O, L


def attn_fwd_varlen(q, k, v, cu_q, cu_k, causal: bool, scale: float):
    """fp64 forward over packed variable-length sequences.

    ``q [Hq, total_q, d]`` and ``k``/``v [Hkv, total_k, d]`` (bf16) hold the sequences one
    after another along the row axis; sequence b owns query rows ``cu_q[b]:cu_q[b+1]`` and
    key rows ``cu_k[b]:cu_k[b+1]``.  Each sequence is an attention problem of its own (the
    packed-sequence scheduling of "FlashAttention-4 explained", section 06, changes only
    the order in which the problems run), computed by ``attn_fwd_kv`` with B = 1, so causal
    is aligned to the sequence's last key.  Returns O ``[Hq, total_q, d]`` and LSE
    ``[Hq, total_q]``; rows of empty sequences do not exist, so nothing is left unset.
    """
    qb, kb, vb = _bits(q), _bits(k), _bits(v)
    cq = np.asarray(cu_q, dtype=np.int64).reshape(-1)
    ck = np.asarray(cu_k, dtype=np.int64).reshape(-1)
    Hq, Tq, d = qb.shape
    Hkv, Tk = kb.shape[0], kb.shape[1]
    if len(cq) != len(ck) or len(cq) < 1:
        raise ValueError("cu_q and cu_k must both hold B + 1 offsets")
    if cq[0] != 0 or ck[0] != 0 or cq[-1] != Tq or ck[-1] != Tk:
        raise ValueError("offsets must start at 0 and end at the packed lengths")
    if np.any(np.diff(cq) < 0) or np.any(np.diff(ck) < 0):
        raise ValueError("offsets must not decrease")
    O = np.zeros((Hq, Tq, d), dtype=np.float64)
    L = np.zeros((Hq, Tq), dtype=np.float64)
    for b in range(len(cq) - 1):
        q0, q1, k0, k1 = int(cq[b]), int(cq[b + 1]), int(ck[b]), int(ck[b + 1])
        if q1 == q0:
            continue
        if k1 == k0:
            raise ValueError(f"sequence {b} has {q1 - q0} queries and no keys")
        Ob, Lb = attn_fwd_kv(np.ascontiguousarray(qb[None, :, q0:q1]), np.ascontiguousarray(kb[None, :, k0:k1]),
                             np.ascontiguousarray(vb[None, :, k0:k1]), causal, scale)
        O[:, q0:q1] = Ob[0]
        L[:, q0:q1] = Lb[0]
    return O, L


def _f64(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float64 values."""
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _bwd_one_head(q, k, v, do, causal: bool, scale: float):
    """The backward of one query head of one sequence, from the definition: q, do [nq,d],
    k, v [nk,d] (fp64); query i sees keys j <= i + nk - nq when causal.
    S = scale Q K^T, P = softmax(S) by rows, O = P V; dV = P^T dO, dP = dO V^T,
    dS = P o (dP - rowsum(dO o O)), dQ = scale dS K, dK = scale dS^T Q."""
    nq, nk = q.shape[0], k.shape[0]
    s = scale * (q @ k.T)
    if causal:
        i = np.arange(nq)[:, None]
        j = np.arange(nk)[None, :]
        s = np.where(j <= i + (nk - nq), s, -np.inf)
    p = np.exp(s - s.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    o = p @ v
    dv = p.T @ do
    dp = do @ v.T
    ds = p * (dp - (do * o).sum(axis=1, keepdims=True))
    return scale * (ds @ k), scale * (ds.T @ q), dv


def attn_bwd_varlen(q, k, v, do, cu_q, cu_k, causal: bool, scale: float):
    """fp64 backward over packed variable-length sequences (layouts and offsets as
    ``attn_fwd_varlen``; ``do`` like ``q``).  Each sequence and query head is differentiated
    on its own from the definition (``_bwd_one_head``, numpy fp64 matrix products); dK and
    dV of a K/V head sum over the query heads of its group.  Keys of a sequence without
    queries get zero gradients.  Returns dQ ``[Hq, total_q, d]``, dK and dV
    ``[Hkv, total_k, d]``."""
    qd, kd, vd, dd = (_f64(_bits(t)) for t in (q, k, v, do))
    cq = np.asarray(cu_q, dtype=np.int64).reshape(-1)
    ck = np.asarray(cu_k, dtype=np.int64).reshape(-1)
    Hq, Tq, d = qd.shape
    Hkv, Tk = kd.shape[0], kd.shape[1]
    g = Hq // Hkv
    if len(cq) != len(ck) or cq[0] != 0 or ck[0] != 0 or cq[-1] != Tq or ck[-1] != Tk:
        raise ValueError("offsets must hold B + 1 entries from 0 to the packed lengths")
    if np.any(np.diff(cq) < 0) or np.any(np.diff(ck) < 0):
        raise ValueError("offsets must not decrease")
    dQ = np.zeros((Hq, Tq, d))
    dK = np.zeros((Hkv, Tk, d))
    dV = np.zeros((Hkv, Tk, d))
    for b in range(len(cq) - 1):
        q0, q1, k0, k1 = int(cq[b]), int(cq[b + 1]), int(ck[b]), int(ck[b + 1])
        if q1 == q0:
            continue
        if k1 == k0 or (causal and k1 - k0 < q1 - q0):
            raise ValueError(f"sequence {b}: some query sees no key")
        for h in range(Hq):
            hk = h // g
            gq, gk, gv = _bwd_one_head(qd[h, q0:q1], kd[hk, k0:k1], vd[hk, k0:k1], dd[h, q0:q1], causal, scale)
            dQ[h, q0:q1] = gq
            dK[hk, k0:k1] += gk
            dV[hk, k0:k1] += gv
    return dQ, dK, dV
