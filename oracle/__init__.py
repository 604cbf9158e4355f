"""fp64 CPU oracle for the exact attention forward pass.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU-baseline / reference arm may import or run anything under
``oracle/``.  The product path (``exact_attention_forward_08_gb300``) never
does, and the two share no code: the only common module is ``synthetic``,
which draws seeded inputs and holds none of the method's arithmetic.

``attn_fwd`` is the plain definition O = softmax(scale * Q K^T) V with the
per-row log-sum-exp, written out row by row in double precision in
``attn_oracle.c`` (see that file for the citations); ``attn_bwd`` is the
chain rule through it (dQ, dK, dV for a given dO), in the same file.  ``online`` restates the
pages' online-softmax algebra (block state, two-block merge, conditional
rescaling) in fp64 for the pins in ``tests/``.

Parity status: pinned (worked example, closed forms, invariants, brute force
and a library routine; see ``tests/test_oracle_pins.py``).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

from . import online  # noqa: F401  (re-exported)

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_LIB_DIR = os.path.join(_HERE, "_build")
_LIB = os.path.join(_LIB_DIR, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc into ``oracle/_build/liboracle.so``."""
    os.makedirs(_LIB_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm", "-lpthread"])
        os.replace(tmp, _LIB)
    return _LIB


def load_library(path: str):
    """Load a compiled oracle library (the default one, or a test's copy)."""
    lib = ctypes.CDLL(path)
    i64 = ctypes.c_int64
    lib.oracle_attn_fwd.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
                                    i64, i64, i64, i64, i64, i64, i64, ctypes.c_int, ctypes.c_double,
                                    ctypes.c_void_p, i64, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
    lib.oracle_attn_fwd.restype = ctypes.c_int
    lib.oracle_attn_bwd.argtypes = [ctypes.c_void_p] * 4 + [ctypes.c_int] + [i64] * 7 + [ctypes.c_int, ctypes.c_double,
                                                                                   ctypes.c_void_p, ctypes.c_void_p,
                                                                                   ctypes.c_void_p, ctypes.c_int]
    lib.oracle_attn_bwd.restype = ctypes.c_int
    return lib


def _load():
    global _lib
    if _lib is None:
        _lib = load_library(build())
    return _lib


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def attn_fwd(q, k, v, causal: bool = False, scale: float | None = None, rows=None, threads: int | None = None,
             lib=None):
    """Reference attention forward.

    q [B,Sq,Hq,dqk], k [B,Sk,Hkv,dqk], v [B,Sk,Hkv,dv]: either float64 arrays or
    ``uint16`` arrays of bf16 bit patterns (decoded exactly).  ``scale`` defaults
    to 1/sqrt(dqk).

    rows=None: returns (O [B,Sq,Hq,dv], LSE [B,Hq,Sq]) as float64.
    rows = int64 array of linear row ids r = (b*Sq + i)*Hq + h: returns
    (O [n, dv], LSE [n]) for those rows only.
    ``lib`` selects another compiled copy of the oracle (used by the tests).
    """
    arrs = [np.ascontiguousarray(x) for x in (q, k, v)]
    kinds = {a.dtype for a in arrs}
    if kinds == {np.dtype(np.uint16)}:
        elem = 1
    elif kinds == {np.dtype(np.float64)}:
        elem = 0
    else:
        raise TypeError(f"q, k, v must all be uint16 (bf16 bits) or all float64, got {kinds}")
    q, k, v = arrs
    B, Sq, Hq, dqk = q.shape
    Bk, Sk, Hkv, dqk2 = k.shape
    Bv, Skv, Hkv2, dv = v.shape
    if not (B == Bk == Bv and dqk == dqk2 and Sk == Skv and Hkv == Hkv2):
        raise ValueError(f"inconsistent shapes q{q.shape} k{k.shape} v{v.shape}")
    if Hq % Hkv:
        raise ValueError("Hq must be a multiple of Hkv")
    if scale is None:
        scale = 1.0 / np.sqrt(dqk)
    full = rows is None
    if full:
        n = B * Sq * Hq
        rows_arr = None
    else:
        rows_arr = np.ascontiguousarray(rows, dtype=np.int64)
        n = rows_arr.size
    o = np.empty((n, dv), dtype=np.float64)
    lse = np.empty((n,), dtype=np.float64)
    rc = (lib or _load()).oracle_attn_fwd(q.ctypes.data, k.ctypes.data, v.ctypes.data, elem, B, Hq, Hkv, Sq, Sk,
                                 dqk, dv, int(bool(causal)), float(scale),
                                 None if full else rows_arr.ctypes.data, n, o.ctypes.data, lse.ctypes.data,
                                 threads or default_threads())
    if rc != 0:
        raise RuntimeError(f"oracle_attn_fwd failed with status {rc}")
    if full:
        return o.reshape(B, Sq, Hq, dv), lse.reshape(B, Sq, Hq).transpose(0, 2, 1).copy()
    return o, lse


def attn_bwd(q, k, v, dout, causal: bool = False, scale: float | None = None, threads: int | None = None, lib=None):
    """Reference attention backward: (dQ, dK, dV) as float64 for a loss with
    dLoss/dO = dout.  q [B,Sq,Hq,dqk], k [B,Sk,Hkv,dqk], v [B,Sk,Hkv,dv],
    dout [B,Sq,Hq,dv]; all float64, or all uint16 bf16 bit patterns."""
    arrs = [np.ascontiguousarray(x) for x in (q, k, v, dout)]
    kinds = {a.dtype for a in arrs}
    if kinds == {np.dtype(np.uint16)}:
        elem = 1
    elif kinds == {np.dtype(np.float64)}:
        elem = 0
    else:
        raise TypeError(f"q, k, v, dout must all be uint16 (bf16 bits) or all float64, got {kinds}")
    q, k, v, dout = arrs
    B, Sq, Hq, dqk = q.shape
    _, Sk, Hkv, _ = k.shape
    dv = v.shape[3]
    if dout.shape != (B, Sq, Hq, dv) or k.shape != (B, Sk, Hkv, dqk) or v.shape[:3] != (B, Sk, Hkv):
        raise ValueError("inconsistent shapes")
    if scale is None:
        scale = 1.0 / np.sqrt(dqk)
    dq = np.empty((B, Sq, Hq, dqk))
    dk = np.empty((B, Sk, Hkv, dqk))
    dvv = np.empty((B, Sk, Hkv, dv))
    rc = (lib or _load()).oracle_attn_bwd(q.ctypes.data, k.ctypes.data, v.ctypes.data, dout.ctypes.data, elem, B, Hq,
                                          Hkv, Sq, Sk, dqk, dv, int(bool(causal)), float(scale), dq.ctypes.data,
                                          dk.ctypes.data, dvv.ctypes.data, threads or default_threads())
    if rc != 0:
        raise RuntimeError(f"oracle_attn_bwd failed with status {rc}")
    return dq, dk, dvv


def attn_bwd_varlen(q, k, v, dout, cu_seqlens_q, cu_seqlens_k, causal: bool = False, scale: float | None = None,
                    threads: int | None = None, lib=None):
    """Reference attention backward of a variable-length batch laid out as
    ``attn_fwd_varlen``'s (dout like its O): ``attn_bwd`` on every sequence as
    a batch of one.  Returns (dQ [total_q,Hq,dqk], dK [total_k,Hkv,dqk],
    dV [total_k,Hkv,dv]) as float64; a sequence without queries has
    dK = dV = 0, one without keys dQ = 0; rows outside every sequence are NaN."""
    cu_q = [int(x) for x in cu_seqlens_q]
    cu_k = [int(x) for x in cu_seqlens_k]
    total_q, Hq, dqk = q.shape
    total_k, Hkv, _ = k.shape
    dvh = v.shape[2]
    dq = np.full((total_q, Hq, dqk), np.nan)
    dk = np.full((total_k, Hkv, dqk), np.nan)
    dv = np.full((total_k, Hkv, dvh), np.nan)
    for b in range(len(cu_q) - 1):
        q0, q1, k0, k1 = cu_q[b], cu_q[b + 1], cu_k[b], cu_k[b + 1]
        if q1 == q0 or k1 == k0:  # nothing flows: the gradients of whatever rows exist are 0
            dq[q0:q1] = 0.0
            dk[k0:k1] = 0.0
            dv[k0:k1] = 0.0
            continue
        g = attn_bwd(q[None, q0:q1], k[None, k0:k1], v[None, k0:k1], dout[None, q0:q1], causal, scale,
                     threads=threads, lib=lib)
        dq[q0:q1], dk[k0:k1], dv[k0:k1] = g[0][0], g[1][0], g[2][0]
    return dq, dk, dv


def row_ids(b, i, h, Sq: int, Hq: int) -> np.ndarray:
    """Linear row ids r = (b*Sq + i)*Hq + h."""
    return (np.asarray(b, dtype=np.int64) * Sq + np.asarray(i, dtype=np.int64)) * Hq + np.asarray(h, dtype=np.int64)


def attn_fwd_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, causal: bool = False, scale: float | None = None,
                    rows=None, threads: int | None = None, lib=None):
    """Reference attention forward of a variable-length batch.

    Sequence b holds queries cu_seqlens_q[b] .. cu_seqlens_q[b+1]-1 of
    q [total_q, Hq, dqk] and keys cu_seqlens_k[b] .. of k [total_k, Hkv, dqk],
    v [total_k, Hkv, dv]; each sequence is its own attention problem (its own
    softmax rows and, with ``causal``, its own bottom-right mask), so this is
    ``attn_fwd`` on every sequence as a batch of one.

    rows=None: returns (O [total_q, Hq, dv], LSE [Hq, total_q]) as float64; query
    rows outside every sequence are NaN.  rows = int64 array of (t, h) pairs
    (shape [n, 2], t a packed query row): returns (O [n, dv], LSE [n]).
    """
    cu_q = [int(x) for x in cu_seqlens_q]
    cu_k = [int(x) for x in cu_seqlens_k]
    total_q, Hq, _ = q.shape
    dv = v.shape[2]
    seq_of = np.full(total_q, -1, dtype=np.int64)
    for b in range(len(cu_q) - 1):
        seq_of[cu_q[b]:cu_q[b + 1]] = b
    if rows is None:
        o = np.full((total_q, Hq, dv), np.nan)
        lse = np.full((Hq, total_q), np.nan)
        for b in range(len(cu_q) - 1):
            q0, q1, k0, k1 = cu_q[b], cu_q[b + 1], cu_k[b], cu_k[b + 1]
            if q1 == q0:
                continue
            ob, lb = attn_fwd(q[None, q0:q1], k[None, k0:k1], v[None, k0:k1], causal, scale, threads=threads, lib=lib)
            o[q0:q1] = ob[0]
            lse[:, q0:q1] = lb[0]
        return o, lse
    rows = np.asarray(rows, dtype=np.int64).reshape(-1, 2)
    o = np.empty((rows.shape[0], dv))
    lse = np.empty(rows.shape[0])
    seqs = seq_of[rows[:, 0]]
    if (seqs < 0).any():
        raise ValueError("a requested row lies outside every sequence")
    for b in np.unique(seqs):
        sel = np.nonzero(seqs == b)[0]
        q0, q1, k0, k1 = cu_q[b], cu_q[b + 1], cu_k[b], cu_k[b + 1]
        ids = row_ids(0, rows[sel, 0] - q0, rows[sel, 1], q1 - q0, Hq)
        ob, lb = attn_fwd(q[None, q0:q1], k[None, k0:k1], v[None, k0:k1], causal, scale, rows=ids, threads=threads,
                          lib=lib)
        o[sel] = ob
        lse[sel] = lb
    return o, lse
