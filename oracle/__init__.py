"""TEST INFRASTRUCTURE ONLY: the fp64 CPU oracle for attention forward
(and its gradients).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The library's product path never
imports it, and it shares no code with the CUDA side.

The arithmetic lives in ``mha_oracle.c`` (plain C, fp64, OpenMP over query
rows); this module compiles it with gcc and marshals numpy arrays.  See the
C file's header for the definition followed and the readings taken.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mha_oracle.c")
_LIB = os.path.join(_HERE, "_build", "libmha_oracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP if the toolchain has it)."""
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    base = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-o", _LIB, _SRC, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        p = ctypes.c_void_p
        i64 = ctypes.c_int64
        lib.oracle_attention_rows.argtypes = [p, p, p, i64, i64, ctypes.c_float, ctypes.c_int,
                                              p, i64, p, p, ctypes.c_int]
        lib.oracle_attention_rows.restype = ctypes.c_int
        lib.oracle_attention_fwd.argtypes = [p, p, p, i64, i64, i64, ctypes.c_float, ctypes.c_int,
                                             p, p, ctypes.c_int]
        lib.oracle_attention_fwd.restype = ctypes.c_int
        lib.oracle_attention_probs.argtypes = [p, p, p, i64, i64, ctypes.c_float, ctypes.c_int,
                                               p, p, p]
        lib.oracle_attention_probs.restype = ctypes.c_int
        lib.oracle_num_threads.restype = ctypes.c_int
        lib.oracle_attention_kv.argtypes = [p, p, p, i64, i64, i64, ctypes.c_float, ctypes.c_int,
                                            p, p, ctypes.c_int]
        lib.oracle_attention_kv.restype = ctypes.c_int
        lib.oracle_attention_bwd.argtypes = [p, p, p, p, i64, i64, i64, ctypes.c_float, ctypes.c_int,
                                             p, p, p, ctypes.c_int]
        lib.oracle_attention_bwd.restype = ctypes.c_int
        _lib = lib
    return _lib


def _bits(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError("oracle inputs are bfloat16 bit patterns (uint16)")
    return a


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def attention_fwd(q, k, v, scale: float, causal: bool, nthreads: int = 0):
    """O [B,H,N,d] float64 and LSE [B,H,N] float64 for bf16-bit inputs."""
    q, k, v = _bits(q), _bits(k), _bits(v)
    if not (q.shape == k.shape == v.shape) or q.ndim != 4:
        raise ValueError("q, k, v must share one [B, H, N, d] shape")
    B, H, N, d = q.shape
    o = np.zeros((B, H, N, d), dtype=np.float64)
    lse = np.zeros((B, H, N), dtype=np.float64)
    rc = _load().oracle_attention_fwd(_ptr(q), _ptr(k), _ptr(v), B * H, N, d,
                                      ctypes.c_float(scale), int(bool(causal)),
                                      _ptr(o), _ptr(lse), int(nthreads))
    if rc != 0:
        raise RuntimeError("oracle_attention_fwd failed")
    return o, lse


def attention_rows(q, k, v, scale: float, causal: bool, bh: int, rows, nthreads: int = 0):
    """O [len(rows), d] and LSE [len(rows)] for query rows of head ``bh``.

    ``bh`` indexes the flattened B*H axis of [B, H, N, d] inputs.
    """
    q, k, v = _bits(q), _bits(k), _bits(v)
    B, H, N, d = q.shape
    qb = q.reshape(B * H, N, d)[bh]
    kb = k.reshape(B * H, N, d)[bh]
    vb = v.reshape(B * H, N, d)[bh]
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    o = np.zeros((rows.size, d), dtype=np.float64)
    lse = np.zeros(rows.size, dtype=np.float64)
    rc = _load().oracle_attention_rows(_ptr(qb), _ptr(kb), _ptr(vb), N, d,
                                       ctypes.c_float(scale), int(bool(causal)),
                                       _ptr(rows), rows.size, _ptr(o), _ptr(lse), int(nthreads))
    if rc != 0:
        raise RuntimeError("oracle_attention_rows failed")
    return o, lse


def attention_probs(q, k, v, scale: float, causal: bool):
    """P [N,N], O [N,d], LSE [N] of a single head given [N, d] inputs."""
    q, k, v = _bits(q), _bits(k), _bits(v)
    N, d = q.shape
    p = np.zeros((N, N), dtype=np.float64)
    o = np.zeros((N, d), dtype=np.float64)
    lse = np.zeros(N, dtype=np.float64)
    rc = _load().oracle_attention_probs(_ptr(q), _ptr(k), _ptr(v), N, d, ctypes.c_float(scale),
                                        int(bool(causal)), _ptr(p), _ptr(o), _ptr(lse))
    if rc != 0:
        raise RuntimeError("oracle_attention_probs failed")
    return p, o, lse


def attention_kv(q, k, v, scale: float, causal: bool, nthreads: int = 0):
    """Nq queries against Nk keys: q [B,H,Nq,d], k/v [B,H,Nk,d] bf16 bits.

    Causal here is bottom-right aligned (the queries are the last Nq
    positions): query i sees keys 0 .. Nk-Nq+i.  Returns O [B,H,Nq,d] and
    LSE [B,H,Nq] in float64.
    """
    q, k, v = _bits(q), _bits(k), _bits(v)
    if q.ndim != 4 or k.shape != v.shape or q.shape[:2] != k.shape[:2] or q.shape[3] != k.shape[3]:
        raise ValueError("q [B,H,Nq,d] and k, v [B,H,Nk,d] expected")
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    o = np.zeros((B, H, Nq, d), dtype=np.float64)
    lse = np.zeros((B, H, Nq), dtype=np.float64)
    lib = _load()
    for bh in range(B * H):
        b, h = divmod(bh, H)
        qb = np.ascontiguousarray(q[b, h])
        kb = np.ascontiguousarray(k[b, h])
        vb = np.ascontiguousarray(v[b, h])
        ob = np.zeros((Nq, d), dtype=np.float64)
        lb = np.zeros(Nq, dtype=np.float64)
        rc = lib.oracle_attention_kv(_ptr(qb), _ptr(kb), _ptr(vb), Nq, Nk, d, ctypes.c_float(scale),
                                     int(bool(causal)), _ptr(ob), _ptr(lb), int(nthreads))
        if rc != 0:
            raise RuntimeError("oracle_attention_kv failed")
        o[b, h] = ob
        lse[b, h] = lb
    return o, lse


def attention_bwd(q, k, v, dout, scale: float, causal: bool, nthreads: int = 0):
    """dQ, dK, dV [B,H,N,d] float64: the gradients of sum(dout * O) for the
    attention output O of ``attention_fwd`` (same scale and mask)."""
    q, k, v, dout = _bits(q), _bits(k), _bits(v), _bits(dout)
    if not (q.shape == k.shape == v.shape == dout.shape) or q.ndim != 4:
        raise ValueError("q, k, v, dout must share one [B, H, N, d] shape")
    B, H, N, d = q.shape
    dq = np.zeros((B, H, N, d), dtype=np.float64)
    dk = np.zeros_like(dq)
    dv = np.zeros_like(dq)
    rc = _load().oracle_attention_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), B * H, N, d,
                                      ctypes.c_float(scale), int(bool(causal)),
                                      _ptr(dq), _ptr(dk), _ptr(dv), int(nthreads))
    if rc != 0:
        raise RuntimeError("oracle_attention_bwd failed")
    return dq, dk, dv
