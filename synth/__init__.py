"""Seeded synthetic inputs shared by the oracle's tests and the GPU path.

This module holds no attention arithmetic: it only turns (seed, tensor id,
element index) into normally distributed values rounded to bfloat16.  Both
sides of every parity check receive the same bf16 bytes from here.

Generator (stated so that any implementation can be checked against it):

* Counter-based SplitMix64 (Steele, Lea & Flood, "Fast splittable
  pseudorandom number generators", OOPSLA 2014; constants as published by
  Vigna).  Word ``w`` of stream ``t`` under ``seed`` is
  ``mix64(base + (w + 1) * GAMMA)`` with ``base = mix64(seed * 4 + t + 1)``
  and ``mix64`` the SplitMix64 finaliser.
* Uniforms ``u = ((w >> 11) + 1) * 2**-53`` lie in ``(0, 1]``.
* Box-Muller: words ``2p`` and ``2p + 1`` give ``u1, u2`` and the pair
  ``r*cos(2*pi*u2), r*sin(2*pi*u2)`` with ``r = sqrt(-2 ln u1)`` becomes
  elements ``2p`` and ``2p + 1`` of the tensor, in row-major order.
* Values are scaled by sigma in float64, rounded to float32, then to bfloat16
  with round-to-nearest-even on the bit pattern.

Stream ids: Q = 0, K = 1, V = 2.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22  # elements generated per numpy pass (bounded temporaries)

STREAM_Q, STREAM_K, STREAM_V = 0, 1, 2


def mix64(z: np.ndarray) -> np.ndarray:
    """SplitMix64 output finaliser on a uint64 array (wrapping arithmetic)."""
    z = z.copy()
    z ^= z >> np.uint64(30)
    z *= _M1
    z ^= z >> np.uint64(27)
    z *= _M2
    z ^= z >> np.uint64(31)
    return z


def _base(seed: int, stream: int) -> np.uint64:
    s = np.array([(seed * 4 + stream + 1) & 0xFFFFFFFFFFFFFFFF], dtype=np.uint64)
    return mix64(s)[0]


def words(seed: int, stream: int, start: int, count: int) -> np.ndarray:
    """Words ``start .. start+count-1`` of stream ``stream`` under ``seed``."""
    with np.errstate(over="ignore"):
        idx = np.arange(start + 1, start + 1 + count, dtype=np.uint64)
        return mix64(_base(seed, stream) + idx * GAMMA)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (nearest, ties to even); returns uint16 bits.

    Inputs are finite (Box-Muller output), so no NaN special case is needed.
    """
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounding = ((b >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((b + rounding) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bfloat16 bit patterns to float32."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def normal_bf16(seed: int, stream: int, n: int, sigma: float = 1.0) -> np.ndarray:
    """``n`` bf16 samples of N(0, sigma^2) as uint16 bit patterns (n even or odd)."""
    out = np.empty(n, dtype=np.uint16)
    npairs = (n + 1) // 2
    pos = 0
    two_pi = 2.0 * np.pi
    for p0 in range(0, npairs, _CHUNK // 2):
        p1 = min(npairs, p0 + _CHUNK // 2)
        w = words(seed, stream, 2 * p0, 2 * (p1 - p0))
        u = ((w >> np.uint64(11)).astype(np.float64) + 1.0) * (2.0 ** -53)
        u1, u2 = u[0::2], u[1::2]
        r = np.sqrt(-2.0 * np.log(u1))
        th = two_pi * u2
        z = np.empty(2 * (p1 - p0), dtype=np.float64)
        z[0::2] = r * np.cos(th)
        z[1::2] = r * np.sin(th)
        z *= sigma
        take = min(z.size, n - pos)
        out[pos:pos + take] = f32_to_bf16_bits(z[:take].astype(np.float32))
        pos += take
    return out


_HERE = os.path.dirname(os.path.abspath(__file__))
_CSRC = os.path.join(_HERE, "synth_gen.c")
_CLIB = os.path.join(_HERE, "_build", "libsynth_gen.so")
_clib = None


def build(force: bool = False) -> str:
    """Compile the C twin of the generator with gcc (OpenMP when available)."""
    os.makedirs(os.path.dirname(_CLIB), exist_ok=True)
    if not force and os.path.exists(_CLIB) and os.path.getmtime(_CLIB) >= os.path.getmtime(_CSRC):
        return _CLIB
    base = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-o", _CLIB, _CSRC, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True)
    return _CLIB


def _c():
    global _clib
    if _clib is None:
        build()
        lib = ctypes.CDLL(_CLIB)
        lib.synth_normal_bf16.argtypes = [ctypes.c_uint64, ctypes.c_int, ctypes.c_int64,
                                          ctypes.c_double, ctypes.c_void_p]
        lib.synth_normal_bf16.restype = None
        _clib = lib
    return _clib


def normal_bf16_c(seed: int, stream: int, n: int, sigma: float = 1.0) -> np.ndarray:
    """Same samples as :func:`normal_bf16`, produced by the compiled twin."""
    out = np.empty(n, dtype=np.uint16)
    _c().synth_normal_bf16(seed & 0xFFFFFFFFFFFFFFFF, stream, n, float(sigma),
                           out.ctypes.data_as(ctypes.c_void_p))
    return out


def qkv(seed: int, B: int, H: int, N: int, d: int,
        sigma_qk: float = 1.0, sigma_v: float = 1.0, compiled: bool = True):
    """Q, K, V as uint16 bf16 bit arrays of shape [B, H, N, d] (row-major).

    ``compiled`` selects the C twin (fast); the numpy path is the readable
    definition that the tests hold the twin to.
    """
    n = B * H * N * d
    shape = (B, H, N, d)
    gen = normal_bf16_c if compiled else normal_bf16
    q = gen(seed, STREAM_Q, n, sigma_qk).reshape(shape)
    k = gen(seed, STREAM_K, n, sigma_qk).reshape(shape)
    v = gen(seed, STREAM_V, n, sigma_v).reshape(shape)
    return q, k, v


# The workloads: (name, B, H, N, d, causal, seed, sigma_qk, sigma_v).
# Shapes, seeds and value distributions follow the benchmark family of the
# ML-Triton page (section 4.2: 32k tokens, head dim 64 or 128) as fixed for
# this library's parity and timing cases.
CONFIGS = {
    "cfg1": dict(B=1, H=2, N=128, d=64, causal=False, seed=0, sigma_qk=1.0, sigma_v=1.0),
    "cfg2": dict(B=16, H=16, N=512, d=64, causal=False, seed=1, sigma_qk=3.0, sigma_v=1.0),
    "cfg3": dict(B=4, H=16, N=2048, d=64, causal=True, seed=2, sigma_qk=1.0, sigma_v=1.0),
    "cfg4a": dict(B=2, H=32, N=4096, d=128, causal=False, seed=3, sigma_qk=1.0, sigma_v=1.0),
    "cfg4b": dict(B=2, H=32, N=4096, d=128, causal=True, seed=3, sigma_qk=1.0, sigma_v=1.0),
    "cfg5": dict(B=1, H=32, N=16384, d=128, causal=True, seed=4, sigma_qk=1.0, sigma_v=1.0),
}


def config_inputs(name: str, compiled: bool = True):
    c = CONFIGS[name]
    return qkv(c["seed"], c["B"], c["H"], c["N"], c["d"], c["sigma_qk"], c["sigma_v"], compiled)


# Decode-shaped workloads for the split-KV path: Nq queries (the newest
# positions) against Nk cached keys; K and V far larger than the 129 MB L2.
DECODE_CONFIGS = {
    "dec0": dict(B=4, H=32, Nq=1, Nk=16384, d=128, causal=False, seed=10),  # 1 GB: profiling size
    "dec1": dict(B=8, H=32, Nq=1, Nk=32768, d=128, causal=False, seed=5),
    "dec2": dict(B=1, H=32, Nq=4, Nk=131072, d=128, causal=True, seed=6),
    "dec3": dict(B=16, H=16, Nq=8, Nk=8192, d=64, causal=True, seed=7),
}


def decode_inputs(name: str, compiled: bool = True):
    """q [B,H,Nq,d], k and v [B,H,Nk,d] as bf16 bit arrays."""
    c = DECODE_CONFIGS[name]
    gen = normal_bf16_c if compiled else normal_bf16
    B, H, Nq, Nk, d = c["B"], c["H"], c["Nq"], c["Nk"], c["d"]
    q = gen(c["seed"], STREAM_Q, B * H * Nq * d).reshape(B, H, Nq, d)
    k = gen(c["seed"], STREAM_K, B * H * Nk * d).reshape(B, H, Nk, d)
    v = gen(c["seed"], STREAM_V, B * H * Nk * d).reshape(B, H, Nk, d)
    return q, k, v


# Paged-cache decode workloads: B sequences whose lengths spread between
# lo and hi keys, pages of `page` keys scattered over the cache.
PAGED_CONFIGS = {
    "pag0": dict(B=8, H=32, Nq=1, d=128, page=64, lo=2048, hi=16384, causal=False, seed=11),  # ~1.2 GB: profiling size
    "pag1": dict(B=32, H=32, Nq=1, d=128, page=16, lo=2048, hi=16384, causal=False, seed=8),
    "pag2": dict(B=32, H=32, Nq=1, d=128, page=64, lo=2048, hi=16384, causal=False, seed=9),
}


def paged_layout(name: str):
    """The paged workload's sequence lengths [B] (int32), block table
    [B, max_blocks] (int32, pages shuffled over the cache, unused entries
    -1) and cache size in blocks, without the cache itself."""
    c = PAGED_CONFIGS[name]
    B, page = c["B"], c["page"]
    w = words(c["seed"], 3, 0, B)  # stream 3: sequence lengths and page placement
    span = c["hi"] - c["lo"] + 1
    seq = (c["lo"] + (w % np.uint64(span)).astype(np.int64)).astype(np.int32)
    pages = (seq.astype(np.int64) + page - 1) // page
    max_blocks = int(pages.max())
    num_blocks = int(pages.sum())
    order = np.argsort(words(c["seed"], 4, 0, num_blocks), kind="stable").astype(np.int32)
    table = np.full((B, max_blocks), -1, dtype=np.int32)
    pos = 0
    for b in range(B):
        table[b, :pages[b]] = order[pos:pos + pages[b]]
        pos += int(pages[b])
    return seq, table, num_blocks


def paged_inputs(name: str):
    """q [B,H,Nq,d], k/v caches [num_blocks,H,page,d] (bf16 bits), block table
    [B, max_blocks] int32 (pages shuffled over the cache) and seq_lens [B]."""
    c = PAGED_CONFIGS[name]
    B, H, Nq, d, page = c["B"], c["H"], c["Nq"], c["d"], c["page"]
    seq, table, num_blocks = paged_layout(name)
    gen = normal_bf16_c
    q = gen(c["seed"], STREAM_Q, B * H * Nq * d).reshape(B, H, Nq, d)
    kc = gen(c["seed"], STREAM_K, num_blocks * H * page * d).reshape(num_blocks, H, page, d)
    vc = gen(c["seed"], STREAM_V, num_blocks * H * page * d).reshape(num_blocks, H, page, d)
    return q, kc, vc, table, seq
