"""Shared helpers for the tests: moving bf16 bit arrays onto the GPU, running
the library through its C ABI, and comparing against the oracle."""
from __future__ import annotations

import math

import numpy as np

import synth

# Agreement bar for the GPU path against the fp64 oracle.
TOL_MAX_O = 2e-2
TOL_MEAN_O = 2e-3
TOL_MAX_LSE = 1e-3


def scale_for(d: int) -> float:
    return float(np.float32(1.0 / math.sqrt(d)))


def to_device(bits: np.ndarray):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
    return t.cuda()


def bf16_to_f64(t) -> np.ndarray:
    """torch bf16 tensor (any device) -> float64 numpy, exactly."""
    import torch
    bits = t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    return synth.bf16_bits_to_f32(bits).astype(np.float64)


def run_gpu(q_bits, k_bits, v_bits, causal: bool, scale: float | None = None, poison: bool = True):
    """Run the C-ABI mha_fwd on bit arrays [B,H,N,d]; returns (O f64, LSE f64)."""
    import torch

    import head_attention_forward_gb300 as mha
    B, H, N, d = q_bits.shape
    if scale is None:
        scale = scale_for(d)
    q, k, v = to_device(q_bits), to_device(k_bits), to_device(v_bits)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    if poison:  # unwritten outputs show up as NaN
        o.fill_(float("nan"))
        lse.fill_(float("nan"))
    mha.mha_fwd(q, k, v, o, lse, B, H, N, d, scale, causal)
    rc, word = mha.mha_device_status()
    assert rc == mha.MHA_OK, f"device status {rc} word {word:#x}"
    return bf16_to_f64(o), lse.cpu().numpy().astype(np.float64)


def assert_close(o_gpu, lse_gpu, o_ref, lse_ref, what: str = ""):
    assert np.isfinite(o_gpu).all(), f"{what}: non-finite O"
    assert np.isfinite(lse_gpu).all(), f"{what}: non-finite LSE"
    do = np.abs(o_gpu - o_ref)
    dl = np.abs(lse_gpu - lse_ref)
    msg = f"{what}: max|dO|={do.max():.3e} mean|dO|={do.mean():.3e} max|dLSE|={dl.max():.3e}"
    assert do.max() <= TOL_MAX_O, msg
    assert do.mean() <= TOL_MEAN_O, msg
    assert dl.max() <= TOL_MAX_LSE, msg
    return do.max(), do.mean(), dl.max()


# Parity figures of the whole-tensor comparisons, printed at the end of the
# session (tests/conftest.py) so that a quiet run still shows them.
PARITY_STATS: list[tuple[str, float, float, float]] = []


def _source_digest() -> str:
    """Digest of the oracle's and the input generator's sources: a cached
    oracle output is reused only while both are unchanged."""
    import hashlib
    import os
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    h = hashlib.sha256()
    for rel in ("oracle/mha_oracle.c", "oracle/__init__.py", "synth/__init__.py", "synth/synth_gen.c"):
        with open(os.path.join(root, rel), "rb") as f:
            h.update(rel.encode() + b"\0" + f.read())
    return h.hexdigest()[:16]


def oracle_fwd_cached(name: str, q, k, v, scale: float, causal: bool):
    """The oracle's O and LSE for a named workload, cached on disk by
    (workload, seed, shape, sources of the oracle and the generator).

    The cache only saves the oracle's minute on a rerun; every value in it
    was written by oracle.attention_fwd.  Directory: $MHA_ORACLE_CACHE, else
    ~/.cache/mha_fwd_oracle.
    """
    import os

    import oracle
    c = synth.CONFIGS[name]
    key = (f"{name}-s{c['seed']}-{'x'.join(map(str, q.shape))}-c{int(bool(causal))}"
           f"-{np.float32(scale).view(np.uint32):08x}-{_source_digest()}")
    root = os.environ.get("MHA_ORACLE_CACHE", os.path.join(os.path.expanduser("~"), ".cache", "mha_fwd_oracle"))
    po, pl = os.path.join(root, key + ".o.npy"), os.path.join(root, key + ".lse.npy")
    if os.path.exists(po) and os.path.exists(pl):
        try:
            o, lse = np.load(po), np.load(pl)
            if o.shape == q.shape and lse.shape == q.shape[:3]:
                return o, lse
        except (OSError, ValueError):
            pass
    o, lse = oracle.attention_fwd(q, k, v, scale, causal)
    try:
        os.makedirs(root, exist_ok=True)
        for path, arr in ((po, o), (pl, lse)):
            tmp = f"{path}.{os.getpid()}.tmp"
            with open(tmp, "wb") as f:
                np.save(f, arr)
            os.replace(tmp, path)
    except OSError:
        pass  # an unwritable cache only costs the next run the oracle's time
    return o, lse
