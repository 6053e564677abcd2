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
