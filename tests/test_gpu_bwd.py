"""Attention backward on the GPU against the oracle's fp64 gradients.

The forward pass (mha_fwd) supplies O and LSE, as a training step would;
mha_bwd then gives dQ, dK, dV, compared element by element with the exact
gradients of the forward definition (oracle.attention_bwd) on the same
seeded inputs.  Gradient magnitudes vary with the shape, so the bar is
relative to each tensor's largest exact entry.
"""
import numpy as np
import pytest

import oracle
import synth
from helpers import bf16_to_f64, scale_for, to_device

pytestmark = pytest.mark.gpu

# max |err| <= TOL_BWD_MAX * max |ref| and mean |err| <= TOL_BWD_MEAN * mean |ref|
TOL_BWD_MAX = 2e-2
TOL_BWD_MEAN = 1e-2


def inputs(seed, B, H, N, d, sigma_qk=1.0):
    n = B * H * N * d
    q = synth.normal_bf16(seed, 0, n, sigma_qk).reshape(B, H, N, d)
    k = synth.normal_bf16(seed, 1, n, sigma_qk).reshape(B, H, N, d)
    v = synth.normal_bf16(seed, 2, n).reshape(B, H, N, d)
    do = synth.normal_bf16(seed, 3, n).reshape(B, H, N, d)
    return q, k, v, do


def run_bwd(q, k, v, do, causal):
    import torch

    import head_attention_forward_gb300 as mha
    B, H, N, d = q.shape
    scale = scale_for(d)
    qd, kd, vd, dod = (to_device(x) for x in (q, k, v, do))
    o = torch.empty_like(qd)
    lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    mha.mha_fwd(qd, kd, vd, o, lse, B, H, N, d, scale, causal)
    grads = [torch.full_like(qd, float("nan")) for _ in range(3)]
    ws_bytes = mha.mha_bwd_workspace_size(B, H, N, d)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    mha.mha_bwd(qd, kd, vd, o, lse, dod, *grads, B, H, N, d, scale, causal, ws, ws_bytes)
    rc, word = mha.mha_device_status()
    assert rc == mha.MHA_OK, f"device status {rc} word {word:#x}"
    return [bf16_to_f64(g) for g in grads]


def check(got, ref, what):
    for name, g, r in zip(("dQ", "dK", "dV"), got, ref):
        assert np.isfinite(g).all(), f"{what} {name}: non-finite"
        err = np.abs(g - r)
        scale_max, scale_mean = np.abs(r).max(), np.abs(r).mean()
        msg = (f"{what} {name}: max|err| {err.max():.3e} (ref max {scale_max:.3e}), "
               f"mean|err| {err.mean():.3e} (ref mean {scale_mean:.3e})")
        print(msg)
        assert err.max() <= TOL_BWD_MAX * scale_max + 1e-6, msg
        assert err.mean() <= TOL_BWD_MEAN * scale_mean + 1e-7, msg


CASES = [
    # (B, H, N, d, causal)
    (1, 2, 128, 64, False), (1, 2, 128, 128, True), (2, 2, 256, 128, False),
    (2, 2, 256, 64, True), (1, 3, 1000, 64, True), (1, 2, 129, 128, False),
    (1, 2, 383, 128, True), (2, 4, 512, 64, False),
]


@pytest.mark.parametrize("case", CASES, ids=[f"B{c[0]}H{c[1]}N{c[2]}d{c[3]}{'c' if c[4] else ''}" for c in CASES])
def test_bwd_against_oracle(case):
    B, H, N, d, causal = case
    q, k, v, do = inputs(100 + N + d, B, H, N, d)
    got = run_bwd(q, k, v, do, causal)
    ref = oracle.attention_bwd(q, k, v, do, scale_for(d), causal)
    check(got, ref, str(case))


def test_bwd_sharp_scores():
    """Scores with a standard deviation near 9 (a sharp softmax)."""
    q, k, v, do = inputs(7, 2, 2, 512, 64, sigma_qk=3.0)
    got = run_bwd(q, k, v, do, False)
    ref = oracle.attention_bwd(q, k, v, do, scale_for(64), False)
    check(got, ref, "sharp")


def test_bwd_single_key():
    """N = 1: dV equals dO up to the bf16 round trip of P = 1, dQ = dK = 0."""
    q, k, v, do = inputs(9, 1, 3, 1, 128)
    dq, dk, dv = run_bwd(q, k, v, do, True)
    dof = synth.bf16_bits_to_f32(do).astype(np.float64)
    assert np.abs(dv - dof).max() <= 1e-2 * np.abs(dof).max()
    assert np.abs(dq).max() <= 1e-3 and np.abs(dk).max() <= 1e-3


def test_bwd_long_sequence_two_heads():
    """N = 2048, d = 128, causal: 16 key tiles and 16 query tiles per head."""
    q, k, v, do = inputs(11, 1, 2, 2048, 128)
    got = run_bwd(q, k, v, do, True)
    ref = oracle.attention_bwd(q, k, v, do, scale_for(128), True)
    check(got, ref, "N2048")


@pytest.mark.parametrize("causal", [False, True])
def test_bwd_tiles_fastest_launch_order(causal):
    """33 tiles per head (N = 4224, ragged): the launch order that keeps one
    head's tiles together."""
    q, k, v, do = inputs(13, 1, 2, 4224, 64)
    got = run_bwd(q, k, v, do, causal)
    ref = oracle.attention_bwd(q, k, v, do, scale_for(64), causal)
    check(got, ref, f"N4224 causal={causal}")


def test_bwd_full_workload_one_head():
    """The whole B=1, H=32, N=16384, d=128 causal workload that the backward
    benchmark times, in the same launch configuration: every gradient finite,
    and one head's dQ, dK, dV compared in full with the oracle's."""
    import torch

    import head_attention_forward_gb300 as mha
    c = synth.CONFIGS["cfg5"]
    B, H, N, d, causal = c["B"], c["H"], c["N"], c["d"], c["causal"]
    q, k, v = synth.qkv(c["seed"], B, H, N, d, c["sigma_qk"], c["sigma_v"])
    do = synth.normal_bf16_c(c["seed"], 3, B * H * N * d).reshape(B, H, N, d)
    scale = scale_for(d)
    qd, kd, vd, dod = (to_device(x) for x in (q, k, v, do))
    o = torch.empty_like(qd)
    lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    mha.mha_fwd(qd, kd, vd, o, lse, B, H, N, d, scale, causal)
    grads = [torch.full_like(qd, float("nan")) for _ in range(3)]
    ws_bytes = mha.mha_bwd_workspace_size(B, H, N, d)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    mha.mha_bwd(qd, kd, vd, o, lse, dod, *grads, B, H, N, d, scale, causal, ws, ws_bytes)
    rc, word = mha.mha_device_status()
    assert rc == mha.MHA_OK, f"device status {rc} word {word:#x}"
    for g in grads:
        assert bool(torch.isfinite(g.float()).all())
    h = 21
    got = [bf16_to_f64(g[:, h:h + 1]) for g in grads]
    one = [np.ascontiguousarray(x[:, h:h + 1]) for x in (q, k, v, do)]
    ref = oracle.attention_bwd(*one, scale, causal)
    check(got, ref, f"cfg5 head {h}")
