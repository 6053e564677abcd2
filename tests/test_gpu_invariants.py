"""Properties the definition fixes, checked on the GPU path with inputs that
are exact in bf16, plus the bounded-wait failure path."""
import math

import numpy as np
import pytest

import synth
from helpers import run_gpu, scale_for

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import head_attention_forward_gb300 as mha
    mha.build()
    mha.lib()


@pytest.mark.parametrize("d", [64, 128])
def test_single_key_is_exact(d):
    """N = 1: P = 1, l = 1, so O = V bit for bit and LSE = the one score."""
    q, k, v = synth.qkv(5, 3, 4, 1, d)
    o, lse = run_gpu(q, k, v, False)
    assert np.array_equal(o, synth.bf16_bits_to_f32(v).astype(np.float64))
    s = scale_for(d) * np.einsum("bhnd,bhnd->bhn", synth.bf16_bits_to_f32(q).astype(np.float64),
                                 synth.bf16_bits_to_f32(k).astype(np.float64))
    np.testing.assert_allclose(lse, s, atol=1e-4)


@pytest.mark.parametrize("d", [64, 128])
def test_causal_row_zero_is_exact(d):
    q, k, v = synth.qkv(6, 2, 2, 300, d)
    o, _ = run_gpu(q, k, v, True)
    assert np.array_equal(o[:, :, 0], synth.bf16_bits_to_f32(v)[:, :, 0].astype(np.float64))


@pytest.mark.parametrize("causal", [False, True])
def test_identical_value_rows(causal):
    """All v_j equal: O_i = v exactly up to bf16 rounding of P and O."""
    B, H, N, d = 1, 2, 700, 128
    q, k, _ = synth.qkv(7, B, H, N, d, sigma_qk=2.0)
    row = synth.normal_bf16(8, 2, d)
    v = np.broadcast_to(row, (B, H, N, d)).copy()
    o, _ = run_gpu(q, k, v, causal)
    ref = np.broadcast_to(synth.bf16_bits_to_f32(row).astype(np.float64), o.shape)
    assert np.abs(o - ref).max() <= 2e-2


@pytest.mark.parametrize("causal", [False, True])
def test_uniform_attention(causal):
    """Q = 0: O is the mean (causal: running mean) of V; LSE = ln |J_i|."""
    B, H, N, d = 1, 1, 513, 64
    _, k, v = synth.qkv(9, B, H, N, d)
    q = np.zeros_like(k)
    o, lse = run_gpu(q, k, v, causal)
    vf = synth.bf16_bits_to_f32(v).astype(np.float64)[0, 0]
    if causal:
        ref = np.cumsum(vf, 0) / np.arange(1, N + 1)[:, None]
        lref = np.log(np.arange(1, N + 1))
    else:
        ref = np.broadcast_to(vf.mean(0), (N, d))
        lref = np.full(N, math.log(N))
    assert np.abs(o[0, 0] - ref).max() <= 2e-2
    assert np.abs(lse[0, 0] - lref).max() <= 1e-3


def test_constant_score_shift():
    """K' = K + 1 u^T (integers, exact in bf16): O unchanged, LSE shifted."""
    rng = np.random.default_rng(3)
    B, H, N, d = 1, 2, 300, 64
    qf = rng.integers(-2, 3, (B, H, N, d)).astype(np.float32)
    kf = rng.integers(-2, 3, (B, H, N, d)).astype(np.float32)
    u = rng.integers(-1, 2, d).astype(np.float32)
    q, k, k2 = (synth.f32_to_bf16_bits(a) for a in (qf, kf, kf + u))
    v = synth.normal_bf16(4, 2, B * H * N * d).reshape(B, H, N, d)
    o1, l1 = run_gpu(q, k, v, False)
    o2, l2 = run_gpu(q, k2, v, False)
    assert np.abs(o2 - o1).max() <= 2e-2
    shift = scale_for(d) * (qf.astype(np.float64) @ u.astype(np.float64))
    assert np.abs((l2 - l1) - shift).max() <= 2e-3


def test_zero_size_is_noop():
    import head_attention_forward_gb300 as mha
    import torch
    x = torch.empty((1, 1, 0, 64), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((1, 1, 0), dtype=torch.float32, device="cuda")
    mha.mha_fwd(x, x, x, x, lse, 1, 1, 0, 64, 0.125, False)


def test_bounded_wait_times_out_and_context_survives():
    """A wait on a barrier nothing completes gives up after its budget,
    reports MHA_ERR_TIMEOUT, and the next launch still works."""
    import head_attention_forward_gb300 as mha
    rc = mha.mha_wait_selftest(2_000_000)
    assert rc == mha.MHA_ERR_TIMEOUT
    rc, word = mha.mha_device_status()
    assert rc == mha.MHA_OK and word == 0
    q, k, v = synth.qkv(1, 1, 1, 130, 64)
    o, lse = run_gpu(q, k, v, True)
    assert np.isfinite(o).all() and np.isfinite(lse).all()
