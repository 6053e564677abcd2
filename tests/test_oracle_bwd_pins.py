"""Pins for the oracle's attention gradients (dQ, dK, dV of sum(dO * O)).

The pages give no attention backward, so the oracle writes out the
derivative of the forward definition (Triton-learning blog, Puzzle 9
problem statement; the ML-Triton paper's FlashAttention-2, section 2.5).
These CPU tests pin it to things that do not reuse its formulas:

* central finite differences of an fp64 forward evaluated on perturbed
  inputs (the derivative itself, coordinate by coordinate);
* torch autograd through fp64 scaled_dot_product_attention;
* closed forms: one key (dV = dO, dQ = dK = 0), uniform attention
  (dV_j = sum over the rows that see key j of dO_i / |J_i|), identical keys
  (dQ = 0), and sum_j dK_j = 0 (softmax is shift invariant in the keys).

A slip such as a dropped D_i term, P in place of P^T, a missing scale, or
the causal mask the wrong way round fails at least one of them.
"""
import math

import numpy as np
import pytest

import oracle
import synth


def rand_bits(seed, stream, shape, sigma=1.0):
    n = int(np.prod(shape))
    return synth.normal_bf16(seed, stream, n, sigma).reshape(shape)


def f64(b):
    return synth.bf16_bits_to_f32(b).astype(np.float64)


def bits(x):
    b = synth.f32_to_bf16_bits(np.asarray(x, dtype=np.float32))
    assert np.array_equal(synth.bf16_bits_to_f32(b), np.asarray(x, dtype=np.float32)), "not bf16-exact"
    return b


def forward_f64(q, k, v, scale, causal):
    """softmax(scale q k^T) v for one head in fp64 on arbitrary (not bf16) inputs."""
    s = scale * (q @ k.T)
    if causal:
        s = np.where(np.tril(np.ones(s.shape, dtype=bool)), s, -np.inf)
    s = s - s.max(axis=1, keepdims=True)
    p = np.exp(s)
    p /= p.sum(axis=1, keepdims=True)
    return p @ v


@pytest.mark.parametrize("causal", [False, True])
def test_finite_differences(causal):
    N, d = 9, 5
    scale = float(np.float32(0.6))  # the oracle takes the scale as fp32
    q, k, v, do = (rand_bits(31, t, (1, 1, N, d)) for t in range(4))
    dq, dk, dv = oracle.attention_bwd(q, k, v, do, scale, causal)
    # the oracle widens bf16 exactly; use the same values, then perturb in fp64
    base = [f64(x)[0, 0] for x in (q, k, v)]
    dof = f64(do)[0, 0]
    grads = [dq[0, 0], dk[0, 0], dv[0, 0]]
    rng = np.random.default_rng(5)
    eps = 1e-6
    for _ in range(30):
        t = int(rng.integers(3))
        i, c = int(rng.integers(N)), int(rng.integers(d))
        plus = [x.copy() for x in base]
        minus = [x.copy() for x in base]
        plus[t][i, c] += eps
        minus[t][i, c] -= eps
        lp = float(np.sum(dof * forward_f64(*plus, scale, causal)))
        lm = float(np.sum(dof * forward_f64(*minus, scale, causal)))
        fd = (lp - lm) / (2 * eps)
        assert abs(fd - grads[t][i, c]) <= 1e-8 * (1 + abs(fd)), (t, i, c, fd, grads[t][i, c])


@pytest.mark.parametrize("causal", [False, True])
def test_torch_autograd_fp64(causal):
    torch = pytest.importorskip("torch")
    import torch.nn.functional as F
    B, H, N, d = 2, 2, 37, 16
    scale = float(np.float32(0.3))  # the oracle takes the scale as fp32
    q, k, v, do = (rand_bits(41, t, (B, H, N, d)) for t in range(4))
    dq, dk, dv = oracle.attention_bwd(q, k, v, do, scale, causal)
    tq, tk, tv = (torch.tensor(f64(x), requires_grad=True) for x in (q, k, v))
    o = F.scaled_dot_product_attention(tq, tk, tv, is_causal=causal, scale=scale)
    o.backward(torch.tensor(f64(do)))
    for ours, ref in ((dq, tq.grad), (dk, tk.grad), (dv, tv.grad)):
        assert np.abs(ours - ref.numpy()).max() <= 1e-10


def test_single_key():
    """N = 1: P = 1, so dV = dO and the softmax has no gradient."""
    q, k, v, do = (rand_bits(51, t, (2, 3, 1, 8)) for t in range(4))
    for causal in (False, True):
        dq, dk, dv = oracle.attention_bwd(q, k, v, do, 0.5, causal)
        assert np.array_equal(dv, f64(do))
        assert np.abs(dq).max() <= 1e-15 and np.abs(dk).max() <= 1e-15


@pytest.mark.parametrize("causal", [False, True])
def test_uniform_attention_dv(causal):
    """Q = 0 gives equal scores: P_ij = 1/|J_i|, so dV_j = sum_{i: j in J_i} dO_i / |J_i|."""
    N, d = 12, 4
    q = bits(np.zeros((1, 1, N, d)))
    k, v, do = (rand_bits(61, t, (1, 1, N, d)) for t in range(1, 4))
    _, _, dv = oracle.attention_bwd(q, k, v, do, 0.7, causal)
    dof = f64(do)[0, 0]
    for j in range(N):
        rows = range(j, N) if causal else range(N)
        want = sum(dof[i] / ((i + 1) if causal else N) for i in rows)
        assert np.abs(dv[0, 0, j] - want).max() <= 1e-13


@pytest.mark.parametrize("causal", [False, True])
def test_identical_keys_give_no_query_gradient(causal):
    """All keys equal: every score in a row is the same whatever q is, so dQ = 0."""
    N, d = 10, 6
    row = rand_bits(71, 1, (d,))
    k = np.broadcast_to(row, (1, 1, N, d)).copy()
    q, v, do = (rand_bits(71, t, (1, 1, N, d)) for t in (0, 2, 3))
    dq, _, _ = oracle.attention_bwd(q, k, v, do, 0.9, causal)
    assert np.abs(dq).max() <= 1e-13


@pytest.mark.parametrize("causal", [False, True])
def test_key_gradients_sum_to_zero(causal):
    """Adding one vector to every key shifts each score row by a constant,
    which softmax ignores; so the key gradients sum to zero."""
    q, k, v, do = (rand_bits(81, t, (1, 2, 23, 8)) for t in range(4))
    _, dk, _ = oracle.attention_bwd(q, k, v, do, 0.4, causal)
    assert np.abs(dk.sum(axis=2)).max() <= 1e-12
    assert np.abs(dk).max() > 1e-3  # not trivially zero


def test_mask_direction():
    """Under the causal mask the last key is seen only by the last query:
    its dV row is P_{N-1,N-1} dO_{N-1}, and changing earlier dO rows leaves it."""
    N, d = 6, 4
    q, k, v, do = (rand_bits(91, t, (1, 1, N, d)) for t in range(4))
    _, _, dv1 = oracle.attention_bwd(q, k, v, do, 0.5, True)
    do2 = do.copy()
    do2[0, 0, :N - 1] = rand_bits(92, 3, (N - 1, d))
    _, _, dv2 = oracle.attention_bwd(q, k, v, do2, 0.5, True)
    assert np.array_equal(dv1[0, 0, N - 1], dv2[0, 0, N - 1])
    assert not np.array_equal(dv1[0, 0, 0], dv2[0, 0, 0])
