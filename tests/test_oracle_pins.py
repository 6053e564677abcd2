"""Pins for the fp64 oracle, checked against what the definition fixes.

Every test here runs on the CPU.  Each pin is chosen so that a plausible
slip in the oracle (a dropped max subtraction, a missing 1/l, the causal
mask the wrong way round or off by one, Q and K swapped, a wrong LSE base)
fails at least one of them.  References:

* definition of the output row: Triton-learning blog, Puzzle 9 problem
  statement (z_i = sum_j softmax(q_i k_1..q_i k_T)_j v_j);
* safe softmax and the online max/sum merge: same blog, Puzzle 8;
* tile-by-tile evaluation: ML-Triton paper, section 2.5, Algorithm 1
  (FlashAttention-2 forward), and the blog's Puzzle 9 rescale rule.
"""
import json
import math
import os
import random

import numpy as np
import pytest

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "puzzle9_hand_cases.json")


def bits(x):
    """float values that are exact in bf16 -> uint16 bit patterns."""
    b = synth.f32_to_bf16_bits(np.asarray(x, dtype=np.float32))
    assert np.array_equal(synth.bf16_bits_to_f32(b), np.asarray(x, dtype=np.float32)), "not bf16-exact"
    return b


def rand_bits(seed, shape, sigma=1.0):
    n = int(np.prod(shape))
    return synth.normal_bf16(seed, 0, n, sigma).reshape(shape)


def f64(b):
    return synth.bf16_bits_to_f32(b).astype(np.float64)


# ---------------------------------------------------------------- golden
def test_hand_derived_cases():
    doc = json.load(open(GOLDEN))
    for c in doc["cases"]:
        q = bits(np.array(c["q"], dtype=np.float32))[None, None]
        k = bits(np.array(c["k"], dtype=np.float32))[None, None]
        v = bits(np.array(c["v"], dtype=np.float32))[None, None]
        o, lse = oracle.attention_fwd(q, k, v, c["scale"], c["causal"])
        np.testing.assert_allclose(o[0, 0], np.array(c["expected_o"]), rtol=0, atol=1e-12, err_msg=c["name"])
        np.testing.assert_allclose(lse[0, 0], np.array(c["expected_lse"]), rtol=0, atol=1e-12, err_msg=c["name"])


# ------------------------------------------------------------ invariants
@pytest.mark.parametrize("causal", [False, True])
def test_probability_rows_sum_to_one(causal):
    N, d = 37, 16
    q, k, v = (rand_bits(s, (N, d), 2.0) for s in (11, 12, 13))
    p, _, _ = oracle.attention_probs(q, k, v, 0.25, causal)
    np.testing.assert_allclose(p.sum(axis=1), 1.0, rtol=0, atol=1e-12)
    assert (p >= 0).all()
    if causal:  # nothing above the diagonal: key j > query i is excluded
        assert np.all(np.triu(p, 1) == 0)
        assert np.all(np.diag(p) > 0)


@pytest.mark.parametrize("causal", [False, True])
def test_identical_value_rows_reproduce_that_row(causal):
    N, d = 41, 8
    q, k = rand_bits(21, (1, 1, N, d), 3.0), rand_bits(22, (1, 1, N, d), 3.0)
    row = rand_bits(23, (d,))
    v = np.broadcast_to(row, (1, 1, N, d)).copy()
    o, _ = oracle.attention_fwd(q, k, v, 0.3, causal)
    np.testing.assert_allclose(o[0, 0], np.broadcast_to(f64(row), (N, d)), rtol=0, atol=1e-12)


def test_single_key_returns_v_and_score():
    d = 24
    q, k, v = (rand_bits(s, (2, 3, 1, d)) for s in (31, 32, 33))
    scale = np.float32(1 / math.sqrt(d))
    o, lse = oracle.attention_fwd(q, k, v, float(scale), False)
    assert np.array_equal(o, f64(v))  # P = 1 exactly
    s00 = float(scale) * np.einsum("bhnd,bhnd->bhn", f64(q), f64(k))
    np.testing.assert_allclose(lse, s00, rtol=0, atol=1e-13)


def test_causal_row_zero_is_v0():
    N, d = 9, 16
    q, k, v = (rand_bits(s, (1, 2, N, d)) for s in (41, 42, 43))
    o, lse = oracle.attention_fwd(q, k, v, 0.25, True)
    assert np.array_equal(o[:, :, 0], f64(v)[:, :, 0])
    s00 = 0.25 * np.einsum("bhd,bhd->bh", f64(q)[:, :, 0], f64(k)[:, :, 0])
    np.testing.assert_allclose(lse[:, :, 0], s00, rtol=0, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_constant_score_shift(causal):
    """K' = K + 1 u^T shifts row i's scores by scale*q_i.u: O fixed, LSE shifted."""
    rng = np.random.default_rng(5)
    N, d, scale = 19, 8, 0.125
    q = bits(rng.integers(-3, 4, (1, 1, N, d)).astype(np.float32))
    k = bits(rng.integers(-3, 4, (1, 1, N, d)).astype(np.float32))
    u = rng.integers(-2, 3, d).astype(np.float32)
    k2 = bits(synth.bf16_bits_to_f32(k) + u)
    v = rand_bits(51, (1, 1, N, d))
    o1, l1 = oracle.attention_fwd(q, k, v, scale, causal)
    o2, l2 = oracle.attention_fwd(q, k2, v, scale, causal)
    np.testing.assert_allclose(o2, o1, rtol=0, atol=1e-12)
    shift = scale * (f64(q)[0, 0] @ u.astype(np.float64))
    np.testing.assert_allclose(l2[0, 0] - l1[0, 0], shift, rtol=0, atol=1e-12)


def test_uniform_attention_closed_form():
    N, d = 33, 8
    z = np.zeros((1, 1, N, d), dtype=np.uint16)  # Q = 0: every score is 0
    k, v = rand_bits(61, (1, 1, N, d)), rand_bits(62, (1, 1, N, d))
    o, lse = oracle.attention_fwd(z, k, v, 0.7, False)
    np.testing.assert_allclose(o[0, 0], np.broadcast_to(f64(v)[0, 0].mean(0), (N, d)), atol=1e-12)
    np.testing.assert_allclose(lse[0, 0], math.log(N), atol=1e-13)
    o, lse = oracle.attention_fwd(z, k, v, 0.7, True)
    cum = np.cumsum(f64(v)[0, 0], axis=0) / np.arange(1, N + 1)[:, None]
    np.testing.assert_allclose(o[0, 0], cum, atol=1e-12)
    np.testing.assert_allclose(lse[0, 0], np.log(np.arange(1, N + 1)), atol=1e-13)


def test_two_keys_logistic():
    d = 4
    q, k, v = (rand_bits(s, (5, d), 2.0) for s in (71, 72, 73))
    q2 = np.ascontiguousarray(q)
    k2 = np.ascontiguousarray(k[:2])
    v2 = np.ascontiguousarray(v[:2])
    p, o, lse = oracle.attention_probs(np.ascontiguousarray(q2[:2]), k2, v2, 0.5, False)
    s = 0.5 * f64(q2[:2]) @ f64(k2).T
    sig = 1.0 / (1.0 + np.exp(-(s[:, 0] - s[:, 1])))
    np.testing.assert_allclose(p[:, 0], sig, atol=1e-14)
    np.testing.assert_allclose(o, sig[:, None] * f64(v2)[0] + (1 - sig)[:, None] * f64(v2)[1], atol=1e-13)


# ----------------------------------------------------------- brute force
def brute_force(qf, kf, vf, scale, causal):
    """Independent restatement: unshifted exponentials, math.fsum, lists."""
    N, d = len(qf), len(qf[0])
    O, L = [], []
    for i in range(N):
        keys = range(i + 1) if causal else range(N)
        w = [math.exp(scale * math.fsum(qf[i][c] * kf[j][c] for c in range(d))) for j in keys]
        tot = math.fsum(w)
        O.append([math.fsum(w[t] * vf[j][c] for t, j in enumerate(keys)) / tot for c in range(d)])
        L.append(math.log(tot))
    return O, L


@pytest.mark.parametrize("trial", range(6))
def test_brute_force_tiny(trial):
    r = random.Random(trial)
    N, d = r.randint(1, 8), r.randint(1, 8)
    causal = bool(trial % 2)
    scale = float(np.float32(1 / math.sqrt(d)))
    q, k, v = (rand_bits(100 * trial + s, (1, 1, N, d)) for s in range(3))
    o, lse = oracle.attention_fwd(q, k, v, scale, causal)
    O, L = brute_force(f64(q)[0, 0].tolist(), f64(k)[0, 0].tolist(), f64(v)[0, 0].tolist(), scale, causal)
    np.testing.assert_allclose(o[0, 0], np.array(O), rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse[0, 0], np.array(L), rtol=0, atol=1e-12)


def test_rows_api_matches_full():
    B, H, N, d = 2, 2, 23, 16
    q, k, v = synth.qkv(7, B, H, N, d, compiled=False)
    o, lse = oracle.attention_fwd(q, k, v, 0.25, True)
    rows = np.array([0, 5, 22, 11])
    o2, l2 = oracle.attention_rows(q, k, v, 0.25, True, 3, rows)
    assert np.array_equal(o2, o.reshape(B * H, N, d)[3][rows])
    assert np.array_equal(l2, lse.reshape(B * H, N)[3][rows])


# ------------------------------------------------- library special case
@pytest.mark.parametrize("causal", [False, True])
def test_torch_sdpa_fp64(causal):
    torch = pytest.importorskip("torch")
    B, H, N, d = 2, 3, 40, 32
    q, k, v = synth.qkv(9, B, H, N, d, compiled=False)
    scale = float(np.float32(1 / math.sqrt(d)))
    o, lse = oracle.attention_fwd(q, k, v, scale, causal)
    tq, tk, tv = (torch.from_numpy(f64(a)) for a in (q, k, v))
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=causal, scale=scale)
    np.testing.assert_allclose(o, ref.numpy(), rtol=0, atol=1e-12)
    s = scale * tq @ tk.transpose(-1, -2)
    if causal:
        s = s.masked_fill(torch.ones(N, N, dtype=torch.bool).triu(1), float("-inf"))
    np.testing.assert_allclose(lse, torch.logsumexp(s, -1).numpy(), rtol=0, atol=1e-12)


# ------------------------------------------------------ online recurrence
def online_recurrence(qf, kf, vf, scale, causal, block):
    """FlashAttention-2 forward, tile by tile (ML-Triton section 2.5,
    Algorithm 1), with the running max/sum merge of Puzzle 8 and the
    output rescale of Puzzle 9, normalised once at the end."""
    N, d = qf.shape
    O = np.zeros((N, d))
    L = np.zeros(N)
    for i in range(N):
        m, l, acc = -np.inf, 0.0, np.zeros(d)
        end = i + 1 if causal else N
        for j0 in range(0, end, block):
            j1 = min(end, j0 + block)
            s = scale * (kf[j0:j1] @ qf[i])
            m_new = max(m, s.max())
            alpha = math.exp(m - m_new) if m != -np.inf else 0.0
            p = np.exp(s - m_new)
            l = l * alpha + p.sum()
            acc = acc * alpha + p @ vf[j0:j1]
            m = m_new
        O[i] = acc / l
        L[i] = m + math.log(l)
    return O, L


@pytest.mark.parametrize("block", [1, 7, 128, 1000])
@pytest.mark.parametrize("causal", [False, True])
def test_online_recurrence_matches(block, causal):
    N, d = 150, 16
    q, k, v = synth.qkv(13, 1, 1, N, d, sigma_qk=2.0, compiled=False)
    o, lse = oracle.attention_fwd(q, k, v, 0.25, causal)
    O, L = online_recurrence(f64(q)[0, 0], f64(k)[0, 0], f64(v)[0, 0], 0.25, causal, block)
    np.testing.assert_allclose(o[0, 0], O, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse[0, 0], L, rtol=0, atol=1e-12)


def test_mask_is_square_top_left():
    """Row i sees exactly keys 0..i: perturbing key i+1 leaves row i alone,
    perturbing key i changes it."""
    N, d = 12, 8
    q, k, v = (rand_bits(s, (1, 1, N, d)) for s in (81, 82, 83))
    o, _ = oracle.attention_fwd(q, k, v, 0.5, True)
    for i in (0, 5, 10):
        v2 = v.copy()
        v2[0, 0, i + 1] = bits(np.full(d, 100.0, np.float32))
        o2, _ = oracle.attention_fwd(q, k, v2, 0.5, True)
        assert np.array_equal(o2[0, 0, : i + 1], o[0, 0, : i + 1])
        assert not np.array_equal(o2[0, 0, i + 1], o[0, 0, i + 1])


# ------------------------------------------- Nq queries against Nk keys
@pytest.mark.parametrize("causal", [False, True])
def test_kv_square_case_is_the_square_oracle(causal):
    q, k, v = synth.qkv(31, 1, 2, 37, 16, compiled=False)
    o1, l1 = oracle.attention_fwd(q, k, v, 0.25, causal)
    o2, l2 = oracle.attention_kv(q, k, v, 0.25, causal)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_kv_last_queries_match_square_rows():
    """The last Nq rows of a square causal problem are exactly the
    bottom-right aligned Nq-query problem over the same keys."""
    N, d, nq = 45, 8, 5
    q, k, v = synth.qkv(32, 1, 2, N, d, compiled=False)
    o1, l1 = oracle.attention_fwd(q, k, v, 0.5, True)
    o2, l2 = oracle.attention_kv(np.ascontiguousarray(q[:, :, N - nq:]), k, v, 0.5, True)
    assert np.array_equal(o2, o1[:, :, N - nq:]) and np.array_equal(l2, l1[:, :, N - nq:])


@pytest.mark.parametrize("causal", [False, True])
def test_kv_brute_force(causal):
    r = random.Random(9 + causal)
    for trial in range(4):
        nq, nk, d = r.randint(1, 6), r.randint(1, 9), r.randint(1, 6)
        q = rand_bits(200 + trial, (1, 1, nq, d))
        k, v = rand_bits(210 + trial, (1, 1, nk, d)), rand_bits(220 + trial, (1, 1, nk, d))
        scale = float(np.float32(0.7))  # the oracle takes the scale as fp32
        o, lse = oracle.attention_kv(q, k, v, scale, causal)
        qf, kf, vf = f64(q)[0, 0], f64(k)[0, 0], f64(v)[0, 0]
        for i in range(nq):
            keys = list(range(min(nk, nk - nq + i + 1))) if causal else list(range(nk))
            if not keys:
                assert np.all(o[0, 0, i] == 0) and lse[0, 0, i] == -np.inf
                continue
            w = [math.exp(scale * math.fsum(qf[i][c] * kf[j][c] for c in range(d))) for j in keys]
            tot = math.fsum(w)
            ref = [math.fsum(w[t] * vf[j][c] for t, j in enumerate(keys)) / tot for c in range(d)]
            np.testing.assert_allclose(o[0, 0, i], ref, rtol=0, atol=1e-12)
            assert abs(lse[0, 0, i] - math.log(tot)) < 1e-12


def test_kv_torch_sdpa_bottom_right():
    torch = pytest.importorskip("torch")
    nq, nk, d = 6, 50, 32
    q = rand_bits(301, (2, 2, nq, d))
    k, v = rand_bits(302, (2, 2, nk, d)), rand_bits(303, (2, 2, nk, d))
    o, lse = oracle.attention_kv(q, k, v, 0.125, True)
    mask = torch.ones(nq, nk, dtype=torch.bool).tril(nk - nq)
    tq, tk, tv = (torch.from_numpy(f64(a)) for a in (q, k, v))
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=mask, scale=0.125)
    np.testing.assert_allclose(o, ref.numpy(), rtol=0, atol=1e-12)
    s = (0.125 * tq @ tk.transpose(-1, -2)).masked_fill(~mask, float("-inf"))
    np.testing.assert_allclose(lse, torch.logsumexp(s, -1).numpy(), rtol=0, atol=1e-12)
