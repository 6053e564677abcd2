"""GPU parity of the split-KV path (a few queries against a long K/V
sequence) against the fp64 oracle, through the C ABI."""
import math

import numpy as np
import pytest

import oracle
import synth
from helpers import TOL_MAX_LSE, TOL_MAX_O, TOL_MEAN_O, bf16_to_f64, scale_for, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import head_attention_forward_gb300 as mha
    mha.build()
    mha.lib()


def run_kv(q_bits, k_bits, v_bits, causal, num_splits=0, scale=None):
    import torch

    import head_attention_forward_gb300 as mha
    B, H, Nq, d = q_bits.shape
    Nk = k_bits.shape[2]
    if scale is None:
        scale = scale_for(d)
    q, k, v = to_device(q_bits), to_device(k_bits), to_device(v_bits)
    o = torch.full_like(q, float("nan"))
    lse = torch.full((B, H, Nq), float("nan"), dtype=torch.float32, device="cuda")
    ws_bytes = mha.mha_fwd_kv_workspace_size(B, H, Nq, Nk, d, num_splits)
    ws = torch.full((max(ws_bytes, 16),), 0xFF, dtype=torch.uint8, device="cuda")  # garbage in
    mha.mha_fwd_kv(q, k, v, o, lse, B, H, Nq, Nk, d, scale, causal, num_splits, ws, ws_bytes)
    rc, word = mha.mha_device_status()
    assert rc == mha.MHA_OK, f"device status {rc} word {word:#x}"
    return bf16_to_f64(o), lse.cpu().numpy().astype(np.float64)


def compare(o, lse, o_ref, lse_ref, what):
    empty = np.isneginf(lse_ref)
    assert np.array_equal(np.isneginf(lse), empty), what
    assert np.all(o[empty] == 0), what
    do = np.abs(o - o_ref)
    dl = np.abs(lse[~empty] - lse_ref[~empty]) if (~empty).any() else np.zeros(1)
    msg = f"{what}: max|dO|={do.max():.3e} mean|dO|={do.mean():.3e} max|dLSE|={dl.max():.3e}"
    assert np.isfinite(o).all(), msg
    assert do.max() <= TOL_MAX_O and do.mean() <= TOL_MEAN_O and dl.max() <= TOL_MAX_LSE, msg


def qkv(seed, B, H, Nq, Nk, d, sigma=1.0):
    q = synth.normal_bf16(seed, synth.STREAM_Q, B * H * Nq * d, sigma).reshape(B, H, Nq, d)
    k = synth.normal_bf16(seed, synth.STREAM_K, B * H * Nk * d, sigma).reshape(B, H, Nk, d)
    v = synth.normal_bf16(seed, synth.STREAM_V, B * H * Nk * d).reshape(B, H, Nk, d)
    return q, k, v


CASES = [
    # (B, H, Nq, Nk, d)
    (1, 1, 1, 1, 64), (1, 2, 1, 63, 128), (2, 1, 3, 64, 64), (1, 1, 16, 65, 128),
    (1, 3, 5, 1000, 64), (2, 2, 1, 4113, 128), (1, 1, 16, 16, 128), (1, 2, 7, 3, 64),
]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("case", CASES)
def test_splitkv_shapes(case, causal):
    B, H, Nq, Nk, d = case
    q, k, v = qkv(50 + Nk, B, H, Nq, Nk, d)
    o, lse = run_kv(q, k, v, causal)
    o_ref, lse_ref = oracle.attention_kv(q, k, v, scale_for(d), causal)
    compare(o, lse, o_ref, lse_ref, f"{case} causal={causal}")


@pytest.mark.parametrize("splits", [1, 2, 5, 64])
def test_splitkv_split_counts(splits):
    q, k, v = qkv(7, 1, 2, 4, 3000, 128, sigma=2.0)
    o, lse = run_kv(q, k, v, True, num_splits=splits)
    o_ref, lse_ref = oracle.attention_kv(q, k, v, scale_for(128), True)
    compare(o, lse, o_ref, lse_ref, f"splits={splits}")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("splits", [0, 3])
def test_splitkv_running_max_paths(d, splits):
    """Scores g_i * f_j with f rising along the keys and per-query slopes
    g_i from [-30, 30]: within one warp some rows' maxima fall behind, some
    rise by less than the rescale threshold per tile and some by more."""
    B, H, Nq, Nk = 1, 3, 16, 3000
    rng = np.random.default_rng(321 + d + splits)
    qf = rng.standard_normal((B, H, Nq, d)).astype(np.float32) * 0.1
    kf = rng.standard_normal((B, H, Nk, d)).astype(np.float32) * 0.1
    qf[..., 0] = rng.uniform(-30.0, 30.0, size=(B, H, Nq))
    kf[..., 0] = np.linspace(0.0, 100.0, Nk, dtype=np.float32)[None, None, :]
    q, k = synth.f32_to_bf16_bits(qf), synth.f32_to_bf16_bits(kf)
    v = synth.f32_to_bf16_bits(rng.standard_normal((B, H, Nk, d)).astype(np.float32))
    for causal in (False, True):
        o, lse = run_kv(q, k, v, causal, num_splits=splits)
        o_ref, lse_ref = oracle.attention_kv(q, k, v, scale_for(d), causal)
        compare(o, lse, o_ref, lse_ref, f"ramp d={d} splits={splits} causal={causal}")


def test_splitkv_square_matches_fused():
    """With Nq == Nk <= 16 both entry points compute the same rows."""
    import torch

    import head_attention_forward_gb300 as mha
    q, k, v = qkv(11, 2, 2, 16, 16, 64)
    o1, l1 = run_kv(q, k, v, True)
    qd, kd, vd = to_device(q), to_device(k), to_device(v)
    o2, l2 = mha.forward(qd, kd, vd, causal=True)
    torch.cuda.synchronize()
    assert np.abs(o1 - bf16_to_f64(o2)).max() <= 2e-2
    assert np.abs(l1 - l2.cpu().numpy()).max() <= 1e-4


def test_splitkv_long_decode_sampled_heads():
    """A long decode-sized problem (one query, 32k keys) on a few heads."""
    B, H, Nq, Nk, d = 1, 8, 1, 32768, 128
    q, k, v = qkv(12, B, H, Nq, Nk, d)
    o, lse = run_kv(q, k, v, False)
    o_ref, lse_ref = oracle.attention_kv(q, k, v, scale_for(d), False)
    compare(o, lse, o_ref, lse_ref, "decode 32k")


@pytest.mark.parametrize("name", ["dec2", "dec3"])
def test_splitkv_full_workload_sampled_heads(name):
    """A whole decode workload in one call (dec2: 4 queries x 128k keys
    causal; dec3: 8 queries x 8k keys, d=64, causal); a few heads checked
    against the oracle, every output checked finite."""
    qb, kb, vb = synth.decode_inputs(name)
    c = synth.DECODE_CONFIGS[name]
    o, lse = run_kv(qb, kb, vb, c["causal"])
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    B, H = qb.shape[:2]
    for (b, h) in {(0, 0), (B - 1, H - 1), (B // 2, H // 3)}:
        o_ref, l_ref = oracle.attention_kv(qb[b:b + 1, h:h + 1], kb[b:b + 1, h:h + 1],
                                           vb[b:b + 1, h:h + 1], scale_for(c["d"]), c["causal"])
        compare(o[b:b + 1, h:h + 1], lse[b:b + 1, h:h + 1], o_ref, l_ref, f"{name} ({b},{h})")


def test_splitkv_in_cuda_graph():
    """The split-KV call captured in a CUDA graph (its counter reset and the
    two dependent kernels) and replayed three times on a dirty workspace gives the
    result of a direct call, bit for bit, and the forward pass captured the
    same way matches its direct call too."""
    import torch

    import head_attention_forward_gb300 as mha
    B, H, Nq, Nk, d = 2, 4, 3, 3000, 128
    q = to_device(synth.normal_bf16(31, 0, B * H * Nq * d).reshape(B, H, Nq, d))
    k = to_device(synth.normal_bf16(31, 1, B * H * Nk * d).reshape(B, H, Nk, d))
    v = to_device(synth.normal_bf16(31, 2, B * H * Nk * d).reshape(B, H, Nk, d))
    scale = scale_for(d)
    ws_bytes = mha.mha_fwd_kv_workspace_size(B, H, Nq, Nk, d, 0)
    ws = torch.full((ws_bytes,), 0xFF, dtype=torch.uint8, device="cuda")
    o_ref = torch.empty_like(q)
    l_ref = torch.empty((B, H, Nq), dtype=torch.float32, device="cuda")
    mha.mha_fwd_kv(q, k, v, o_ref, l_ref, B, H, Nq, Nk, d, scale, True, 0, ws, ws_bytes)
    o = torch.full_like(q, float("nan"))
    lse = torch.full_like(l_ref, float("nan"))
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            mha.mha_fwd_kv(q, k, v, o, lse, B, H, Nq, Nk, d, scale, True, 0, ws, ws_bytes, side)
    for _ in range(3):
        ws.fill_(0xFF)
        graph.replay()
    torch.cuda.synchronize()
    rc, word = mha.mha_device_status()
    assert rc == mha.MHA_OK, f"device status {rc} word {word:#x}"
    assert torch.equal(o, o_ref) and torch.equal(lse, l_ref)

    N = 1000
    qf = to_device(synth.normal_bf16(32, 0, B * H * N * d).reshape(B, H, N, d))
    kf = to_device(synth.normal_bf16(32, 1, B * H * N * d).reshape(B, H, N, d))
    vf = to_device(synth.normal_bf16(32, 2, B * H * N * d).reshape(B, H, N, d))
    of_ref, lf_ref = torch.empty_like(qf), torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    mha.mha_fwd(qf, kf, vf, of_ref, lf_ref, B, H, N, d, scale, True)
    of, lf = torch.full_like(qf, float("nan")), torch.full_like(lf_ref, float("nan"))
    torch.cuda.synchronize()
    graph2 = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph2, stream=side):
            mha.mha_fwd(qf, kf, vf, of, lf, B, H, N, d, scale, True, side)
    graph2.replay()
    torch.cuda.synchronize()
    assert torch.equal(of, of_ref) and torch.equal(lf, lf_ref)
