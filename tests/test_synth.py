"""The seeded input generator: determinism, the C twin, bf16 rounding."""
import numpy as np
import pytest

import synth


def test_c_twin_matches_numpy_definition():
    for seed, stream, n, sigma in [(0, 0, 1001, 1.0), (1, 1, 4096, 3.0), (4, 2, 7, 1.0)]:
        a = synth.normal_bf16(seed, stream, n, sigma)
        b = synth.normal_bf16_c(seed, stream, n, sigma)
        assert np.array_equal(a, b)


def test_deterministic_and_streams_differ():
    a = synth.normal_bf16(3, 0, 512)
    assert np.array_equal(a, synth.normal_bf16(3, 0, 512))
    assert not np.array_equal(a, synth.normal_bf16(3, 1, 512))
    assert not np.array_equal(a, synth.normal_bf16(4, 0, 512))


def test_prefix_stable():
    """Element e does not depend on how many elements are drawn."""
    a = synth.normal_bf16(5, 2, 100)
    b = synth.normal_bf16(5, 2, 333)
    assert np.array_equal(a, b[:100])


@pytest.mark.parametrize("sigma", [1.0, 3.0])
def test_moments(sigma):
    x = synth.bf16_bits_to_f32(synth.normal_bf16_c(11, 0, 1 << 20, sigma)).astype(np.float64)
    assert abs(x.mean()) < 5 * sigma / 1024
    assert abs(x.std() / sigma - 1) < 0.01
    # tail mass beyond 2 sigma of a normal distribution is 4.55%
    assert abs((np.abs(x) > 2 * sigma).mean() - 0.0455) < 0.002


def test_bf16_rounding_matches_torch():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(0)
    x = (rng.standard_normal(1 << 16) * 10).astype(np.float32)
    # include exact ties to exercise round-half-to-even
    x[:4] = np.array([1.00390625, 1.01171875, -1.00390625, 3.0], dtype=np.float32)
    ours = synth.f32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


def test_config_shapes():
    for name, c in synth.CONFIGS.items():
        assert c["d"] in (64, 128)
    q, k, v = synth.config_inputs("cfg1")
    assert q.shape == (1, 2, 128, 64) and q.dtype == np.uint16
