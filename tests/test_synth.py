"""The seeded input generators (CPU): splitmix64 against its published
sequence, counter-form consistency, the distributions, determinism and
stream independence, the rounding to the storage dtype, and the rotary tables."""
import math

import numpy as np
import torch

import synth


def test_splitmix64_reference_sequence():
    """With key 0 the counter form is plain SplitMix64 seeded with 0, whose first
    outputs are published with the generator (Steele, Lea & Flood, OOPSLA 2014;
    the reference C implementation's test vector)."""
    want = [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]
    with np.errstate(over="ignore"):
        got = [int(synth._mix(np.array([synth.GAMMA * np.uint64(i + 1)], dtype=np.uint64))[0])
               for i in range(3)]
    assert got == want


def test_counter_form_offsets_and_chunks():
    long = synth.words(7, 3, 5000)
    np.testing.assert_array_equal(synth.words(7, 3, 100, offset=1234), long[1234:1334])
    old = synth._CHUNK
    try:
        synth._CHUNK = 64                     # force many chunks: same stream
        np.testing.assert_array_equal(synth.words(7, 3, 5000), long)
        np.testing.assert_array_equal(synth.normal(7, 3, 999), _normal_unchunked(7, 3, 999))
    finally:
        synth._CHUNK = old


def _normal_unchunked(seed, stream, count):
    n = (count + 1) // 2
    u = ((synth.words(seed, stream, 2 * n) >> np.uint64(11)).astype(np.float64) + 1.0) * 2.0 ** -53
    r = np.sqrt(-2.0 * np.log(u[0::2]))
    z = np.empty(2 * n)
    z[0::2], z[1::2] = r * np.cos(2 * np.pi * u[1::2]), r * np.sin(2 * np.pi * u[1::2])
    return z[:count]


def test_distributions():
    n = 1 << 20
    u = synth.uniform(1, 0, n)
    assert u.min() > 0.0 and u.max() <= 1.0
    assert abs(u.mean() - 0.5) < 4 * math.sqrt(1 / 12 / n)
    z = synth.normal(1, 1, n)
    assert abs(z.mean()) < 4 / math.sqrt(n)
    assert abs(z.var() - 1.0) < 4 * math.sqrt(2 / n)
    assert abs(np.mean(np.abs(z) < 1.0) - 0.6826894921370859) < 4 * math.sqrt(0.25 / n)


def test_determinism_and_stream_independence():
    a = synth.attention_inputs(1, 2, 33, 16, "bf16", seed=5)
    b = synth.attention_inputs(1, 2, 33, 16, "bf16", seed=5)
    for x, y in zip(a, b):
        assert torch.equal(x, y)
    q, k, v = a
    assert not torch.equal(q, k) and not torch.equal(k, v)
    c = synth.attention_inputs(1, 2, 33, 16, "bf16", seed=6)
    assert not torch.equal(a[0], c[0])
    corr = np.corrcoef(synth.normal(5, 0, 50000), synth.normal(5, 1, 50000))[0, 1]
    assert abs(corr) < 4 / math.sqrt(50000)


def test_rounding_to_storage_dtype():
    """Draws are rounded through float32 to the storage dtype, both steps to
    nearest even; every value is exactly representable afterwards."""
    x = synth.normal(2, 0, 4096)
    t = synth.as_dtype(x, (4096,), "bf16")
    assert t.dtype == torch.bfloat16
    assert torch.equal(t, torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16))
    assert torch.equal(t.float().to(torch.bfloat16), t)


def test_outliers_and_signs():
    q, _, _ = synth.outlier_inputs(1, 4, 1024, 128, "fp32", seed=3)
    big = (q.abs() > 6).float().mean().item()
    assert 0.0002 < big < 0.002                  # ~0.1 % outliers of sigma 10, few N(0,1) tails
    s = synth.hadamard_signs(16, 128, seed=1)
    assert s.dtype == torch.int8 and set(s.unique().tolist()) == {-1, 1}
    assert abs(s.float().mean().item()) < 4 / math.sqrt(16 * 128)


def test_rotary_tables():
    c, s = synth.rotary_tables(50, 64, offset=0)
    assert c.shape == s.shape == (50, 32) and c.dtype == torch.float32
    np.testing.assert_allclose((c ** 2 + s ** 2).numpy(), 1.0, rtol=0, atol=2e-7)
    assert torch.all(c[0] == 1) and torch.all(s[0] == 0)    # position 0: zero angles
    c7, s7 = synth.rotary_tables(43, 64, offset=7)
    assert torch.equal(c7, c[7:]) and torch.equal(s7, s[7:])
    np.testing.assert_allclose(s[:, 0].numpy(), np.sin(np.arange(50)).astype(np.float32), rtol=0, atol=1e-7)
