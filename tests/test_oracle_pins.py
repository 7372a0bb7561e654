"""The float64 oracle against what the pages and the mathematics fix (CPU only)."""
from __future__ import annotations

import math

import numpy as np
import pytest
import scipy.linalg
import torch

import oracle
import synth
from tests import pins


def _attn(q, k, v, causal, scale, rows=None):
    return oracle.attention(q, k, v, causal=causal, scale=scale, rows=rows)


@pytest.mark.parametrize("check", pins.ALL_CHECKS, ids=lambda c: c.__name__)
def test_attention_pin(check):
    check(_attn)


def test_thread_count_does_not_change_results():
    q, k, v = synth.attention_inputs(1, 3, 67, 16, "bf16", seed=5)
    o1, l1 = oracle.attention(q, k, v, causal=True, nthreads=1)
    o2, l2, used = oracle.attention(q, k, v, causal=True, nthreads=5, return_threads=True)
    assert used == 5
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)


# ----------------------------------------------------------------- E4M3 codec

# Points of the OCP 8-bit floating point specification, E4M3 column: zero, the
# smallest subnormal 2^-9, the largest subnormal 7 * 2^-9, the smallest normal
# 2^-6, one, the largest finite 448 = 1.75 * 2^8, and the NaN encodings.
_OCP_POINTS = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6, 0x38: 1.0,
               0x3F: 1.875, 0x40: 2.0, 0x7E: 448.0, 0x80: -0.0, 0xFE: -448.0}


def test_e4m3_decode_spec_points():
    vals = oracle.e4m3_decode(np.arange(256, dtype=np.uint8))
    for code, want in _OCP_POINTS.items():
        assert vals[code] == want and math.copysign(1, vals[code]) == math.copysign(1, want), hex(code)
    assert math.isnan(vals[0x7F]) and math.isnan(vals[0xFF])


def test_e4m3_decode_matches_library():
    """All 256 codes against PyTorch's float8_e4m3fn (same OCP format)."""
    ours = oracle.e4m3_decode(np.arange(256, dtype=np.uint8))
    lib = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    np.testing.assert_array_equal(ours, lib)


def test_e4m3_encode_round_trip_and_ties():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    back = oracle.e4m3_encode(oracle.e4m3_decode(codes))
    np.testing.assert_array_equal(back, codes)
    # ties go to the even mantissa: 1 + 1/16 lies halfway between 1 and 1.125
    assert oracle.e4m3_encode(np.array([1.0625]))[0] == 0x38
    assert oracle.e4m3_encode(np.array([1.1875]))[0] == 0x3A  # between 1.125 and 1.25 -> 1.25
    # saturation instead of overflow
    np.testing.assert_array_equal(oracle.e4m3_encode(np.array([449.0, 1e9, -1e9, 465.0])),
                                  np.array([0x7E, 0x7E, 0xFE, 0x7E], dtype=np.uint8))


def test_e4m3_encode_matches_library_in_range():
    """Random and midpoint values below the overflow threshold against PyTorch's
    round-to-nearest-even float32 -> float8_e4m3fn conversion."""
    grid = np.sort(oracle.e4m3_decode(np.arange(0x00, 0x7F, dtype=np.uint8)))
    mids = (grid[:-1] + grid[1:]) / 2
    rnd = np.random.default_rng(7).standard_normal(20000) * np.exp2(
        np.random.default_rng(8).uniform(-12, 8, 20000))
    x = np.concatenate([mids, -mids, rnd, grid, -grid]).astype(np.float32)
    x = x[np.abs(x) < 448.0]
    ours = oracle.e4m3_encode(x.astype(np.float64))
    lib = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(ours, lib)


# ---------------------------------------------------------- Hadamard rotation

@pytest.mark.parametrize("d", [1, 2, 4, 8, 64, 128, 256])
def test_hadamard_matrix_is_sylvester(d):
    h = oracle.hadamard_matrix(d)
    np.testing.assert_array_equal(h, scipy.linalg.hadamard(d))
    np.testing.assert_array_equal(h @ h.T, d * np.eye(d))


def test_hadamard_rotate_matches_dense_product():
    B, H, N, d = 1, 3, 9, 64
    x = np.random.default_rng(3).standard_normal((B, H, N, d))
    signs = synth.hadamard_signs(H, d, seed=4).numpy()
    got = oracle.hadamard_rotate(x, signs)
    hd = scipy.linalg.hadamard(d).astype(np.float64)
    for h in range(H):
        want = (x[0, h] * signs[h]) @ hd / math.sqrt(d)
        np.testing.assert_allclose(got[0, h], want, rtol=0, atol=1e-12)
    np.testing.assert_allclose(np.linalg.norm(got, axis=-1), np.linalg.norm(x, axis=-1), rtol=1e-13)


def test_rotation_leaves_attention_unchanged():
    """The rotation is orthogonal and shared by Q and K, so Q K^T is unchanged
    (the reason it is legal, "Incoherent Processing for FP8 Accuracy")."""
    q, k, v = synth.attention_inputs(1, 2, 70, 128, "bf16", seed=9)
    signs = synth.hadamard_signs(2, 128, seed=9)
    qr, kr = oracle.hadamard_rotate(q, signs), oracle.hadamard_rotate(k, signs)
    for causal in (False, True):
        o1, l1 = oracle.attention(q, k, v, causal=causal)
        o2, l2 = oracle.attention(qr, kr, v, causal=causal)
        np.testing.assert_allclose(o2, o1, rtol=0, atol=1e-11)
        np.testing.assert_allclose(l2, l1, rtol=0, atol=1e-11)


def test_rotation_spreads_outliers():
    """A single spike becomes a flat +-spike/sqrt(d) vector: the peak drops by sqrt(d)."""
    d = 128
    x = np.zeros((1, 1, 1, d))
    x[0, 0, 0, 17] = 100.0
    y = oracle.hadamard_rotate(x, np.ones((1, d), dtype=np.int8))
    np.testing.assert_allclose(np.abs(y), 100.0 / math.sqrt(d), rtol=1e-14)


# -------------------------------------------------------- block quantisation

def test_block_quantize_scales_and_error_bound():
    B, H, N, d = 1, 2, 300, 64   # ragged last block (300 = 2 * 128 + 44)
    x = synth.outlier_inputs(B, H, N, d, "bf16", seed=2)[0].double().numpy()
    codes, scales = oracle.block_quantize(x)
    assert scales.shape == (B, H, 3) and scales.dtype == np.float32
    for h in range(H):
        for b in range(3):
            blk = x[0, h, b * 128:(b + 1) * 128]
            assert scales[0, h, b] == np.float32(np.float32(np.abs(blk).max()) / np.float32(448.0))
            arg = np.unravel_index(np.abs(blk).argmax(), blk.shape)
            assert codes[0, h, b * 128 + arg[0], arg[1]] & 0x7F == 0x7E   # amax -> +-448
    deq = oracle.dequantize(codes, scales)
    s = np.repeat(scales.astype(np.float64), 128, axis=-1)[..., :N, None]
    # half a step of E4M3: 2^-4 relative for normals, 2^-10 * s below 2^-6 * s
    bound = np.maximum(np.abs(x) * 2.0 ** -4, s * 2.0 ** -10) * (1 + 1e-6)
    assert np.all(np.abs(deq - x) <= bound)


def test_block_quantize_matches_library_rounding():
    x = np.random.default_rng(11).standard_normal((1, 1, 256, 32)) * 3
    codes, scales = oracle.block_quantize(x)
    for b in range(2):
        blk = torch.from_numpy(x[0, 0, b * 128:(b + 1) * 128].astype(np.float32))
        want = (blk / torch.tensor(scales[0, 0, b])).to(torch.float8_e4m3fn).view(torch.uint8)
        np.testing.assert_array_equal(codes[0, 0, b * 128:(b + 1) * 128], want.numpy())


def test_block_quantize_blocks_are_independent():
    x = np.random.default_rng(12).standard_normal((1, 1, 256, 16))
    c1, s1 = oracle.block_quantize(x)
    x2 = x.copy()
    x2[0, 0, 200, 3] = 1000.0       # only the second block changes
    c2, s2 = oracle.block_quantize(x2)
    np.testing.assert_array_equal(c1[0, 0, :128], c2[0, 0, :128])
    assert s1[0, 0, 0] == s2[0, 0, 0] and s1[0, 0, 1] != s2[0, 0, 1]


def test_per_tensor_scale_and_zero_input():
    x = np.random.default_rng(13).standard_normal((2, 2, 50, 8))
    _, s = oracle.block_quantize(x, per_tensor=True)
    assert s.shape == (1,) and s[0] == np.float32(np.float32(np.abs(x).max()) / np.float32(448.0))
    c0, s0 = oracle.block_quantize(np.zeros((1, 1, 5, 8)))
    assert np.all(c0 == 0) and np.all(s0 == 1.0)


def test_fp8_pipeline_is_close_to_exact_attention():
    """Without outliers the quantised pipeline stays within a few 1e-3 RMS."""
    q, k, v = synth.attention_inputs(1, 2, 256, 128, "bf16", seed=3)
    signs = synth.hadamard_signs(2, 128, seed=3)
    o_ref, _ = oracle.attention(q, k, v)
    o8, _ = oracle.fp8_pipeline(q, k, v, signs)
    rms = float(np.sqrt(np.mean((o8 - o_ref) ** 2)))
    assert rms < 5e-3


def test_rows_without_keys_are_rejected():
    """A row that sees no key has no softmax: Nk = 0, or the end-aligned mask
    with more queries than keys."""
    q, k = np.zeros((1, 1, 4, 2)), np.zeros((1, 1, 3, 2))
    with pytest.raises(RuntimeError):
        oracle.attention(q, k, k, causal=2, scale=1.0)
    with pytest.raises(RuntimeError):
        oracle.attention(q, np.zeros((1, 1, 0, 2)), np.zeros((1, 1, 0, 2)), scale=1.0)
    o, lse = oracle.attention(q, k, k, causal=1, scale=1.0)  # rows 3.. see all 3 keys
    np.testing.assert_allclose(lse[0, 0], np.log([1, 2, 3, 3]), rtol=0, atol=1e-15)


def test_rotary_is_complex_multiplication():
    pins.check_rotary_complex(lambda x, c, s, inter: oracle.rotary(x, c, s, interleaved=inter))


def test_rotary_zero_angle_is_identity_and_norms_are_kept():
    x = np.random.default_rng(82).standard_normal((1, 2, 7, 16))
    one, zero = np.ones((7, 8), np.float32), np.zeros((7, 8), np.float32)
    for inter in (False, True):
        np.testing.assert_array_equal(oracle.rotary(x, one, zero, inter), x)
        c, s = synth.rotary_tables(7, 16, offset=3)
        y = oracle.rotary(x, c, s, inter)
        # cos^2 + sin^2 of the float32 table entries is 1 to ~1e-7.
        np.testing.assert_allclose(np.linalg.norm(y, axis=-1), np.linalg.norm(x, axis=-1), rtol=2e-7)


def test_rotary_scores_depend_on_relative_position_only():
    """<R_m q, R_n k> = <R_{m+s} q, R_{n+s} k>: shifting every position by s
    (tables with an offset) leaves every logit unchanged, up to the float32
    rounding of the tables."""
    N, d = 40, 64
    q = np.random.default_rng(83).standard_normal((1, 1, N, d))
    k = np.random.default_rng(84).standard_normal((1, 1, N, d))
    for inter in (False, True):
        c0, s0 = synth.rotary_tables(N, d, offset=0)
        c1, s1 = synth.rotary_tables(N, d, offset=57)
        l0 = oracle.rotary(q, c0, s0, inter)[0, 0] @ oracle.rotary(k, c0, s0, inter)[0, 0].T
        l1 = oracle.rotary(q, c1, s1, inter)[0, 0] @ oracle.rotary(k, c1, s1, inter)[0, 0].T
        np.testing.assert_allclose(l1, l0, rtol=0, atol=1e-4)
        # ... while the logits themselves do change with the relative position.
        plain = q[0, 0] @ k[0, 0].T
        assert np.abs(l0 - plain).max() > 1.0


def _bwd(q, k, v, g, causal, scale):
    return oracle.attention_bwd(q, k, v, g, causal=causal, scale=scale)


@pytest.mark.parametrize("check", pins.BWD_CHECKS, ids=lambda c: c.__name__)
def test_attention_bwd_pin(check):
    check(_attn, _bwd)


@pytest.mark.parametrize("causal", [0, 1, 2])
def test_attention_bwd_matches_autograd(causal):
    """The same gradients from PyTorch's float64 autograd through an explicit
    masked softmax (an independent implementation of the chain rule)."""
    B, H, Nq, Nk, d = 2, 2, 7, 11, 5
    rng = np.random.default_rng(110 + causal)
    q, k, v, g = (rng.standard_normal(s) for s in ((B, H, Nq, d), (B, H, Nk, d), (B, H, Nk, d), (B, H, Nq, d)))
    qt, kt, vt = (torch.tensor(a, requires_grad=True) for a in (q, k, v))
    s = 0.6 * qt @ kt.transpose(-1, -2)
    i = torch.arange(Nq)[:, None]
    j = torch.arange(Nk)[None, :]
    limit = {0: torch.full((Nq, 1), Nk - 1), 1: i, 2: i + (Nk - Nq)}[causal]
    s = s.masked_fill(j > limit, float("-inf"))
    (torch.softmax(s, dim=-1) @ vt).backward(torch.tensor(g))
    for mine, ref in zip(oracle.attention_bwd(q, k, v, g, causal=causal, scale=0.6), (qt, kt, vt)):
        np.testing.assert_allclose(mine, ref.grad.numpy(), rtol=0, atol=1e-12)


def test_attention_bwd_rejects_rows_without_keys():
    q, k = np.zeros((1, 1, 4, 2)), np.zeros((1, 1, 3, 2))
    with pytest.raises(RuntimeError):
        oracle.attention_bwd(q, k, k, q, causal=2, scale=1.0)
