"""FP8 path on the GPU: the pre-pass against the oracle's rotation and block
quantisation, the FP8 attention kernel against exact attention on the
dequantised operands, and the end-to-end error against exact attention on the
16-bit inputs next to the naive per-tensor FP8 baseline."""
import math

import numpy as np
import pytest
import torch

import exact_attention_forward_05_gb300 as attn
import oracle
import synth

pytestmark = pytest.mark.gpu

D = 128
FP8_RMS = 2.5e-2     # error bound of the FP8 path against exact attention (target)


def _np(t):
    return t.detach().cpu().numpy()


def _e4m3_step(x):
    """Spacing of E4M3 values around |x| (2^-9 in the subnormal range)."""
    a = np.maximum(np.abs(x), 2.0 ** -6)
    return 2.0 ** (np.floor(np.log2(a)) - 3)


def _assert_codes_within_one_step(codes_gpu, scales_gpu, codes_ref, scales_ref):
    """Rotated (or rotary-embedded) rows: the device's float32 arithmetic and
    the oracle's float64 arithmetic round differently, so the block scale
    differs by float32 rounding and a code may land on the neighbouring E4M3
    value at a rounding midpoint.  The two effects are checked apart: scales to
    float32 rounding, codes (scale-free) within one E4M3 step, and only a small
    fraction of codes different."""
    np.testing.assert_allclose(scales_gpu, scales_ref, rtol=1e-5, atol=0)
    vg, vr = oracle.e4m3_decode(codes_gpu), oracle.e4m3_decode(codes_ref)
    assert np.all(np.abs(vg - vr) <= _e4m3_step(vr))
    assert np.mean(codes_gpu != codes_ref) < 0.01


PREP_D = [64, 128, 256]


@pytest.mark.parametrize("d", PREP_D)
@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_prepare_without_rotation_is_bit_exact(dtype, d):
    """No rotation: both sides divide the same float32 value by the same scale
    and round to nearest even, so every code and every scale is identical.
    A ragged last block."""
    q, k, v = synth.outlier_inputs(2, 3, 300, d, dtype, seed=1)
    out = attn.fp8_prepare(q.cuda(), k.cuda(), v.cuda(), signs=None)
    torch.cuda.synchronize()
    for x, c, s in zip((q, k, v), out[:3], out[3:]):
        codes, scales = oracle.block_quantize(x)
        np.testing.assert_array_equal(_np(c), codes)
        np.testing.assert_array_equal(_np(s), scales)


@pytest.mark.parametrize("d", PREP_D)
@pytest.mark.parametrize("per_tensor", [False, True])
def test_prepare_keeps_the_sign_of_zero(d, per_tensor):
    """Exact zeros of either sign (and the smallest subnormals) in unrotated
    tensors: code = RNE(x / s) keeps the sign, so -0 gives 0x80 and +0 gives
    0x00, bit-exact against the oracle."""
    q, k, v = synth.outlier_inputs(2, 3, 300, d, "fp16", seed=14)
    g = torch.Generator().manual_seed(14)
    for t in (q, k, v):
        flat = t.view(-1)
        idx = torch.randperm(flat.numel(), generator=g)[:4000]
        flat[idx[:1000]] = -0.0
        flat[idx[1000:2000]] = 0.0
        flat[idx[2000:3000]] = -2.0 ** -24
        flat[idx[3000:]] = 2.0 ** -24
    out = attn.fp8_prepare(q.cuda(), k.cuda(), v.cuda(), signs=None, per_tensor=per_tensor)
    torch.cuda.synchronize()
    for x, c, s in zip((q, k, v), out[:3], out[3:]):
        codes, scales = oracle.block_quantize(x, per_tensor=per_tensor)
        assert np.sum(codes == 0x80) >= 1000
        np.testing.assert_array_equal(_np(s), scales)
        np.testing.assert_array_equal(_np(c), codes)


@pytest.mark.parametrize("d", PREP_D)
def test_prepare_per_tensor_is_bit_exact(d):
    q, k, v = synth.outlier_inputs(1, 4, 257, d, "bf16", seed=2)
    out = attn.fp8_prepare(q.cuda(), k.cuda(), v.cuda(), per_tensor=True)
    torch.cuda.synchronize()
    for x, c, s in zip((q, k, v), out[:3], out[3:]):
        codes, scales = oracle.block_quantize(x, per_tensor=True)
        assert _np(s).shape == (1,)
        np.testing.assert_array_equal(_np(s), scales)
        np.testing.assert_array_equal(_np(c), codes)


@pytest.mark.parametrize("d", PREP_D)
def test_prepare_with_rotation_matches_oracle(d):
    """With the Hadamard rotation the kernel's float32 butterflies and the
    oracle's float64 dense product round differently, so a code may land on the
    neighbouring E4M3 value when the quotient sits at a rounding midpoint: the
    scales agree to float32 rounding, dequantised values to one E4M3 step, and
    only a small fraction of codes differ.  V is not rotated: bit-exact."""
    B, H, N = 2, 4, 385
    q, k, v = synth.outlier_inputs(B, H, N, d, "bf16", seed=3)
    signs = synth.hadamard_signs(H, d, seed=3)
    out = attn.fp8_prepare(q.cuda(), k.cuda(), v.cuda(), signs=signs.cuda())
    torch.cuda.synchronize()
    for i, x in enumerate((q, k)):
        rot = oracle.hadamard_rotate(x, signs)
        codes, scales = oracle.block_quantize(rot)
        _assert_codes_within_one_step(_np(out[i]), _np(out[3 + i]), codes, scales)
    codes, scales = oracle.block_quantize(v)
    np.testing.assert_array_equal(_np(out[2]), codes)
    np.testing.assert_array_equal(_np(out[5]), scales)


def test_prepare_rotation_is_orthogonal_on_device():
    """Dequantised rotated Q and K keep Q K^T: compare the logits of the
    dequantised codes with those of the 16-bit inputs (up to quantisation)."""
    q, k, v = synth.attention_inputs(1, 2, 256, D, "bf16", seed=4)
    signs = synth.hadamard_signs(2, D, seed=4)
    q8, k8, _, qs, ks, _ = attn.fp8_prepare(q.cuda(), k.cuda(), v.cuda(), signs=signs.cuda())
    qd = oracle.dequantize(_np(q8), _np(qs))
    kd = oracle.dequantize(_np(k8), _np(ks))
    s_fp8 = np.einsum("bhid,bhjd->bhij", qd, kd)
    s_ref = np.einsum("bhid,bhjd->bhij", q.double().numpy(), k.double().numpy())
    assert np.sqrt(np.mean((s_fp8 - s_ref) ** 2)) < 0.05 * np.sqrt(np.mean(s_ref ** 2))


@pytest.mark.parametrize("d", PREP_D)
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [128, 300, 1100])
def test_fp8_kernel_on_oracle_quantised_operands(N, causal, d):
    """The FP8 kernel on operands quantised by the oracle, against exact
    attention on the dequantised operands.  lse does not depend on the E4M3
    rounding of P (the running sum adds the float32 weights; the products of
    two E4M3 codes are exact in float32): 1e-3.  O: the weights are rounded
    to E4M3 (relative half step 2^-4), so its RMS error is a few percent of
    the RMS of O."""
    B, H = 2, 2
    q, k, v = synth.outlier_inputs(B, H, N, d, "bf16", seed=5)
    signs = synth.hadamard_signs(H, d, seed=5)
    qr, kr = oracle.hadamard_rotate(q, signs), oracle.hadamard_rotate(k, signs)
    (qc, qs), (kc, ks), (vc, vs) = (oracle.block_quantize(t) for t in (qr, kr, v))
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    o, lse = attn.attn_fwd_fp8(dev(qc), dev(kc), dev(vc), dev(qs), dev(ks), dev(vs), causal=causal)
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle.attention(oracle.dequantize(qc, qs), oracle.dequantize(kc, ks),
                                      oracle.dequantize(vc, vs), causal=causal, scale=d ** -0.5)
    d = o.double().cpu().numpy() - o_ref
    assert np.isfinite(d).all()
    assert np.abs(lse.double().cpu().numpy() - lse_ref).max() <= 1e-3
    assert np.sqrt(np.mean(d ** 2)) <= 0.08 * np.sqrt(np.mean(o_ref ** 2))
    assert attn.device_status() == attn.ATTN_OK


@pytest.mark.parametrize("causal", [False, True])
def test_fp8_kernel_negative_scale(causal):
    """As above with a negative softmax scale: the per-block multiplier of S is
    negative, so the row extreme taken from S is its minimum."""
    B, H, N, d = 1, 2, 1100, 128
    q, k, v = synth.outlier_inputs(B, H, N, d, "bf16", seed=8)
    (qc, qs), (kc, ks), (vc, vs) = (oracle.block_quantize(t) for t in (q, k, v))
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    scale = -(d ** -0.5)
    o, lse = attn.attn_fwd_fp8(dev(qc), dev(kc), dev(vc), dev(qs), dev(ks), dev(vs), causal=causal, scale=scale)
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle.attention(oracle.dequantize(qc, qs), oracle.dequantize(kc, ks),
                                      oracle.dequantize(vc, vs), causal=causal, scale=scale)
    diff = o.double().cpu().numpy() - o_ref
    assert np.isfinite(diff).all()
    assert np.abs(lse.double().cpu().numpy() - lse_ref).max() <= 1e-3
    assert np.sqrt(np.mean(diff ** 2)) <= 0.08 * np.sqrt(np.mean(o_ref ** 2))
    assert attn.device_status() == attn.ATTN_OK


@pytest.mark.parametrize("d", PREP_D)
def test_fp8_weights_layout_through_identity_values(d):
    """V = identity (N = 128 keys, one key block; d = 64 sees the first 64
    weights of each row, d = 256 all 128 and zero columns after them): O
    equals the rounded softmax weights themselves, so every weight is checked
    at its position: within an E4M3 half step (2^-4 relative, 2^-10 absolute
    below 2^-6) of the exact one."""
    N = 128
    q, k, _ = synth.attention_inputs(1, 2, N, d, "bf16", seed=6)
    v = torch.eye(N, d, dtype=torch.bfloat16).expand(1, 2, N, d).contiguous()
    for causal in (False, True):
        o, lse = attn.attn_fwd_fp8_pipeline(q.cuda(), k.cuda(), v.cuda(), signs=None, causal=causal)
        torch.cuda.synchronize()
        q8, k8, v8, qs, ks, vs = attn.fp8_prepare(q.cuda(), k.cuda(), v.cuda())
        deq = [oracle.dequantize(_np(c), _np(s)) for c, s in ((q8, qs), (k8, ks), (v8, vs))]
        w_ref, lse_ref = oracle.attention(deq[0], deq[1], deq[2], causal=causal, scale=d ** -0.5)
        w = o.double().cpu().numpy()
        # The kernel's running sum is >= 1 (the row maximum contributes 2^0), so
        # a weight below the E4M3 normal range (2^-6) is off by at most 2^-10.
        tol = 2.0 ** -4 * w_ref + 2.0 ** -10 + 2.0 ** -8 * w_ref + 1e-6
        assert np.all(np.abs(w - w_ref) <= tol), (causal, np.abs(w - w_ref).max())


@pytest.mark.parametrize("N", [1024, 2048, 4096, 8192, 16384])
def test_fp8_error_against_exact_attention(N):
    """FP8 path with per-block scales and the Hadamard rotation on inputs with
    0.1 % outliers (B = 16384 / N, H = 16, d = 128): RMS <= 2.5e-2 against
    exact attention on the 16-bit inputs.  The RMS runs over 256 seeded query
    rows of every head for N <= 4096, and over 64 rows of 8 heads spread over
    the batch above that.  The naive per-tensor FP8 baseline is computed on the
    same rows and reported next to it."""
    B, H = 16384 // N, 16
    q, k, v = synth.outlier_inputs(B, H, N, D, "bf16", seed=0)
    signs = synth.hadamard_signs(H, D, seed=0)
    if N <= 4096:
        rows = synth.sample_rows(N, 256, seed=0, salt=N)
        heads = list(range(B * H))
    else:
        rows = synth.sample_rows(N, 64, seed=0, salt=N)
        heads = [int(i) for i in np.linspace(0, B * H - 1, 8).round()]
    qc, kc, vc = q.cuda(), k.cuda(), v.cuda()
    o8, _ = attn.attn_fwd_fp8_pipeline(qc, kc, vc, signs=signs.cuda())
    ob, _ = attn.attn_fwd_fp8_pipeline(qc, kc, vc, signs=None, per_tensor=True)
    torch.cuda.synchronize()
    assert bool(torch.isfinite(o8).all()) and bool(torch.isfinite(ob).all())
    flat = lambda t: t.reshape(1, B * H, N, D)
    hsel = torch.as_tensor(heads)
    o_ref, _ = oracle.attention(flat(q)[:, hsel], flat(k)[:, hsel], flat(v)[:, hsel], scale=D ** -0.5,
                                rows=rows)
    idx = torch.as_tensor(rows, device="cuda")
    pick = lambda o: flat(o)[:, hsel.cuda()][:, :, idx].double().cpu().numpy()
    rms8 = float(np.sqrt(np.mean((pick(o8) - o_ref) ** 2)))
    rmsb = float(np.sqrt(np.mean((pick(ob) - o_ref) ** 2)))
    print(f"N={N}: {len(rows)} rows x {len(heads)} heads: FP8 per-block + Hadamard RMS {rms8:.3e}; "
          f"naive per-tensor FP8 RMS {rmsb:.3e}; ratio {rmsb / rms8:.2f}")
    assert rms8 <= FP8_RMS
    assert attn.device_status() == attn.ATTN_OK


@pytest.mark.parametrize("N", [1024, 4096])
@pytest.mark.parametrize("d", [64, 256])
def test_fp8_error_other_head_dims(d, N):
    """The FP8 path at d = 64 and 256 (shapes of the bf16 sweep: B = 16384 / N,
    H = 2048 / d; inputs with 0.1 % outliers): RMS <= 2.5e-2 against exact
    attention on the 16-bit inputs over 256 seeded rows of every head, the
    naive per-tensor FP8 baseline on the same rows beside it."""
    B, H = 16384 // N, 2048 // d
    q, k, v = synth.outlier_inputs(B, H, N, d, "bf16", seed=0)
    signs = synth.hadamard_signs(H, d, seed=0)
    rows = synth.sample_rows(N, 256, seed=0, salt=N + d)
    qc, kc, vc = q.cuda(), k.cuda(), v.cuda()
    o8, _ = attn.attn_fwd_fp8_pipeline(qc, kc, vc, signs=signs.cuda())
    ob, _ = attn.attn_fwd_fp8_pipeline(qc, kc, vc, signs=None, per_tensor=True)
    torch.cuda.synchronize()
    assert bool(torch.isfinite(o8).all()) and bool(torch.isfinite(ob).all())
    o_ref, _ = oracle.attention(q, k, v, scale=d ** -0.5, rows=rows)
    idx = torch.as_tensor(rows, device="cuda")
    rms8 = float(np.sqrt(np.mean((o8[:, :, idx].double().cpu().numpy() - o_ref) ** 2)))
    rmsb = float(np.sqrt(np.mean((ob[:, :, idx].double().cpu().numpy() - o_ref) ** 2)))
    print(f"d={d} N={N}: FP8 per-block + Hadamard RMS {rms8:.3e}; naive per-tensor FP8 RMS {rmsb:.3e}")
    assert rms8 <= FP8_RMS
    assert attn.device_status() == attn.ATTN_OK


@pytest.mark.parametrize("d", [64, 128])
def test_fp8_stream_k_schedule(d):
    """The FP8 kernel under the stream-K schedule (a workspace, 160 units on
    the SMs, so most units are done in two parts): on operands quantised by
    the oracle, against exact attention on the dequantised operands with the
    FP8 kernel's own bounds (lse 1e-3; O RMS within 8 % of RMS(O)), for both
    schedules; lse of the two schedules equal to float32 summation order (the
    logits and the running sums are the same numbers).  O of the two
    schedules is not compared element by element: each part rounds its
    weights to E4M3 against its own maximum and V scale, so rows dominated by
    an outlier differ by as much as the FP8 error itself."""
    B, H, N = 4, 10, 1024
    q, k, v = synth.outlier_inputs(B, H, N, d, "bf16", seed=13)
    signs = synth.hadamard_signs(H, d, seed=13)
    qr, kr = oracle.hadamard_rotate(q, signs), oracle.hadamard_rotate(k, signs)
    (qc, qs), (kc, ks), (vc, vs) = (oracle.block_quantize(t) for t in (qr, kr, v))
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    bufs = [dev(a) for a in (qc, kc, vc, qs, ks, vs)]
    ws = torch.empty(attn.workspace_bytes(d), dtype=torch.uint8, device="cuda")
    o_sk, l_sk = attn.attn_fwd_fp8(*bufs, workspace=ws)
    o_rr, l_rr = attn.attn_fwd_fp8(*bufs)
    torch.cuda.synchronize()
    o_ref, l_ref = oracle.attention(oracle.dequantize(qc, qs), oracle.dequantize(kc, ks),
                                    oracle.dequantize(vc, vs), scale=d ** -0.5)
    for name, o, l in (("stream-K", o_sk, l_sk), ("round-robin", o_rr, l_rr)):
        e = o.double().cpu().numpy() - o_ref
        assert np.isfinite(e).all(), name
        assert np.abs(l.double().cpu().numpy() - l_ref).max() <= 1e-3, name
        assert np.sqrt(np.mean(e ** 2)) <= 0.08 * np.sqrt(np.mean(o_ref ** 2)), name
    assert (l_sk - l_rr).abs().max().item() <= 1e-4
    assert attn.device_status() == attn.ATTN_OK


def test_fp8_empty_and_bad_arguments():
    z = torch.empty((1, 1, 0, D), dtype=torch.bfloat16, device="cuda")
    attn.fp8_prepare(z, z, z)
    q = torch.zeros((1, 1, 16, 96), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(attn.AttnError) as e:
        attn.fp8_prepare(q, q, q)
    assert e.value.status == attn.ATTN_ERR_UNSUPPORTED


@pytest.mark.parametrize("d", PREP_D)
def test_prepare_many_items_per_cta(d):
    """A problem with many more (block, tensor, head) items than CTAs: at
    d = 128 every CTA of the streaming pre-pass walks a long range of items
    through its ring of copies (crossing block boundaries); codes and scales
    bit-exact against the oracle without rotation."""
    B, H, N = 4, 8, 2048 + 77
    q, k, v = synth.outlier_inputs(B, H, N, d, "bf16", seed=12)
    out = attn.fp8_prepare(q.cuda(), k.cuda(), v.cuda(), signs=None)
    torch.cuda.synchronize()
    for x, c, s in zip((q, k, v), out[:3], out[3:]):
        codes, scales = oracle.block_quantize(x)
        np.testing.assert_array_equal(_np(c), codes)
        np.testing.assert_array_equal(_np(s), scales)
    assert attn.device_status() == attn.ATTN_OK


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("rope", [None, "half", "interleaved"])
def test_prepare_rotation_many_items_per_cta(rope, dtype):
    """d = 128 streams (block, tensor, head) items through a ring of copies on
    a grid of two CTAs per SM: with many items per CTA, Q and K with the
    rotation (and the rotary embedding) against the oracle within one E4M3
    step, V bit-exact, and a ragged last block."""
    B, H, N, d = 4, 8, 2048 + 77, 128
    q, k, v = synth.outlier_inputs(B, H, N, d, dtype, seed=13)
    signs = synth.hadamard_signs(H, d, seed=13)
    tables = synth.rotary_tables(N, d, offset=3) if rope else None
    out = attn.fp8_prepare(q.cuda(), k.cuda(), v.cuda(), signs=signs.cuda(),
                           rope=None if tables is None else tuple(t.cuda() for t in tables),
                           rope_interleaved=rope == "interleaved")
    torch.cuda.synchronize()
    for i, x in enumerate((q, k)):
        ref = x if tables is None else oracle.rotary(x, *tables, rope == "interleaved")
        codes, scales = oracle.block_quantize(oracle.hadamard_rotate(ref, signs))
        _assert_codes_within_one_step(_np(out[i]), _np(out[3 + i]), codes, scales)
    codes, scales = oracle.block_quantize(v)
    np.testing.assert_array_equal(_np(out[2]), codes)
    np.testing.assert_array_equal(_np(out[5]), scales)
    assert attn.device_status() == attn.ATTN_OK


@pytest.mark.parametrize("B, H, N", [(1, 64, 100), (3, 5, 1), (2, 40, 257)])
@pytest.mark.parametrize("rope", [None, "half"])
def test_prepare_many_heads_and_short_sequences(B, H, N, rope):
    """d = 128 streaming pre-pass with the per-unit sign tables: many heads
    (the table of the next unit's head is filled while the current one is
    used, wrapping from the last head to the first), sequences shorter than one
    128-row block, a single row.  Q, K within one E4M3 step of the oracle, V
    bit-exact."""
    d = 128
    q, k, v = synth.outlier_inputs(B, H, N, d, "fp16", seed=16 + H)
    signs = synth.hadamard_signs(H, d, seed=16 + H)
    tables = synth.rotary_tables(N, d, offset=1) if rope else None
    out = attn.fp8_prepare(q.cuda(), k.cuda(), v.cuda(), signs=signs.cuda(),
                           rope=None if tables is None else tuple(t.cuda() for t in tables))
    torch.cuda.synchronize()
    for i, x in enumerate((q, k)):
        ref = x if tables is None else oracle.rotary(x, *tables, False)
        codes, scales = oracle.block_quantize(oracle.hadamard_rotate(ref, signs))
        _assert_codes_within_one_step(_np(out[i]), _np(out[3 + i]), codes, scales)
    codes, scales = oracle.block_quantize(v)
    np.testing.assert_array_equal(_np(out[2]), codes)
    np.testing.assert_array_equal(_np(out[5]), scales)
    assert attn.device_status() == attn.ATTN_OK


def test_prepare_code_buffers_off_32_byte_boundaries():
    """Code buffers that start 16 bytes past a 32-byte boundary take 16-byte
    stores instead of 32-byte ones: the same codes and scales."""
    B, H, N, d = 2, 4, 640, 128
    q, k, v = (t.cuda() for t in synth.outlier_inputs(B, H, N, d, "bf16", seed=15))
    signs = synth.hadamard_signs(H, d, seed=15).cuda()
    ref = attn.fp8_prepare(q, k, v, signs=signs)
    n = B * H * N * d
    raw = [torch.empty(n + 64, dtype=torch.uint8, device="cuda") for _ in range(3)]
    codes = [r[16:16 + n].view(B, H, N, d) for r in raw]
    assert all(c.data_ptr() % 32 == 16 for c in codes)
    scales = [torch.empty((B, H, N // 128), dtype=torch.float32, device="cuda") for _ in range(3)]
    out = attn.fp8_prepare(q, k, v, signs=signs, out=codes + scales)
    torch.cuda.synchronize()
    for a, b in zip(ref, out):
        assert torch.equal(a, b)


@pytest.mark.parametrize("d", PREP_D)
@pytest.mark.parametrize("interleaved", [False, True])
@pytest.mark.parametrize("rotate", [False, True])
def test_prepare_with_rotary_matches_oracle(interleaved, rotate, d):
    """Rotary embedding fused in front of the rotation: Q and K against the
    oracle's rotary -> rotation -> block quantisation (float32 on the device,
    float64 in the oracle: scales to float32 rounding, dequantised values within
    one E4M3 step, few codes different); V untouched, bit-exact.  N = 385 leaves
    a ragged last block (rows past N skip the table loads)."""
    B, H, N = 2, 3, 385
    q, k, v = synth.outlier_inputs(B, H, N, d, "bf16", seed=7)
    signs = synth.hadamard_signs(H, d, seed=7) if rotate else None
    cos, sin = synth.rotary_tables(N, d, offset=5)
    out = attn.fp8_prepare(q.cuda(), k.cuda(), v.cuda(), signs=None if signs is None else signs.cuda(),
                           rope=(cos.cuda(), sin.cuda()), rope_interleaved=interleaved)
    torch.cuda.synchronize()
    for i, x in enumerate((q, k)):
        ref = oracle.rotary(x, cos, sin, interleaved)
        if rotate:
            ref = oracle.hadamard_rotate(ref, signs)
        codes, scales = oracle.block_quantize(ref)
        _assert_codes_within_one_step(_np(out[i]), _np(out[3 + i]), codes, scales)
    codes, scales = oracle.block_quantize(v)
    np.testing.assert_array_equal(_np(out[2]), codes)
    np.testing.assert_array_equal(_np(out[5]), scales)


def test_prepare_without_tables_is_unchanged():
    """No tables: the rotary entry point is the plain pre-pass, bit for bit."""
    q, k, v = (t.cuda() for t in synth.outlier_inputs(1, 2, 300, D, "bf16", seed=8))
    signs = synth.hadamard_signs(2, D, seed=8).cuda()
    a = attn.fp8_prepare(q, k, v, signs=signs)
    b = attn.fp8_prepare(q, k, v, signs=signs, rope=None)
    cos, sin = (torch.zeros(300, 64, device="cuda") for _ in range(2))
    cos += 1.0  # zero angles: the embedding is the identity, exactly
    c = attn.fp8_prepare(q, k, v, signs=signs, rope=(cos, sin))
    torch.cuda.synchronize()
    for x, y, z in zip(a, b, c):
        assert torch.equal(x, y) and torch.equal(x, z)


@pytest.mark.parametrize("interleaved", [False, True])
def test_fp8_pipeline_with_rotary_against_exact_attention(interleaved):
    """End to end: FP8 pipeline with the fused rotary embedding against exact
    attention on the rotary-embedded 16-bit inputs (sampled rows), within the
    FP8 bound."""
    B, H, N = 1, 4, 2048
    q, k, v = synth.outlier_inputs(B, H, N, D, "bf16", seed=9)
    signs = synth.hadamard_signs(H, D, seed=9)
    cos, sin = synth.rotary_tables(N, D)
    o, _ = attn.attn_fwd_fp8_pipeline(q.cuda(), k.cuda(), v.cuda(), signs=signs.cuda(),
                                      rope=(cos.cuda(), sin.cuda()), rope_interleaved=interleaved)
    torch.cuda.synchronize()
    rows = synth.sample_rows(N, 32, seed=9)
    qr, kr = oracle.rotary(q, cos, sin, interleaved), oracle.rotary(k, cos, sin, interleaved)
    o_ref, _ = oracle.attention(qr, kr, v, scale=D ** -0.5, rows=rows)
    err = _np(o.float())[:, :, rows] - o_ref
    assert math.sqrt(np.mean(err ** 2)) <= FP8_RMS
