"""GPU parity of the backward kernel (attn_bwd): dQ, dK, dV against the float64
oracle's gradients (oracle.attention_bwd, the chain rule through the
definition), every element, on the same rounded inputs and dO.  O and lse come
from the forward kernel.

Tolerance (derived from the arithmetic; the pages fix none for gradients): each gradient is
rounded once to the 16-bit type at the end (relative error up to u, RMS about
u / sqrt(3) for uniformly spread rounding), and P, dS and O (inside D) carry one
rounding each into float32 sums whose terms mostly do not cancel.  Checked per
gradient tensor: RMS(error) <= 2 u RMS(ref) and max |error| <= 4 u max|ref|,
u = 2^-8 (bf16), 2^-11 (fp16).  Measured: RMS 0.6 u, max up to 1.2 u."""
import numpy as np
import pytest
import torch

import exact_attention_forward_05_gb300 as attn
import oracle
import synth
from tests import parity

pytestmark = pytest.mark.gpu


def _check(B, H, N, d, dtype, causal, seed=0, what=""):
    q, k, v = parity.inputs(B, H, N, d, dtype, seed=seed)
    g = synth.attention_inputs(B, H, N, d, dtype, seed=seed + 1000)[0]  # dL/dO, same recipe
    qc, kc, vc, gc = q.cuda(), k.cuda(), v.cuda(), g.cuda()
    scale = d ** -0.5
    o, lse = attn.attn_fwd(qc, kc, vc, causal=causal, scale=scale)
    dq, dk, dv = attn.attn_bwd(qc, kc, vc, o, gc, lse, causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert attn.device_status() == attn.ATTN_OK
    rq, rk, rv = oracle.attention_bwd(q, k, v, g, causal=causal, scale=scale)
    _assert_grads(((dq, rq), (dk, rk), (dv, rv)), dtype, what)


def _assert_grads(pairs, dtype, what):
    u = 2.0 ** -8 if dtype == "bf16" else 2.0 ** -11
    for name, (got, ref) in zip(("dQ", "dK", "dV"), pairs):
        x = got.double().cpu().numpy()
        assert np.isfinite(x).all(), f"{what} {name}: non-finite"
        e = x - ref
        rms, rms_ref = float(np.sqrt(np.mean(e ** 2))), float(np.sqrt(np.mean(ref ** 2)))
        mx, mx_ref = float(np.abs(e).max()), float(np.abs(ref).max())
        print(f"{what} {name}: RMS err / RMS ref = {rms / rms_ref:.2e}, max err / max ref = {mx / mx_ref:.2e} "
              f"(bounds {2 * u:.2e}, {4 * u:.2e})")
        assert rms <= 2 * u * rms_ref, f"{what} {name}: RMS {rms:.3e} > {2 * u:.2e} x {rms_ref:.3e}"
        assert mx <= 4 * u * mx_ref, f"{what} {name}: max {mx:.3e} > {4 * u:.2e} x {mx_ref:.3e}"


@pytest.mark.parametrize("causal", [False, True])
def test_bwd_tiny_fp16_config(causal):
    """fp16, B=1, H=2, N=256, d=64 (the tiny forward configuration)."""
    _check(1, 2, 256, 64, "fp16", causal, what=f"tiny causal={causal}")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N", [128, 200, 384])
@pytest.mark.parametrize("causal", [False, True])
def test_bwd_ragged_bf16(d, N, causal):
    _check(2, 3, N, d, "bf16", causal, seed=N + d, what=f"d={d} N={N} causal={causal}")


@pytest.mark.parametrize("causal", [False, True])
def test_bwd_b4_h16_n2048_d128(causal):
    """bf16, B=4, H=16, N=2048, d=128: every element of every gradient."""
    _check(4, 16, 2048, 128, "bf16", causal, what=f"B4 H16 N2048 causal={causal}")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_bwd_fp16_long_ragged(d, causal):
    """fp16, one head pair with N = 4096 + 37: 33 query blocks per key block (the
    Q / dO ring and the dQ staging wrap many times within a unit), a ragged
    last block, every element."""
    _check(1, 2, 4096 + 37, d, "fp16", causal, seed=40 + d, what=f"fp16 d={d} N=4133 causal={causal}")


def test_bwd_bench_shape_one_head():
    """bf16, B=2, H=16, N=8192, d=128, non-causal: the backward bench line's
    launch over the whole problem, and every element of the last head's
    gradients against the oracle run on that head alone (it sees no other)."""
    B, H, N, d = 2, 16, 8192, 128
    q, k, v = parity.inputs(B, H, N, d, "bf16", seed=7)
    g = synth.attention_inputs(B, H, N, d, "bf16", seed=1007)[0]
    scale = d ** -0.5
    qc, kc, vc, gc = q.cuda(), k.cuda(), v.cuda(), g.cuda()
    o, lse = attn.attn_fwd(qc, kc, vc, scale=scale)
    dq, dk, dv = attn.attn_bwd(qc, kc, vc, o, gc, lse, scale=scale)
    torch.cuda.synchronize()
    assert attn.device_status() == attn.ATTN_OK
    for t in (dq, dk, dv):
        assert bool(torch.isfinite(t).all())
    last = lambda t: t.reshape(1, B * H, N, d)[:, -1:]
    rq, rk, rv = oracle.attention_bwd(last(q), last(k), last(v), last(g), causal=False, scale=scale)
    _assert_grads(((last(dq.cpu()), rq), (last(dk.cpu()), rk), (last(dv.cpu()), rv)), "bf16", "bench shape, last head")
