"""Element-by-element comparison of the CUDA path with the float64 oracle.

Tolerances for 16-bit inputs: max |dO| <= 1e-2, RMS(dO) <= 2e-3, max |dlse| <=
1e-3 (absolute).  Both sides read the same rounded inputs, so the only
differences are the kernel's float32 accumulation, its 16-bit rounding of the
softmax weights P and of O.
"""
from __future__ import annotations

import numpy as np
import torch

import exact_attention_forward_05_gb300 as attn
import oracle
import synth

MAX_ABS, RMS, LSE_ABS = 1e-2, 2e-3, 1e-3


def metrics(o_gpu, lse_gpu, o_ref, lse_ref):
    o = o_gpu.double().cpu().numpy() if hasattr(o_gpu, "cpu") else np.asarray(o_gpu, np.float64)
    l = lse_gpu.double().cpu().numpy() if hasattr(lse_gpu, "cpu") else np.asarray(lse_gpu, np.float64)
    d = o - o_ref
    return {"max_abs": float(np.abs(d).max()) if d.size else 0.0,
            "rms": float(np.sqrt(np.mean(d ** 2))) if d.size else 0.0,
            "lse_abs": float(np.abs(l - lse_ref).max()) if l.size else 0.0,
            "finite": bool(np.isfinite(o).all() and np.isfinite(l).all())}


def assert_close(m, what=""):
    assert m["finite"], f"{what}: non-finite output"
    assert m["max_abs"] <= MAX_ABS, f"{what}: max |dO| {m['max_abs']:.3e} > {MAX_ABS}"
    assert m["rms"] <= RMS, f"{what}: RMS {m['rms']:.3e} > {RMS}"
    assert m["lse_abs"] <= LSE_ABS, f"{what}: max |dlse| {m['lse_abs']:.3e} > {LSE_ABS}"


def run_gpu(q, k, v, causal, scale, device="cuda"):
    o, lse = attn.attn_fwd(q.to(device), k.to(device), v.to(device), causal=causal, scale=scale)
    torch.cuda.synchronize()
    return o, lse


# Unit roundoff of the 16-bit formats (significand bits incl. the hidden bit: 8, 11).
UNIT_ROUNDOFF = {torch.bfloat16: 2.0 ** -8, torch.float16: 2.0 ** -11}


def assert_within_rounding(o_gpu, o_ref, v, what=""):
    """Bound for outputs of any magnitude, derived from the arithmetic: O is
    rounded once to the 16-bit format (relative error <= u |O|) and every
    softmax weight once (|dO| <= u max|v| since the weights sum to one), plus
    the 1e-2 float32 accumulation allowance."""
    u = UNIT_ROUNDOFF[o_gpu.dtype]
    o = o_gpu.double().cpu().numpy()
    vmax = float(v.double().abs().max())
    bound = MAX_ABS + u * (np.abs(o_ref) + vmax)
    excess = np.abs(o - o_ref) - bound
    assert np.all(excess <= 0), f"{what}: exceeds the rounding bound by {excess.max():.3e}"


def assert_close_elementwise(o_gpu, lse_gpu, o_ref, lse_ref, q, k, v, causal, scale, rows=None, what=""):
    """The fixed tolerances, except that an element of O whose fixed 1e-2
    bound is below what the kernel's two roundings allow is held to that
    instead.  The kernel rounds every softmax weight to the 16-bit input type
    before P V and rounds O once at the end, so element e of O may differ from
    the exact value by u (|O_e| + A_e) with A = P |V| (the weighted mean of
    |v|, computed by the oracle) and u the unit roundoff (2^-8 bf16, 2^-11
    fp16), plus float32 accumulation (1e-4 allowance).  In early causal rows
    (few keys) |O| reaches 2-4, where one bf16 rounding of O alone can exceed
    1e-2.  RMS <= 2e-3 and max |dlse| <= 1e-3 are never relaxed, and the extra
    oracle pass runs only when some element misses the fixed bound."""
    m = metrics(o_gpu, lse_gpu, o_ref, lse_ref)
    assert m["finite"], f"{what}: non-finite output"
    assert m["rms"] <= RMS, f"{what}: RMS {m['rms']:.3e} > {RMS}"
    assert m["lse_abs"] <= LSE_ABS, f"{what}: max |dlse| {m['lse_abs']:.3e} > {LSE_ABS}"
    if m["max_abs"] <= MAX_ABS:
        return m
    u = UNIT_ROUNDOFF[o_gpu.dtype]
    a_ref, _ = oracle.attention(q, k, v.abs(), causal=causal, scale=scale, rows=rows)
    o = o_gpu.double().cpu().numpy()
    bound = np.maximum(MAX_ABS, u * (np.abs(o_ref) + a_ref) + 1e-4)
    excess = np.abs(o - o_ref) - bound
    assert np.all(excess <= 0), f"{what}: max |dO| {m['max_abs']:.3e} exceeds the rounding bound by {excess.max():.3e}"
    return dict(m, rounding_bound_used=True)


def check_case(q, k, v, causal, scale=None, rows=None, what="", large_outputs=False):
    """Run the kernel, compare every output row (or the sampled ``rows``) with
    the oracle; returns the metrics.  ``large_outputs`` replaces the fixed
    max-abs bound by the rounding bound above (for inputs whose outputs reach
    several units, where one bf16 ulp alone exceeds 1e-2)."""
    d = q.shape[-1]
    scale = d ** -0.5 if scale is None else scale
    o, lse = run_gpu(q, k, v, causal, scale)
    o_ref, lse_ref = oracle.attention(q, k, v, causal=causal, scale=scale, rows=rows)
    if rows is not None:
        idx = torch.as_tensor(rows, device=o.device)
        o, lse = o[:, :, idx], lse[:, :, idx]
    m = metrics(o, lse, o_ref, lse_ref)
    if large_outputs:
        assert_within_rounding(o, o_ref, v, what)
        m = dict(m, max_abs=0.0)
    assert_close(m, what)
    st = attn.device_status()
    assert st == attn.ATTN_OK, f"{what}: device status {attn.status_string(st)}"
    return m


def inputs(B, H, N, d, dtype="bf16", seed=0):
    return synth.attention_inputs(B, H, N, d, dtype, seed)
