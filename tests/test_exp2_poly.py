"""CPU check of the polynomial 2^x the kernels use on the FMA pipe
(exp2_poly2 in csrc/sm103.cuh).  The coefficients are read from the source,
so this checks what the kernel compiles.  A float32 model of the whole
function -- clamp, rounding by the 1.5 * 2^23 constant, reduction to
f in [-1/2, 1/2], Horner evaluation, exponent add -- is compared with
float64 2**x on a dense grid: maximum relative error below 7.6e-5.  The
GPU test of the device function itself is in test_exp2_poly_gpu.py."""
import os
import re

import numpy as np

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                   "exact_attention_forward_05_gb300", "csrc", "sm103.cuh")
BOUND = 7.6e-5


def coefficients():
    text = open(SRC).read()
    got = {k: float(v) for k, v in re.findall(r"kExp2(C[0-3]) = ([0-9.eE+-]+)f", text)}
    magic = float(re.search(r"kExp2Magic = ([0-9.]+)f", text).group(1))
    return [got["C0"], got["C1"], got["C2"], got["C3"]], magic


def model(x):
    """float32 model of exp2_poly2, elementwise."""
    c, magic = coefficients()
    f32 = np.float32
    x = np.maximum(x.astype(f32), f32(-125.0))
    t = (x + f32(magic)).astype(f32)
    f = (x - (t - f32(magic)).astype(f32)).astype(f32)
    p = (f * f32(c[3]) + f32(c[2])).astype(f32)   # fma rounding differs from mul+add by < 1 ulp
    p = (p * f + f32(c[1])).astype(f32)
    p = (p * f + f32(c[0])).astype(f32)
    bits = p.view(np.uint32) + (t.view(np.uint32) << np.uint32(23))
    return bits.astype(np.uint32).view(np.float32)


def test_magic_constant_and_bound_of_the_cubic():
    c, magic = coefficients()
    assert magic == 1.5 * 2 ** 23
    f = np.linspace(-0.5, 0.5, 1_000_001)
    p = ((c[3] * f + c[2]) * f + c[1]) * f + c[0]
    assert np.max(np.abs(p / 2.0 ** f - 1)) < BOUND
    # the cubic is close to the Taylor coefficients of 2^f = e^(f ln 2)
    ln2 = np.log(2.0)
    for got, want in zip(c, [1.0, ln2, ln2 ** 2 / 2, ln2 ** 3 / 6]):
        assert abs(got - want) < 0.02 * max(want, 0.05)


def test_whole_function_on_a_dense_grid():
    x = np.concatenate([np.linspace(-125.0, 8.0, 4_000_001),
                        np.arange(-125, 9).astype(np.float64),           # integers
                        np.arange(-125, 8).astype(np.float64) + 0.5])    # rounding ties
    y = model(x).astype(np.float64)
    ref = 2.0 ** x.astype(np.float32).astype(np.float64)
    assert np.all(np.isfinite(y)) and np.all(y > 0)
    assert np.max(np.abs(y / ref - 1)) < BOUND


def test_clamp_below_the_normal_range():
    x = np.array([-125.0, -126.0, -150.0, -1e30, -np.inf], dtype=np.float32)
    y = model(x).astype(np.float64)
    assert np.all(np.abs(y / 2.0 ** -125 - 1) < BOUND)   # clamped to 2^-125, still normal
