"""Seeded synthetic workloads for exact attention (shared by tests and bench).

This module only draws random numbers and rounds them to the storage dtype.
It holds none of the attention arithmetic: both the float64 oracle and the
CUDA path take its outputs as inputs.

Generator (documented so that anyone can regenerate the exact stream):

* splitmix64 (Steele, Lea & Flood, "Fast splittable pseudorandom number
  generators", OOPSLA 2014) in counter form: for a key ``k`` the i-th word is
  ``mix(k + (i + 1) * GAMMA)`` with ``GAMMA = 0x9E3779B97F4A7C15`` and
  ``mix(z) = z3`` where ``z1 = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9``,
  ``z2 = (z1 ^ (z1 >> 27)) * 0x94D049BB133111EB``, ``z3 = z2 ^ (z2 >> 31)``
  (all arithmetic modulo 2**64).
* one key per (seed, stream): ``k = mix(seed * GAMMA + stream * 0xD1B54A32D192ED03 + 1)``.
* uniforms in (0, 1]: ``u = ((word >> 11) + 1) * 2**-53``.
* standard normals by the Box-Muller transform on consecutive pairs
  ``(u1, u2)``: ``r = sqrt(-2 ln u1)``, ``z0 = r cos(2 pi u2)``, ``z1 = r sin(2 pi u2)``.

Streams: Q=0, K=1, V=2; outlier masks 3..5; outlier magnitudes 6..8;
Hadamard signs 9; sampled query rows 10.

Workload recipes follow the sequence-length sweep of the FlashAttention-3
evaluation (iid N(0, 1) inputs) and its FP8 accuracy experiment (0.1 % of the
entries of Q, K and V replaced by large outliers), as described in
"FlashAttention-3: Fast & Accurate Attention with Asynchrony & Low-Precision"
(section "Incoherent Processing for FP8 Accuracy") and in the comrad404 review
(section "Ограничения и критика").
"""
from __future__ import annotations

import numpy as np
import torch

GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_STREAM_MUL = np.uint64(0xD1B54A32D192ED03)

STREAM_Q, STREAM_K, STREAM_V = 0, 1, 2
STREAM_OUTLIER_MASK = 3  # + tensor index (0, 1, 2)
STREAM_OUTLIER_MAG = 6   # + tensor index
STREAM_SIGNS = 9
STREAM_ROWS = 10

_CHUNK = 1 << 22  # words generated per numpy pass (bounds temporary memory)


def _mix(z: np.ndarray) -> np.ndarray:
    with np.errstate(over="ignore"):
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def stream_key(seed: int, stream: int) -> np.uint64:
    with np.errstate(over="ignore"):
        z = (np.uint64(seed & 0xFFFFFFFFFFFFFFFF) * GAMMA
             + np.uint64(stream) * _STREAM_MUL + np.uint64(1))
    return _mix(np.array([z], dtype=np.uint64))[0]


def words(seed: int, stream: int, count: int, offset: int = 0) -> np.ndarray:
    """``count`` splitmix64 words of (seed, stream), starting at word ``offset``."""
    key = stream_key(seed, stream)
    out = np.empty(count, dtype=np.uint64)
    for start in range(0, count, _CHUNK):
        n = min(_CHUNK, count - start)
        idx = np.arange(offset + start + 1, offset + start + 1 + n, dtype=np.uint64)
        with np.errstate(over="ignore"):
            out[start:start + n] = _mix(key + idx * GAMMA)
    return out


def uniform(seed: int, stream: int, count: int) -> np.ndarray:
    """Uniform doubles in (0, 1]."""
    w = words(seed, stream, count)
    return ((w >> np.uint64(11)).astype(np.float64) + 1.0) * (2.0 ** -53)


def normal(seed: int, stream: int, count: int) -> np.ndarray:
    """Standard normal float64 draws by Box-Muller on consecutive uniform pairs."""
    npairs = (count + 1) // 2
    out = np.empty(2 * npairs, dtype=np.float64)
    for p0 in range(0, npairs, _CHUNK // 2):
        n = min(_CHUNK // 2, npairs - p0)
        w = words(seed, stream, 2 * n, offset=2 * p0)
        u = ((w >> np.uint64(11)).astype(np.float64) + 1.0) * (2.0 ** -53)
        u1, u2 = u[0::2], u[1::2]
        r = np.sqrt(-2.0 * np.log(u1))
        t = 2.0 * np.pi * u2
        out[2 * p0:2 * (p0 + n):2] = r * np.cos(t)
        out[2 * p0 + 1:2 * (p0 + n):2] = r * np.sin(t)
    return out[:count]


_TORCH_DTYPES = {"fp16": torch.float16, "bf16": torch.bfloat16, "fp32": torch.float32}


def as_dtype(x: np.ndarray, shape, dtype: str) -> torch.Tensor:
    """Round float64 draws to the storage dtype: to float32, then to the 16-bit
    type, each step to nearest even."""
    t = torch.from_numpy(x.astype(np.float32, copy=False)).reshape(shape)
    return t.to(_TORCH_DTYPES[dtype]).contiguous()


def attention_inputs(B: int, H: int, N: int, d: int, dtype: str = "bf16", seed: int = 0):
    """Q, K, V of shape [B, H, N, d], iid N(0, 1), rounded to ``dtype`` (CPU tensors)."""
    shape = (B, H, N, d)
    n = B * H * N * d
    return tuple(as_dtype(normal(seed, s, n), shape, dtype)
                 for s in (STREAM_Q, STREAM_K, STREAM_V))


def outlier_inputs(B: int, H: int, N: int, d: int, dtype: str = "bf16", seed: int = 0,
                   sigma: float = 10.0, prob: float = 0.001):
    """Q, K, V = N(0, 1) + N(0, sigma**2) * Bernoulli(prob), rounded to ``dtype``.

    sigma = 10 reads "N(0,100)" as a variance of 100; sigma = 100 is the
    other reading, kept as a sensitivity case.
    """
    shape = (B, H, N, d)
    n = B * H * N * d
    out = []
    for i, s in enumerate((STREAM_Q, STREAM_K, STREAM_V)):
        x = normal(seed, s, n)
        hit = uniform(seed, STREAM_OUTLIER_MASK + i, n) <= prob
        x[hit] += sigma * normal(seed, STREAM_OUTLIER_MAG + i, n)[hit]
        out.append(as_dtype(x, shape, dtype))
    return tuple(out)


def hadamard_signs(H: int, d: int, seed: int = 0) -> torch.Tensor:
    """Random +-1 signs, one vector of length d per head, int8 [H, d]."""
    w = words(seed, STREAM_SIGNS, H * d)
    s = np.where((w >> np.uint64(63)) == 0, 1, -1).astype(np.int8)
    return torch.from_numpy(s.reshape(H, d)).contiguous()


def rotary_tables(N: int, d: int, base: float = 10000.0, offset: int = 0):
    """cos / sin tables [N, d/2] float32 of a rotary embedding cache: entry
    (n, i) of the angle (n + offset) * base^(-2i/d), evaluated in float64 and
    rounded once.  Deterministic: a caller-side input, like the signs."""
    pos = np.arange(offset, offset + N, dtype=np.float64)[:, None]
    inv_freq = base ** (-np.arange(0, d, 2, dtype=np.float64) / d)[None, :]
    ang = pos * inv_freq
    return (torch.from_numpy(np.cos(ang).astype(np.float32)).contiguous(),
            torch.from_numpy(np.sin(ang).astype(np.float32)).contiguous())


def sample_rows(N: int, count: int, seed: int = 0, salt: int = 0) -> np.ndarray:
    """``count`` distinct query rows in [0, N), sorted (seeded partial shuffle)."""
    count = min(count, N)
    w = words(seed, STREAM_ROWS + 16 * salt, count)
    perm = np.arange(N, dtype=np.int64)
    for i in range(count):  # Fisher-Yates, first ``count`` positions only
        j = i + int(w[i] % np.uint64(N - i))
        perm[i], perm[j] = perm[j], perm[i]
    return np.sort(perm[:count])
