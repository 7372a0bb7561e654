"""Float64 CPU oracle for the exact attention forward -- TEST INFRASTRUCTURE.

Only the test suite, the smoke check and the benchmark's CPU-baseline leg may
import this package.  It shares no code with the CUDA library: the C source
``oracle.c`` is compiled here by gcc, and this module only marshals arrays.

Definitions (each cited where it is computed, in ``oracle.c``):

* ``attention``: softmax(scale * Q K^T [+ causal mask]) V and the per-row
  logsumexp, exactly as the "Standard Attention" section of "FlashAttention --
  one, two, three!" lays it out (three plain passes, Nq x Nk scores per head;
  for Nq != Nk the causal mask is aligned at the first positions, causal=1 or
  True, or at the last positions, causal=2).
* ``e4m3_encode`` / ``e4m3_decode``: OCP E4M3 codec, round to nearest even,
  saturating at +-448.
* ``hadamard_rotate``: x -> (x * sigma) H_d / sqrt(d) with the Sylvester
  Hadamard matrix, the random-sign rotation of "Incoherent Processing for FP8
  Accuracy" (FlashAttention-3 podcast page).
* ``attention_bwd``: dQ, dK, dV of ``attention`` for a given dL/dO, the chain
  rule through the definition (the pages name the backward pass and its
  recomputation, "FlashAttention v1.", but print no gradient formulas).
* ``rotary``: the rotary position embedding that the same section names as the
  memory-bound step the rotation is fused into; the pages do not define it, so
  it is RoFormer's pairwise rotation by position-dependent angles, with the
  angles given as cos / sin tables and either pairing convention.
* ``block_quantize``: per-block (or per-tensor) amax scaling to E4M3, the block
  quantisation of the comrad404 review, "Метод", item 3.
* ``fp8_pipeline``: the composition of the three steps above followed by exact
  attention on the dequantised operands (what the FP8 path computes apart from
  its own rounding of P and its accumulation order).

Parity pins for every function live in ``tests/test_oracle_pins.py``.  The
FP8 error-reduction ratio the pages report is context only: parity unpinned.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "liboracle.so")
_lock = threading.Lock()
_lib = None

E4M3_MAX = 448.0
QUANT_BLOCK = 128


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` with gcc into ``oracle/_build/liboracle.so``."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
           "-fvisibility=hidden", "-D_GNU_SOURCE", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64, dp, i32 = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int
            lib.oracle_attention.argtypes = [dp, dp, dp, dp, dp, i64, i64, i64, i32,
                                             ctypes.c_double, dp, i64, i32, dp]
            lib.oracle_attention.restype = i32
            lib.oracle_attention_qk.argtypes = [dp, dp, dp, dp, dp, i64, i64, i64, i64, i32,
                                                ctypes.c_double, dp, i64, i32, dp]
            lib.oracle_attention_qk.restype = i32
            lib.oracle_e4m3_decode.argtypes = [dp, dp, i64]
            lib.oracle_e4m3_encode.argtypes = [dp, dp, i64]
            lib.oracle_hadamard_entry.argtypes = [i64, i64]
            lib.oracle_hadamard_entry.restype = i32
            lib.oracle_hadamard_rotate.argtypes = [dp, dp, dp, i64, i64, i64, i64]
            lib.oracle_hadamard_rotate.restype = i32
            lib.oracle_attention_bwd.argtypes = [dp, dp, dp, dp, dp, dp, dp, i64, i64, i64, i64, i32,
                                                 ctypes.c_double, i32]
            lib.oracle_attention_bwd.restype = i32
            lib.oracle_rotary.argtypes = [dp, dp, dp, dp, i64, i64, i64, i32]
            lib.oracle_rotary.restype = i32
            lib.oracle_block_quantize.argtypes = [dp, dp, dp, i64, i64, i64, i64, i32]
            lib.oracle_block_quantize.restype = i32
            _lib = lib
    return _lib


def _f64(x) -> np.ndarray:
    if hasattr(x, "detach"):  # torch tensor (CPU): widen exactly to float64
        x = x.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(x, dtype=np.float64)


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


def attention(q, k, v, causal: bool = False, scale: float | None = None, rows=None,
              nthreads: int = 0, return_threads: bool = False):
    """Exact attention in float64.

    q: [B, H, Nq, d], k, v: [B, H, Nk, d] (torch CPU tensors or numpy arrays,
    any float dtype; values are widened exactly).  ``causal``: False / 0 (no
    mask), True / 1 (query i sees keys j <= i), 2 (query i sees keys
    j <= i + Nk - Nq).  ``rows``: optional sorted query-row subset, applied to
    every head.  Returns (O [B, H, R, d], lse [B, H, R]) float64, plus the
    thread count when ``return_threads``.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, N, d = q.shape
    if k.shape != v.shape or k.shape[:2] != (B, H) or k.shape[3] != d:
        raise ValueError("k, v must be [B, H, Nk, d] with q's B, H and d")
    Nk = k.shape[2]
    mode = int(causal)
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    rows_arr = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    R = N if rows_arr is None else len(rows_arr)
    o = np.empty((B, H, R, d), dtype=np.float64)
    lse = np.empty((B, H, R), dtype=np.float64)
    used = ctypes.c_int(0)
    st = _load().oracle_attention_qk(
        _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B * H, N, Nk, d, mode,
        float(scale), None if rows_arr is None else _ptr(rows_arr), R, int(nthreads),
        ctypes.cast(ctypes.pointer(used), ctypes.c_void_p))
    if st != 0:
        raise RuntimeError(f"oracle_attention failed with status {st}")
    return (o, lse, used.value) if return_threads else (o, lse)


def e4m3_decode(codes) -> np.ndarray:
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    out = np.empty(c.shape, dtype=np.float64)
    _load().oracle_e4m3_decode(_ptr(c), _ptr(out), c.size)
    return out


def e4m3_encode(x) -> np.ndarray:
    a = _f64(x)
    out = np.empty(a.shape, dtype=np.uint8)
    _load().oracle_e4m3_encode(_ptr(a), _ptr(out), a.size)
    return out


def hadamard_matrix(d: int) -> np.ndarray:
    """Sylvester Hadamard matrix H_d (entries +-1) as the oracle defines it."""
    lib = _load()
    return np.array([[lib.oracle_hadamard_entry(i, j) for j in range(d)] for i in range(d)],
                    dtype=np.float64)


def hadamard_rotate(x, signs) -> np.ndarray:
    """x [B, H, N, d] -> (x * sigma_h) H_d / sqrt(d) per head, float64."""
    a = _f64(x)
    B, H, N, d = a.shape
    s = np.ascontiguousarray(signs.numpy() if hasattr(signs, "numpy") else signs, dtype=np.int8)
    out = np.empty_like(a)
    st = _load().oracle_hadamard_rotate(_ptr(a), _ptr(s), _ptr(out), B * H, H, N, d)
    if st != 0:
        raise ValueError("hadamard_rotate: d must be a power of two")
    return out


def attention_bwd(q, k, v, dout, causal=False, scale: float | None = None, nthreads: int = 0):
    """Gradients (dQ, dK, dV) of ``attention`` for dL/dO = ``dout``, float64.

    q, dout: [B, H, Nq, d]; k, v: [B, H, Nk, d]; ``causal`` as for
    ``attention``.  lse is an auxiliary output: no gradient flows through it.
    """
    q, k, v, g = _f64(q), _f64(k), _f64(v), _f64(dout)
    B, H, N, d = q.shape
    if k.shape != v.shape or k.shape[:2] != (B, H) or k.shape[3] != d or g.shape != q.shape:
        raise ValueError("k, v must be [B, H, Nk, d] and dout like q")
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    dq, dk, dv = np.empty_like(q), np.empty_like(k), np.empty_like(v)
    st = _load().oracle_attention_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(dq), _ptr(dk), _ptr(dv),
                                      B * H, N, k.shape[2], d, int(causal), float(scale), int(nthreads))
    if st != 0:
        raise RuntimeError(f"oracle_attention_bwd failed with status {st}")
    return dq, dk, dv


def rotary(x, cos, sin, interleaved: bool = False) -> np.ndarray:
    """x [B, H, N, d] -> the rotary position embedding of every row, float64;
    cos, sin: [N, d/2] tables (float32 values), pair i = (2i, 2i+1) when
    ``interleaved`` else (i, i + d/2)."""
    a = _f64(x)
    B, H, N, d = a.shape
    c = np.ascontiguousarray(_np32(cos))
    s = np.ascontiguousarray(_np32(sin))
    if c.shape != (N, d // 2) or s.shape != (N, d // 2):
        raise ValueError("cos, sin must be [N, d/2]")
    out = np.empty_like(a)
    st = _load().oracle_rotary(_ptr(a), _ptr(c), _ptr(s), _ptr(out), B * H, N, d, int(bool(interleaved)))
    if st != 0:
        raise RuntimeError(f"oracle_rotary failed with status {st}")
    return out


def _np32(t) -> np.ndarray:
    t = t.cpu().numpy() if hasattr(t, "cpu") else np.asarray(t)
    return t.astype(np.float32)


def block_quantize(x, block: int = QUANT_BLOCK, per_tensor: bool = False):
    """E4M3 codes [B, H, N, d] and float32 scales [B, H, ceil(N/block)] (or [1])."""
    a = _f64(x)
    B, H, N, d = a.shape
    codes = np.empty(a.shape, dtype=np.uint8)
    nblk = (N + block - 1) // block
    scales = np.empty(1 if per_tensor else (B, H, nblk), dtype=np.float32)
    st = _load().oracle_block_quantize(_ptr(a), _ptr(codes), _ptr(scales), B * H, N, d,
                                       block, int(bool(per_tensor)))
    if st != 0:
        raise ValueError("block_quantize: bad block size")
    return codes, scales


def dequantize(codes, scales, block: int = QUANT_BLOCK) -> np.ndarray:
    """codes * scale of their block, float64."""
    vals = e4m3_decode(codes)
    s = np.asarray(scales, dtype=np.float64)
    if s.size == 1:
        return vals * float(s.reshape(-1)[0])
    rep = np.repeat(s, block, axis=-1)[..., :vals.shape[2]]
    return vals * rep[..., None]


def fp8_pipeline(q, k, v, signs=None, causal: bool = False, scale: float | None = None,
                 per_tensor: bool = False, rows=None, block: int = QUANT_BLOCK, rope=None):
    """Rotary embedding of Q and K (if ``rope`` = (cos, sin, interleaved)), their
    Hadamard rotation (if ``signs``), E4M3 quantisation of Q, K, V, then exact
    attention on the dequantised operands.  Returns (O, lse) like ``attention``."""
    qf, kf, vf = _f64(q), _f64(k), _f64(v)
    if rope is not None:
        qf, kf = (rotary(t, rope[0], rope[1], rope[2]) for t in (qf, kf))
    if signs is not None:
        qf, kf = hadamard_rotate(qf, signs), hadamard_rotate(kf, signs)
    deq = []
    for t in (qf, kf, vf):
        c, s = block_quantize(t, block, per_tensor)
        deq.append(dequantize(c, s, block))
    return attention(deq[0], deq[1], deq[2], causal=causal, scale=scale, rows=rows)
