"""GB300 (sm_103a) exact attention forward -- Python binding of the C ABI.

Argument marshalling only: every step of the computation runs in the CUDA
kernels of ``_build/libattn_gb300.so`` (declared in ``include/attn.h``).
PyTorch supplies device memory and streams.  There is no fallback: if the
library is missing or a call fails, an exception is raised.

The operation is exact attention, O = softmax(scale * Q K^T [+ causal mask]) V
with the per-row logsumexp ("FlashAttention -- one, two, three!", section
"Standard Attention"), computed by one fused tiled kernel.
"""
from __future__ import annotations

import ctypes
import math
import os
import re
import threading

import torch

from . import build as _build

__all__ = ["attn_fwd", "workspace_bytes", "attn_bwd", "bwd_workspace_bytes", "attn_fwd_host", "fp8_prepare", "attn_fwd_fp8", "attn_fwd_fp8_pipeline", "host_workspace_bytes", "device_status",
           "set_wait_timeout_ns", "set_schedule", "debug_bounded_wait", "debug_fail_host_chunk", "debug_exp2_poly", "debug_tmem_ld_red",
           "attn_fwd_host_noalloc", "status_string", "library_path",
           "AttnError", "ATTN_OK", "ATTN_ERR_INVALID_ARG", "ATTN_ERR_UNSUPPORTED",
           "ATTN_ERR_MISALIGNED", "ATTN_ERR_CUDA", "ATTN_ERR_TIMEOUT", "exported_symbols",
           "LAYOUT_BHND", "LAYOUT_BNHD", "CAUSAL_NONE", "CAUSAL_TOP_LEFT", "CAUSAL_BOTTOM_RIGHT"]

ATTN_OK, ATTN_ERR_INVALID_ARG, ATTN_ERR_UNSUPPORTED, ATTN_ERR_MISALIGNED, ATTN_ERR_CUDA, \
    ATTN_ERR_TIMEOUT = range(6)
LAYOUT_BHND, LAYOUT_BNHD = 0, 1  # [B, H, N, d] / [B, N, H, d] for q, k, v and o
_LAYOUTS = {"bhnd": LAYOUT_BHND, "bnhd": LAYOUT_BNHD}
CAUSAL_NONE, CAUSAL_TOP_LEFT, CAUSAL_BOTTOM_RIGHT = 0, 1, 2
_CAUSAL_NAMES = {"none": CAUSAL_NONE, "top_left": CAUSAL_TOP_LEFT, "bottom_right": CAUSAL_BOTTOM_RIGHT}


def _causal_mode(causal) -> int:
    """False / True / 0 / 1 / 2 or a name in _CAUSAL_NAMES -> CAUSAL_*."""
    mode = _CAUSAL_NAMES.get(causal, -1) if isinstance(causal, str) else int(causal)
    if mode not in (CAUSAL_NONE, CAUSAL_TOP_LEFT, CAUSAL_BOTTOM_RIGHT):
        raise ValueError("causal must be False, True, 'top_left' or 'bottom_right'")
    return mode
ATTN_FP16, ATTN_BF16 = 0, 1
_DTYPES = {torch.float16: ATTN_FP16, torch.bfloat16: ATTN_BF16}

_lock = threading.Lock()
_lib = None


class AttnError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})")


def library_path() -> str:
    return _build.LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            path = _build.LIB_PATH
            if not os.path.exists(path):
                raise RuntimeError(f"{path} is not built; run __graft_entry__.build() "
                                   "(the CUDA library is required, there is no fallback)")
            lib = ctypes.CDLL(path)
            vp, i32, f32, u64, sz = (ctypes.c_void_p, ctypes.c_int, ctypes.c_float,
                                     ctypes.c_uint64, ctypes.c_size_t)
            lib.attn_fwd.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, f32, i32, vp]
            lib.attn_fwd.restype = i32
            lib.attn_fwd_ex.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, i32, f32, i32, i32, vp]
            lib.attn_fwd_ex.restype = i32
            lib.attn_fwd_ws.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, f32, i32, vp, sz, vp]
            lib.attn_fwd_ws.restype = i32
            lib.attn_fwd_workspace_bytes.argtypes = [i32]
            lib.attn_fwd_workspace_bytes.restype = sz
            lib.attn_fwd_fp8_ws.argtypes = [vp, vp, vp, vp, vp, vp, i32, vp, vp, i32, i32, i32, i32,
                                            i32, f32, vp, sz, vp]
            lib.attn_fwd_fp8_ws.restype = i32
            lib.attn_fwd_host_workspace_bytes.argtypes = [i32, i32, i32, i32, i32]
            lib.attn_fwd_host_workspace_bytes.restype = sz
            lib.attn_fwd_host.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, f32, i32,
                                          vp, sz, vp]
            lib.attn_fwd_host.restype = i32
            lib.attn_fp8_prepare.argtypes = [vp, vp, vp, i32, vp, vp, vp, vp, vp, vp, vp, i32,
                                             i32, i32, i32, i32, vp]
            lib.attn_fp8_prepare.restype = i32
            lib.attn_fp8_prepare_rotary.argtypes = [vp, vp, vp, i32, vp, vp, vp, vp, vp, vp, vp, i32,
                                                    vp, vp, i32, i32, i32, i32, i32, vp]
            lib.attn_fp8_prepare_rotary.restype = i32
            lib.attn_fwd_fp8.argtypes = [vp, vp, vp, vp, vp, vp, i32, vp, vp, i32, i32, i32, i32,
                                         i32, f32, vp]
            lib.attn_fwd_fp8.restype = i32
            lib.attn_bwd_workspace_bytes.argtypes = [i32, i32, i32, i32]
            lib.attn_bwd_workspace_bytes.restype = sz
            lib.attn_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, f32, i32,
                                     vp, sz, vp]
            lib.attn_bwd.restype = i32
            lib.attn_get_device_status.argtypes = [vp]
            lib.attn_get_device_status.restype = i32
            lib.attn_set_wait_timeout_ns.argtypes = [u64]
            lib.attn_set_wait_timeout_ns.restype = None
            lib.attn_set_schedule.argtypes = [i32]
            lib.attn_debug_bounded_wait.argtypes = [u64, vp]
            lib.attn_debug_bounded_wait.restype = i32
            lib.attn_debug_exp2_poly.argtypes = [vp, vp, vp, i32, vp]
            lib.attn_debug_exp2_poly.restype = i32
            lib.attn_debug_tmem_ld_red.argtypes = [vp, vp, vp, i32, i32, vp]
            lib.attn_debug_tmem_ld_red.restype = i32
            lib.attn_debug_fail_host_chunk.argtypes = [i32]
            lib.attn_debug_fail_host_chunk.restype = None
            lib.attn_fwd_host_noalloc.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, f32, i32, vp]
            lib.attn_fwd_host_noalloc.restype = i32
            lib.attn_last_cuda_error.argtypes = []
            lib.attn_last_cuda_error.restype = i32
            lib.attn_status_string.argtypes = [i32]
            lib.attn_status_string.restype = ctypes.c_char_p
            lib.attn_version.argtypes = []
            lib.attn_version.restype = ctypes.c_char_p
            _lib = lib
    return _lib


def lib():
    """The loaded ctypes library (raises if it is not built)."""
    return _load()


def exported_symbols():
    """Names of the functions ``include/attn.h`` declares."""
    hdr = os.path.join(os.path.dirname(_build.PKG), "include", "attn.h")
    text = open(hdr).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(attn_[a-z0-9_]+)\s*\(", text)))


def status_string(status: int) -> str:
    return _load().attn_status_string(int(status)).decode()


def _stream_handle(stream, device) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream)


def _check(st: int, what: str):
    if st != ATTN_OK:
        raise AttnError(st, what)


def _shape_of(q, k, v):
    if q.dim() != 4 or q.shape != k.shape or q.shape != v.shape:
        raise ValueError("q, k, v must share one [B, H, N, d] shape")
    if not (q.dtype == k.dtype == v.dtype) or q.dtype not in _DTYPES:
        raise ValueError("q, k, v must all be float16 or all bfloat16")
    for t in (q, k, v):
        if not t.is_contiguous():
            raise ValueError("q, k, v must be contiguous [B, H, N, d]")
    return tuple(int(s) for s in q.shape)


def _qkv_shapes(q, k, v, layout):
    """(B, H, Nq, Nk, d) of q [B, H, Nq, d] and k, v [B, H, Nk, d] (or the
    [B, N, H, d] forms)."""
    if q.dim() != 4 or k.dim() != 4 or k.shape != v.shape:
        raise ValueError("q, k, v must be 4-D, k and v of one shape")
    if not (q.dtype == k.dtype == v.dtype) or q.dtype not in _DTYPES:
        raise ValueError("q, k, v must all be float16 or all bfloat16")
    for t in (q, k, v):
        if not t.is_contiguous():
            raise ValueError("q, k, v must be contiguous")
    if layout == "bnhd":
        (B, Nq, H, d), (Bk, Nk, Hk, dk) = q.shape, k.shape
    else:
        (B, H, Nq, d), (Bk, Hk, Nk, dk) = q.shape, k.shape
    if (B, H, d) != (Bk, Hk, dk):
        raise ValueError("q, k, v must share B, H and d")
    return int(B), int(H), int(Nq), int(Nk), int(d)


def workspace_bytes(d: int, device=None) -> int:
    """Bytes of the workspace that balances full attention over the SMs
    (attn_fwd_workspace_bytes) for head dimension d on ``device``."""
    device = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with torch.cuda.device(device):
        return int(_load().attn_fwd_workspace_bytes(int(d)))


def _check_workspace(ws, device):
    if ws.dtype != torch.uint8 or not ws.is_contiguous() or ws.device != device:
        raise ValueError("workspace must be a contiguous uint8 tensor on q's device")


def attn_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, causal=False,
             scale: float | None = None, out: torch.Tensor | None = None,
             lse: torch.Tensor | None = None, return_lse: bool = True, stream=None,
             layout: str = "bhnd", workspace: torch.Tensor | None = None):
    """Exact attention forward on CUDA tensors (fp16 or bf16).

    q: [B, H, Nq, d], k, v: [B, H, Nk, d]; with ``layout="bnhd"`` they are
    [B, Nq, H, d] and [B, Nk, H, d] (no transpose needed).  ``causal``: False,
    True (query i sees keys j <= i) or "bottom_right" (query i sees keys
    j <= i + Nk - Nq: the queries are the last Nq positions).  Returns (O, lse)
    with O like q and lse float32 [B, H, Nq] in either layout (None when
    ``return_lse`` is false and no ``lse`` buffer is given).  ``workspace``
    (uint8 CUDA tensor of workspace_bytes(d)) selects attn_fwd_ws, which
    balances full self-attention in [B, H, N, d] over the SMs.
    """
    if layout not in _LAYOUTS:
        raise ValueError("layout must be 'bhnd' or 'bnhd'")
    mode = _causal_mode(causal)
    B, H, N, Nk, d = _qkv_shapes(q, k, v, layout)
    if not (q.is_cuda and k.device == q.device and v.device == q.device):
        raise ValueError("q, k, v must be CUDA tensors on one device")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    if (out.shape != q.shape or out.dtype != q.dtype or out.device != q.device
            or not out.is_contiguous()):
        raise ValueError("out must be a contiguous tensor like q")
    if lse is None and return_lse:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    if lse is not None and (lse.dtype != torch.float32 or not lse.is_contiguous()
                            or tuple(lse.shape) != (B, H, N) or lse.device != q.device):
        raise ValueError("lse must be a contiguous float32 [B, H, N] tensor on q's device")
    if workspace is not None:
        if layout != "bhnd" or N != Nk or mode == CAUSAL_BOTTOM_RIGHT:
            raise ValueError("a workspace is taken for [B, H, N, d] self-attention only")
        _check_workspace(workspace, q.device)
        with torch.cuda.device(q.device):
            st = _load().attn_fwd_ws(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                     None if lse is None else lse.data_ptr(), B, H, N, d, mode,
                                     float(scale), _DTYPES[q.dtype], workspace.data_ptr(),
                                     workspace.numel(), _stream_handle(stream, q.device))
        _check(st, "attn_fwd_ws")
        return out, lse
    with torch.cuda.device(q.device):
        st = _load().attn_fwd_ex(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                 None if lse is None else lse.data_ptr(), B, H, N, Nk, d,
                                 mode, float(scale), _DTYPES[q.dtype], _LAYOUTS[layout],
                                 _stream_handle(stream, q.device))
    _check(st, "attn_fwd")
    return out, lse


def host_workspace_bytes(B: int, H: int, N: int, d: int, dtype=torch.bfloat16) -> int:
    return int(_load().attn_fwd_host_workspace_bytes(B, H, N, d, _DTYPES[dtype]))


def attn_fwd_host(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, causal: bool = False,
                  scale: float | None = None, workspace: torch.Tensor | None = None,
                  out: torch.Tensor | None = None, lse: torch.Tensor | None = None,
                  device=None, stream=None):
    """The same operation on host tensors (pinned memory recommended): the
    library copies the inputs to ``workspace`` on the device, runs the kernel
    and copies O and lse back, synchronising the stream before it returns."""
    B, H, N, d = _shape_of(q, k, v)
    if q.is_cuda:
        raise ValueError("attn_fwd_host takes host tensors")
    device = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    need = host_workspace_bytes(B, H, N, d, q.dtype)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=device)
    if out is None:
        out = torch.empty_like(q, pin_memory=q.is_pinned())
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, pin_memory=q.is_pinned())
    with torch.cuda.device(device):
        st = _load().attn_fwd_host(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                   lse.data_ptr(), B, H, N, d, int(bool(causal)), float(scale),
                                   _DTYPES[q.dtype], workspace.data_ptr(), workspace.numel(),
                                   _stream_handle(stream, device))
    _check(st, "attn_fwd_host")
    return out, lse


FP8_BLOCK = 128  # rows per quantisation scale block


def fp8_prepare(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, signs: torch.Tensor | None = None,
                per_tensor: bool = False, stream=None, out=None, rope=None, rope_interleaved: bool = False):
    """FP8 pre-pass on CUDA tensors [B, H, N, d], d = 64, 128 or 256 (fp16 or
    bf16): rotary embedding of Q and K (when ``rope`` = (cos, sin), float32
    [N, d/2] CUDA tables; pairs (2i, 2i+1) if ``rope_interleaved`` else
    (i, i + d/2)), then
    their random-sign Hadamard rotation (when ``signs`` [H, d] int8 is given)
    and E4M3 quantisation with one float32 scale per 128 rows of a head (or one
    per tensor).  Returns (q8, k8, v8, q_scale, k_scale, v_scale); the codes are
    uint8 tensors [B, H, N, 128].  ``out`` may pass those six tensors in."""
    B, H, N, d = _shape_of(q, k, v)
    if not q.is_cuda:
        raise ValueError("fp8_prepare takes CUDA tensors")
    nblk = (N + FP8_BLOCK - 1) // FP8_BLOCK
    sshape = (1,) if per_tensor else (B, H, nblk)
    if out is not None:
        codes, scales = list(out[:3]), list(out[3:])
        for c in codes:
            if c.dtype != torch.uint8 or tuple(c.shape) != (B, H, N, d) or not c.is_contiguous():
                raise ValueError("code tensors must be contiguous uint8 [B, H, N, d]")
        for sc in scales:
            if sc.dtype != torch.float32 or tuple(sc.shape) != sshape or not sc.is_contiguous():
                raise ValueError(f"scale tensors must be contiguous float32 {sshape}")
    else:
        codes = [torch.empty((B, H, N, d), dtype=torch.uint8, device=q.device) for _ in range(3)]
        scales = [torch.empty(sshape, dtype=torch.float32, device=q.device) for _ in range(3)]
    if signs is not None:
        if signs.dtype != torch.int8 or tuple(signs.shape) != (H, d):
            raise ValueError("signs must be an int8 [H, d] tensor of +1 / -1")
        signs = signs.to(q.device).contiguous()
    rc = rs = None
    if rope is not None:
        rc, rs = rope
        for t in (rc, rs):
            if (t.dtype != torch.float32 or tuple(t.shape) != (N, d // 2) or not t.is_contiguous()
                    or t.device != q.device):
                raise ValueError("rope tables must be contiguous float32 [N, d/2] on q's device")
    with torch.cuda.device(q.device):
        st = _load().attn_fp8_prepare_rotary(
            q.data_ptr(), k.data_ptr(), v.data_ptr(), _DTYPES[q.dtype],
            *(c.data_ptr() for c in codes), *(sc.data_ptr() for sc in scales),
            None if signs is None else signs.data_ptr(), int(bool(per_tensor)),
            None if rc is None else rc.data_ptr(), None if rs is None else rs.data_ptr(),
            int(bool(rope_interleaved)), B, H, N, d, _stream_handle(stream, q.device))
    _check(st, "attn_fp8_prepare")
    return (*codes, *scales)


def attn_fwd_fp8(q8, k8, v8, q_scale, k_scale, v_scale, causal: bool = False,
                 scale: float | None = None, out: torch.Tensor | None = None,
                 lse: torch.Tensor | None = None, return_lse: bool = True, stream=None,
                 workspace: torch.Tensor | None = None):
    """Exact attention on E4M3 codes (uint8 [B, H, N, d], d = 64, 128, 256)
    and float32 scales (per block [B, H, ceil(N/128)] or per tensor [1]); bf16
    output.  ``workspace`` as for attn_fwd (attn_fwd_fp8_ws)."""
    if q8.dim() != 4 or q8.shape != k8.shape or q8.shape != v8.shape:
        raise ValueError("q8, k8, v8 must share one [B, H, N, d] shape")
    B, H, N, d = (int(s_) for s_ in q8.shape)
    per_tensor = q_scale.numel() == 1
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty((B, H, N, d), dtype=torch.bfloat16, device=q8.device)
    if lse is None and return_lse:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q8.device)
    if workspace is not None:
        _check_workspace(workspace, q8.device)
    with torch.cuda.device(q8.device):
        st = _load().attn_fwd_fp8_ws(q8.data_ptr(), k8.data_ptr(), v8.data_ptr(), q_scale.data_ptr(),
                                     k_scale.data_ptr(), v_scale.data_ptr(), int(per_tensor),
                                     out.data_ptr(), None if lse is None else lse.data_ptr(),
                                     B, H, N, d, int(bool(causal)), float(scale),
                                     None if workspace is None else workspace.data_ptr(),
                                     0 if workspace is None else workspace.numel(),
                                     _stream_handle(stream, q8.device))
    _check(st, "attn_fwd_fp8")
    return out, lse


def attn_fwd_fp8_pipeline(q, k, v, signs=None, causal: bool = False, scale: float | None = None,
                          per_tensor: bool = False, stream=None, rope=None, rope_interleaved: bool = False):
    """fp8_prepare followed by attn_fwd_fp8 (the quantised operands are
    allocated here, as torch tensors)."""
    q8, k8, v8, qs, ks, vs = fp8_prepare(q, k, v, signs=signs, per_tensor=per_tensor, stream=stream,
                                         rope=rope, rope_interleaved=rope_interleaved)
    return attn_fwd_fp8(q8, k8, v8, qs, ks, vs, causal=causal, scale=scale, stream=stream)


def bwd_workspace_bytes(B: int, H: int, N: int, d: int) -> int:
    return int(_load().attn_bwd_workspace_bytes(B, H, N, d))


def attn_bwd(q, k, v, o, dout, lse, causal: bool = False, scale: float | None = None,
             workspace: torch.Tensor | None = None, out=None, stream=None):
    """Gradients (dQ, dK, dV) of attn_fwd for dL/dO = ``dout`` on CUDA tensors
    [B, H, N, d] (d = 64 or 128, fp16 or bf16), given attn_fwd's ``o`` and
    ``lse``; the softmax weights are recomputed from Q, K and lse.  ``out``
    may pass (dq, dk, dv); ``workspace`` (uint8, bwd_workspace_bytes) is
    allocated here when not given."""
    B, H, N, d = _shape_of(q, k, v)
    for t in (o, dout):
        if t.shape != q.shape or t.dtype != q.dtype or not t.is_contiguous() or t.device != q.device:
            raise ValueError("o and dout must be contiguous tensors like q")
    if lse.dtype != torch.float32 or tuple(lse.shape) != (B, H, N) or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous float32 [B, H, N] tensor")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dq, dk, dv = out if out is not None else (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v))
    if workspace is None:
        workspace = torch.empty(max(bwd_workspace_bytes(B, H, N, d), 1), dtype=torch.uint8, device=q.device)
    with torch.cuda.device(q.device):
        st = _load().attn_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), dout.data_ptr(),
                              lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, N, d,
                              int(bool(causal)), float(scale), _DTYPES[q.dtype], workspace.data_ptr(),
                              workspace.numel(), _stream_handle(stream, q.device))
    _check(st, "attn_bwd")
    return dq, dk, dv


def device_status(stream=None) -> int:
    """Synchronise ``stream``; return and clear the device status word."""
    dev = torch.cuda.current_device()
    return int(_load().attn_get_device_status(_stream_handle(stream, dev)))


def set_wait_timeout_ns(ns: int) -> None:
    _load().attn_set_wait_timeout_ns(int(ns))


SCHEDULE_PINGPONG, SCHEDULE_ONE_TILE, SCHEDULE_BALANCED = 0, 1, 2


def set_schedule(mode: int) -> None:
    """Work schedule of later launches with d <= 128: SCHEDULE_PINGPONG (two Q
    tiles per CTA, softmax of one overlapping the products of the other; the
    default) or SCHEDULE_ONE_TILE (one tile at a time, the overlap ablation)."""
    _check(_load().attn_set_schedule(int(mode)), "attn_set_schedule")


def debug_exp2_poly(x: torch.Tensor):
    """(polynomial 2^x of the FP8 weights, CUDA exp2f) of a float32 CUDA
    tensor, elementwise (a test hook)."""
    if x.dtype != torch.float32 or not x.is_cuda or not x.is_contiguous():
        raise ValueError("x must be a contiguous float32 CUDA tensor")
    yp, yr = torch.empty_like(x), torch.empty_like(x)
    with torch.cuda.device(x.device):
        _check(_load().attn_debug_exp2_poly(x.data_ptr(), yp.data_ptr(), yr.data_ptr(), x.numel(),
                                            _stream_handle(None, x.device)), "attn_debug_exp2_poly")
    return yp, yr


def debug_tmem_ld_red(x: torch.Tensor, use_min: bool = False):
    """(values, extremes) of a float32 [128, 32] or [128, 128] CUDA tensor put
    into TMEM and read back by the reducing load of the attention softmax (its
    32- or 128-column form): the values unchanged and each row's maximum
    (minimum with ``use_min``) (a test hook)."""
    if (x.dtype != torch.float32 or not x.is_cuda or not x.is_contiguous() or x.dim() != 2
            or x.shape[0] != 128 or x.shape[1] not in (32, 128)):
        raise ValueError("x must be a contiguous float32 CUDA tensor of shape [128, 32] or [128, 128]")
    vals, ext = torch.empty_like(x), torch.empty(128, dtype=torch.float32, device=x.device)
    with torch.cuda.device(x.device):
        _check(_load().attn_debug_tmem_ld_red(x.data_ptr(), vals.data_ptr(), ext.data_ptr(), int(x.shape[1]),
                                              int(bool(use_min)), _stream_handle(None, x.device)),
               "attn_debug_tmem_ld_red")
    return vals, ext


def debug_fail_host_chunk(chunk: int) -> None:
    """Arm (chunk >= 0) or disarm (-1) the one-shot host-side failure of the
    next host-buffer call at pipeline chunk ``chunk`` (a test hook)."""
    _load().attn_debug_fail_host_chunk(int(chunk))


def debug_bounded_wait(timeout_ns: int, stream=None) -> None:
    dev = torch.cuda.current_device()
    _check(_load().attn_debug_bounded_wait(int(timeout_ns), _stream_handle(stream, dev)),
           "attn_debug_bounded_wait")


NOALLOC_SCRATCH_BYTES = 64 * 1024 * 1024  # ATTN_NOALLOC_SCRATCH_BYTES in include/attn.h


def attn_fwd_host_noalloc(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, causal: bool = False,
                          scale: float | None = None, out: torch.Tensor | None = None,
                          lse: torch.Tensor | None = None, device=None, stream=None):
    """attn_fwd_host without a workspace, for callers that cannot allocate
    device memory (a host framework that owns every device allocation, device
    memory fully reserved by another allocator, or a latency-critical path where
    cudaMalloc could synchronise the device).  The library keeps the device
    copies in one fixed array of NOALLOC_SCRATCH_BYTES shared by every call:
    larger problems raise ATTN_ERR_INVALID_ARG, and calls whose GPU work
    overlaps race on the array.  Host output tensors are created here when not
    given (host memory only)."""
    B, H, N, d = _shape_of(q, k, v)
    if q.is_cuda:
        raise ValueError("attn_fwd_host_noalloc takes host tensors")
    device = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q, pin_memory=q.is_pinned())
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, pin_memory=q.is_pinned())
    fn = _load().attn_fwd_host_noalloc
    with torch.cuda.device(device):
        st = fn(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(), B, H, N, d,
                int(bool(causal)), float(scale), _DTYPES[q.dtype], _stream_handle(stream, device))
    _check(st, "attn_fwd_host_noalloc")
    return out, lse
