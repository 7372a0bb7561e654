"""The host-buffer entry point that allocates nothing (attn_fwd_host_noalloc).

It serves callers that cannot allocate device memory -- a host framework that
owns every device allocation, device memory already reserved by another
allocator, or a latency-critical path where cudaMalloc could synchronise the
device -- by keeping its device copies in one fixed array inside the library.
Called through the C ABI on two calls in a row with different problems (the
array keeps the previous call's contents), its output must match both the
float64 oracle and the workspace entry point (attn_fwd_host) within the parity
tolerances, and each call must leave the device status clean.  A further test
checks the property the entry point exists for: once the library is loaded
and the array's address looked up, a call leaves the device's free memory
unchanged.  This file is collected last, so a run that stops at the first
failure has already run every other test.
"""
import ctypes

import pytest
import torch

import exact_attention_forward_05_gb300 as attn
import oracle
from tests import parity

pytestmark = pytest.mark.gpu


def _noalloc(lib, q, k, v, causal, scale, o=None, lse=None):
    B, H, N, d = q.shape
    o = torch.empty_like(q).pin_memory() if o is None else o
    lse = torch.empty((B, H, N), dtype=torch.float32).pin_memory() if lse is None else lse
    fn = lib.attn_fwd_host_noalloc
    vp, i32 = ctypes.c_void_p, ctypes.c_int
    fn.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, ctypes.c_float, i32, vp]
    fn.restype = i32
    dt = attn.ATTN_BF16 if q.dtype == torch.bfloat16 else attn.ATTN_FP16
    st = fn(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, N, d,
            int(causal), float(scale), dt, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return st, o, lse


CASES = [((2, 4, 520, 128, "bf16"), False, 1), ((1, 3, 333, 64, "fp16"), True, 2)]


def test_noalloc_matches_oracle_and_workspace_entry_point_on_two_calls():
    lib = attn.lib()
    for (B, H, N, d, dt), causal, seed in CASES:
        what = (B, H, N, d, dt, causal)
        q, k, v = (t.pin_memory() for t in parity.inputs(B, H, N, d, dt, seed=seed))
        scale = d ** -0.5
        st, o, lse = _noalloc(lib, q, k, v, causal, scale)
        assert st == attn.ATTN_OK, attn.status_string(st)
        # A clean return means the copies and the kernel ran; the device status
        # rules out a kernel whose internal wait timed out.
        assert attn.device_status() == attn.ATTN_OK
        o_ref, lse_ref = oracle.attention(q, k, v, causal=causal, scale=scale)
        parity.assert_close(parity.metrics(o, lse, o_ref, lse_ref), f"noalloc vs oracle {what}")
        o_ws, lse_ws = attn.attn_fwd_host(q, k, v, causal=causal, scale=scale)
        m = parity.metrics(o, lse, o_ws.double().numpy(), lse_ws.double().numpy())
        parity.assert_close(m, f"noalloc vs workspace entry point {what}")


def test_noalloc_call_leaves_free_device_memory_unchanged():
    lib = attn.lib()
    (B, H, N, d, dt), causal, seed = CASES[0]
    q, k, v = (t.pin_memory() for t in parity.inputs(B, H, N, d, dt, seed=seed))
    o = torch.empty_like(q).pin_memory()
    lse = torch.empty((B, H, N), dtype=torch.float32).pin_memory()
    # The first call of this shape on the device looks up the array's address
    # and loads the kernel; the calls after it must allocate nothing.
    st, _, _ = _noalloc(lib, q, k, v, causal, d ** -0.5, o, lse)
    assert st == attn.ATTN_OK
    torch.cuda.synchronize()
    free_before = torch.cuda.mem_get_info()[0]
    for _ in range(3):
        st, _, _ = _noalloc(lib, q, k, v, causal, d ** -0.5, o, lse)
        assert st == attn.ATTN_OK
    torch.cuda.synchronize()
    free_after = torch.cuda.mem_get_info()[0]
    assert free_after == free_before, (free_before, free_after)
    assert attn.device_status() == attn.ATTN_OK


def test_noalloc_rejects_problems_beyond_the_array():
    lib = attn.lib()
    fn = lib.attn_fwd_host_noalloc
    vp, i32 = ctypes.c_void_p, ctypes.c_int
    fn.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, ctypes.c_float, i32, vp]
    fn.restype = i32
    # 4 x (1 x 64 x 4096 x 128 x 2 bytes) = 256 MiB > 64 MiB: rejected before any copy.
    st = fn(0x1000, 0x2000, 0x3000, 0x4000, 0x5000, 1, 64, 4096, 128, 0, 0.1, attn.ATTN_BF16, None)
    assert st == attn.ATTN_ERR_INVALID_ARG
    assert attn.NOALLOC_SCRATCH_BYTES == 64 * 1024 * 1024
