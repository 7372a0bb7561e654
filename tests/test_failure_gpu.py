"""Failure detection without a GPU fault: a kernel wait that nothing completes
runs out its time limit, the kernel returns, and the host reads
ATTN_ERR_TIMEOUT from the device status word; the context stays usable."""
import time

import pytest
import torch

import exact_attention_forward_05_gb300 as attn
from tests import parity

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives():
    assert attn.device_status() == attn.ATTN_OK
    t0 = time.time()
    attn.debug_bounded_wait(20_000_000)  # 20 ms limit on a barrier nobody signals
    assert attn.device_status() == attn.ATTN_ERR_TIMEOUT
    assert time.time() - t0 < 10
    assert attn.device_status() == attn.ATTN_OK  # reading clears the word
    q, k, v = parity.inputs(1, 2, 130, 64, "bf16", seed=1)
    parity.check_case(q, k, v, True, what="after timeout")


def test_wait_limit_setting_round_trip():
    attn.set_wait_timeout_ns(5_000_000_000)
    try:
        q, k, v = parity.inputs(1, 1, 256, 128, "bf16", seed=2)
        parity.check_case(q, k, v, False, what="custom limit")
    finally:
        attn.set_wait_timeout_ns(0)


@pytest.mark.parametrize("chunk", [0, 3, 7])
def test_host_pipeline_error_path_then_next_call_is_correct(chunk):
    """A host-side failure injected at pipeline chunk `chunk` (before that
    chunk's kernel is enqueued; nothing faults on the device) makes
    attn_fwd_host return ATTN_ERR_CUDA after draining what it had enqueued.
    The hook is one-shot: the next call on the same streams, workspace and
    host buffers runs every chunk and matches the oracle."""
    import oracle
    B, H, N, d = 2, 8, 384, 128  # 16 (batch, head) pairs: 8 pipeline chunks
    q, k, v = (t.pin_memory() for t in parity.inputs(B, H, N, d, "bf16", seed=chunk))
    scale = d ** -0.5
    ws = torch.empty(attn.host_workspace_bytes(B, H, N, d, q.dtype), dtype=torch.uint8, device="cuda")
    out = torch.full_like(q, float("nan")).pin_memory()
    lse = torch.full((B, H, N), float("nan"), dtype=torch.float32).pin_memory()
    attn.debug_fail_host_chunk(chunk)
    with pytest.raises(attn.AttnError) as e:
        attn.attn_fwd_host(q, k, v, causal=True, scale=scale, workspace=ws, out=out, lse=lse)
    assert e.value.status == attn.ATTN_ERR_CUDA
    # Chunks after the failing one were never launched: their outputs are untouched.
    last = out.reshape(B * H, N, d)[-1]
    assert bool(torch.isnan(last.float()).all())
    o, l = attn.attn_fwd_host(q, k, v, causal=True, scale=scale, workspace=ws, out=out, lse=lse)
    o_ref, lse_ref = oracle.attention(q, k, v, causal=True, scale=scale)
    parity.assert_close(parity.metrics(o, l, o_ref, lse_ref), f"after injected failure at chunk {chunk}")
    assert attn.device_status() == attn.ATTN_OK


def test_noalloc_error_path_then_next_call_is_correct():
    import oracle
    B, H, N, d = 1, 8, 256, 64
    q, k, v = (t.pin_memory() for t in parity.inputs(B, H, N, d, "fp16", seed=9))
    attn.debug_fail_host_chunk(5)
    with pytest.raises(attn.AttnError) as e:
        attn.attn_fwd_host_noalloc(q, k, v, causal=False)
    assert e.value.status == attn.ATTN_ERR_CUDA
    o, l = attn.attn_fwd_host_noalloc(q, k, v, causal=False)
    o_ref, lse_ref = oracle.attention(q, k, v, causal=False, scale=d ** -0.5)
    parity.assert_close(parity.metrics(o, l, o_ref, lse_ref), "noalloc after injected failure")
    assert attn.device_status() == attn.ATTN_OK
