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
