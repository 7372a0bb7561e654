"""Full-size workloads on the GPU, checked on seeded samples of query rows.

* sequence-length sweep: N in {512, ..., 16384} x d in {64, 128, 256} with
  B = 16384 / N and H = 2048 / d, bf16, causal and non-causal (the launch
  configuration the benchmark times for N = 8192, d = 128);
* long context: B = 1, H = 16, N = 32768, d = 128, causal, 64 random query
  rows per head.
The oracle computes the sampled rows one by one; every other row is checked
for finiteness.
"""
import pytest
import torch

import synth
from tests import parity

pytestmark = pytest.mark.gpu

SWEEP_N = [512, 1024, 2048, 4096, 8192, 16384]
SWEEP_D = [64, 128, 256]


@pytest.mark.parametrize("d", SWEEP_D)
@pytest.mark.parametrize("N", SWEEP_N)
def test_sequence_sweep(N, d):
    B, H = 16384 // N, 2048 // d
    q, k, v = synth.attention_inputs(B, H, N, d, "bf16", seed=0)
    rows = synth.sample_rows(N, 64, seed=0, salt=N + d)
    for causal in (False, True):
        parity.check_case(q, k, v, causal, rows=rows, what=f"sweep N={N} d={d} causal={causal}")


def test_long_context_causal():
    B, H, N, d = 1, 16, 32768, 128
    q, k, v = synth.attention_inputs(B, H, N, d, "bf16", seed=0)
    rows = synth.sample_rows(N, 64, seed=0, salt=5)
    m = parity.check_case(q, k, v, True, rows=rows, what="long context")
    assert m["finite"]
