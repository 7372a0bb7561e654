"""Full-size workloads on the GPU, checked against the float64 oracle.

* sequence-length sweep: N in {512, ..., 16384} x d in {64, 128, 256} with
  B = 16384 / N and H = 2048 / d, bf16, causal and non-causal (the launch
  configuration the benchmark times for N = 8192, d = 128).  For N <= 2048
  every output row of every head is compared with the oracle.  Above that,
  one whole head (every row) is compared, plus 64 seeded query rows of every
  other head.
* long context: B = 1, H = 16, N = 32768, d = 128, causal, 64 random query
  rows per head plus every row of the last head.
* longest sequence: B = 1, H = 2, N = 131072, d = 128 (1024 key blocks per
  row), causal and not, the first and last rows and 62 seeded ones per head.
Before any slicing, the whole O and lse of the launch are checked to be
finite, so rows the oracle does not recompute are still covered for NaN or
infinity.
"""
import numpy as np
import pytest
import torch

import exact_attention_forward_05_gb300 as attn
import oracle
import synth
from tests import parity

pytestmark = pytest.mark.gpu

SWEEP_N = [512, 1024, 2048, 4096, 8192, 16384]
SWEEP_D = [64, 128, 256]
FULL_ROWS_UP_TO = 2048


def _launch(q, k, v, causal, scale):
    o, lse = attn.attn_fwd(q.cuda(), k.cuda(), v.cuda(), causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert bool(torch.isfinite(o).all()), "non-finite O"
    assert bool(torch.isfinite(lse).all()), "non-finite lse"
    st = attn.device_status()
    assert st == attn.ATTN_OK, attn.status_string(st)
    return o.cpu(), lse.cpu()


def _check_heads(q, k, v, o, lse, causal, scale, whole_head, rows, what):
    """Every row of head `whole_head` (flattened b * H + h index), and `rows`
    of every head."""
    B, H, N, d = q.shape
    flat = lambda t: t.reshape(1, B * H, *t.shape[2:])
    qf, kf, vf, of, lf = (flat(t) for t in (q, k, v, o, lse))
    h = slice(whole_head, whole_head + 1)
    o_ref, lse_ref = oracle.attention(qf[:, h], kf[:, h], vf[:, h], causal=causal, scale=scale)
    parity.assert_close_elementwise(of[:, h], lf[:, h], o_ref, lse_ref, qf[:, h], kf[:, h], vf[:, h], causal,
                                    scale, what=f"{what} head {whole_head}")
    o_ref, lse_ref = oracle.attention(qf, kf, vf, causal=causal, scale=scale, rows=rows)
    idx = torch.as_tensor(rows)
    parity.assert_close_elementwise(of[:, :, idx], lf[:, :, idx], o_ref, lse_ref, qf, kf, vf, causal, scale,
                                    rows=rows, what=f"{what} sampled rows")


@pytest.mark.parametrize("d", SWEEP_D)
@pytest.mark.parametrize("N", SWEEP_N)
def test_sequence_sweep(N, d):
    B, H = 16384 // N, 2048 // d
    q, k, v = synth.attention_inputs(B, H, N, d, "bf16", seed=0)
    scale = d ** -0.5
    for causal in (False, True):
        what = f"sweep N={N} d={d} causal={causal}"
        o, lse = _launch(q, k, v, causal, scale)
        if N <= FULL_ROWS_UP_TO:
            o_ref, lse_ref = oracle.attention(q, k, v, causal=causal, scale=scale)
            parity.assert_close_elementwise(o, lse, o_ref, lse_ref, q, k, v, causal, scale, what=what)
        else:
            rows = synth.sample_rows(N, 64, seed=0, salt=N + d)
            whole = (N + d + int(causal)) % (B * H)
            _check_heads(q, k, v, o, lse, causal, scale, whole, rows, what)


def test_long_context_causal():
    B, H, N, d = 1, 16, 32768, 128
    q, k, v = synth.attention_inputs(B, H, N, d, "bf16", seed=0)
    rows = synth.sample_rows(N, 64, seed=0, salt=5)
    o, lse = _launch(q, k, v, True, d ** -0.5)
    _check_heads(q, k, v, o, lse, True, d ** -0.5, H - 1, rows, "long context")


@pytest.mark.parametrize("causal", [False, True])
def test_longest_sequence(causal):
    B, H, N, d = 1, 2, 131072, 128
    q, k, v = synth.attention_inputs(B, H, N, d, "bf16", seed=3)
    scale = d ** -0.5
    rows = np.unique(np.concatenate([[0, N - 1], synth.sample_rows(N, 62, seed=3, salt=11)]))
    o, lse = _launch(q, k, v, causal, scale)
    o_ref, lse_ref = oracle.attention(q, k, v, causal=causal, scale=scale, rows=rows)
    idx = torch.as_tensor(rows)
    parity.assert_close_elementwise(o[:, :, idx], lse[:, :, idx], o_ref, lse_ref, q, k, v, causal, scale,
                                    rows=rows, what=f"N={N} causal={causal}")
