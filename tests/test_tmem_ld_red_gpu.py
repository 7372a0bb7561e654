"""The reducing tensor-memory load (tcgen05.ld.red, sm_103a) that gives the
attention softmax its row maximum: through the library's test hook, which
runs the kernel's own load helper, every row's 32 values come back unchanged
and its extreme equals the maximum (or, for a negative scale, the minimum) of
those values, with infinities, signed zeros and one-sided rows included."""
import pytest
import torch

import exact_attention_forward_05_gb300 as attn

pytestmark = pytest.mark.gpu


def _rows():
    g = torch.Generator().manual_seed(0)
    x = torch.randn(128, 32, generator=g) * 10
    x[1, 5] = float("-inf")             # one masked-looking entry
    x[2, :] = float("-inf")             # a row with no finite value
    x[3, :] = -5.0
    x[3, 7] = -1.0                      # all negative, one larger
    x[4, :] = 0.0
    x[4, 9] = -0.0                      # zeros of both signs
    x[5, 31] = 1e30                     # extreme in the last column
    x[6, 0] = float("inf")              # extreme in the first column
    x[7, :] = torch.arange(32, dtype=torch.float32) - 40
    x[8, :] = 3.0                       # constant row
    x[9, 16] = -1e30
    return x


@pytest.mark.parametrize("use_min", [False, True])
def test_reducing_load_gives_row_extreme(use_min):
    x = _rows()
    vals, ext = attn.debug_tmem_ld_red(x.cuda(), use_min=use_min)
    torch.cuda.synchronize()
    assert torch.equal(vals.cpu(), x)
    ref = x.min(dim=1).values if use_min else x.max(dim=1).values
    assert torch.equal(ext.cpu(), ref)
    assert attn.device_status() == attn.ATTN_OK


def test_reducing_load_rejects_bad_arguments():
    with pytest.raises(ValueError):
        attn.debug_tmem_ld_red(torch.zeros(128, 16, device="cuda"))
