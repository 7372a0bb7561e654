"""The reducing tensor-memory load (tcgen05.ld.red, sm_103a) that gives the
attention softmax its row maximum, in its 32-column form (16-bit kernels) and
its 128-column form (E4M3 kernel): through the library's test hook, which
runs the kernel's own load helpers, every row's values come back unchanged
and its extreme equals the maximum (or, for a negative scale, the minimum) of
all of them, with infinities, signed zeros and one-sided rows included."""
import pytest
import torch

import exact_attention_forward_05_gb300 as attn

pytestmark = pytest.mark.gpu


def _rows(cols):
    g = torch.Generator().manual_seed(cols)
    x = torch.randn(128, cols, generator=g) * 10
    x[1, 5] = float("-inf")             # one masked-looking entry
    x[2, :] = float("-inf")             # a row with no finite value
    x[3, :] = -5.0
    x[3, 7] = -1.0                      # all negative, one larger
    x[4, :] = 0.0
    x[4, 9] = -0.0                      # zeros of both signs
    x[5, 31] = 1e30                     # extreme in column 31
    x[6, 0] = float("inf")              # extreme in the first column
    x[7, :] = torch.arange(cols, dtype=torch.float32) - 200
    x[8, :] = 3.0                       # constant row
    x[9, 16] = -1e30
    x[10, cols - 1] = 1e20              # extreme in the last column of the widest load
    x[11, cols // 2] = 1e21
    return x


@pytest.mark.parametrize("cols", [32, 128])
@pytest.mark.parametrize("use_min", [False, True])
def test_reducing_load_gives_row_extreme(use_min, cols):
    x = _rows(cols)
    vals, ext = attn.debug_tmem_ld_red(x.cuda(), use_min=use_min)
    torch.cuda.synchronize()
    assert torch.equal(vals.cpu(), x)
    ref = x.min(dim=1).values if use_min else x.max(dim=1).values
    assert torch.equal(ext.cpu(), ref)
    assert attn.device_status() == attn.ATTN_OK


def test_reducing_load_rejects_bad_arguments():
    with pytest.raises(ValueError):
        attn.debug_tmem_ld_red(torch.zeros(128, 64, device="cuda"))
