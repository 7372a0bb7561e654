"""The polynomial 2^x of the FP8 softmax weights (exp2_poly2), evaluated on
the GPU through a test hook, against float64 2**x and against CUDA's exp2f
over a sweep of the arguments the weights take (-125 <= x <= 8, plus the
clamp below): relative error below the 7.6e-5 bound that the CPU test of the
same coefficients derives."""
import numpy as np
import pytest
import torch

import exact_attention_forward_05_gb300 as attn

pytestmark = pytest.mark.gpu
BOUND = 7.6e-5


def test_device_polynomial_against_float64_and_exp2f():
    x = np.concatenate([np.linspace(-125.0, 8.0, 2_000_001), np.arange(-125, 9) + 0.5,
                        np.arange(-125, 9), [-125.0, -126.0, -200.0, -3e38]]).astype(np.float32)
    xd = torch.from_numpy(x).cuda()
    yp, yr = attn.debug_exp2_poly(xd)
    torch.cuda.synchronize()
    yp, yr = yp.cpu().double().numpy(), yr.cpu().double().numpy()
    ref = 2.0 ** np.maximum(x.astype(np.float64), -125.0)
    assert np.all(np.isfinite(yp)) and np.all(yp > 0)
    assert np.max(np.abs(yp / ref - 1)) < BOUND
    ok = x >= -125
    assert np.max(np.abs(yp[ok] / yr[ok] - 1)) < BOUND + 2e-7   # exp2f is within an ulp or two
    assert attn.device_status() == attn.ATTN_OK
