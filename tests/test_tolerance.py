"""The tolerance helper itself: bf16 spacing and the two error measures."""

import numpy as np
import torch

from tolerance import assert_close, errors, half_ulp_bf16


def test_half_ulp_values():
    assert half_ulp_bf16(1.0) == 2.0 ** -8
    assert half_ulp_bf16(1.99) == 2.0 ** -8
    assert half_ulp_bf16(2.0) == 2.0 ** -7
    assert half_ulp_bf16(-0.75) == 2.0 ** -9
    assert half_ulp_bf16(0.0) == 0.0


def test_correctly_rounded_output_has_no_excess():
    rng = np.random.default_rng(0)
    x = rng.standard_normal(200000) * np.exp(rng.standard_normal(200000))
    xr = torch.from_numpy(x.astype(np.float32)).bfloat16().double().numpy()
    rel, excess, rms = errors(xr, x, bf16_output=True)
    assert excess <= 1e-7 * rms and rel < 3e-3
    # the plain max-abs measure is not met by bf16 rounding of a heavy-tailed tensor
    _, plain, _ = errors(xr, x, bf16_output=False)
    assert plain > 2e-2 * rms


def test_assert_close_rejects_real_errors():
    rng = np.random.default_rng(1)
    x = rng.standard_normal(10000)
    y = x.copy()
    y[17] += 0.05 * np.sqrt(np.mean(x ** 2))   # one element off by 5% of RMS
    try:
        assert_close(y, x, "planted", bf16_output=True)
    except AssertionError:
        pass
    else:
        raise AssertionError("a 5%-of-RMS error was accepted")
    assert_close(x + 1e-4, x, "tiny shift")
