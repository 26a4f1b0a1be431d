"""The comparison helpers themselves (CPU): the bf16 rounding allowance is zero
below magnitude 8 and exactly the rounding beyond 1/64 above it, and fp32
results get none."""
import numpy as np
import pytest
import torch

from tests.parity_util import TOL_BF16, assert_close, bf16_excess_rounding, errors


def test_excess_rounding_is_zero_below_eight():
    v = np.array([0.0, 1e-3, 1.0, 3.99, 4.0, 7.999])
    assert np.all(bf16_excess_rounding(v) == 0.0)
    assert bf16_excess_rounding(np.array(8.0)) == 2.0 ** -5 - 2.0 ** -6
    assert bf16_excess_rounding(np.array(-12.5)) == 2.0 ** -5 - 2.0 ** -6
    assert bf16_excess_rounding(np.array(16.0)) == 2.0 ** -4 - 2.0 ** -6


def test_allowance_only_for_bf16_results():
    ref = np.array([8.09, 1.0])
    x = torch.tensor([8.0625, 1.0], dtype=torch.bfloat16)   # 8.0625: the nearest bf16
    assert errors(x, ref)[0] < 2e-2
    x32 = x.float()
    assert errors(x32, ref)[0] > 2e-2                          # fp32 results: no allowance
    bad = torch.tensor([8.0625, 1.03125], dtype=torch.bfloat16)  # 0.031 off below 8
    with pytest.raises(AssertionError):
        assert_close(bad, ref, TOL_BF16, "below eight")
