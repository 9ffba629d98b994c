"""The comparison rule the parity tests apply (no GPU): literal max-abs 1e-2
where bf16 can meet it; where its spacing cannot (|o| >= 4), half a bf16
step plus 2^-9 |o| of slack for the kernels' error before the final
rounding; rel-L2 2e-3 throughout."""
import numpy as np
import pytest
import torch

from helpers import bf16_step, compare


def test_step_sizes():
    assert bf16_step(np.array([1.0]))[0] == 2.0 ** -7
    assert bf16_step(np.array([3.99]))[0] == 2.0 ** -6
    assert bf16_step(np.array([-4.0]))[0] == 2.0 ** -5
    assert bf16_step(np.array([100.0]))[0] == 2.0 ** -1


def test_correct_rounding_passes_where_one_e_minus_two_cannot():
    # -4.04985 rounds to -4.0625 (1.27e-2 away): no bf16 value is within 1e-2
    ref = np.ones(2000)
    ref[0] = -4.04985
    out = torch.tensor(ref).to(torch.bfloat16)
    assert float(out[0]) == -4.0625
    compare(out, ref)
    out[0] = -4.09375  # two steps away is not a rounding of it
    with pytest.raises(AssertionError):
        compare(out, ref)


def test_one_step_off_above_four_fails():
    # exact 6.0001: correctly rounded 6.0; a result one step (1/32) away, 6.03125,
    # exceeds half a step (1/64) plus 2^-9 x 6 of slack
    ref = np.ones(2000)
    ref[0] = 6.0001
    out = torch.tensor(ref).to(torch.bfloat16)
    compare(out, ref)
    out[0] = 6.03125
    with pytest.raises(AssertionError):
        compare(out, ref)


def test_literal_bound_below_four():
    ref = np.full(1000, 1.0)
    ref[0] = 3.0
    out = torch.tensor(ref).to(torch.bfloat16)
    out[0] = 3.015625  # one step (1/64) above 3: 1.56e-2 > 1e-2
    with pytest.raises(AssertionError):
        compare(out, ref)


def test_rel_l2_still_applies():
    ref = np.ones(100)
    with pytest.raises(AssertionError):
        compare(torch.full((100,), 1.0078125, dtype=torch.bfloat16), ref)  # rel 7.8e-3
