"""The per-element parity bound (host logic of the GPU parity tests)."""

import numpy as np

from gpu_util import TOL, bf16_ulp, elementwise_bound


def test_bf16_ulp():
    assert bf16_ulp(np.array([1.0]))[0] == 2 ** -7
    assert bf16_ulp(np.array([3.9]))[0] == 2 ** -6
    assert bf16_ulp(np.array([-4.0]))[0] == 2 ** -5


def test_bound_is_the_stated_tolerance_below_4():
    x = np.array([0.0, 0.3, -1.5, 2.0, 3.99])
    assert np.all(elementwise_bound(x, TOL["bf16"].max_o) == 1e-2)
    assert np.all(elementwise_bound(x, TOL["fp8"].max_o) == 4e-2)


def test_bound_is_one_step_where_half_a_step_exceeds_it():
    x = np.array([4.0, -5.5, 7.9])
    assert np.all(elementwise_bound(x, TOL["bf16"].max_o) == 2 ** -5)
    # FP8's 4e-2 is above half a BF16 step up to |O| < 8: unchanged
    assert np.all(elementwise_bound(x, TOL["fp8"].max_o) == 4e-2)
