"""The parity bound of the GPU tests, checked on the CPU.

The outputs are bf16.  The bound is the stated atol wherever half the bf16
spacing at the reference is below atol (|ref| < 4 for atol 1e-2); above that,
half a spacing plus a small allowance for the error before the final
rounding.  These checks pin it: it equals atol below the threshold, a
correctly rounded bf16 value (torch's conversion) always meets it, and a
value one whole spacing off does not where the bound is the half spacing.
"""
import numpy as np
import torch

from tests.gpu_util import ROUND_EPS, allowed_err, bf16_ulp, excess


def test_bound_is_atol_below_the_threshold():
    x = np.array([0.0, 1e-3, -0.7, 1.999, 2.0, -3.0, 3.9999, -3.9999])
    assert np.all(allowed_err(x, 1e-2) == 1e-2)
    assert np.all(allowed_err(x * 4, 5e-2) == 5e-2)       # |ref| < 16 for atol 5e-2


def test_bound_above_the_threshold_is_half_a_spacing():
    assert bf16_ulp(np.array([4.0]))[0] == 2.0 ** -5
    assert bf16_ulp(np.array([3.99]))[0] == 2.0 ** -6
    assert allowed_err(np.array([4.0]), 1e-2)[0] == 2.0 ** -6 + ROUND_EPS
    assert allowed_err(np.array([-100.0]), 1e-2)[0] == 2.0 ** -2 + ROUND_EPS


def test_correctly_rounded_values_pass_and_a_whole_spacing_fails():
    rng = np.random.default_rng(0)
    ref = np.concatenate([rng.normal(0, 3, 20000), rng.uniform(-64, 64, 20000)])
    got = torch.from_numpy(ref).to(torch.float32).to(torch.bfloat16).double().numpy()
    assert excess(got, ref, 1e-2) <= 1.0
    big = ref[np.abs(ref) >= 4]
    off = big + np.sign(big) * bf16_ulp(big)                 # one whole spacing away
    assert np.all(np.abs(off - big) > allowed_err(big, 1e-2))
    small = ref[np.abs(ref) < 4]
    assert np.all(np.abs((small + 0.011) - small) > allowed_err(small, 1e-2))
