"""The parity tolerance's allowance for outputs whose 16-bit format cannot
meet the absolute bound (CPU): one unit in the last place of bf16 / f16 at
the oracle value, checked against numpy's own spacing of the formats."""
import numpy as np
import torch

from parity_util import TOL, max_error, output_ulp


def test_output_ulp_is_the_format_spacing():
    x = np.array([0.3, 1.0, 1.7, 2.0, 3.99, 4.4, 7.0, 100.0])
    # f16: numpy's own spacing
    assert np.array_equal(output_ulp(x, "f16"), np.spacing(x.astype(np.float16)).astype(np.float64))
    # bf16: the gap from torch's bf16 value to the next code up (all x positive, same binade)
    b = torch.tensor(x, dtype=torch.bfloat16)
    nxt = (b.view(torch.int16) + 1).view(torch.bfloat16)
    gap = (nxt.double() - b.double()).numpy()
    assert np.array_equal(output_ulp(x, "bf16"), gap)


def test_max_error_allows_only_the_format_spacing():
    ref = np.array([0.25, 4.4])
    # small outputs: the plain absolute bound
    assert max_error(np.array([0.25 + 0.009, 4.4]), ref, "bf16", TOL["bf16"]) <= TOL["bf16"]
    assert max_error(np.array([0.25 + 0.011, 4.4]), ref, "bf16", TOL["bf16"]) > TOL["bf16"]
    # at 4.4 bf16's spacing is 2^-5: one unit passes, two do not
    assert max_error(np.array([0.25, 4.4 + 0.03125]), ref, "bf16", TOL["bf16"]) <= TOL["bf16"] + 1e-15
    assert max_error(np.array([0.25, 4.4 + 0.0625]), ref, "bf16", TOL["bf16"]) > TOL["bf16"]
    # f16 keeps 2e-3 up to |out| < 4
    assert max_error(np.array([3.0 + 0.0025]), np.array([3.0]), "f16", TOL["f16"]) > TOL["f16"]
