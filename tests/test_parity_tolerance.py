"""The parity tolerance's allowance for outputs whose 16-bit format cannot
meet the absolute bound (CPU).  Only where half a unit in the last place of
bf16 / f16 at the oracle value exceeds the bound (bf16 |out| >= 4 at 1e-2,
f16 |out| >= 8 at 2e-3) does the bound become that half unit plus the
float32 term; the unit itself is checked against numpy's and torch's own
spacing of the formats."""
import numpy as np
import torch

from parity_util import FP32_TERM, TOL, max_error, output_ulp, relaxed_bound


def test_output_ulp_is_the_format_spacing():
    x = np.array([0.3, 1.0, 1.7, 2.0, 3.99, 4.4, 7.0, 100.0])
    # f16: numpy's own spacing
    assert np.array_equal(output_ulp(x, "f16"), np.spacing(x.astype(np.float16)).astype(np.float64))
    # bf16: the gap from torch's bf16 value to the next code up (all x positive, same binade)
    b = torch.tensor(x, dtype=torch.bfloat16)
    nxt = (b.view(torch.int16) + 1).view(torch.bfloat16)
    gap = (nxt.double() - b.double()).numpy()
    assert np.array_equal(output_ulp(x, "bf16"), gap)


def test_plain_bound_wherever_the_format_can_meet_it():
    tol = TOL["bf16"]
    # small outputs
    assert max_error(np.array([0.25 + 0.009]), np.array([0.25]), "bf16", tol) <= tol
    assert max_error(np.array([0.25 + 0.011]), np.array([0.25]), "bf16", tol) > tol
    # bf16 in [2, 4): half an ulp is 2^-7 < 1e-2, so the plain bound holds
    assert max_error(np.array([3.0 + 0.0095]), np.array([3.0]), "bf16", tol) <= tol
    assert max_error(np.array([3.0 + 0.0105]), np.array([3.0]), "bf16", tol) > tol
    assert np.all(relaxed_bound(np.array([2.0, 3.99]), "bf16", tol, 8.0) == tol)
    # f16 keeps 2e-3 up to |out| < 8 (half an ulp in [4, 8) is 2^-9 < 2e-3)
    assert max_error(np.array([3.0 + 0.0025]), np.array([3.0]), "f16", TOL["f16"]) > TOL["f16"]
    assert max_error(np.array([5.0 + 0.0021]), np.array([5.0]), "f16", TOL["f16"]) > TOL["f16"]
    assert max_error(np.array([5.0 + 0.0019]), np.array([5.0]), "f16", TOL["f16"]) <= TOL["f16"]


def test_half_ulp_plus_float32_term_where_it_cannot():
    tol = TOL["bf16"]
    ref = np.array([0.25, 4.4])
    # at 4.4 bf16's spacing is 2^-5: half a unit (the correctly rounded
    # result's worst case) passes, a whole unit does not
    assert max_error(np.array([0.25, 4.4 + 0.015625]), ref, "bf16", tol) <= tol
    assert max_error(np.array([0.25, 4.4 - 0.015625]), ref, "bf16", tol) <= tol
    assert max_error(np.array([0.25, 4.4 + 0.03125]), ref, "bf16", tol) > tol
    # the float32 term: twice 2^-14 of the largest |V|
    vmax = 4.5
    b = relaxed_bound(np.array([4.4]), "bf16", tol, vmax)[0]
    assert b == 2.0 ** -6 + 2 * FP32_TERM * vmax
    assert max_error(np.array([4.4 + b * 0.999]), np.array([4.4]), "bf16", tol, vmax) <= tol
    assert max_error(np.array([4.4 + b * 1.001]), np.array([4.4]), "bf16", tol, vmax) > tol
    # f16 at 9.0: half an ulp is 2^-8 > 2e-3
    assert max_error(np.array([9.0 + 2.0 ** -8]), np.array([9.0]), "f16", TOL["f16"]) <= TOL["f16"]
    assert max_error(np.array([9.0 + 2.0 ** -7]), np.array([9.0]), "f16", TOL["f16"]) > TOL["f16"]


def test_correctly_rounded_outputs_always_pass():
    """Whatever the value, rounding the exact result to the output format
    passes the bound (this is what the allowance exists for), for both
    formats and across the binades around the switch."""
    rng = np.random.default_rng(3)
    x = np.concatenate([rng.uniform(-16, 16, 20000), rng.uniform(-0.5, 0.5, 2000)])
    for dt, tdt in (("bf16", torch.bfloat16), ("f16", torch.float16)):
        r = torch.tensor(x, dtype=torch.float64).to(tdt).double().numpy()
        assert max_error(r, x, dt, TOL[dt]) <= TOL[dt]
