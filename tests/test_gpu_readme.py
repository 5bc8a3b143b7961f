"""The README's Python example runs as written on the GPU, and its output
matches the float64 oracle on the same pools."""
import os
import re

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_readme_example_runs_and_matches_oracle():
    import oracle
    from parity_util import TOL, host_bits, max_error
    text = open(os.path.join(ROOT, "README.md")).read()
    code = re.search(r"```python\n(.*?)```", text, re.S).group(1)
    env = {}
    exec(compile(code, "README.md example", "exec"), env)
    # the oracle on the pools as the example left them
    kp, vp = host_bits(env["k_cache"]), host_bits(env["v_cache"])
    ref = oracle.paged_decode(host_bits(env["q"]), "bf16", kp, vp, "bf16", env["tables"], env["lens"],
                              env["D"] ** -0.5)
    got = oracle.dequantize(host_bits(env["out"]), "bf16")
    assert max_error(got, ref, "bf16", TOL["bf16"]) <= TOL["bf16"]
    # the appended rows are the inputs, bit for bit
    for s in range(2):
        blk, off = divmod(int(env["slots"][s]), 16)
        assert np.array_equal(kp[blk, :, off], host_bits(env["k_new"])[s])
        assert np.array_equal(vp[blk, :, off], host_bits(env["v_new"])[s])
