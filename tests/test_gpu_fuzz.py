"""Seeded random decode and prefill batches against the float64 oracle:
batch size, length mix (empty rows, single tokens, block and partition
boundaries, long tails), head ratio, head size, pool and query types,
partition size, CTA order (grid or host plan) and the fused or separate
append, all drawn per case.  PKV_FUZZ_CASES sets the number of cases per
test (default 12)."""
import os

import numpy as np
import pytest
import torch

from parity_util import TOL, check_step, host_bits, max_error

pytestmark = pytest.mark.gpu
N = int(os.environ.get("PKV_FUZZ_CASES", "12"))


@pytest.fixture(scope="module")
def lib():
    from paged_kv_cache_10_gb300 import build, pagedkv
    build.build()
    pagedkv.lib()
    return pagedkv


def _lens(rng, S, cap):
    kind = rng.integers(0, 4)
    if kind == 0:  # around block and partition boundaries
        base = rng.choice([1, 15, 16, 17, 255, 256, 257, 511, 512, 513], S)
        return np.minimum(base + rng.integers(-1, 2, S), cap).clip(0)
    if kind == 1:  # many short rows, a few long ones
        L = rng.integers(0, 40, S)
        L[rng.integers(0, S, max(1, S // 8))] = rng.integers(cap // 2, cap + 1, max(1, S // 8))
        return L
    if kind == 2:
        return rng.integers(0, cap + 1, S)
    return np.full(S, rng.integers(1, cap + 1))


@pytest.mark.parametrize("case", range(N))
def test_fuzz_decode(lib, case):
    from paged_kv_cache_10_gb300 import workloads
    from paged_kv_cache_10_gb300.step import DecodeStep
    rng = np.random.default_rng(7000 + case)
    D = int(rng.choice([64, 128]))
    kv = str(rng.choice(["bf16", "f16", "e4m3"]))
    qd = str(rng.choice(["bf16", "f16"])) if kv == "e4m3" else kv
    G = int(rng.choice([1, 2, 4, 8]))
    Hkv = int(rng.choice([1, 2, 3]))
    S = int(rng.integers(1, 48))
    lens = _lens(rng, S, int(rng.choice([64, 700, 2100])))
    P = int(rng.choice([0, 16, 64, 512]))
    wl = workloads.custom(f"fuzz{case}", 7100 + case, lens.tolist(), Hkv * G, Hkv, D, kv_dtype=kv, q_dtype=qd,
                          partition_tokens=P)
    fused = bool(rng.integers(0, 2))
    plan = bool(rng.integers(0, 2)) and fused
    st = DecodeStep(wl, device="cuda", fused=fused, plan=plan)
    st.run()
    torch.cuda.synchronize()
    assert lib.get_device_error() == 0
    err, mx = check_step(st)
    assert err <= TOL[kv], (err, mx, dict(D=D, kv=kv, qd=qd, G=G, Hkv=Hkv, S=S, P=P, fused=fused, plan=plan))


@pytest.mark.parametrize("case", range(N))
def test_fuzz_prefill(lib, case):
    import oracle
    from paged_kv_cache_10_gb300 import workloads
    from paged_kv_cache_10_gb300.step import PrefillStep
    rng = np.random.default_rng(8000 + case)
    D = int(rng.choice([64, 128]))
    dtype = str(rng.choice(["bf16", "f16"]))
    G = int(rng.choice([1, 2, 4, 8]))
    Hkv = int(rng.choice([1, 2]))
    S = int(rng.integers(1, 7))
    ctx = rng.integers(0, 600, S) * rng.integers(0, 2, S)
    qlens = rng.integers(0, 300, S)
    qlens[rng.integers(0, S)] = max(1, int(qlens.max()))
    wl = workloads.prefill(f"pfuzz{case}", 8100 + case, ctx.tolist(), qlens.tolist(), Hkv * G, Hkv, D=D, dtype=dtype)
    st = PrefillStep(wl, device="cuda", plan=bool(rng.integers(0, 2)))
    st.run()
    torch.cuda.synchronize()
    assert lib.get_device_error() == 0
    kp, vp = host_bits(st.k_cache), host_bits(st.v_cache)
    ref = oracle.paged_prefill(wl.q, wl.dtype, st.query_start, kp, vp, wl.dtype, st.tables, st.seq_lens, wl.scale)
    got = oracle.dequantize(host_bits(st.out), wl.dtype)
    assert max_error(got, ref, dtype, TOL[dtype]) <= TOL[dtype], dict(D=D, dtype=dtype, G=G, Hkv=Hkv, S=S)
