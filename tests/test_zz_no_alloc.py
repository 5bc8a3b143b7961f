"""The allocation-free decode entry point (a scratch array inside the
library instead of a caller workspace), for callers that cannot allocate
device memory.  Its output is checked against the float64 oracle and, bit
for bit, against the regular entry point with a torch-allocated workspace
(same kernels, same partitions); before the checked calls, a larger split-K
call on other values fills the shared array with leftovers, so a partial
that was read without being written would show.  Collected last on purpose
(``zz``): it must pass both alone in a fresh process and after every other
test has run."""
import numpy as np
import pytest
import torch

from parity_util import TOL, check_step, host_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pk():
    from paged_kv_cache_10_gb300 import build, pagedkv
    build.build()
    pagedkv.lib()
    return pagedkv


def _noalloc(pk, st, P):
    wl = st.wl
    out = torch.full_like(st.out, 0xFFFF)
    pk.paged_attention_decode_noalloc(st.q, st.k_cache, st.v_cache, st.desc, st.d_tables, st.d_lens,
                                      st.max_seq_len, wl.scale, out, partition_tokens=P, q_dtype=wl.q_dtype)
    torch.cuda.synchronize()
    return out


def _fill_scratch_with_leftovers(pk):
    """A split-K call with more rows x heads x partitions than the checked
    ones, on other values: it writes partials over the whole region the
    checked calls use."""
    from paged_kv_cache_10_gb300 import workloads
    from paged_kv_cache_10_gb300.step import DecodeStep
    wl = workloads.custom("noalloc_fill", 77, [4096] * 8, 64, 8, 128, kv_dtype="bf16", partition_tokens=64)
    st = DecodeStep(wl, device="cuda")
    st.run()
    torch.cuda.synchronize()
    _noalloc(pk, st, 64)
    return pk.decode_workspace_bytes(wl.S, wl.Hq, wl.D, st.max_seq_len, 64)  # 17 MiB of the 32


@pytest.mark.parametrize("kv,Hq,Hkv,P", [("bf16", 32, 8, 64), ("bf16", 16, 16, 48), ("e4m3", 64, 8, 512),
                                         ("e4m3", 64, 8, 0)])
def test_noalloc_matches_oracle_and_workspace_decode_on_two_calls(pk, kv, Hq, Hkv, P):
    from paged_kv_cache_10_gb300 import workloads
    from paged_kv_cache_10_gb300.step import DecodeStep

    # P = 0: the library picks the partition size; the long fp8 rows make it split
    lens = [700, 1300, 64, 2049, 1] if kv != "e4m3" else [32768, 20000, 3000]
    wl = workloads.custom("noalloc", 31, lens, Hq, Hkv, 128, kv_dtype=kv, partition_tokens=P)
    st = DecodeStep(wl, device="cuda", plan=False)
    used_P = st.effective_partition()
    need = pk.decode_workspace_bytes(wl.S, wl.Hq, wl.D, st.max_seq_len, used_P)
    assert need > 0  # really split-K
    st.run()  # regular entry point, torch workspace (and the step's appends)
    torch.cuda.synchronize()
    assert pk.get_device_error() == 0
    err, mx = check_step(st)  # the workspace path itself against the oracle
    assert err <= TOL[kv], (err, mx)
    ref = host_bits(st.out).copy()
    assert _fill_scratch_with_leftovers(pk) > need
    for _ in range(2):
        out = _noalloc(pk, st, P)
        assert pk.get_device_error() == 0
        assert np.array_equal(host_bits(out), ref)  # bit for bit the workspace path's output
        st.out.copy_(out)
        err, mx = check_step(st)  # and against the oracle
        assert err <= TOL[kv], (err, mx)


def test_noalloc_rejects_scratch_beyond_its_maximum(pk):
    from paged_kv_cache_10_gb300 import workloads
    from paged_kv_cache_10_gb300.step import DecodeStep
    wl = workloads.custom("noalloc_small", 32, [40], 8, 2, 128, kv_dtype="bf16")
    st = DecodeStep(wl, device="cuda")
    # 4096 sequences x 64 heads x 256 partitions of 16 tokens need far more than 32 MiB:
    # the size check happens on the host before anything is read or launched
    big_S, big_L = 4096, 4096
    assert pk.decode_workspace_bytes(big_S, 64, 128, big_L, 16) > (32 << 20)
    q = torch.empty((big_S, 64, 128), dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(q)
    tables = torch.zeros((big_S, 256), dtype=torch.int32, device="cuda")
    lens = torch.zeros(big_S, dtype=torch.int32, device="cuda")
    desc = pk.CacheDesc(num_blocks=wl.NB, num_kv_heads=8, head_size=128, kv_dtype="bf16")
    with pytest.raises(pk.PagedKVError) as e:
        pk.paged_attention_decode_noalloc(q, st.k_cache, st.v_cache, desc, tables, lens, big_L, 0.1, out,
                                          partition_tokens=16)
    assert e.value.status == pk.ERR_WORKSPACE
