"""Shared-prefix (cascade) decode on the GPU: the same function as plain
decode, checked against the float64 oracle (which knows nothing about
groups) on fork trees, the full-size prefix-sharing workload, several group
sizes and both attention kernels underneath."""
import numpy as np
import pytest
import torch

from parity_util import TOL, check_step, host_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    from paged_kv_cache_10_gb300 import build, pagedkv
    build.build()
    pagedkv.lib()
    return pagedkv


def run(wl, **kw):
    from paged_kv_cache_10_gb300.step import DecodeStep
    st = DecodeStep(wl, device="cuda", **kw)
    st.run()
    torch.cuda.synchronize()
    return st


@pytest.mark.parametrize("kv", ["bf16", "f16"])
@pytest.mark.parametrize("G", [1, 2, 4, 8])
@pytest.mark.parametrize("min_blocks", [1, 16])
def test_cascade_fork_trees_match_oracle(lib, kv, G, min_blocks):
    from paged_kv_cache_10_gb300 import workloads
    Hkv = 2
    # prefixes of 2, 20 and 33 blocks (one and three prefix partitions), a lone fork, singles
    wl = workloads.fork_groups("forks", 60 + G, [(32, 3), (320, 5), (528, 4), (96, 1)], 3, Hkv * G, Hkv,
                               kv_dtype=kv)
    st = run(wl, cascade=True, cascade_min_blocks=min_blocks)
    assert lib.get_device_error() == 0
    g = st.groups
    assert g.num_groups >= (3 if min_blocks == 1 else 2)
    err, mx = check_step(st)
    assert err <= TOL[kv], (err, mx)


def test_cascade_prefix_share_full_size(lib):
    from paged_kv_cache_10_gb300 import workloads
    wl = workloads.prefix_share()
    st = run(wl, cascade=True)
    assert lib.get_device_error() == 0
    assert st.groups.num_groups == 1 and st.groups.max_blocks == 128 and st.groups.max_members == 128
    err, mx = check_step(st)
    assert err <= TOL["bf16"], (err, mx)


def test_cascade_equals_plain_decode(lib):
    from paged_kv_cache_10_gb300 import workloads
    import oracle
    wl = workloads.fork_groups("eq", 71, [(256, 6), (64, 3)], 2, 32, 8)
    a = run(wl, cascade=True, cascade_min_blocks=1)
    b = run(wl)
    fa = oracle.dequantize(host_bits(a.out), "bf16")
    fb = oracle.dequantize(host_bits(b.out), "bf16")
    assert np.max(np.abs(fa - fb)) <= 4e-3


def test_cascade_without_groups_is_plain_decode(lib):
    from paged_kv_cache_10_gb300 import workloads
    wl = workloads.custom("nogroups", 72, [1, 17, 300, 0], 16, 2, 128, kv_dtype="bf16")
    st = run(wl, cascade=True)
    assert st.groups.num_groups == 0
    err, _ = check_step(st)
    assert err <= TOL["bf16"]
    assert np.all(host_bits(st.out)[3] == 0)


def test_cascade_rejects_fp8(lib):
    from paged_kv_cache_10_gb300 import workloads
    wl = workloads.custom("fp8c", 73, [40, 50], 16, 2, 128, kv_dtype="e4m3")
    with pytest.raises(lib.PagedKVError) as e:
        run(wl, cascade=True)
    assert e.value.status == lib.ERR_UNSUPPORTED


def test_cascade_graph_replay_and_stream_order(lib):
    """The prefix pass runs on the library's own stream, forked from the
    caller's and joined before the merge: captured into a CUDA graph the step
    replays to the same bits as eager, and on a non-default caller stream the
    eager result is the same too."""
    from paged_kv_cache_10_gb300 import workloads
    from paged_kv_cache_10_gb300.step import DecodeStep
    wl = workloads.fork_groups("cgraph", 74, [(320, 5), (96, 3)], 2, 32, 8)
    st = DecodeStep(wl, device="cuda", cascade=True, cascade_min_blocks=1)
    assert st.groups.num_groups >= 1
    g = st.capture()  # runs one eager step first, then captures
    eager = host_bits(st.out).copy()
    err, mx = check_step(st)
    assert err <= TOL["bf16"], (err, mx)
    for _ in range(2):
        st.out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(host_bits(st.out), eager)
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        st.out.zero_()
        st.decode(stream=side)
    torch.cuda.synchronize()
    assert lib.get_device_error() == 0
    assert np.array_equal(host_bits(st.out), eager)
