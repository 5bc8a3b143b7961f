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


@pytest.mark.parametrize("qd", ["bf16", "f16"])
@pytest.mark.parametrize("G", [1, 2, 4, 8])
def test_cascade_fp8_fork_trees_match_oracle(lib, qd, G):
    """fp8 E4M3 pools: the prefix pass reads a 16-bit copy of every group's
    shared blocks (made by the call), the own tokens use the fp8 decode
    kernels; judged against the oracle on the dequantised codes."""
    from paged_kv_cache_10_gb300 import workloads
    Hkv = 2
    wl = workloads.fork_groups("forks_fp8", 160 + G, [(32, 3), (320, 5), (528, 4), (96, 1)], 3, Hkv * G, Hkv,
                               kv_dtype="e4m3", q_dtype=qd)
    assert wl.k_scale != wl.v_scale
    st = run(wl, cascade=True, cascade_min_blocks=1)
    assert lib.get_device_error() == 0
    assert st.groups.num_groups >= 3 and st.kernel_launches() == 5  # append, staging, prefix, decode, merge
    err, mx = check_step(st)
    assert err <= TOL["e4m3"], (err, mx)


@pytest.mark.parametrize("kv,qd", [("bf16", "bf16"), ("f16", "f16"), ("e4m3", "bf16")])
@pytest.mark.parametrize("G", [1, 4, 8])
def test_cascade_head_size_64_matches_oracle(lib, kv, qd, G):
    from paged_kv_cache_10_gb300 import workloads
    Hkv = 2
    wl = workloads.fork_groups("forks_d64", 260 + G, [(64, 4), (400, 6), (1040, 3)], 2, Hkv * G, Hkv, D=64,
                               kv_dtype=kv, q_dtype=qd)
    st = run(wl, cascade=True, cascade_min_blocks=1)
    assert lib.get_device_error() == 0
    assert st.groups.num_groups >= 3
    err, mx = check_step(st)
    assert err <= TOL[kv], (err, mx)


def test_cascade_fp8_prefix_share_full_size(lib):
    """prefix_share over an fp8 pool at full size: 128 rows, one group of a
    2048-token prefix read once per KV head through the staged copy; every
    row against the oracle and equal, within the bound, to plain decode."""
    import oracle
    from paged_kv_cache_10_gb300 import workloads
    wl = workloads.prefix_share(kv_dtype="e4m3")
    st = run(wl, cascade=True)
    assert lib.get_device_error() == 0
    assert st.groups.num_groups == 1 and st.groups.max_blocks == 128
    err, mx = check_step(st)
    assert err <= TOL["e4m3"], (err, mx)
    plain = run(wl)
    fa = oracle.dequantize(host_bits(st.out), "bf16")
    fb = oracle.dequantize(host_bits(plain.out), "bf16")
    assert np.max(np.abs(fa - fb)) <= TOL["e4m3"]


def test_cascade_fp8_workspace_must_hold_the_staging(lib):
    """The staged prefix copy follows the partials in the workspace; a
    workspace of the partials alone is refused before any launch."""
    from paged_kv_cache_10_gb300 import workloads
    from paged_kv_cache_10_gb300.step import DecodeStep
    wl = workloads.fork_groups("fp8_ws", 171, [(320, 4)], 1, 16, 2, kv_dtype="e4m3")
    st = DecodeStep(wl, device="cuda", cascade=True, cascade_min_blocks=1)
    g = st.groups
    part = lib.decode_cascade_workspace_bytes(wl.S, wl.Hq, wl.D, st.max_seq_len, st.partition_tokens, g.max_blocks)
    stage = lib.decode_cascade_staging_bytes("e4m3", wl.S, st.max_blocks, g.num_groups, g.max_blocks, wl.Hkv, wl.D)
    assert stage > 0 and lib.decode_cascade_staging_bytes("bf16", wl.S, st.max_blocks, g.num_groups, g.max_blocks,
                                                          wl.Hkv, wl.D) == 0
    short = torch.empty(part, dtype=torch.uint8, device="cuda")
    with pytest.raises(lib.PagedKVError) as e:
        lib.paged_attention_decode_cascade(st.q, st.k_cache, st.v_cache, st.desc, st.d_tables, st.d_lens,
                                           st.max_seq_len, wl.scale, st.out, st.d_seq_group, st.d_group_blocks,
                                           st.d_group_offsets, st.d_group_members, g.max_members, g.max_blocks,
                                           short, partition_tokens=st.partition_tokens, q_dtype="bf16")
    assert e.value.status == lib.ERR_WORKSPACE
    st.run()
    torch.cuda.synchronize()
    assert lib.get_device_error() == 0
    err, mx = check_step(st)
    assert err <= TOL["e4m3"], (err, mx)


def test_cascade_graph_replay_and_stream_order(lib):
    """The prefix pass, the own-token decode (its programmatic dependent)
    and the merge all run on the caller's stream: captured into a CUDA graph
    the step replays to the same bits as eager, and on a non-default caller
    stream the eager result is the same too."""
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


def test_cascade_merge_waits_for_the_prefix_pass(lib):
    """The merge must see the prefix pass's partials, which only the decode
    grid's join CTA orders before it.  The workspace is filled with NaN bits
    before every call (so a partial read too early is wrong, not a stale
    copy of the right one), on a batch whose prefix pass outlasts the
    own-token decode (32 rows over an 8192-token shared prefix: 64 prefix
    CTAs of 8 key tiles, one wave of short own-token CTAs).  Eager calls and
    CUDA-graph replays of fill + call give the oracle-checked bits every
    time."""
    from paged_kv_cache_10_gb300 import workloads
    from paged_kv_cache_10_gb300.step import DecodeStep
    wl = workloads.fork_groups("cjoin", 75, [(8192, 32)], 0, 32, 8)
    st = DecodeStep(wl, device="cuda", cascade=True)
    assert st.groups.num_groups == 1 and st.workspace is not None
    st.workspace.fill_(255)
    st.run()
    torch.cuda.synchronize()
    err, mx = check_step(st)
    assert err <= TOL["bf16"], (err, mx)
    ref = host_bits(st.out).copy()

    def call():
        st.workspace.fill_(255)
        st.decode()

    for _ in range(30):
        st.out.zero_()
        call()
        torch.cuda.synchronize()
        assert np.array_equal(host_bits(st.out), ref)
    call()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call()
    torch.cuda.synchronize()
    for _ in range(100):
        st.out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(host_bits(st.out), ref)
    assert lib.get_device_error() == 0
