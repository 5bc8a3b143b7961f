"""GPU parity: the CUDA path through the C ABI against the float64 oracle.

Append and copy-on-write must match bit for bit (whole pools compared);
attention within max-abs 2e-3 (fp16) / 1e-2 (bf16, fp8 KV judged on the
dequantised values).  Small cases span several blocks, partitions and warps
with ragged tails; the five named workloads run at full size with the
launch configuration the benchmark uses, every row checked.
"""
import numpy as np
import pytest
import torch

from parity_util import TOL, check_step, host_bits, max_error

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    from paged_kv_cache_10_gb300 import build, pagedkv
    build.build()
    pagedkv.lib()
    return pagedkv


def run(wl, partition=None, fused=True):
    from paged_kv_cache_10_gb300.step import DecodeStep
    st = DecodeStep(wl, device="cuda", partition_tokens=partition, fused=fused)
    st.run()
    torch.cuda.synchronize()
    return st


EDGE_LENS = [1, 15, 16, 17, 31, 33, 100, 255, 511, 512, 513, 1000]

CASES = [
    # (kv dtype, q dtype, head size)
    ("f16", "f16", 64),
    ("bf16", "bf16", 128),
    ("e4m3", "bf16", 128),
    ("f16", "f16", 128),
    ("bf16", "bf16", 64),
    ("e4m3", "f16", 64),
    ("e4m3", "f16", 128),
]


# path 0: the automatic choice (tensor cores for G >= 2 at D = 128); path 1:
# the CUDA-core kernel forced, only where the automatic choice differs
SMALL = [(kv, qd, D, G, path) for kv, qd, D in CASES for G in (1, 2, 4, 8) for path in (0, 1)
         if path == 0 or (G > 1 and D == 128)]


@pytest.mark.parametrize("kv,qd,D,G,path", SMALL)
@pytest.mark.parametrize("partition", [0, 16, 64, 512])
def test_small_cases_match_oracle(lib, kv, qd, D, G, partition, path):
    """Every element of a small edge-length batch against the oracle, for
    each dtype / head size / group size / partition size and kernel."""
    from paged_kv_cache_10_gb300 import workloads
    Hkv = 2
    wl = workloads.custom(f"edge_{kv}_{D}_{G}", 7 + G + D, EDGE_LENS, Hkv * G, Hkv, D, kv_dtype=kv,
                          q_dtype=qd, partition_tokens=partition)
    with lib.decode_path(path):
        st = run(wl)
    assert lib.get_device_error() == 0
    err, mx = check_step(st)
    assert err <= TOL[kv], (err, mx)


@pytest.mark.parametrize("kv,qd", [("bf16", "bf16"), ("f16", "f16"), ("e4m3", "bf16")])
def test_tensor_core_and_cuda_core_kernels_agree(lib, kv, qd):
    from paged_kv_cache_10_gb300 import workloads
    import oracle
    wl = workloads.custom("paths", 21, [1, 16, 17, 300, 1029], 32, 8, 128, kv_dtype=kv, q_dtype=qd)
    with lib.decode_path(2):
        a = run(wl)
    with lib.decode_path(1):
        b = run(wl)
    ea, _ = check_step(a)
    eb, _ = check_step(b)
    assert ea <= TOL[kv] and eb <= TOL[kv]
    fa = oracle.dequantize(host_bits(a.out), qd)
    fb = oracle.dequantize(host_bits(b.out), qd)
    assert np.max(np.abs(fa - fb)) <= TOL[kv]


def test_tensor_core_path_rejects_what_it_cannot_serve(lib):
    from paged_kv_cache_10_gb300 import workloads
    wl = workloads.custom("mha", 22, [40], 4, 4, 128, kv_dtype="bf16")  # G = 1
    with lib.decode_path(2):
        with pytest.raises(lib.PagedKVError):
            run(wl)


def test_stale_nan_bytes_past_the_sequence_end_are_ignored(lib):
    """Slots past a sequence's last token may hold anything (here NaN bit
    patterns); neither kernel may let them reach the output."""
    from paged_kv_cache_10_gb300 import workloads
    from paged_kv_cache_10_gb300.step import DecodeStep
    wl = workloads.custom("nan", 23, [5, 21, 16], 16, 2, 128, kv_dtype="bf16")
    for path in (1, 2):
        st = DecodeStep(wl, device="cuda")
        for s in range(wl.S):
            L = int(st.seq_lens[s])
            last = int(st.tables[s, (L - 1) // 16])
            off = L % 16
            if off:
                st.k_cache[last, :, off:] = 0x7FC0  # bf16 quiet NaN
                st.v_cache[last, :, off:] = 0x7FC0
        with lib.decode_path(path):
            st.run()
        torch.cuda.synchronize()
        got = host_bits(st.out)
        import oracle
        assert np.all(np.isfinite(oracle.dequantize(got, "bf16"))), path


def test_zero_length_rows_and_padding_slots(lib):
    from paged_kv_cache_10_gb300 import workloads
    wl = workloads.custom("zeros", 3, [0, 5, 0, 40], 8, 2, 128, kv_dtype="bf16")
    st = run(wl)
    assert lib.get_device_error() == 0
    err, _ = check_step(st)
    assert err <= TOL["bf16"]
    out = host_bits(st.out)
    assert np.all(out[0] == 0) and np.all(out[2] == 0)
    assert st.slots[0] == -1 and st.slots[2] == -1


# 2049 tokens in P-token partitions: 129 (three merge chunks of a warp), 43,
# 26, 13 and 5 partitions, i.e. every warps-per-row choice of the merge
@pytest.mark.parametrize("P", [16, 48, 80, 160, 512, 0])
def test_split_and_unsplit_agree(lib, P):
    from paged_kv_cache_10_gb300 import workloads
    wl = workloads.custom("split", 11, [700, 1300, 64, 2049], 32, 8, 128, kv_dtype="bf16", partition_tokens=P)
    a = run(wl)
    b = run(wl, partition=2064)  # one partition for every row
    ea, _ = check_step(a)
    eb, _ = check_step(b)
    assert ea <= TOL["bf16"] and eb <= TOL["bf16"]
    import oracle
    fa = oracle.dequantize(host_bits(a.out), "bf16")
    fb = oracle.dequantize(host_bits(b.out), "bf16")
    # the two reductions differ in summation order and, on the tensor-core
    # path, in where P is rounded to bf16 (relative to a partition's running
    # max): a few bf16 ulps of the outputs, far inside the tolerance
    assert np.max(np.abs(fa - fb)) <= 4e-3


@pytest.mark.parametrize("name", ["tiny_fp16", "llama7b_mha", "llama3_8b_gqa", "longctx_fp8", "prefix_share"])
def test_named_workloads_full_size(lib, name):
    """Each named workload at full size, in the launch configuration the
    benchmark times (host plan where it pays, automatic or stated
    partitions, fused append): every row and head against the oracle, pools
    bit for bit."""
    from paged_kv_cache_10_gb300 import workloads
    wl = workloads.NAMED[name]()
    st = run(wl)
    assert lib.get_device_error() == 0
    if name == "prefix_share":
        assert len(st.pairs) >= 50  # copy-on-write really happens
    err, mx = check_step(st)
    assert err <= TOL[wl.kv_dtype], (name, err, mx)
    del st
    torch.cuda.empty_cache()


def test_literal_prefix_share_has_no_copy(lib):
    from paged_kv_cache_10_gb300 import workloads
    wl = workloads.prefix_share(literal=True, pairs=16)
    st = run(wl)
    assert len(st.pairs) == 0
    err, _ = check_step(st)
    assert err <= TOL["bf16"]


def test_device_errors_are_reported_not_trapped(lib):
    """Out-of-range ids set bits in the device error word; the kernels skip
    the access and the context stays usable."""
    from paged_kv_cache_10_gb300 import workloads
    wl = workloads.custom("errs", 5, [20, 40], 4, 2, 128, kv_dtype="bf16")
    from paged_kv_cache_10_gb300.step import DecodeStep
    st = DecodeStep(wl, device="cuda")
    assert lib.get_device_error() == 0
    # a block id outside the pool in row 1
    bad = st.d_tables.clone()
    bad[1, 1] = wl.NB + 5
    st.decode(tables=bad)
    assert lib.get_device_error() & lib.DEVERR_BLOCK_ID
    # a seq_len beyond the block table
    lens = st.d_lens.clone()
    lens[0] = st.max_blocks * 16 + 7
    st.decode(lens=lens)
    assert lib.get_device_error() & lib.DEVERR_SEQ_LEN
    # a slot outside the pool; -1 is padding and silent
    slots = torch.tensor([wl.NB * 16 + 3, -1], dtype=torch.int64, device="cuda")
    lib.paged_kv_append(st.k_new, st.v_new, slots, st.k_cache, st.v_cache, st.desc, in_dtype="bf16")
    assert lib.get_device_error() == lib.DEVERR_SLOT
    # a copy pair outside the pool
    pairs = torch.tensor([[0, wl.NB]], dtype=torch.int32, device="cuda")
    lib.copy_blocks(st.k_cache, st.v_cache, st.desc, pairs)
    assert lib.get_device_error() == lib.DEVERR_COPY_PAIR
    # the context still works: a clean step matches the oracle
    st2 = run(wl)
    assert lib.get_device_error() == 0
    err, _ = check_step(st2)
    assert err <= TOL["bf16"]


@pytest.mark.parametrize("Hq,Hkv", [(8, 8), (32, 8)])
def test_many_sequences_and_a_full_block_table(lib, Hq, Hkv):
    """3000 short sequences (a large grid and 3000 x Hq merge rows) around
    one 2048-token sequence whose block table is exactly full, split into
    256-token partitions; every row against the oracle, pools bit-exact."""
    from paged_kv_cache_10_gb300 import workloads
    rng = np.random.default_rng(97)
    lens = rng.integers(0, 40, 3000).tolist()
    lens[1234] = 2048  # 128 blocks: the widest table, every entry used
    wl = workloads.custom("many", 98 + Hq, lens, Hq, Hkv, 128, kv_dtype="bf16", partition_tokens=256)
    st = run(wl)
    assert lib.get_device_error() == 0
    assert st.tables.shape[1] == 128 and np.all(st.tables[1234] >= 0)
    err, mx = check_step(st)
    assert err <= TOL["bf16"], (err, mx)


def test_library_is_loaded_from_the_tree(lib):
    import os
    maps = open("/proc/self/maps").read()
    assert os.path.realpath(lib.LIB_PATH) in maps


def test_graph_replay_matches_eager(lib):
    """A captured step replays the same kernels: outputs and pools identical."""
    from paged_kv_cache_10_gb300 import workloads
    from paged_kv_cache_10_gb300.step import DecodeStep
    wl = workloads.custom("graph", 81, [1, 33, 700, 2100], 32, 8, 128, kv_dtype="bf16")
    st = DecodeStep(wl, device="cuda")
    g = st.capture()
    st.out.zero_()
    g.replay()
    torch.cuda.synchronize()
    err, _ = check_step(st)
    assert err <= TOL["bf16"]
    first = host_bits(st.out).copy()
    g.replay()
    torch.cuda.synchronize()
    assert np.array_equal(host_bits(st.out), first)


def test_swap_round_trip_preserves_sequences(lib):
    """Swap two sequences out to a pinned host pool, let other data overwrite
    their old device blocks, swap them back into new blocks: the host copy is
    bit-exact and decode of the swapped-in sequences matches the oracle on the
    original data."""
    import oracle
    from paged_kv_cache_10_gb300 import workloads
    from paged_kv_cache_10_gb300.step import DecodeStep
    wl = workloads.custom("swap", 91, [40, 300, 17, 700], 16, 2, 128, kv_dtype="bf16")
    st = DecodeStep(wl, device="cuda")
    st.run()
    torch.cuda.synchronize()
    NH = 64
    k_host = torch.zeros((NH, wl.Hkv, 16, wl.D), dtype=torch.uint16).pin_memory()
    v_host = torch.zeros_like(k_host).pin_memory()
    host = lib.Allocator(NH, 16)
    orig_k, orig_v = host_bits(st.k_cache).copy(), host_bits(st.v_cache).copy()
    moved = {}
    for s in (1, 3):
        old_table = st.alloc.block_table(s)
        pairs = st.alloc.swap_out(host, s)
        assert [p[0] for p in pairs.tolist()] == old_table
        lib.swap_blocks(st.k_cache, st.v_cache, st.desc, k_host, v_host,
                        torch.from_numpy(pairs).cuda(), lib.SWAP_OUT)
        moved[s] = pairs
    torch.cuda.synchronize()
    kh = k_host.view(torch.int16).numpy().view(np.uint16)
    vh = v_host.view(torch.int16).numpy().view(np.uint16)
    for s, pairs in moved.items():
        for d, h in pairs.tolist():
            assert np.array_equal(kh[h], orig_k[d]) and np.array_equal(vh[h], orig_v[d])
    # freed device blocks get overwritten by other work
    st.k_cache.view(torch.int16).random_(0, 30000)
    st.v_cache.view(torch.int16).random_(0, 30000)
    keep_k, keep_v = host_bits(st.k_cache).copy(), host_bits(st.v_cache).copy()
    for s in (3, 1):
        pairs = st.alloc.swap_in(host, s)
        lib.swap_blocks(st.k_cache, st.v_cache, st.desc, k_host, v_host,
                        torch.from_numpy(pairs).cuda(), lib.SWAP_IN)
        for d, h in pairs.tolist():
            keep_k[d], keep_v[d] = kh[h], vh[h]
    torch.cuda.synchronize()
    assert lib.get_device_error() == 0
    assert np.array_equal(host_bits(st.k_cache), keep_k) and np.array_equal(host_bits(st.v_cache), keep_v)
    # decode the swapped-in sequences from their new blocks
    rows = np.array([1, 3])
    tables, lens = st.alloc.export(rows, st.max_blocks)
    q = st.q.view(torch.int16)[torch.from_numpy(rows).cuda()].contiguous().view(torch.uint16)
    out = torch.empty_like(q)
    ws = torch.empty(max(lib.decode_workspace_bytes(2, wl.Hq, wl.D, int(lens.max()), 0), 16), dtype=torch.uint8,
                     device="cuda")
    lib.paged_attention_decode(q, st.k_cache, st.v_cache, st.desc, torch.from_numpy(tables).cuda(),
                               torch.from_numpy(lens).cuda(), int(lens.max()), wl.scale, out, workspace=ws,
                               q_dtype="bf16")
    torch.cuda.synchronize()
    ref = oracle.paged_decode(np.ascontiguousarray(wl.q[rows]), "bf16", keep_k, keep_v, "bf16", tables, lens,
                              wl.scale)
    got = oracle.dequantize(host_bits(out), "bf16")
    assert max_error(got, ref, "bf16", TOL["bf16"]) <= TOL["bf16"]
    # and it is the attention of the original data (old tables, original pools)
    ref0 = oracle.paged_decode(np.ascontiguousarray(wl.q[rows]), "bf16", orig_k, orig_v, "bf16",
                               st.tables[rows], st.seq_lens[rows], wl.scale)
    assert np.max(np.abs(got - ref0)) <= TOL["bf16"]


def test_swap_rejects_unpinned_host_memory(lib):
    from paged_kv_cache_10_gb300 import workloads
    from paged_kv_cache_10_gb300.step import DecodeStep
    wl = workloads.custom("swap2", 92, [40], 4, 2, 128, kv_dtype="bf16")
    st = DecodeStep(wl, device="cuda")
    k_host = torch.zeros((4, 2, 16, 128), dtype=torch.uint16)
    with pytest.raises(ValueError):
        lib.swap_blocks(st.k_cache, st.v_cache, st.desc, k_host, k_host,
                        torch.zeros((1, 2), dtype=torch.int32, device="cuda"), lib.SWAP_OUT)


@pytest.mark.parametrize("kv,qd,D,G", [("f16", "f16", 64, 1), ("bf16", "bf16", 128, 4), ("e4m3", "bf16", 128, 8),
                                       ("e4m3", "f16", 64, 2)])
def test_separate_append_kernel_matches_oracle(lib, kv, qd, D, G):
    """The step with the append as its own kernel (the fused path is the
    default everywhere else): pools bit for bit, attention within tolerance."""
    from paged_kv_cache_10_gb300 import workloads
    Hkv = 2
    wl = workloads.custom(f"unfused_{kv}_{D}_{G}", 40 + G, EDGE_LENS, Hkv * G, Hkv, D, kv_dtype=kv, q_dtype=qd)
    st = run(wl, fused=False)
    assert lib.get_device_error() == 0
    err, mx = check_step(st)
    assert err <= TOL[kv], (err, mx)


def test_fused_append_rejects_a_slot_off_the_last_position(lib):
    """A slot that is not the block table's slot of position seq_len - 1 is
    flagged and not written; the other rows are unaffected."""
    from paged_kv_cache_10_gb300 import workloads
    from paged_kv_cache_10_gb300.step import DecodeStep
    wl = workloads.custom("fused_bad_slot", 77, [20, 40, 9], 8, 2, 128, kv_dtype="bf16")
    st = DecodeStep(wl, device="cuda")
    k_before = st.k_cache.clone()
    bad = st.d_slots.clone()
    bad[1] = bad[1] + 1  # next offset in the same block: not position L - 1
    lib.paged_attention_decode_append(st.k_new, st.v_new, bad, st.q, st.k_cache, st.v_cache, st.desc, st.d_tables,
                                      st.d_lens, st.max_seq_len, wl.scale, st.out, workspace=st.workspace,
                                      q_dtype="bf16", in_dtype="bf16")
    torch.cuda.synchronize()
    assert lib.get_device_error() & lib.DEVERR_SLOT
    # row 1's slot (and the wrong one) untouched, rows 0 and 2 written
    b, o = int(bad[1]) // 16, int(bad[1]) % 16
    assert torch.equal(st.k_cache[b, :, o], k_before[b, :, o])
    b1, o1 = int(st.d_slots[1]) // 16, int(st.d_slots[1]) % 16
    assert torch.equal(st.k_cache[b1, :, o1], k_before[b1, :, o1])
    b0, o0 = int(st.d_slots[0]) // 16, int(st.d_slots[0]) % 16
    assert torch.equal(st.k_cache[b0, :, o0], st.k_new[0])


def test_fused_copy_on_write_rejects_a_bad_source(lib):
    """A copy-on-write source outside the pool is flagged and the row is not
    written; the context stays usable."""
    from paged_kv_cache_10_gb300 import workloads
    from paged_kv_cache_10_gb300.step import DecodeStep
    wl = workloads.prefix_share(pairs=4, prefix=64)
    st = DecodeStep(wl, device="cuda")
    assert len(st.pairs) > 0
    bad = st.d_cow_src.clone()
    row = int(np.nonzero(st.cow_src >= 0)[0][0])
    bad[row] = wl.NB + 1
    st.decode(cow_src=bad)
    torch.cuda.synchronize()
    assert lib.get_device_error() & lib.DEVERR_COPY_PAIR
    st2 = DecodeStep(wl, device="cuda")
    st2.run()
    torch.cuda.synchronize()
    assert lib.get_device_error() == 0
    err, _ = check_step(st2)
    assert err <= TOL["bf16"]


def _scale_q(wl, factor):
    """q of the workload times `factor`, re-rounded to its 16-bit type (test
    input generation only)."""
    import oracle
    x = oracle.dequantize(wl.q, wl.q_dtype) * factor
    t = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16 if wl.q_dtype == "bf16" else torch.float16)
    wl.q = t.view(torch.int16).numpy().view(np.uint16).copy()


@pytest.mark.parametrize("kv,G,partition", [("bf16", 1, 0), ("bf16", 4, 0), ("bf16", 4, 256), ("e4m3", 8, 256),
                                            ("f16", 2, 64)])
def test_sharp_softmax_matches_oracle(lib, kv, G, partition):
    """q scaled by 30: scores spread over ~150 log2 units, so the running
    maximum moves by large steps inside blocks, across warps and across
    split-K partitions (merge weights underflow to 0), and few keys dominate
    each row.  The tensor-core kernels carry the probabilities as a 16-bit
    head plus a 16-bit tail, so the plain bound holds here too."""
    from paged_kv_cache_10_gb300 import workloads
    Hkv = 2
    wl = workloads.custom(f"sharp_{kv}", 111 + G, [1, 17, 200, 1500, 3000], Hkv * G, Hkv, 128, kv_dtype=kv,
                          partition_tokens=partition)
    _scale_q(wl, 30.0)
    st = run(wl)
    assert lib.get_device_error() == 0
    err, mx = check_step(st)
    assert err <= TOL[kv], (err, mx)


@pytest.mark.parametrize("kv,G,partition", [("bf16", 1, 64), ("bf16", 4, 0), ("e4m3", 8, 256), ("f16", 2, 16)])
def test_decode_in_plan_order_matches_oracle(lib, kv, G, partition):
    """The fused decode with its CTAs in the host plan's longest-first order:
    same rows, pools and appends as the grid order, every element against
    the oracle; a unit outside the batch is flagged."""
    from paged_kv_cache_10_gb300 import workloads
    from paged_kv_cache_10_gb300.step import DecodeStep
    Hkv = 2
    wl = workloads.custom(f"plan_{kv}", 131 + G, EDGE_LENS + [0, 2050], Hkv * G, Hkv, 128, kv_dtype=kv,
                          partition_tokens=partition)
    st = DecodeStep(wl, device="cuda", plan=True)
    assert st.work is not None and len(set(st.work_host.tolist())) == len(st.work_host)
    st.run()
    torch.cuda.synchronize()
    assert lib.get_device_error() == 0
    err, mx = check_step(st)
    assert err <= TOL[kv], (err, mx)
    bad = torch.from_numpy(np.concatenate([st.work_host, np.array([10 ** 6], np.int32)])).cuda()
    st.work = bad
    st.decode()
    torch.cuda.synchronize()
    assert lib.get_device_error() & lib.DEVERR_SEQ_LEN


@pytest.mark.parametrize("which", [0, 1])
def test_bounded_wait_gives_up_and_reports(lib, which):
    """A pipeline wait that can never be satisfied (a barrier nothing arrives
    at, no copy in flight) gives up after its bound, sets DEVERR_TIMEOUT and
    lets its kernel return; the context stays usable and the next step
    matches the oracle."""
    import time
    from paged_kv_cache_10_gb300 import workloads
    assert lib.get_device_error() == 0
    t0 = time.perf_counter()
    lib.check_wait_timeout(which)
    torch.cuda.synchronize()
    waited = time.perf_counter() - t0
    assert lib.get_device_error() == lib.DEVERR_TIMEOUT
    assert waited < 30.0, waited
    with pytest.raises(lib.PagedKVError):
        lib.check_wait_timeout(2)
    wl = workloads.custom("after_timeout", 6, [20, 300], 8, 2, 128, kv_dtype="bf16")
    st = run(wl)
    assert lib.get_device_error() == 0
    err, mx = check_step(st)
    assert err <= TOL["bf16"], (err, mx)
