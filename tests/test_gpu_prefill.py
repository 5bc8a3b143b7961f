"""Paged (chunked) prefill attention on the GPU against the float64 oracle:
every output element on small mixed batches (several query and key tiles,
ragged tails, empty chunks, all group sizes, both 16-bit types, fp8 E4M3
pools with per-tensor scales), every token of the full-size workloads, the
appended pool bytes, and the error paths."""
import numpy as np
import pytest
import torch

import oracle
from oracle.allocator_model import AllocatorModel
from parity_util import TOL, host_bits, max_error

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    from paged_kv_cache_10_gb300 import build, pagedkv
    build.build()
    pagedkv.lib()
    return pagedkv


def run(wl, plan=True):
    from paged_kv_cache_10_gb300.step import PrefillStep
    st = PrefillStep(wl, device="cuda", plan=plan)
    st.run()
    torch.cuda.synchronize()
    return st


def model(wl):
    """Slots, block tables and lengths from the independent allocator model."""
    m = AllocatorModel(wl.NB, wl.b, wl.free_order)
    for s, c in enumerate(wl.ctx):
        m.seq_new(s, c)
    slots = []
    for s, n in enumerate(wl.qlens):
        for _ in range(n):
            slot, cow = m.append_slot(s)
            assert cow is None
            slots.append(slot)
    tables = np.full((wl.S, wl.max_blocks), -1, np.int32)
    lens = np.zeros(wl.S, np.int32)
    for s in range(wl.S):
        t = m.block_table(s)
        tables[s, :len(t)] = t
        lens[s] = m.lens[s]
    return np.array(slots, np.int64), tables, lens


def oracle_pools(wl, slots):
    kp, vp = wl.k_pool.copy(), wl.v_pool.copy()
    oracle.append(wl.k_new, wl.v_new, wl.dtype, slots, kp, vp, wl.kv_dtype, wl.k_scale, wl.v_scale)
    return kp, vp


def check_full(st):
    wl = st.wl
    slots, tables, lens = model(wl)
    assert np.array_equal(st.slots, slots)
    assert np.array_equal(st.tables, tables)
    assert np.array_equal(st.seq_lens, lens)
    kp, vp = oracle_pools(wl, slots)
    assert np.array_equal(host_bits(st.k_cache), kp)
    assert np.array_equal(host_bits(st.v_cache), vp)
    ref = oracle.paged_prefill(wl.q, wl.dtype, st.query_start, kp, vp, wl.kv_dtype, tables, lens, wl.scale,
                               wl.k_scale, wl.v_scale)
    got = oracle.dequantize(host_bits(st.out), wl.dtype)
    assert np.all(np.isfinite(got))
    return max_error(got, ref, wl.dtype, TOL[wl.kv_dtype]), float(np.max(np.abs(ref)))


CASES = [
    # ctx, qlens: ragged query tiles, key tiles, empty chunks, single tokens
    ([0, 37, 5, 300, 0, 129], [20, 45, 1, 130, 0, 128]),
    ([700, 0, 16, 255], [1, 300, 17, 257]),
]


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("G", [1, 2, 4, 8])
@pytest.mark.parametrize("case", [0, 1])
@pytest.mark.parametrize("D", [128, 64])
@pytest.mark.parametrize("plan", [True, False])
def test_prefill_matches_oracle_every_element(lib, dtype, G, case, D, plan):
    """plan: CTAs in the host plan's longest-first order, or in grid order."""
    from paged_kv_cache_10_gb300 import workloads
    ctx, qlens = CASES[case]
    Hkv = 2
    wl = workloads.prefill("prefill_small", 2000 + 10 * G + case + D, ctx, qlens, Hkv * G, Hkv, D=D, dtype=dtype)
    st = run(wl, plan)
    assert lib.get_device_error() == 0
    err, mx = check_full(st)
    assert err <= TOL[dtype], (err, mx)


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("G", [1, 4, 8])
@pytest.mark.parametrize("case", [0, 1])
@pytest.mark.parametrize("D", [128, 64])
def test_prefill_fp8_cache_matches_oracle_every_element(lib, dtype, G, case, D):
    """fp8 E4M3 pools with per-tensor scales: the new tokens are encoded by
    the append, the attention pass reads 16-bit copies of the reached blocks;
    every output element against the oracle over the same codes."""
    from paged_kv_cache_10_gb300 import workloads
    ctx, qlens = CASES[case]
    Hkv = 2
    wl = workloads.prefill("prefill_fp8", 2300 + 10 * G + case + D, ctx, qlens, Hkv * G, Hkv, D=D, dtype=dtype,
                           kv_dtype="e4m3")
    assert wl.k_scale != wl.v_scale  # a swapped scale would show
    st = run(wl)
    assert st.workspace is not None
    assert lib.get_device_error() == 0
    err, mx = check_full(st)
    assert err <= TOL["e4m3"], (err, mx)


def test_prefill_fp8_cache_ignores_nan_codes_past_the_sequence_end(lib):
    """E4M3 NaN codes (0x7f, 0xff) in the slots no sequence has written reach
    the 16-bit copy as NaN and must still get probability 0."""
    from paged_kv_cache_10_gb300 import workloads
    wl = workloads.prefill("prefill_fp8_nan", 2398, [0, 0, 0], [10, 7, 150], 8, 2, dtype="bf16", kv_dtype="e4m3")
    wl.k_pool[:] = 0x7f
    wl.v_pool[:] = 0xff
    st = run(wl)
    assert lib.get_device_error() == 0
    err, mx = check_full(st)
    assert err <= TOL["e4m3"], (err, mx)


def test_prefill_fp8_cache_errors(lib):
    """A block id outside the pool is flagged (its copy reads as zeros), a
    short workspace is refused before any launch, and the next correct call
    still matches."""
    from paged_kv_cache_10_gb300 import workloads
    wl = workloads.prefill("prefill_fp8_err", 2399, [40, 0], [9, 30], 8, 2, dtype="bf16", kv_dtype="e4m3")
    st = run(wl)
    assert lib.get_device_error() == 0
    bad_tables = st.d_tables.clone()
    bad_tables[0, 0] = wl.NB + 5
    lib.paged_attention_prefill(st.q, st.k_cache, st.v_cache, st.desc, st.d_query_start, wl.max_query_len,
                                bad_tables, st.d_lens, wl.scale, st.out, q_dtype="bf16", workspace=st.workspace)
    torch.cuda.synchronize()
    assert lib.get_device_error() & lib.DEVERR_BLOCK_ID
    with pytest.raises(lib.PagedKVError):
        lib.paged_attention_prefill(st.q, st.k_cache, st.v_cache, st.desc, st.d_query_start, wl.max_query_len,
                                    st.d_tables, st.d_lens, wl.scale, st.out, q_dtype="bf16",
                                    workspace=st.workspace[:-1])
    with pytest.raises(lib.PagedKVError):
        lib.paged_attention_prefill(st.q, st.k_cache, st.v_cache, st.desc, st.d_query_start, wl.max_query_len,
                                    st.d_tables, st.d_lens, wl.scale, st.out, q_dtype="bf16")
    st.out.zero_()
    st.attend()
    torch.cuda.synchronize()
    assert lib.get_device_error() == 0
    err, mx = check_full(st)
    assert err <= TOL["e4m3"], (err, mx)


@pytest.mark.parametrize("name", ["prefill_chunked_gqa", "prefill_prompt_gqa", "prefill_prompt_mha",
                                  "prefill_chunked_gqa_fp8"])
def test_prefill_full_size_every_token(lib, name):
    """The full-size prefill workloads in the launch configuration the
    benchmark times: every token and head against the oracle's causal
    prefill, the appended pool bytes bit for bit."""
    from paged_kv_cache_10_gb300 import workloads
    wl = workloads.PREFILL[name]()
    st = run(wl)
    assert lib.get_device_error() == 0
    err, mx = check_full(st)
    assert err <= TOL[wl.kv_dtype], (err, mx)


def test_prefill_ignores_nan_bytes_past_the_sequence_end(lib):
    """Pool slots past a sequence's last token (never written) may hold NaN
    bit patterns; they get probability 0 and must not reach the output."""
    from paged_kv_cache_10_gb300 import workloads
    # no earlier context: every key is appended in the step, so every other
    # pool byte (the rest of each last block, unused blocks) may be NaN
    wl = workloads.prefill("prefill_nan", 2101, [0, 0, 0], [10, 7, 150], 8, 2, dtype="bf16")
    wl.k_pool[:] = 0x7fc1
    wl.v_pool[:] = 0x7fc1
    st = run(wl)
    assert lib.get_device_error() == 0
    err, mx = check_full(st)
    assert err <= TOL["bf16"], (err, mx)


def test_prefill_work_list_runs_exactly_its_units(lib):
    """A work list runs only the units it names, in any order; a unit id
    outside the batch is flagged and skipped."""
    from paged_kv_cache_10_gb300 import workloads
    wl = workloads.prefill("prefill_units", 2103, [40, 0, 300], [70, 129, 33], 8, 2, dtype="bf16")
    st = run(wl)
    assert lib.get_device_error() == 0
    err, mx = check_full(st)
    assert err <= TOL["bf16"], (err, mx)
    full = host_bits(st.out).copy()
    plan = st.work_host
    assert len(plan) == len(set(plan.tolist()))
    # run only the second half of the plan, reversed, into a cleared output
    part = plan[len(plan) // 2:][::-1].copy()
    st.out.zero_()
    lib.paged_attention_prefill(st.q, st.k_cache, st.v_cache, st.desc, st.d_query_start, wl.max_query_len,
                                st.d_tables, st.d_lens, wl.scale, st.out, q_dtype="bf16",
                                work_units=torch.from_numpy(part).cuda())
    torch.cuda.synchronize()
    assert lib.get_device_error() == 0
    got = host_bits(st.out)
    rows_per_unit = 2 * (128 // (wl.Hq // wl.Hkv))
    nq = -(-wl.max_query_len // rows_per_unit)
    done = np.zeros(wl.T, bool)
    for u in part.tolist():
        s, qt = divmod(u, nq)
        a = st.query_start[s] + qt * rows_per_unit
        done[a:min(a + rows_per_unit, st.query_start[s + 1])] = True
    assert np.array_equal(got[done], full[done])
    assert np.all(got[~done] == 0)
    # an out-of-range unit: flagged, the valid ones still run
    bad = np.concatenate([plan[:1], np.array([wl.S * nq + 3], np.int32)])
    lib.paged_attention_prefill(st.q, st.k_cache, st.v_cache, st.desc, st.d_query_start, wl.max_query_len,
                                st.d_tables, st.d_lens, wl.scale, st.out, q_dtype="bf16",
                                work_units=torch.from_numpy(bad).cuda())
    torch.cuda.synchronize()
    assert lib.get_device_error() & lib.DEVERR_SEQ_LEN


def test_prefill_rejects_bad_arguments(lib):
    from paged_kv_cache_10_gb300 import workloads
    from paged_kv_cache_10_gb300.step import PrefillStep
    wl = workloads.prefill("prefill_err", 2102, [5, 0], [9, 30], 8, 2, dtype="bf16")
    st = PrefillStep(wl, device="cuda")
    st.run()
    torch.cuda.synchronize()
    assert lib.get_device_error() == 0
    # more new tokens than the sequence holds: flagged, sequence skipped
    bad_lens = st.d_lens.clone()
    bad_lens[1] = 10
    lib.paged_attention_prefill(st.q, st.k_cache, st.v_cache, st.desc, st.d_query_start, wl.max_query_len,
                                st.d_tables, bad_lens, wl.scale, st.out, q_dtype="bf16")
    torch.cuda.synchronize()
    assert lib.get_device_error() & lib.DEVERR_SEQ_LEN
    # a grid bound below the longest chunk: flagged
    lib.paged_attention_prefill(st.q, st.k_cache, st.v_cache, st.desc, st.d_query_start, 8,
                                st.d_tables, st.d_lens, wl.scale, st.out, q_dtype="bf16")
    torch.cuda.synchronize()
    assert lib.get_device_error() & lib.DEVERR_SEQ_LEN
    # block id outside the pool: flagged
    bad_tables = st.d_tables.clone()
    bad_tables[0, 0] = wl.NB + 5
    lib.paged_attention_prefill(st.q, st.k_cache, st.v_cache, st.desc, st.d_query_start, wl.max_query_len,
                                bad_tables, st.d_lens, wl.scale, st.out, q_dtype="bf16")
    torch.cuda.synchronize()
    assert lib.get_device_error() & lib.DEVERR_BLOCK_ID
    # unsupported: q type differing from the pool, head_size 96
    with pytest.raises(lib.PagedKVError):
        lib.paged_attention_prefill(st.q, st.k_cache, st.v_cache, st.desc, st.d_query_start, wl.max_query_len,
                                    st.d_tables, st.d_lens, wl.scale, st.out, q_dtype="f16")
    d96 = lib.CacheDesc(num_blocks=wl.NB, num_kv_heads=2, head_size=96, kv_dtype="bf16")
    with pytest.raises(lib.PagedKVError):
        lib.paged_attention_prefill(st.q, st.k_cache, st.v_cache, d96, st.d_query_start, wl.max_query_len,
                                    st.d_tables, st.d_lens, wl.scale, st.out, q_dtype="bf16")
    # the context is still usable and the correct call still matches
    st.attend()
    torch.cuda.synchronize()
    assert lib.get_device_error() == 0
    err, mx = check_full(st)
    assert err <= TOL["bf16"], (err, mx)


@pytest.mark.parametrize("dtype,G", [("bf16", 4), ("f16", 1)])
def test_prefill_sharp_softmax(lib, dtype, G):
    """q scaled by 30: the row maximum jumps by far more than the lazy
    rebase threshold (2^8) between key tiles, in prompts and in chunks over
    earlier context, and few keys dominate each row; with the probabilities
    carried as a 16-bit head plus tail the plain bound holds."""
    import oracle as orc
    from paged_kv_cache_10_gb300 import workloads
    Hkv = 2
    wl = workloads.prefill("prefill_sharp", 2200 + G, [0, 300, 0], [257, 130, 40], Hkv * G, Hkv, dtype=dtype)
    x = orc.dequantize(wl.q, dtype) * 30.0
    t = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16 if dtype == "bf16" else torch.float16)
    wl.q = t.view(torch.int16).numpy().view(np.uint16).copy()
    st = run(wl)
    assert lib.get_device_error() == 0
    err, mx = check_full(st)
    assert err <= TOL[dtype], (err, mx)


def test_prefill_persistent_grid_counters_graphs_and_streams(lib):
    """The persistent prefill takes units from a per-call device counter that
    its last CTA puts back to zero.  More calls in a row than there are
    counters, replays of a captured call, and two calls running at once on two
    streams all reproduce the eager result bit for bit."""
    from paged_kv_cache_10_gb300 import workloads
    from paged_kv_cache_10_gb300.step import PrefillStep
    wl = workloads.prefill("prefill_persist", 2500, [700, 0, 40, 2000, 5], [300, 600, 129, 77, 1000], 32, 8)
    st = run(wl)
    assert lib.get_device_error() == 0
    err, mx = check_full(st)
    assert err <= TOL["bf16"], (err, mx)
    eager = host_bits(st.out).copy()
    for _ in range(1100):  # wraps the library's 1024 counters
        st.attend()
    torch.cuda.synchronize()
    assert lib.get_device_error() == 0
    assert np.array_equal(host_bits(st.out), eager)
    # a captured call, replayed
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        st.attend(stream=side)  # warm-up outside the capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        st.attend()
    for _ in range(3):
        st.out.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert lib.get_device_error() == 0
        assert np.array_equal(host_bits(st.out), eager)
    # an output 16 bytes (not 32) into its buffer takes the 16-byte stores
    buf = torch.zeros(st.out.numel() + 8, dtype=torch.uint16, device="cuda")
    out16 = buf[8:].view(st.out.shape)
    assert out16.data_ptr() % 32 == 16
    lib.paged_attention_prefill(st.q, st.k_cache, st.v_cache, st.desc, st.d_query_start, wl.max_query_len,
                                st.d_tables, st.d_lens, wl.scale, out16, q_dtype="bf16", work_units=st.work)
    torch.cuda.synchronize()
    assert lib.get_device_error() == 0
    assert np.array_equal(host_bits(out16), eager)
    assert np.all(host_bits(buf[:8]) == 0)
    # two calls at once on two streams (each holds its own counter)
    st2 = PrefillStep(wl, device="cuda")
    st2.run()
    torch.cuda.synchronize()
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    st.out.zero_()
    st2.out.zero_()
    torch.cuda.synchronize()
    for _ in range(20):
        with torch.cuda.stream(s1):
            st.attend(stream=s1)
        with torch.cuda.stream(s2):
            st2.attend(stream=s2)
    torch.cuda.synchronize()
    assert lib.get_device_error() == 0
    assert np.array_equal(host_bits(st.out), eager)
    assert np.array_equal(host_bits(st2.out), eager)
