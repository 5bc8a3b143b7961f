"""Host work plan of the paged prefill (pkv_prefill_plan): every non-empty
(sequence, query tile pair) unit exactly once, sorted by the causal key range
of the unit's last row, longest first, and the error paths.  CPU only."""
import numpy as np
import pytest


@pytest.fixture(scope="module")
def pk():
    from paged_kv_cache_10_gb300 import build, pagedkv
    build.build()
    return pagedkv


def expected_units(qs, lens, G, maxq):
    """The plan restated: units s * nq + qt with qt * r < n_s, r = 256 / G
    query tokens per unit, key range ctx_s + min(n_s, (qt + 1) r)."""
    r = 2 * (128 // G)
    nq = -(-maxq // r)
    units = []
    for s in range(len(lens)):
        n = int(qs[s + 1] - qs[s])
        ctx = int(lens[s]) - n
        for qt in range(-(-n // r)):
            units.append((ctx + min(n, (qt + 1) * r), s, qt, s * nq + qt))
    # longest first, then sequence and query tile ascending
    units.sort(key=lambda t: (-t[0], t[1], t[2]))
    return np.array([u[3] for u in units], np.int32)


@pytest.mark.parametrize("G", [1, 2, 4, 8])
def test_plan_orders_every_unit_longest_first(pk, G):
    rng = np.random.default_rng(7 + G)
    S = 37
    qlens = rng.integers(0, 700, S)
    qlens[3] = 0
    ctx = rng.integers(0, 5000, S)
    qs = np.zeros(S + 1, np.int32)
    qs[1:] = np.cumsum(qlens)
    lens = (ctx + qlens).astype(np.int32)
    maxq = int(qlens.max()) + 5
    got = pk.prefill_plan(qs, lens, 8 * G, 8, maxq)
    want = expected_units(qs, lens, G, maxq)
    assert np.array_equal(got, want)
    # a permutation of the non-empty units, and key ranges non-increasing
    r = 2 * (128 // G)
    nq = -(-maxq // r)
    assert len(set(got.tolist())) == len(got) == sum(-(-int(n) // r) for n in qlens)
    s, qt = got // nq, got % nq
    keys = (lens[s] - qlens[s]) + np.minimum(qlens[s], (qt + 1) * r)
    assert np.all(np.diff(keys) <= 0)


def test_plan_equal_prompts_go_by_query_tile(pk):
    # equal chunks from empty contexts: the last query tiles of every sequence first
    qs = np.array([0, 512, 1024], np.int32)
    lens = np.array([512, 512], np.int32)
    got = pk.prefill_plan(qs, lens, 32, 8, 512)  # G = 4: 64 tokens per unit, 8 per sequence
    assert got.tolist() == [7, 15, 6, 14, 5, 13, 4, 12, 3, 11, 2, 10, 1, 9, 0, 8]


def test_plan_errors(pk):
    import ctypes
    L = pk.lib()
    qs = np.array([0, 10, 30], np.int32)
    lens = np.array([10, 25], np.int32)
    n = ctypes.c_int32(-1)
    out = np.zeros(1, np.int32)
    # too small an output: the count comes back with PKV_ERR_WORKSPACE
    st = L.pkv_prefill_plan(pk._np_ptr(qs), pk._np_ptr(lens), 2, 8, 8, 20, pk._np_ptr(out), 1, ctypes.byref(n))
    assert st == 5 and n.value == 2
    # a chunk longer than max_query_len, or than the sequence: invalid
    with pytest.raises(pk.PagedKVError):
        pk.prefill_plan(qs, lens, 8, 8, 15)
    with pytest.raises(pk.PagedKVError):
        pk.prefill_plan(qs, np.array([10, 19], np.int32), 8, 8, 20)
    # head ratio 3: unsupported; ratio not integral: invalid
    with pytest.raises(pk.PagedKVError):
        pk.prefill_plan(qs, lens, 24, 8, 20)
    with pytest.raises(pk.PagedKVError):
        pk.prefill_plan(qs, lens, 12, 8, 20)
    # nothing to do
    assert pk.prefill_plan(np.array([0], np.int32), np.zeros(0, np.int32), 8, 8, 20).size == 0


def test_decode_plan_lists_every_unit_longest_first(pk):
    rng = np.random.default_rng(5)
    lens = rng.integers(0, 5000, 300).astype(np.int32)
    lens[7] = 0
    P = 512
    got = pk.decode_plan(lens, 8, int(lens.max()), P)
    NP = -(-int(lens.max()) // P)
    want = []
    for s, L in enumerate(lens.tolist()):
        n = -(-L // P) if L > 0 else 1
        for p in range(n):
            want.append((-min(P, L - p * P), s * NP + p))
    want.sort()
    assert got.tolist() == [u for _, u in want]
    # lengths beyond the bound: invalid; more units than the cap: the count comes back
    with pytest.raises(pk.PagedKVError):
        pk.decode_plan(np.array([10, 600], np.int32), 8, 500, 512)
    import ctypes
    n = ctypes.c_int32(-1)
    out = np.zeros(1, np.int32)
    st = pk.lib().pkv_decode_plan(pk._np_ptr(lens), lens.size, 8, int(lens.max()), P, pk._np_ptr(out), 1,
                                  ctypes.byref(n))
    assert st == 5 and n.value == len(want)


def test_fp8_prefill_workload_codes_and_scales():
    """The fp8 prefill workload stores E4M3 codes under per-tensor scales
    max|x| / 448 of each pool's N(0,1) source: finite codes only (no NaN,
    0x7f / 0xff), the largest magnitude code reached, the same context
    lengths and queries as the bf16 batch of the same seed, and a staging
    workspace sized for its tables."""
    import oracle
    from paged_kv_cache_10_gb300 import pagedkv as pk, workloads
    wl = workloads.PREFILL["prefill_chunked_gqa_fp8"]()
    ref = workloads.PREFILL["prefill_chunked_gqa"]()
    assert wl.kv_dtype == "e4m3" and wl.dtype == "bf16"
    assert wl.ctx == ref.ctx and wl.qlens == ref.qlens
    assert np.array_equal(wl.q, ref.q)
    for pool, scale in ((wl.k_pool, wl.k_scale), (wl.v_pool, wl.v_scale)):
        assert pool.dtype == np.uint8
        assert not np.any((pool & 0x7f) == 0x7f)
        vals = oracle.dequantize(pool.ravel()[:1 << 20], "e4m3")
        assert np.all(np.isfinite(vals))
        assert np.max(np.abs(vals)) <= 448.0
        assert scale > 0
    assert np.max(np.abs(oracle.dequantize(wl.k_pool, "e4m3"))) == 448.0
    assert wl.k_scale != wl.v_scale
    need = pk.prefill_workspace_bytes("e4m3", wl.S, wl.Hkv, wl.D, wl.max_blocks)
    copy = wl.S * wl.max_blocks * wl.Hkv * 16 * wl.D * 2
    assert need >= 2 * copy + wl.S * wl.max_blocks * 4
    assert pk.prefill_workspace_bytes("bf16", wl.S, wl.Hkv, wl.D, wl.max_blocks) == 0
