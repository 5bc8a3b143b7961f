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
