"""Automatic prefix caching on the host (CPU only): the cascaded block hash
pinned to the published FNV-1a test vectors and checked between the C++
library and the independent Python model; the page's lookup / touch /
commit / evict cycle on worked scenarios (system-prompt reuse, cache salt
and extra hashes isolating requests, leaf-first LRU eviction); and random
operation sequences compared operation by operation."""
import json
import os

import numpy as np
import pytest

from oracle.allocator_model import AllocatorModel, OutOfBlocks, block_hash, fnv1a64, prefix_block_hashes

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "fnv1a64_vectors.json")


@pytest.fixture(scope="module")
def pk():
    from paged_kv_cache_10_gb300 import build, pagedkv
    build.build()
    pagedkv.lib()
    return pagedkv


def test_fnv1a64_matches_published_vectors():
    for v in json.load(open(GOLDEN))["vectors"]:
        assert fnv1a64(v["input"].encode()) == int(v["fnv1a64"], 16)


def test_block_hash_library_equals_model(pk):
    rng = np.random.default_rng(7)
    for _ in range(200):
        parent = int(rng.integers(0, 2**63)) * 2 + int(rng.integers(0, 2))
        toks = rng.integers(-2**31, 2**31, size=int(rng.integers(0, 40))).astype(np.int32)
        ex = rng.integers(0, 2**63, size=int(rng.integers(0, 4))).astype(np.uint64)
        assert pk.block_hash(parent, toks, ex) == block_hash(parent, toks.tolist(), [int(e) for e in ex])
    toks = rng.integers(0, 50000, size=100).astype(np.int32)
    for extras, salt in [((), None), ((12345,), None), ((), 99), ((7, 8), 2**63 + 5)]:
        a = pk.prefix_block_hashes(toks, 16, extras, salt)
        b = prefix_block_hashes(toks.tolist(), 16, list(extras), salt)
        assert a.tolist() == b and len(b) == 6


def test_hash_chain_depends_on_every_part():
    toks = list(range(48))
    base = prefix_block_hashes(toks)
    assert len(set(base)) == 3
    # a change in block 1 changes blocks 1 and 2 (parent chaining), not 0
    t2 = list(toks)
    t2[20] += 1
    h2 = prefix_block_hashes(t2)
    assert h2[0] == base[0] and h2[1] != base[1] and h2[2] != base[2]
    # salt: every block differs (it enters the first, the rest chain from it)
    hs = prefix_block_hashes(toks, salt=1)
    assert all(a != b for a, b in zip(hs, base))
    # extra hash (e.g. an adapter id): every block differs
    he = prefix_block_hashes(toks, extras=[3])
    assert all(a != b for a, b in zip(he, base))


def _both(pk, NB, free=None):
    free = np.arange(NB, dtype=np.int32) if free is None else free
    return pk.Allocator(NB, 16, free), AllocatorModel(NB, 16, free)


def test_system_prompt_reuse_salt_and_extras(pk):
    a, m = _both(pk, 40)
    system = list(range(1000, 1048))  # 3 full blocks
    req_a = system + list(range(50))  # 98 tokens: 6 full blocks + 2
    ha = pk.prefix_block_hashes(np.array(req_a, np.int32))
    assert a.seq_new_prefix(1, ha, len(req_a)) == 0 == m.seq_new_prefix(1, ha.tolist(), len(req_a))
    # after the prefill has written the KV: commit the full blocks
    assert a.commit(1, ha) == 6 == m.commit(1, ha.tolist())
    blocks_a = a.block_table(1)
    a.free(1)
    m.free_seq(1)
    assert a.num_cached() == 6 == m.num_cached()
    assert a.num_free() == 40 == m.num_free()
    # same system prompt: its three blocks are found and shared, no recompute
    req_b = system + list(range(900, 940))
    hb = pk.prefix_block_hashes(np.array(req_b, np.int32))
    assert a.lookup(hb) == 3
    assert a.seq_new_prefix(2, hb, len(req_b)) == 3 == m.seq_new_prefix(2, hb.tolist(), len(req_b))
    assert a.block_table(2)[:3] == blocks_a[:3] == m.block_table(2)[:3]
    assert [a.refcount(b) for b in blocks_a[:3]] == [1, 1, 1]
    assert a.num_cached() == 3 == m.num_cached()  # A's own three blocks are still cached
    # another salt, or another extra hash: nothing shared
    assert a.lookup(pk.prefix_block_hashes(np.array(req_b, np.int32), salt=77)) == 0
    assert a.lookup(pk.prefix_block_hashes(np.array(req_b, np.int32), extras=[5])) == 0
    # a block committed under another hash is refused
    with pytest.raises(pk.PagedKVError):
        a.commit(2, np.array([hb[0] ^ 1], np.uint64))


def test_eviction_is_lru_with_leaf_blocks_first(pk):
    a, m = _both(pk, 10)
    p1 = list(range(64))         # 4 blocks
    p2 = list(range(500, 548))   # 3 blocks
    for sid, toks in ((1, p1), (2, p2)):
        h = pk.prefix_block_hashes(np.array(toks, np.int32))
        a.seq_new_prefix(sid, h, len(toks))
        m.seq_new_prefix(sid, h.tolist(), len(toks))
        a.commit(sid, h)
        m.commit(sid, h.tolist())
    t1, t2 = a.block_table(1), a.block_table(2)
    a.free(1); m.free_seq(1)   # released first: evicted first, leaf end first
    a.free(2); m.free_seq(2)
    assert a.num_cached() == 7 and a.num_free() == 10
    # 3 never-cached blocks go first, then p1's chain from its last block
    a.seq_new(3, 16 * 5)
    m.seq_new(3, 16 * 5)
    got = a.block_table(3)
    assert got == m.block_table(3)
    assert set(got[3:]) == {t1[3], t1[2]}
    assert all(a.block_hash_of(b) is None for b in (t1[3], t1[2]))
    # p1's root blocks and all of p2 are still found
    assert a.lookup(pk.prefix_block_hashes(np.array(p1, np.int32))) == 2
    assert a.lookup(pk.prefix_block_hashes(np.array(p2, np.int32))) == 3
    # touching p2 (a new request) protects it: the next evictions take p1's root
    h2 = pk.prefix_block_hashes(np.array(p2 + [1], np.int32))
    assert a.seq_new_prefix(4, h2, 49) == 3 == m.seq_new_prefix(4, h2.tolist(), 49)
    assert a.block_table(4)[:3] == t2
    a.seq_new(5, 16)
    m.seq_new(5, 16)
    assert a.block_table(5) == m.block_table(5) and a.block_table(5)[0] in (t1[1], t1[0])


def test_seq_new_prefix_is_all_or_nothing(pk):
    a, m = _both(pk, 6)
    toks = np.arange(64, dtype=np.int32)
    h = pk.prefix_block_hashes(toks)
    a.seq_new_prefix(1, h, 64)
    a.commit(1, h)
    a.free(1)
    before = (a.num_free(), a.num_cached(), a.lookup(h))
    with pytest.raises(pk.OutOfBlocks):
        a.seq_new_prefix(2, h[:2], 16 * 9)  # 2 hits + 7 new > 6 - 2
    assert (a.num_free(), a.num_cached(), a.lookup(h)) == before
    a.fail_after(1)
    with pytest.raises(pk.OutOfBlocks):
        a.seq_new_prefix(3, h[:1], 16 * 3)
    assert (a.num_free(), a.num_cached(), a.lookup(h)) == before
    assert a.seq_new_prefix(4, h[:1], 16 * 3) == 1


@pytest.mark.parametrize("seed", range(4))
def test_random_prefix_cache_sequences_match_model(pk, seed):
    rng = np.random.default_rng(500 + seed)
    NB = 60
    free = rng.permutation(NB).astype(np.int32)
    a, m = _both(pk, NB, free)
    templates = [rng.integers(0, 1000, size=int(rng.integers(16, 120))).tolist() for _ in range(4)]
    live, nxt = [], 0
    for step in range(300):
        op = rng.random()
        if op < 0.45:
            t = templates[int(rng.integers(0, 4))]
            toks = t[: int(rng.integers(1, len(t) + 1))] + rng.integers(0, 1000, size=int(rng.integers(0, 40))).tolist()
            salt = None if rng.random() < 0.8 else int(rng.integers(0, 3))
            h = prefix_block_hashes(toks, 16, [], salt)
            hc = pk.prefix_block_hashes(np.array(toks, np.int32), 16, (), salt)
            assert hc.tolist() == h
            try:
                k_model = m.seq_new_prefix(nxt, h, len(toks))
            except OutOfBlocks:
                k_model = None
            try:
                k_lib = a.seq_new_prefix(nxt, hc, len(toks))
            except pk.OutOfBlocks:
                k_lib = None
            assert k_lib == k_model
            if k_lib is not None:
                live.append((nxt, h))
                nxt += 1
        elif op < 0.7 and live:
            sid, h = live[int(rng.integers(0, len(live)))]
            n = int(rng.integers(0, len(h) + 1))
            assert a.commit(sid, np.array(h[:n], np.uint64)) == m.commit(sid, h[:n])
        elif op < 0.9 and live:
            sid, _ = live.pop(int(rng.integers(0, len(live))))
            a.free(sid)
            m.free_seq(sid)
        elif live:
            sid, h = live[int(rng.integers(0, len(live)))]
            try:
                want = m.append_slot(sid)
            except OutOfBlocks:
                want = None
            try:
                got = a.append_slot(sid)
            except pk.OutOfBlocks:
                got = None
            assert (got is None) == (want is None)
            if got is not None:
                assert got[0] == want[0]
        assert a.num_free() == m.num_free() and a.num_cached() == m.num_cached()
        for sid, _ in live:
            assert a.block_table(sid) == m.block_table(sid)
    for b in range(NB):
        assert a.block_hash_of(b) == m.hash_of.get(b)
        assert a.refcount(b) == m.ref[b]
    a.reset_prefix_cache()
    m.reset_prefix_cache()
    assert a.num_cached() == 0 == m.num_cached() and a.num_free() == m.num_free()
