"""Host block allocator (C++, through the C ABI) against the independent
Python model in ``oracle/allocator_model.py`` and the pages' worked examples.
CPU only: the allocator touches no device memory.
"""
import json
import os

import numpy as np
import pytest

from oracle.allocator_model import AllocatorModel, OutOfBlocks

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "block_table_examples.json")


@pytest.fixture(scope="module")
def pk():
    from paged_kv_cache_10_gb300 import build, pagedkv
    build.build()
    return pagedkv


def test_worked_examples_block_counts(pk):
    g = json.load(open(GOLDEN))
    for ex in g["examples"]:
        a = pk.Allocator(64, ex["block_size"])
        a.seq_new(7, ex["tokens"])
        assert len(a.block_table(7)) == ex["blocks"], ex["cite"]
        if "logical_ranges" in ex:
            for j, (lo, hi) in enumerate(ex["logical_ranges"]):
                assert lo // 16 == j and hi // 16 == j
        m = AllocatorModel(64, ex["block_size"])
        m.seq_new(7, ex["tokens"])
        assert len(m.block_table(7)) == ex["blocks"]


def test_worked_example_prefix_sharing(pk):
    ps = json.load(open(GOLDEN))["prefix_sharing"]
    a = pk.Allocator(32, ps["block_size"])
    a.seq_new(100, ps["prefix_tokens"])
    prefix = a.block_table(100)
    assert len(prefix) == ps["prefix_blocks"]
    for r in range(len(ps["requests"])):
        a.fork(100, r)
    a.free(100)
    for blk in prefix:
        assert a.refcount(blk) == ps["shared_refcount"]
    for r in range(len(ps["requests"])):
        assert a.block_table(r) == prefix
    # the first request to write into the shared partial block gets a private copy
    slot, cow = a.append_slot(0)
    assert cow is not None and cow[0] == prefix[-1]
    assert a.refcount(prefix[-1]) == ps["shared_refcount"] - 1
    assert slot == cow[1] * 16 + ps["prefix_tokens"] % 16


def test_waste_bound_and_on_demand_growth(pk):
    a = pk.Allocator(1000, 16)
    a.seq_new(1, 0)
    for L in range(1, 200):
        slot, cow = a.append_slot(1)
        assert cow is None
        n = len(a.block_table(1))
        assert n == -(-L // 16)
        assert n * 16 - L <= 15  # at most b-1 unused slots, all in the last block
        assert slot == a.block_table(1)[-1] * 16 + (L - 1) % 16


def _random_ops(rng, steps, num_blocks):
    live, next_id, ops = [], 0, []
    for _ in range(steps):
        r = rng.random()
        if r < 0.2 or not live:
            ops.append(("new", next_id, int(rng.integers(0, 70))))
            live.append(next_id)
            next_id += 1
        elif r < 0.35:
            ops.append(("fork", int(rng.choice(live)), next_id))
            live.append(next_id)
            next_id += 1
        elif r < 0.85:
            ops.append(("append", int(rng.choice(live))))
        elif r < 0.93:
            ops.append(("batch", [int(x) for x in rng.choice(live, size=min(len(live), 5), replace=False)]))
        else:
            s = int(rng.choice(live))
            ops.append(("free", s))
            live.remove(s)
    return ops


def _check_invariants(pk_alloc, model, num_blocks):
    refs = [pk_alloc.refcount(b) for b in range(num_blocks)]
    assert refs == model.ref
    assert pk_alloc.num_free() == model.num_free()
    counted = [0] * num_blocks
    for seq, table in model.tables.items():
        assert pk_alloc.block_table(seq) == table
        assert pk_alloc.seq_len(seq) == model.lens[seq]
        assert len(table) == -(-model.lens[seq] // 16)
        for b in table:
            counted[b] += 1
    assert counted == refs  # refcount == number of table references
    free = set(model.free)
    assert all((refs[b] == 0) == (b in free) for b in range(num_blocks))


@pytest.mark.parametrize("seed", range(6))
def test_random_operation_sequences_match_model(pk, seed):
    rng = np.random.default_rng(seed)
    NB = 48
    order = rng.permutation(NB).astype(np.int32)
    a = pk.Allocator(NB, 16, order)
    m = AllocatorModel(NB, 16, order)
    for op in _random_ops(rng, 400, NB):
        kind = op[0]
        if kind == "new":
            try:
                m.seq_new(op[1], op[2])
                ok = True
            except OutOfBlocks:
                ok = False
            if ok:
                a.seq_new(op[1], op[2])
            else:
                with pytest.raises(pk.OutOfBlocks):
                    a.seq_new(op[1], op[2])
                m.tables.pop(op[1], None)
                m.lens.pop(op[1], None)
        elif kind == "fork":
            if op[1] not in m.tables:
                continue
            m.fork(op[1], op[2])
            a.fork(op[1], op[2])
        elif kind == "append":
            if op[1] not in m.tables:
                continue
            try:
                want = m.append_slot(op[1])
            except OutOfBlocks:
                with pytest.raises(pk.OutOfBlocks):
                    a.append_slot(op[1])
                continue
            assert a.append_slot(op[1]) == want
        elif kind == "batch":
            ids = [s for s in op[1] if s in m.tables]
            snapshot = (list(m.free), list(m.ref), {k: list(v) for k, v in m.tables.items()}, dict(m.lens))
            want_slots, want_pairs = [], []
            try:
                for s in ids:
                    slot, cow = m.append_slot(s)
                    want_slots.append(slot)
                    if cow:
                        want_pairs.append(cow)
                oom = False
            except OutOfBlocks:
                oom = True
                m.free, m.ref, m.tables, m.lens = snapshot
            if oom:
                with pytest.raises(pk.OutOfBlocks):
                    a.append_batch(ids)
            else:
                slots, pairs = a.append_batch(ids)
                assert slots.tolist() == want_slots
                assert [tuple(p) for p in pairs.tolist()] == want_pairs
        elif kind == "free":
            if op[1] not in m.tables:
                continue
            m.free_seq(op[1])
            a.free(op[1])
        _check_invariants(a, m, NB)


def test_oom_leaves_state_unchanged_and_fault_injection(pk):
    a = pk.Allocator(4, 16)
    a.seq_new(1, 40)  # 3 blocks, last one partial
    with pytest.raises(pk.OutOfBlocks):
        a.seq_new(2, 33)  # needs 3, 1 free
    assert a.num_free() == 1 and a.num_seqs() == 1
    a.fork(1, 3)  # the partial block is now shared
    snap = lambda: ([a.block_table(s) for s in (1, 3)], [a.seq_len(s) for s in (1, 3)],
                    [a.refcount(b) for b in range(4)], a.num_free())
    before = snap()
    a.fail_after(1)  # the copy-on-write allocation of seq 1 fails
    with pytest.raises(pk.OutOfBlocks):
        a.append_batch([1, 3])
    assert snap() == before
    slots, pairs = a.append_batch([1, 3])  # injection was one-shot
    assert len(pairs) == 1 and pairs[0, 0] == before[0][0][-1]
    assert slots[1] == before[0][0][-1] * 16 + 40 % 16  # last holder writes in place


def test_batch_rollback_restores_exact_state(pk):
    a = pk.Allocator(10, 16)
    a.seq_new(0, 16)   # full block -> next append allocates
    a.seq_new(1, 16)
    a.seq_new(2, 16)
    a.seq_new(3, 5)
    before = ([a.block_table(s) for s in range(4)], [a.seq_len(s) for s in range(4)],
              [a.refcount(b) for b in range(10)], a.num_free())
    a.fail_after(3)  # seq 0 and 1 get blocks, seq 2's allocation fails
    with pytest.raises(pk.OutOfBlocks):
        a.append_batch([0, 1, 2, 3])
    after = ([a.block_table(s) for s in range(4)], [a.seq_len(s) for s in range(4)],
             [a.refcount(b) for b in range(10)], a.num_free())
    assert after == before
    # and the free-list order is intact: the next allocations match a fresh model
    m = AllocatorModel(10, 16)
    for s, n in ((0, 16), (1, 16), (2, 16), (3, 5)):
        m.seq_new(s, n)
    slots, _ = a.append_batch([0, 1, 2, 3])
    assert slots.tolist() == [m.append_slot(s)[0] for s in range(4)]


def test_invalid_calls(pk):
    a = pk.Allocator(8, 16)
    with pytest.raises(pk.PagedKVError):
        a.fork(5, 6)  # unknown parent
    a.seq_new(1, 3)
    with pytest.raises(pk.PagedKVError):
        a.seq_new(1, 3)  # duplicate id
    with pytest.raises(pk.PagedKVError):
        a.append_batch([1, 1])  # a sequence twice in one batch
    a.fork(1, 2)
    with pytest.raises(pk.PagedKVError):
        a.extend(2, 4)  # would write into a shared partial block
    with pytest.raises(pk.PagedKVError):
        pk.Allocator(4, 16, [0, 1, 1, 3])  # not a permutation
    tables, lens = a.export([1, -1, 2], 2)
    assert lens.tolist() == [3, 0, 3] and tables[1].tolist() == [-1, -1]
    with pytest.raises(pk.PagedKVError):
        a.export([1], 0)


def test_prefix_share_workload_script_produces_copy_on_write(pk):
    from paged_kv_cache_10_gb300 import workloads
    wl = workloads.prefix_share()
    a = pk.Allocator(wl.NB, 16, wl.free_order)
    pk.apply_setup(a, wl.setup)
    m = AllocatorModel(wl.NB, 16, wl.free_order)
    for op in wl.setup:
        if op[0] == "new":
            m.seq_new(op[1], op[2])
        elif op[0] == "fork":
            m.fork(op[1], op[2])
        elif op[0] == "extend":
            for _ in range(op[2]):
                assert m.append_slot(op[1])[1] is None
        else:
            m.free_seq(op[1])
    prefix = a.block_table(0)[:128]
    assert all(a.refcount(b) == 128 for b in prefix)
    slots, pairs = a.append_batch(wl.step_seqs)
    want = [m.append_slot(s) for s in wl.step_seqs]
    assert slots.tolist() == [w[0] for w in want]
    assert [tuple(p) for p in pairs.tolist()] == [w[1] for w in want if w[1]]
    assert 50 <= len(pairs) <= 64
    tables, lens = a.export(np.arange(wl.S), wl.max_blocks)
    assert lens.tolist() == wl.seq_lens


def _groups_model(tables, lens, min_blocks, b=16):
    """Independent restatement of the grouping rule for cascade decode."""
    order, buckets = [], {}
    for i, (t, L) in enumerate(zip(tables, lens)):
        if t is None or L // b < min_blocks:
            continue
        if t[0] not in buckets:
            buckets[t[0]] = []
            order.append(t[0])
        buckets[t[0]].append(i)
    out = []
    for key in order:
        rows = buckets[key]
        if len(rows) < 2:
            continue
        full = min(lens[r] // b for r in rows)
        lcp = 0
        while lcp < full and len({tables[r][lcp] for r in rows}) == 1:
            lcp += 1
        if lcp >= min_blocks:
            out.append((lcp, rows))
    return out


@pytest.mark.parametrize("seed", range(4))
def test_prefix_groups_match_model(pk, seed):
    from paged_kv_cache_10_gb300 import workloads
    wl = workloads.fork_groups("g", 50 + seed, [(64, 3), (160, 5), (32, 1)], 4, 8, 2, 128)
    a = pk.Allocator(wl.NB, 16, wl.free_order)
    pk.apply_setup(a, wl.setup)
    a.append_batch(wl.step_seqs)
    rows = list(range(wl.S)) + [-1]
    for min_blocks in (1, 2, 4, 10):
        g = a.prefix_groups(rows, min_blocks)
        tables = [a.block_table(r) for r in range(wl.S)] + [None]
        lens = [a.seq_len(r) for r in range(wl.S)] + [0]
        want = _groups_model(tables, lens, min_blocks)
        got = [(int(g.group_blocks[k]), g.group_members[g.group_offsets[k]:g.group_offsets[k + 1]].tolist())
               for k in range(g.num_groups)]
        assert got == want
        for k, (lcp, members) in enumerate(got):
            assert all(g.seq_group[r] == k for r in members)
        grouped = {r for _, ms in got for r in ms}
        assert all(g.seq_group[r] == -1 for r in range(len(rows)) if r not in grouped)


@pytest.mark.parametrize("seed", range(3))
def test_swap_out_and_in_match_model(pk, seed):
    rng = np.random.default_rng(100 + seed)
    dev, host = pk.Allocator(40, 16, rng.permutation(40)), pk.Allocator(24, 16, rng.permutation(24))
    mdev, mhost = AllocatorModel(40, 16, dev._order), AllocatorModel(24, 16, host._order)
    for s in range(6):
        n = int(rng.integers(1, 90))
        dev.seq_new(s, n)
        mdev.seq_new(s, n)
    dev.fork(0, 9)
    mdev.fork(0, 9)
    with pytest.raises(pk.PagedKVError):
        dev.swap_out(host, 0)  # shared blocks cannot move
    for s in (1, 3, 4):
        got = dev.swap_out(host, s)
        assert [tuple(x) for x in got.tolist()] == mdev.move_to(mhost, s)
    assert dev.num_free() == mdev.num_free() and host.num_free() == mhost.num_free()
    slot, _ = dev.append_slot(2)  # the device pool keeps working meanwhile
    assert slot == mdev.append_slot(2)[0]
    for s in (3, 1):
        got = dev.swap_in(host, s)  # pairs are (device block, host block)
        want = [(new, old) for old, new in mhost.move_to(mdev, s)]
        assert [tuple(x) for x in got.tolist()] == want
        assert dev.block_table(s) == mdev.block_table(s) and dev.seq_len(s) == mdev.lens[s]
    assert [dev.refcount(b) for b in range(40)] == mdev.ref
    assert [host.refcount(b) for b in range(24)] == mhost.ref


def test_swap_out_is_all_or_nothing(pk):
    dev, host = pk.Allocator(20, 16), pk.Allocator(2, 16)
    dev.seq_new(1, 70)  # 5 blocks, host has 2
    before = (dev.block_table(1), dev.num_free(), host.num_free())
    with pytest.raises(pk.OutOfBlocks):
        dev.swap_out(host, 1)
    assert (dev.block_table(1), dev.num_free(), host.num_free()) == before


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_append_tokens_matches_model(pk, seed):
    """Chunked-prefill slot reservation equals the model's append_slot one
    token at a time, including copy-on-write of a shared partial block by a
    sequence's first new token."""
    rng = np.random.default_rng(300 + seed)
    NB = 200
    free = rng.permutation(NB).astype(np.int32)
    a, m = pk.Allocator(NB, 16, free), AllocatorModel(NB, 16, free)
    for s in range(6):
        L = int(rng.integers(0, 90))
        a.seq_new(s, L)
        m.seq_new(s, L)
    a.fork(2, 10)
    m.fork(2, 10)
    seqs = [10, 0, 3, 2, 5]
    counts = [int(rng.integers(0, 60)) for _ in seqs]
    slots, pairs = a.append_tokens(seqs, counts)
    want_slots, want_pairs = [], []
    for s, c in zip(seqs, counts):
        for _ in range(c):
            slot, cow = m.append_slot(s)
            want_slots.append(slot)
            if cow:
                want_pairs.append(cow)
    assert slots.tolist() == want_slots
    assert [tuple(p) for p in pairs.tolist()] == want_pairs
    for s in list(range(6)) + [10]:
        assert a.block_table(s) == m.block_table(s)
    assert a.num_free() == m.num_free()


def test_append_tokens_is_all_or_nothing(pk):
    a = pk.Allocator(6, 16)
    a.seq_new(0, 20)
    a.seq_new(1, 5)
    before = (a.block_table(0), a.block_table(1), a.num_free())
    with pytest.raises(pk.OutOfBlocks):
        a.append_tokens([0, 1], [30, 60])  # needs 2 + 4 blocks, 3 free
    assert (a.block_table(0), a.block_table(1), a.num_free()) == before
    with pytest.raises(pk.PagedKVError):
        a.append_tokens([0, 0], [1, 1])  # a sequence twice
    with pytest.raises(pk.PagedKVError):
        a.append_tokens([0], [-1])
