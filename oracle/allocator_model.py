"""Independent pure-Python model of the host block allocator.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).  It is written from the
pages, not from the C++ allocator, and is compared against it operation by
operation.

Sources:
  * "vLLM：大语言模型推理与服务库" section 4.2, "Block Pool": a pool pre-split into
    fixed-size blocks, a free list, O(1) allocate (take the LAST free id, fail
    when empty) and O(1) free (append the id to the free list).
  * same page, section 4.3: a block is allocated only when the current last
    block is full, then the block table is updated and the KV written.
  * "vLLM 高性能大语言模型推理引擎深度技术评估与分布式架构展望", section
    "束搜索与并行采样的三大调度原语": fork copies the parent's block table (same
    physical ids); append with copy-on-write gives a sequence a private copy
    of a shared block it is about to modify; free decrements reference
    counts and a block whose count reaches zero goes back to the free list.
  * "vLLM 深度解析：从 PagedAttention 到生产部署", "Prefix Caching 与
    Copy-on-Write": shared blocks carry a reference count > 1 and are copied
    only when modified.

  * "vLLM 高性能大语言模型推理引擎深度技术评估与分布式架构展望", sections
    "基于级联哈希的缓存结构设计" and "缓存分配、触碰与驱逐闭环" (automatic
    prefix caching): a full block is keyed by hash(parent hash, block
    tokens, extra hashes), the cache salt joining the first block's hash;
    lookup finds the cached leading blocks of a prompt, touch takes a
    reference on them and takes them off the free queue, a filled block is
    committed to the table, and when blocks run short the least recently
    used count-0 cached blocks are evicted, leaf blocks of long chains first.

Readings: the free list is a stack (the C++ sketch's back()/pop_back()); a
write into a *partial* last block whose count is > 1 copies it first, a full
last block just gets a fresh block; blocks of a freed sequence are released
from its last block to its first; OOM leaves the state unchanged.
Prefix cache: the hash is 64-bit FNV-1a over the little-endian bytes of
parent (8), token count (4), token ids (4 each), extra count (4), extras (8
each); the salt is appended to the first block's extras.  Never-cached free
blocks are used before any cached one is evicted; eviction takes the cached
count-0 block released longest ago -- with a sequence released last block
first, that is LRU with the leaf end of a chain before its root.  A commit
skips a hash that another block already holds.
"""
from __future__ import annotations


class OutOfBlocks(Exception):
    pass


FNV_OFFSET = 0xCBF29CE484222325
FNV_PRIME = 0x100000001B3
MASK64 = (1 << 64) - 1


def fnv1a64(data: bytes) -> int:
    """64-bit FNV-1a: for each byte, xor it in, then multiply by the prime."""
    h = FNV_OFFSET
    for b in data:
        h ^= b
        h = (h * FNV_PRIME) & MASK64
    return h


def block_hash(parent: int, tokens, extras=()) -> int:
    data = bytearray()
    data += int(parent).to_bytes(8, "little")
    data += len(tokens).to_bytes(4, "little")
    for t in tokens:
        data += (int(t) & 0xFFFFFFFF).to_bytes(4, "little")
    data += len(extras).to_bytes(4, "little")
    for e in extras:
        data += int(e).to_bytes(8, "little")
    return fnv1a64(bytes(data))


def prefix_block_hashes(tokens, block_size=16, extras=(), salt=None) -> list:
    out, parent = [], 0
    for i in range(len(tokens) // block_size):
        ex = list(extras) + ([salt] if (i == 0 and salt is not None) else [])
        parent = block_hash(parent, tokens[i * block_size:(i + 1) * block_size], ex)
        out.append(parent)
    return out


class AllocatorModel:
    def __init__(self, num_blocks: int, block_size: int, free_order=None):
        self.block_size = block_size
        self.num_blocks = num_blocks
        # allocation takes from the end of this list
        self.free = list(range(num_blocks)) if free_order is None else [int(x) for x in free_order]
        assert sorted(self.free) == list(range(num_blocks))
        self.ref = [0] * num_blocks
        self.tables: dict[int, list[int]] = {}
        self.lens: dict[int, int] = {}
        # prefix cache
        self.hash_of: dict[int, int] = {}    # committed block -> hash
        self.cached: dict[int, int] = {}     # hash -> block
        self.evictable: dict[int, int] = {}  # count-0 committed block -> release time
        self.clock = 0

    # -- helpers
    def _take(self) -> int:
        if self.free:
            blk = self.free.pop()
        elif self.evictable:
            blk = min(self.evictable, key=self.evictable.get)  # released longest ago
            del self.evictable[blk]
            del self.cached[self.hash_of.pop(blk)]
        else:
            raise OutOfBlocks()
        self.ref[blk] = 1
        return blk

    def _release(self, blk: int) -> None:
        self.ref[blk] -= 1
        if self.ref[blk] == 0:
            if blk in self.hash_of:
                self.evictable[blk] = self.clock
                self.clock += 1
            else:
                self.free.append(blk)

    # -- primitives
    def seq_new(self, seq: int, num_tokens: int) -> None:
        assert seq not in self.tables
        need = -(-num_tokens // self.block_size)
        if need > self.num_free():
            raise OutOfBlocks()
        self.tables[seq] = [self._take() for _ in range(need)]
        self.lens[seq] = num_tokens

    def fork(self, parent: int, child: int) -> None:
        assert child not in self.tables
        self.tables[child] = list(self.tables[parent])
        self.lens[child] = self.lens[parent]
        for blk in self.tables[child]:
            self.ref[blk] += 1

    def append_slot(self, seq: int):
        """Returns (slot, cow) where cow is None or (src, dst)."""
        table = self.tables[seq]
        pos = self.lens[seq]
        off = pos % self.block_size
        cow = None
        if off == 0:
            table.append(self._take())
        else:
            last = table[-1]
            if self.ref[last] > 1:
                dst = self._take()
                self.ref[last] -= 1
                table[-1] = dst
                cow = (last, dst)
        self.lens[seq] = pos + 1
        return table[-1] * self.block_size + off, cow

    def free_seq(self, seq: int) -> None:
        table = self.tables.pop(seq)
        self.lens.pop(seq)
        for blk in reversed(table):
            self._release(blk)

    def move_to(self, other: "AllocatorModel", seq: int):
        """Moves seq into another pool (swap out / in): one new block per
        block, all held by this sequence alone; returns (old, new) pairs."""
        table = self.tables[seq]
        assert all(self.ref[b] == 1 for b in table)
        if len(table) > other.num_free():
            raise OutOfBlocks()
        new = [other._take() for _ in table]
        other.tables[seq] = new
        other.lens[seq] = self.lens[seq]
        pairs = list(zip(table, new))
        self.free_seq(seq)
        return pairs

    # -- views
    def block_table(self, seq: int) -> list[int]:
        return list(self.tables[seq])

    def num_free(self) -> int:
        return len(self.free) + len(self.evictable)

    # -- prefix cache
    def lookup(self, hashes) -> int:
        k = 0
        while k < len(hashes) and int(hashes[k]) in self.cached:
            k += 1
        return k

    def seq_new_prefix(self, seq: int, hashes, num_tokens: int) -> int:
        assert seq not in self.tables and len(hashes) * self.block_size <= num_tokens
        k = self.lookup(hashes)
        hits = [self.cached[int(h)] for h in hashes[:k]]
        need = -(-num_tokens // self.block_size) - k
        if need > self.num_free() - sum(1 for b in hits if b in self.evictable):
            raise OutOfBlocks()
        for b in hits:  # touch
            self.evictable.pop(b, None)
            self.ref[b] += 1
        self.tables[seq] = hits + [self._take() for _ in range(need)]
        self.lens[seq] = num_tokens
        return k

    def commit(self, seq: int, hashes) -> int:
        table = self.tables[seq]
        assert len(hashes) * self.block_size <= self.lens[seq]
        for i, h in enumerate(hashes):
            if table[i] in self.hash_of and self.hash_of[table[i]] != int(h):
                raise ValueError("block committed under another hash")
        n = 0
        for i, h in enumerate(hashes):
            b, h = table[i], int(h)
            if b in self.hash_of or h in self.cached:
                continue
            self.hash_of[b] = h
            self.cached[h] = b
            n += 1
        return n

    def num_cached(self) -> int:
        return len(self.evictable)

    def reset_prefix_cache(self) -> None:
        for b in sorted(self.evictable, key=self.evictable.get):
            self.free.append(b)
        self.evictable.clear()
        self.cached.clear()
        self.hash_of.clear()
