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

Readings: the free list is a stack (the C++ sketch's back()/pop_back()); a
write into a *partial* last block whose count is > 1 copies it first, a full
last block just gets a fresh block; blocks of a freed sequence are released
from its last block to its first; OOM leaves the state unchanged.
"""
from __future__ import annotations


class OutOfBlocks(Exception):
    pass


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

    # -- helpers
    def _take(self) -> int:
        if not self.free:
            raise OutOfBlocks()
        blk = self.free.pop()
        self.ref[blk] = 1
        return blk

    def _release(self, blk: int) -> None:
        self.ref[blk] -= 1
        if self.ref[blk] == 0:
            self.free.append(blk)

    # -- primitives
    def seq_new(self, seq: int, num_tokens: int) -> None:
        assert seq not in self.tables
        need = -(-num_tokens // self.block_size)
        if need > len(self.free):
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
        if len(table) > len(other.free):
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
        return len(self.free)
