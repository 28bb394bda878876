"""Physical block pool and per-sequence block tables (oracle; test infrastructure only).

Sources:

* "Series 03: why the KV cache eats memory ..." section 3.1: the cache is cut
  into fixed-size physical blocks (16 tokens by default) kept in one pool;
  each request keeps a block table mapping its logical block i to a physical
  block, and physical blocks need not be contiguous.
* Same page, section 3.2: blocks are taken from a global free list on demand,
  one more whenever the current block is full, so a sequence wastes at most
  the unused tail of its last block.
* Same page, section 3.3: several block tables may reference one physical
  block (shared prefixes, beam search); such blocks stay shared until a write.
* "What a KV cache is ..." section 3.2: the pool is preallocated at start-up
  (2048 blocks of 16 tokens = 32768 tokens); a 1200-token prompt takes 75
  blocks.  Section 4.2: writing past the capacity raises RuntimeError.

Allocation policy (a reading; the pages fix none): the free list is a LIFO
stack whose initial order hands out block 0 first, then 1, 2, ...; a freed
block is the next one handed out.  The C-ABI host pool follows the same policy
so the two can be compared id for id.
"""
from __future__ import annotations


class PoolExhausted(RuntimeError):
    """Raised when an allocation finds no free block (the cache overflow of
    "What a KV cache is ..." section 4.2 is a RuntimeError too)."""


def blocks_needed(n_tokens: int, block_size: int = 16) -> int:
    """Blocks holding ``n_tokens`` tokens: the ceiling of n / block_size."""
    if n_tokens < 0 or block_size <= 0:
        raise ValueError("n_tokens must be >= 0 and block_size > 0")
    return -(-n_tokens // block_size)


class BlockPool:
    """A pool of ``num_blocks`` physical block ids with reference counts."""

    def __init__(self, num_blocks: int, block_size: int = 16) -> None:
        if num_blocks < 0 or block_size <= 0:
            raise ValueError("num_blocks must be >= 0 and block_size > 0")
        self.num_blocks = num_blocks
        self.block_size = block_size
        self._free = list(range(num_blocks - 1, -1, -1))   # top of stack = 0
        self._ref = [0] * num_blocks

    @property
    def num_free(self) -> int:
        return len(self._free)

    @property
    def capacity_tokens(self) -> int:
        return self.num_blocks * self.block_size

    def refcount(self, block_id: int) -> int:
        return self._ref[block_id]

    def alloc(self) -> int:
        if not self._free:
            raise PoolExhausted("no free KV block")
        block_id = self._free.pop()
        self._ref[block_id] = 1
        return block_id

    def incref(self, block_id: int) -> None:
        if not (0 <= block_id < self.num_blocks) or self._ref[block_id] == 0:
            raise ValueError(f"block {block_id} is not allocated")
        self._ref[block_id] += 1

    def decref(self, block_id: int) -> None:
        if not (0 <= block_id < self.num_blocks) or self._ref[block_id] == 0:
            raise ValueError(f"block {block_id} is not allocated")
        self._ref[block_id] -= 1
        if self._ref[block_id] == 0:
            self._free.append(block_id)


class SequenceTable:
    """One sequence's block table, grown on demand as tokens are appended."""

    def __init__(self, pool: BlockPool) -> None:
        self.pool = pool
        self.blocks: list[int] = []
        self.length = 0

    def reserve(self, n_new: int) -> None:
        """Make room for ``n_new`` more tokens, taking blocks only when the
        last one is full.  On exhaustion nothing is changed and
        PoolExhausted is raised."""
        need = blocks_needed(self.length + n_new, self.pool.block_size) - len(self.blocks)
        if need > self.pool.num_free:
            raise PoolExhausted(f"need {need} blocks, {self.pool.num_free} free")
        for _ in range(need):
            self.blocks.append(self.pool.alloc())

    def append_tokens(self, n_new: int) -> list[int]:
        """Reserve room, advance the length and return the logical positions
        the new tokens occupy."""
        self.reserve(n_new)
        start = self.length
        self.length += n_new
        return list(range(start, self.length))

    def share_prefix_from(self, other: "SequenceTable", n_blocks: int) -> None:
        """Reference the first ``n_blocks`` physical blocks of ``other``
        (copy-free sharing, "Series 03 ..." section 3.3).  Only whole blocks
        are shared, so the new sequence starts at a block boundary."""
        if self.blocks:
            raise ValueError("prefix sharing starts an empty table")
        for block_id in other.blocks[:n_blocks]:
            self.pool.incref(block_id)
            self.blocks.append(block_id)
        self.length = n_blocks * self.pool.block_size

    def fork(self) -> "SequenceTable":
        """A new sequence that shares every block of this one: a beam-search
        branch or a parallel sample ("Series 03 ..." section 3.3: branches
        share the prefix blocks and nothing is copied).  Same length, same
        physical blocks, each block's reference count one higher."""
        child = SequenceTable(self.pool)
        for block_id in self.blocks:
            self.pool.incref(block_id)
            child.blocks.append(block_id)
        child.length = self.length
        return child

    def prepare_write(self, position: int):
        """Copy-on-write before writing the token at logical ``position``
        ("Series 03 ..." section 3.3: when a branch writes its first token of
        its own into a shared block, a new block is taken, the old contents
        are copied into it and the token is written there; the other branches
        keep the old block).  If the block holding ``position`` is shared
        (reference count > 1), take a fresh block, point this table at it,
        drop one reference from the old block and return ``(old, new)``: the
        caller copies block ``old`` into block ``new`` before writing.
        A private block needs nothing: None.  On exhaustion nothing changes
        and PoolExhausted is raised."""
        logical_block = position // self.pool.block_size
        if not (0 <= logical_block < len(self.blocks)):
            raise ValueError(f"position {position} lies outside the reserved blocks")
        old = self.blocks[logical_block]
        if self.pool.refcount(old) <= 1:
            return None
        new = self.pool.alloc()
        self.pool.decref(old)
        self.blocks[logical_block] = new
        return old, new

    def release(self) -> None:
        for block_id in self.blocks:
            self.pool.decref(block_id)
        self.blocks = []
        self.length = 0

    def wasted_slots(self) -> int:
        return len(self.blocks) * self.pool.block_size - self.length
