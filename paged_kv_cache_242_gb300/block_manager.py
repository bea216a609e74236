"""Host-side KV block manager: block tables, free list, reference counts.

This is the scheduler-side half of paged KV storage described in "vLLM
PagedAttention & continuous batching" (sections "PagedAttention: fixed
blocks, non-contiguous physical memory" and "Sharing with reference counts
and copy-on-write"):

* a block table maps each logical block of a sequence to a physical block;
  logical blocks fill left to right and a new physical block is allocated
  only when the previous one is full;
* every physical block carries a reference count; ``fork`` maps a child's
  logical blocks onto the parent's physical blocks;
* a sequence that must write into a block whose count is above one gets a
  freshly allocated block, the old block is copied into it (a copy-on-write
  pair for the ``copy_blocks`` kernel) and the old count drops by one;
* ``free`` drops every reference of a sequence; a block whose count reaches
  zero returns to the free list (and never while still referenced).

The manager produces the device inputs of the kernels: block tables,
sequence lengths, slot mappings (slot = physical block * B + offset) and
copy-on-write (src, dst) pairs.  The kernels see physical block ids only,
never the sharing policy.
"""
from __future__ import annotations

from collections import deque
from typing import Dict, Iterable, List, Optional, Sequence, Tuple

import numpy as np


class OutOfBlocks(RuntimeError):
    """The pool has no free physical block left."""


class BlockManager:
    def __init__(self, num_blocks: int, block_size: int,
                 free_order: Optional[Iterable[int]] = None) -> None:
        if num_blocks <= 0 or block_size <= 0:
            raise ValueError("num_blocks and block_size must be positive")
        self.num_blocks = int(num_blocks)
        self.block_size = int(block_size)
        order = list(range(num_blocks)) if free_order is None else [int(b) for b in free_order]
        if sorted(order) != list(range(num_blocks)):
            raise ValueError("free_order must be a permutation of range(num_blocks)")
        self._free = deque(order)
        self.refcount = np.zeros(num_blocks, dtype=np.int64)
        self.tables: Dict[int, List[int]] = {}
        self.lengths: Dict[int, int] = {}

    # -- pool -------------------------------------------------------------
    @property
    def num_free(self) -> int:
        return len(self._free)

    def _allocate(self) -> int:
        if not self._free:
            raise OutOfBlocks("no free physical block")
        block = self._free.popleft()
        assert self.refcount[block] == 0
        self.refcount[block] = 1
        return block

    def _drop(self, block: int) -> None:
        if self.refcount[block] <= 0:
            raise RuntimeError(f"reference count of block {block} would go negative")
        self.refcount[block] -= 1
        if self.refcount[block] == 0:
            self._free.append(block)

    # -- sequences --------------------------------------------------------
    def _slot(self, seq_id: int, position: int) -> int:
        table = self.tables[seq_id]
        return table[position // self.block_size] * self.block_size + position % self.block_size

    def add_sequence(self, seq_id: int, num_tokens: int) -> List[int]:
        """Allocate ceil(n / B) blocks for an n-token prompt; return its slots."""
        if seq_id in self.tables:
            raise KeyError(f"sequence {seq_id} exists")
        if num_tokens < 0:
            raise ValueError("num_tokens must be >= 0")
        needed = -(-num_tokens // self.block_size)
        if needed > len(self._free):
            raise OutOfBlocks(f"prompt needs {needed} blocks, {len(self._free)} free")
        self.tables[seq_id] = [self._allocate() for _ in range(needed)]
        self.lengths[seq_id] = num_tokens
        return [self._slot(seq_id, p) for p in range(num_tokens)]

    def append_slot(self, seq_id: int) -> Tuple[int, Optional[Tuple[int, int]]]:
        """Reserve the slot of the next token of ``seq_id``.

        Returns ``(slot, cow)`` where ``cow`` is a (src, dst) block pair that
        must be copied before the write, or None.
        """
        table = self.tables[seq_id]
        position = self.lengths[seq_id]
        cow = None
        if position % self.block_size == 0:
            table.append(self._allocate())
        else:
            last = table[-1]
            if self.refcount[last] > 1:
                fresh = self._allocate()
                self.refcount[last] -= 1  # still referenced by others: never freed here
                table[-1] = fresh
                cow = (last, fresh)
        self.lengths[seq_id] = position + 1
        return self._slot(seq_id, position), cow

    def fork(self, parent: int, child: int) -> None:
        """The child shares every physical block of the parent."""
        if child in self.tables:
            raise KeyError(f"sequence {child} exists")
        self.tables[child] = list(self.tables[parent])
        self.lengths[child] = self.lengths[parent]
        for block in self.tables[child]:
            self.refcount[block] += 1

    def free(self, seq_id: int) -> None:
        """Drop every reference held by ``seq_id`` (cancellation / completion)."""
        for block in self.tables.pop(seq_id):
            self._drop(block)
        del self.lengths[seq_id]

    # -- device inputs ----------------------------------------------------
    def block_table_array(self, seq_ids: Sequence[int], max_blocks: Optional[int] = None,
                          pad: int = 0) -> np.ndarray:
        width = max((len(self.tables[s]) for s in seq_ids), default=0)
        if max_blocks is None:
            max_blocks = max(width, 1)
        if width > max_blocks:
            raise ValueError("max_blocks smaller than the longest block table")
        out = np.full((len(seq_ids), max_blocks), pad, dtype=np.int32)
        for row, s in enumerate(seq_ids):
            table = self.tables[s]
            out[row, :len(table)] = table
        return out

    def seq_lens_array(self, seq_ids: Sequence[int]) -> np.ndarray:
        return np.asarray([self.lengths[s] for s in seq_ids], dtype=np.int32)
