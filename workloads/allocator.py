"""Host-side block allocator for a paged KV pool (harness logic, no GPU).

Follows the block manager described on habr.com/ru/articles/1021832, section 4
"Вспомним PagedAttention" (fixed 16-token blocks; a block table maps logical to
physical blocks; physical blocks are handed out in any order, "scattered, that is
fine"; the worked example of a 1024-token prompt plus 10 generated tokens), and the
reference-counted sharing of that section's copy-on-write paragraph and of
gotacat.dev/blog/prompt-caching-kv-cache-vllm ("ref_cnt").

It only hands out ids and counts slots; it never touches K/V values.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Dict, List, Optional, Sequence

import torch

BLOCK_SIZE = 16


def blocks_for_tokens(num_tokens: int, block_size: int = BLOCK_SIZE) -> int:
    """Blocks needed to hold num_tokens tokens (the last one may be partial)."""
    return (num_tokens + block_size - 1) // block_size


def wasted_slots(num_tokens: int, block_size: int = BLOCK_SIZE) -> int:
    """Allocated but unused slots: the tail of the last, partial block."""
    return blocks_for_tokens(num_tokens, block_size) * block_size - num_tokens


def position_to_block(pos: int, block_size: int = BLOCK_SIZE) -> tuple[int, int]:
    """(logical block, offset in block) of 0-based token position pos."""
    return pos // block_size, pos % block_size


def slot_of(block_table_row: Sequence[int], pos: int, block_size: int = BLOCK_SIZE) -> int:
    """Flat pool slot (physical_block * block_size + offset) of token position pos."""
    j, off = position_to_block(pos, block_size)
    return int(block_table_row[j]) * block_size + off


@dataclass
class BlockPool:
    """A pool of num_blocks physical block ids with reference counts.

    Free ids are handed out in the order of a seeded random permutation, so the
    physical placement of consecutive logical blocks is scattered.
    """

    num_blocks: int
    block_size: int = BLOCK_SIZE
    generator: Optional[torch.Generator] = None
    ref_cnt: Dict[int, int] = field(default_factory=dict)

    def __post_init__(self) -> None:
        if self.generator is None:
            order = list(range(self.num_blocks))
        else:
            order = torch.randperm(self.num_blocks, generator=self.generator).tolist()
        self._free: List[int] = order[::-1]  # pop() from the end gives order[0] first

    @property
    def num_free(self) -> int:
        return len(self._free)

    def allocate(self, n: int) -> List[int]:
        if n > len(self._free):
            raise MemoryError(f"pool exhausted: need {n} blocks, {len(self._free)} free")
        ids = [self._free.pop() for _ in range(n)]
        for i in ids:
            self.ref_cnt[i] = 1
        return ids

    def share(self, ids: Sequence[int]) -> List[int]:
        """Take another reference to already-allocated blocks (prefix sharing / fork)."""
        for i in ids:
            if self.ref_cnt.get(i, 0) <= 0:
                raise ValueError(f"block {i} is not allocated")
            self.ref_cnt[i] += 1
        return list(ids)

    def release(self, ids: Sequence[int]) -> None:
        for i in ids:
            c = self.ref_cnt.get(i, 0)
            if c <= 0:
                raise ValueError(f"block {i} released more often than taken")
            if c == 1:
                del self.ref_cnt[i]
                self._free.append(i)
            else:
                self.ref_cnt[i] = c - 1


@dataclass
class Sequence_:
    """One decode sequence: its length (cached tokens including the one appended this
    step) and its block table row (physical ids of logical blocks 0..)."""

    length: int
    blocks: List[int]

    def slot(self, pos: int, block_size: int = BLOCK_SIZE) -> int:
        return slot_of(self.blocks, pos, block_size)


def allocate_private(pool: BlockPool, length: int) -> Sequence_:
    return Sequence_(length, pool.allocate(blocks_for_tokens(length, pool.block_size)))


def allocate_with_prefix(pool: BlockPool, prefix_blocks: Sequence[int], length: int) -> Sequence_:
    """A sequence whose first len(prefix_blocks) full blocks are shared (ref_cnt + 1);
    only full blocks are shared, so the private part starts in a fresh block."""
    bs = pool.block_size
    shared = len(prefix_blocks)
    if length < shared * bs:
        raise ValueError("sequence shorter than its shared prefix")
    own = blocks_for_tokens(length, bs) - shared
    return Sequence_(length, pool.share(prefix_blocks) + pool.allocate(own))


def fork(pool: BlockPool, seq: Sequence_) -> Sequence_:
    """A new sequence sharing every block of seq (parallel sampling / beam search: the
    pages' copy-on-write paragraph), including a partially filled tail block."""
    return Sequence_(seq.length, pool.share(seq.blocks))


def copy_on_write(pool: BlockPool, seq: Sequence_, logical_block: int):
    """Before seq writes into its logical block j: if that physical block is shared, give
    seq a fresh block and return (src, dst) for the device copy; else return None."""
    blk = seq.blocks[logical_block]
    if pool.ref_cnt.get(blk, 0) <= 1:
        return None
    new = pool.allocate(1)[0]
    pool.release([blk])
    seq.blocks[logical_block] = new
    return blk, new


def sampling_token_counts(prompt_tokens: int, generated_tokens: int, samples: int) -> tuple[int, int]:
    """Cached tokens for `samples` parallel samples of one prompt: without sharing
    (every sample keeps its own copy of the prompt) and with the prompt shared."""
    unshared = samples * (prompt_tokens + generated_tokens)
    shared = prompt_tokens + samples * generated_tokens
    return unshared, shared


def sampling_block_counts(prompt_tokens: int, generated_tokens: int, samples: int,
                          block_size: int = BLOCK_SIZE) -> tuple[int, int]:
    """Same count in blocks: only the prompt's full blocks can be shared."""
    unshared = samples * blocks_for_tokens(prompt_tokens + generated_tokens, block_size)
    full = prompt_tokens // block_size
    private = blocks_for_tokens(prompt_tokens + generated_tokens, block_size) - full
    return unshared, full + samples * private
