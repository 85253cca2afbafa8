"""Plain-Python model of the block manager with a prefix cache (TEST INFRASTRUCTURE).

Only the tests may use this module.  It shares no code with the library's C++ manager;
hashing uses Python's hashlib.

What it follows:

* habr.com/ru/articles/1021832, section 7 "Тот самый Cache Read" (Automatic Prefix
  Caching): the hash of a block covers every token up to the end of that block; a flat table maps block hash to
  physical block; a request hashes its blocks, looks them up from block 0 and stops at the
  first miss, and the hits are reused with their reference count raised; finished
  requests leave their blocks in the table with count 0; when no free block is left the
  least recently used block with count 0 is evicted; cached blocks are immutable; the
  worked example (2000-token prompt = 125 blocks, plus 200 tokens = 13 blocks, 138 in all;
  the second request reuses 125).
* gotacat.dev/blog/prompt-caching-kv-cache-vllm, "Хэш-цепочка в стиле git": block
  hash = hash(parent hash, the block's token ids, extra keys), the first block's parent a
  fixed seed; the lookup is capped at num_tokens - 1 tokens ("at least the last token must
  be computed"); section "Этот кэш не твой": a salt goes into the extra keys of the
  first block only.

Readings where the pages are silent:

* Byte format hashed (the pages leave the serialisation to the hash function):
  parent (32 bytes) || u32 little-endian block size || each token id as i32 little-endian
  || u32 little-endian length of the extra keys || the extra keys; SHA-256 (the pages name
  sha256 as the default).
* The free queue is a plain list: new blocks start in id order; a block whose count drops
  to zero goes to the end; allocation takes the front (the least recently freed, so LRU).
  One request's blocks are released from its last block to its first, so among blocks
  freed together the end of a chain is evicted first.
* A hash already owned by another block leaves the second block uncached (the table keeps
  the first owner).  Writing into a block that is shared or cached needs a fresh copy.
"""
from __future__ import annotations

import hashlib
import struct
from typing import Dict, List, Optional, Sequence, Tuple


def block_hash(parent: bytes, block_tokens: Sequence[int], extra: bytes = b"") -> bytes:
    msg = parent + struct.pack("<I", len(block_tokens))
    msg += b"".join(struct.pack("<i", int(t)) for t in block_tokens)
    msg += struct.pack("<I", len(extra)) + extra
    return hashlib.sha256(msg).digest()


def chain_hashes(tokens: Sequence[int], block_size: int = 16, seed: bytes = bytes(32),
                 salt: Optional[bytes] = None) -> List[bytes]:
    """Hashes of the full blocks of tokens, each chained to the previous one."""
    out, parent = [], seed
    for i in range(len(tokens) // block_size):
        parent = block_hash(parent, tokens[i * block_size:(i + 1) * block_size], (salt or b"") if i == 0 else b"")
        out.append(parent)
    return out


class PrefixCacheModel:
    def __init__(self, num_blocks: int, block_size: int = 16, seed: Optional[bytes] = None):
        self.block_size = block_size
        self.seed = seed if seed is not None else bytes(32)
        self.ref: List[int] = [0] * num_blocks
        self.hash_of: Dict[int, bytes] = {}  # cached block -> its hash
        self.table: Dict[bytes, int] = {}  # hash -> block
        self.free: List[int] = list(range(num_blocks))  # front = next to be taken

    @property
    def num_free(self) -> int:
        return len(self.free)

    def allocate(self, n: int) -> List[int]:
        if n > len(self.free):
            raise MemoryError("not enough free blocks")
        got = []
        for _ in range(n):
            b = self.free.pop(0)
            if b in self.hash_of:  # evict
                del self.table[self.hash_of.pop(b)]
            self.ref[b] = 1
            got.append(b)
        return got

    def get_computed_blocks(self, tokens: Sequence[int], salt: Optional[bytes] = None) -> List[int]:
        limit = max(len(tokens) - 1, 0) // self.block_size
        hits = []
        for h in chain_hashes(tokens, self.block_size, self.seed, salt)[:limit]:
            b = self.table.get(h)
            if b is None:
                break
            if self.ref[b] == 0:
                self.free.remove(b)
            self.ref[b] += 1
            hits.append(b)
        return hits

    def cache_full_blocks(self, tokens: Sequence[int], table: Sequence[int], salt: Optional[bytes] = None) -> int:
        hs = chain_hashes(tokens, self.block_size, self.seed, salt)
        if len(hs) > len(table):
            raise ValueError("table shorter than the full blocks")
        for b, h in zip(table, hs):
            if self.ref[b] <= 0:
                raise ValueError("block not held")
            if b in self.hash_of and self.hash_of[b] != h:
                raise ValueError("block holds another hash")
        for b, h in zip(table, hs):
            if b not in self.hash_of and h not in self.table:
                self.hash_of[b] = h
                self.table[h] = b
        return sum(1 for b in table[:len(hs)] if b in self.hash_of)

    def release(self, blocks: Sequence[int]) -> None:
        need: Dict[int, int] = {}
        for b in blocks:
            need[b] = need.get(b, 0) + 1
            if need[b] > self.ref[b]:
                raise ValueError("released more often than held")
        for b in reversed(list(blocks)):
            self.ref[b] -= 1
            if self.ref[b] == 0:
                self.free.append(b)

    def share(self, blocks: Sequence[int]) -> None:
        if any(self.ref[b] <= 0 for b in blocks):
            raise ValueError("block not held")
        for b in blocks:
            self.ref[b] += 1

    def copy_on_write(self, block: int) -> Tuple[int, bool]:
        if self.ref[block] <= 0:
            raise ValueError("block not held")
        if self.ref[block] == 1 and block not in self.hash_of:
            return block, False
        fresh = self.allocate(1)[0]
        self.ref[block] -= 1
        if self.ref[block] == 0:
            self.free.append(block)
        return fresh, True
