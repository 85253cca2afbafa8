"""Python binding of the host block manager (include/pkv_block_manager.h).

Argument marshalling only: the reference counts, the chained block hashes, the prefix
lookup and the LRU free queue live in ``libpkv.so`` (``csrc/block_manager.cpp``).  The
manager hands out the physical block ids that ``paged_kv_append`` writes and that the
block tables of ``paged_decode_attention`` list.
"""
from __future__ import annotations

import ctypes
from typing import List, Optional, Sequence, Tuple

import numpy as np

from . import PKV_OK, PkvError, lib  # noqa: F401  (PkvError re-exported)

EXPORTED_SYMBOLS = (
    "pkv_sha256", "pkv_bm_chain_hashes", "pkv_bm_create", "pkv_bm_destroy", "pkv_bm_allocate",
    "pkv_bm_get_computed_blocks", "pkv_bm_cache_full_blocks", "pkv_bm_free", "pkv_bm_share",
    "pkv_bm_copy_on_write", "pkv_bm_num_free", "pkv_bm_num_cached", "pkv_bm_ref_count", "pkv_bm_block_hash",
    "pkv_bm_lookup", "pkv_bm_free_queue",
)

_P, _i32, _i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
_sigs = {
    "pkv_sha256": (None, [_P, _i64, _P]),
    "pkv_bm_chain_hashes": (ctypes.c_int, [_P, _i32, _P, _i64, _P, _i64, _P]),
    "pkv_bm_create": (ctypes.c_int, [_i64, _i32, _P, ctypes.POINTER(_P)]),
    "pkv_bm_destroy": (None, [_P]),
    "pkv_bm_allocate": (ctypes.c_int, [_P, _i64, _P]),
    "pkv_bm_get_computed_blocks": (ctypes.c_int, [_P, _P, _i64, _P, _i64, _P, _i64, ctypes.POINTER(_i64)]),
    "pkv_bm_cache_full_blocks": (ctypes.c_int, [_P, _P, _i64, _P, _i64, _P, _i64, ctypes.POINTER(_i64)]),
    "pkv_bm_free": (ctypes.c_int, [_P, _P, _i64]),
    "pkv_bm_share": (ctypes.c_int, [_P, _P, _i64]),
    "pkv_bm_copy_on_write": (ctypes.c_int, [_P, _i32, ctypes.POINTER(_i32), ctypes.POINTER(_i32)]),
    "pkv_bm_num_free": (_i64, [_P]),
    "pkv_bm_num_cached": (_i64, [_P]),
    "pkv_bm_ref_count": (_i32, [_P, _i32]),
    "pkv_bm_block_hash": (_i32, [_P, _i32, _P]),
    "pkv_bm_lookup": (_i32, [_P, _P]),
    "pkv_bm_free_queue": (_i64, [_P, _P, _i64]),
}
for _name, (_res, _args) in _sigs.items():
    _f = getattr(lib, _name)
    _f.restype = _res
    _f.argtypes = _args


def _check(status: int) -> None:
    if status != PKV_OK:
        raise PkvError(status, lib.pkv_last_error().decode() or lib.pkv_status_string(status).decode())


def _i32_array(values: Sequence[int]) -> np.ndarray:
    a = np.asarray(values, dtype=np.int64).reshape(-1)
    if a.size and (a.min() < -2**31 or a.max() >= 2**31):
        raise ValueError("token and block ids must fit in int32")
    return np.ascontiguousarray(a.astype(np.int32))


def _ptr(a: np.ndarray) -> Optional[int]:
    return a.ctypes.data if a.size else None


def _bytes(b: Optional[bytes]) -> Tuple[Optional[bytes], int]:
    return (None, 0) if not b else (bytes(b), len(b))


def sha256(data: bytes) -> bytes:
    out = ctypes.create_string_buffer(32)
    lib.pkv_sha256(data if data else None, len(data), out)
    return out.raw


def chain_hashes(tokens: Sequence[int], block_size: int = 16, seed: bytes = bytes(32),
                 salt: Optional[bytes] = None) -> List[bytes]:
    """Hashes of the full blocks of `tokens` (the first block's parent is `seed`)."""
    if len(seed) != 32:
        raise ValueError("seed must be 32 bytes")
    toks = _i32_array(tokens)
    n = len(toks) // block_size if block_size > 0 else 0
    out = ctypes.create_string_buffer(max(1, 32 * n))
    s, sl = _bytes(salt)
    _check(lib.pkv_bm_chain_hashes(seed, block_size, _ptr(toks), len(toks), s, sl, out))
    return [out.raw[32 * i:32 * i + 32] for i in range(n)]


class BlockManager:
    """Reference-counted physical blocks with a hash-chained prefix cache (host only)."""

    def __init__(self, num_blocks: int, block_size: int = 16, seed: Optional[bytes] = None):
        if seed is not None and len(seed) != 32:
            raise ValueError("seed must be 32 bytes")
        h = _P()
        _check(lib.pkv_bm_create(num_blocks, block_size, seed, ctypes.byref(h)))
        self._h = h
        self.num_blocks = num_blocks
        self.block_size = block_size

    def close(self) -> None:
        if self._h:
            lib.pkv_bm_destroy(self._h)
            self._h = _P()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def allocate(self, n: int) -> List[int]:
        out = np.empty(max(n, 0), dtype=np.int32)
        _check(lib.pkv_bm_allocate(self._h, n, _ptr(out)))
        return out.tolist()

    def get_computed_blocks(self, tokens: Sequence[int], salt: Optional[bytes] = None) -> List[int]:
        toks = _i32_array(tokens)
        cap = max(len(toks) // self.block_size, 0)
        out = np.empty(cap, dtype=np.int32)
        hit = _i64(0)
        s, sl = _bytes(salt)
        _check(lib.pkv_bm_get_computed_blocks(self._h, _ptr(toks), len(toks), s, sl, _ptr(out), cap,
                                              ctypes.byref(hit)))
        return out[: hit.value].tolist()

    def cache_full_blocks(self, tokens: Sequence[int], block_table: Sequence[int],
                          salt: Optional[bytes] = None) -> int:
        toks = _i32_array(tokens)
        table = _i32_array(block_table)
        n = _i64(0)
        s, sl = _bytes(salt)
        _check(lib.pkv_bm_cache_full_blocks(self._h, _ptr(toks), len(toks), s, sl, _ptr(table), len(table),
                                            ctypes.byref(n)))
        return n.value

    def free(self, blocks: Sequence[int]) -> None:
        b = _i32_array(blocks)
        _check(lib.pkv_bm_free(self._h, _ptr(b), len(b)))

    def share(self, blocks: Sequence[int]) -> List[int]:
        b = _i32_array(blocks)
        _check(lib.pkv_bm_share(self._h, _ptr(b), len(b)))
        return list(blocks)

    def copy_on_write(self, block: int) -> Tuple[int, bool]:
        """(block to write into, whether the caller must copy `block` into it first)."""
        out, need = _i32(0), _i32(0)
        _check(lib.pkv_bm_copy_on_write(self._h, block, ctypes.byref(out), ctypes.byref(need)))
        return out.value, bool(need.value)

    @property
    def num_free(self) -> int:
        return int(lib.pkv_bm_num_free(self._h))

    @property
    def num_cached(self) -> int:
        return int(lib.pkv_bm_num_cached(self._h))

    def ref_count(self, block: int) -> int:
        return int(lib.pkv_bm_ref_count(self._h, block))

    def block_hash(self, block: int) -> Optional[bytes]:
        out = ctypes.create_string_buffer(32)
        r = lib.pkv_bm_block_hash(self._h, block, out)
        if r < 0:
            raise ValueError(f"block {block} outside the pool")
        return out.raw if r == 1 else None

    def lookup(self, block_hash: bytes) -> int:
        if len(block_hash) != 32:
            raise ValueError("a block hash is 32 bytes")
        return int(lib.pkv_bm_lookup(self._h, block_hash))

    def free_queue(self) -> List[int]:
        out = np.empty(self.num_blocks, dtype=np.int32)
        n = lib.pkv_bm_free_queue(self._h, _ptr(out), self.num_blocks)
        return out[:n].tolist()
