"""CPU oracle for paged KV append and paged decode attention (TEST INFRASTRUCTURE).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py``
may import this package.  It wraps ``pkv_oracle.c`` (plain C, fp64) with ctypes and
numpy; it shares no code with the CUDA library and never calls it.

Every function follows a passage of the pages the method comes from; see the header
of ``pkv_oracle.c`` for the citations and the readings taken where they are silent.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pkv_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "liborcl.so")

KV_BF16 = 0
KV_E4M3 = 1


def build(force: bool = False) -> str:
    """Compile pkv_oracle.c into a shared library with plain IEEE arithmetic."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp.%d" % os.getpid()
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math", "-ffp-contract=off",
               "-D_GNU_SOURCE", _SRC, "-o", tmp, "-lm", "-lpthread"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


_lib: Optional[ctypes.CDLL] = None


def _L() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i32, i64, dbl = ctypes.c_int, ctypes.c_int64, ctypes.c_double
        lib.orc_bf16_to_f64.restype = dbl
        lib.orc_bf16_to_f64.argtypes = [ctypes.c_uint16]
        lib.orc_e4m3_decode.restype = dbl
        lib.orc_e4m3_decode.argtypes = [ctypes.c_uint8]
        lib.orc_e4m3_encode.restype = ctypes.c_uint8
        lib.orc_e4m3_encode.argtypes = [ctypes.c_float]
        lib.orc_append.restype = i32
        lib.orc_append.argtypes = [P, P, i64, i32, i32, i32, i32, P, P, P, i64, P]
        lib.orc_gather.restype = None
        lib.orc_gather.argtypes = [P, i32, P, i32, i32, i32, P, i32, i32, P]
        lib.orc_attention_one.restype = None
        lib.orc_attention_one.argtypes = [P, P, P, i32, i32, dbl, P]
        lib.orc_decode_pairs.restype = i32
        lib.orc_decode_pairs.argtypes = [P, P, P, i32, P, i32, i32, i32, i32, P, i32, P, dbl, P, i64,
                                         P, i32]
        lib.orc_copy_blocks.restype = i32
        lib.orc_copy_blocks.argtypes = [P, P, i64, i64, P, i64]
        lib.orc_kv_bytes_per_token.restype = i64
        lib.orc_kv_bytes_per_token.argtypes = [i64, i64, i64, i64]
        _lib = lib
    return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data


# ------------------------------------------------------------------ element codecs

def bf16_to_f64(bits: int) -> float:
    return _L().orc_bf16_to_f64(int(bits))


def e4m3_decode(code: int) -> float:
    return _L().orc_e4m3_decode(int(code))


def e4m3_encode(x: float) -> int:
    return int(_L().orc_e4m3_encode(float(np.float32(x))))


def e4m3_encode_array(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    f = _L().orc_e4m3_encode
    return np.array([f(float(v)) for v in x.ravel()], dtype=np.uint8).reshape(x.shape)


def kv_bytes_per_token(layers: int, kv_heads: int, head_dim: int, bytes_per_elem: int) -> int:
    return int(_L().orc_kv_bytes_per_token(layers, kv_heads, head_dim, bytes_per_elem))


# ------------------------------------------------------------------ append / gather / attention

def append(k_cache: np.ndarray, v_cache: np.ndarray, k: np.ndarray, v: np.ndarray,
           slot_mapping: np.ndarray, kv_dtype: int, scales: Optional[np.ndarray] = None) -> int:
    """In-place append of new K/V rows into the pools (numpy arrays, modified).

    k_cache/v_cache: [num_blocks, block_size, Hkv, D] as uint16 (bf16 bits) or uint8 (e4m3).
    k, v: [T, Hkv, D] uint16 (bf16 bits).  slot_mapping: [T] int64.  scales: [2, Hkv] f32.
    """
    nb, bs, hkv, d = k_cache.shape
    k = np.ascontiguousarray(k, dtype=np.uint16)
    v = np.ascontiguousarray(v, dtype=np.uint16)
    sm = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    sc = None if scales is None else np.ascontiguousarray(scales, dtype=np.float32)
    if kv_dtype == KV_BF16:
        assert k_cache.dtype == np.uint16 and v_cache.dtype == np.uint16
    else:
        assert k_cache.dtype == np.uint8 and v_cache.dtype == np.uint8 and sc is not None
    return _L().orc_append(_ptr(k_cache), _ptr(v_cache), nb, bs, hkv, d, kv_dtype, _ptr(k), _ptr(v),
                           _ptr(sm), sm.shape[0], None if sc is None else _ptr(sc))


def copy_blocks(k_cache: np.ndarray, v_cache: np.ndarray, pairs: np.ndarray) -> int:
    """In-place block copy (copy-on-write) for rows (src, dst) of pairs [n, 2] int64."""
    assert k_cache.shape == v_cache.shape and k_cache.dtype == v_cache.dtype
    nb = k_cache.shape[0]
    block_bytes = k_cache[0].nbytes
    pr = np.ascontiguousarray(pairs, dtype=np.int64).reshape(-1, 2)
    return _L().orc_copy_blocks(_ptr(k_cache), _ptr(v_cache), nb, block_bytes, _ptr(pr), pr.shape[0])


def gather(pool: np.ndarray, kv_dtype: int, block_table_row: np.ndarray, length: int, h: int,
           scales_row: Optional[np.ndarray] = None) -> np.ndarray:
    """Contiguous fp64 [length, D] view of kv head h of one sequence."""
    nb, bs, hkv, d = pool.shape
    row = np.ascontiguousarray(block_table_row, dtype=np.int32)
    out = np.empty((length, d), dtype=np.float64)
    sc = None if scales_row is None else np.ascontiguousarray(scales_row, dtype=np.float32)
    _L().orc_gather(_ptr(pool), kv_dtype, None if sc is None else _ptr(sc), bs, hkv, d, _ptr(row),
                    length, h, _ptr(out))
    return out


def attention_one(q: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float) -> np.ndarray:
    """softmax(scale * q K^T) V for one fp64 query over contiguous fp64 K, V [n, D]."""
    q = np.ascontiguousarray(q, dtype=np.float64)
    K = np.ascontiguousarray(K, dtype=np.float64)
    V = np.ascontiguousarray(V, dtype=np.float64)
    n, d = K.shape
    out = np.empty(d, dtype=np.float64)
    _L().orc_attention_one(_ptr(q), _ptr(K), _ptr(V), n, d, float(scale), _ptr(out))
    return out


def decode_pairs(q: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray, kv_dtype: int,
                 block_tables: np.ndarray, context_lens: np.ndarray, softmax_scale: float,
                 pairs: np.ndarray, scales: Optional[np.ndarray] = None,
                 nthreads: int = 1) -> np.ndarray:
    """fp64 decode attention for the listed (b, hq) pairs; returns [num_pairs, D].

    q: [B, Hq, D] uint16 (bf16 bits); pools [NB, bs, Hkv, D]; block_tables [B, M] int32;
    context_lens [B] int32; pairs [P, 2] int32.
    """
    q = np.ascontiguousarray(q, dtype=np.uint16)
    B, hq, d = q.shape
    nb, bs, hkv, d2 = k_cache.shape
    assert d == d2
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    pr = np.ascontiguousarray(pairs, dtype=np.int32).reshape(-1, 2)
    sc = None if scales is None else np.ascontiguousarray(scales, dtype=np.float32)
    out = np.empty((pr.shape[0], d), dtype=np.float64)
    rc = _L().orc_decode_pairs(_ptr(q), _ptr(k_cache), _ptr(v_cache), kv_dtype,
                               None if sc is None else _ptr(sc), bs, hkv, hq, d, _ptr(bt),
                               bt.shape[1], _ptr(cl), float(softmax_scale), _ptr(pr), pr.shape[0],
                               _ptr(out), int(nthreads))
    if rc != 0:
        raise ValueError("oracle decode: bad head configuration")
    return out


def decode_all(q: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray, kv_dtype: int,
               block_tables: np.ndarray, context_lens: np.ndarray, softmax_scale: float,
               scales: Optional[np.ndarray] = None, nthreads: int = 1) -> np.ndarray:
    """fp64 decode attention for every (b, hq); returns [B, Hq, D]."""
    B, hq, d = q.shape
    pairs = np.array([(b, h) for b in range(B) for h in range(hq)], dtype=np.int32)
    out = decode_pairs(q, k_cache, v_cache, kv_dtype, block_tables, context_lens, softmax_scale,
                       pairs, scales=scales, nthreads=nthreads)
    return out.reshape(B, hq, d)
