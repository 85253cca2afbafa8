"""Paged KV-cache decode for GB300 (sm_103a): Python binding of the C ABI in include/pkv.h.

Two calls make one decode step of one attention layer:

* ``paged_kv_append(k, v, slot_mapping, k_cache, v_cache, kv_dtype, scales)`` scatters the
  step's new K/V rows into the block-paged pool (bf16 copy, or E4M3 quantise-on-write);
* ``paged_decode_attention(q, k_cache, v_cache, block_tables, context_lens, softmax_scale,
  out)`` runs GQA decode attention over each sequence's cached K/V, gathered through its
  block table.

This module only marshals arguments: it takes shapes, dtypes and device pointers from
torch tensors and passes the current CUDA stream.  Every step of the computation runs in
the CUDA kernels of ``libpkv.so``; there is no fallback, and importing this module fails
loudly if the library has not been built (``python -m paged_kv_cache_17_gb300._build``).
"""
from __future__ import annotations

import ctypes
import os
from typing import Dict, Optional, Tuple

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libpkv.so")

PKV_OK = 0
PKV_ERR_INVALID_ARG = 1
PKV_ERR_UNSUPPORTED = 2
PKV_ERR_WORKSPACE = 3
PKV_ERR_CUDA = 4
PKV_ERR_DEVICE_CHECK = 5
KV_BF16 = 0
KV_FP8_E4M3 = 1
OUT_BF16 = 0
OUT_FP32 = 1

DEVFLAG_BAD_SLOT = 0x1
DEVFLAG_BAD_CONTEXT_LEN = 0x2
DEVFLAG_BAD_BLOCK_ID = 0x4
DEVFLAG_WAIT_TIMEOUT = 0x8

EXPORTED_SYMBOLS = (
    "pkv_paged_kv_append", "pkv_decode_workspace_size",
    "pkv_decode_partition_tokens", "pkv_paged_decode_attention", "pkv_check_device_status",
    "pkv_status_string", "pkv_last_error", "pkv_version", "pkv_paged_decode_attention_noalloc",
    "pkv_copy_blocks", "pkv_cascade_workspace_size", "pkv_cascade_decode_attention", "pkv_paged_kv_checksum",
    "pkv_paged_append_decode", "pkv_stage_copy",
)


class PkvError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"pkv error {status}: {message}")
        self.status = status


class CacheDesc(ctypes.Structure):
    _fields_ = [("k_cache", ctypes.c_void_p), ("v_cache", ctypes.c_void_p), ("num_blocks", ctypes.c_int64),
                ("block_size", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("kv_dtype", ctypes.c_int), ("scales", ctypes.c_void_p)]


class PrefixDesc(ctypes.Structure):
    _fields_ = [("prefix_tables", ctypes.c_void_p), ("max_prefix_blocks", ctypes.c_int32),
                ("prefix_lens", ctypes.c_void_p), ("num_prefixes", ctypes.c_int32),
                ("member_indptr", ctypes.c_void_p), ("member_seqs", ctypes.c_void_p),
                ("max_members", ctypes.c_int32), ("max_prefix_len", ctypes.c_int32),
                ("seq_prefix", ctypes.c_void_p)]


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libpkv.so is not built ({LIB_PATH}); run python -m paged_kv_cache_17_gb300._build")
    lib = ctypes.CDLL(LIB_PATH)
    P, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    lib.pkv_paged_kv_append.restype = ctypes.c_int
    lib.pkv_paged_kv_append.argtypes = [ctypes.POINTER(CacheDesc), P, P, P, i64, P]
    lib.pkv_decode_workspace_size.restype = sz
    lib.pkv_decode_workspace_size.argtypes = [i32, i32, i32, i32, i32]
    lib.pkv_decode_partition_tokens.restype = i32
    lib.pkv_decode_partition_tokens.argtypes = [i32, i32, i32]
    lib.pkv_paged_decode_attention.restype = ctypes.c_int
    lib.pkv_paged_decode_attention.argtypes = [ctypes.POINTER(CacheDesc), P, P, i32, P, i32, i32, i32,
                                               ctypes.c_float, P, ctypes.c_int, P, sz, P]
    lib.pkv_paged_decode_attention_noalloc.restype = ctypes.c_int
    lib.pkv_paged_decode_attention_noalloc.argtypes = [ctypes.POINTER(CacheDesc), P, P, i32, P, i32, i32, i32,
                                                       ctypes.c_float, P, ctypes.c_int, P]
    lib.pkv_cascade_workspace_size.restype = sz
    lib.pkv_cascade_workspace_size.argtypes = [i32, i32, i32, i32, i32, i32, i32, i32]
    lib.pkv_cascade_decode_attention.restype = ctypes.c_int
    lib.pkv_cascade_decode_attention.argtypes = [ctypes.POINTER(CacheDesc), P, ctypes.POINTER(PrefixDesc), P, i32, P,
                                                 i32, i32, i32, ctypes.c_float, P, ctypes.c_int, P, sz, P]
    lib.pkv_paged_append_decode.restype = ctypes.c_int
    lib.pkv_paged_append_decode.argtypes = [ctypes.POINTER(CacheDesc), P, P, P, P, P, i32, P, i32, i32, i32,
                                            ctypes.c_float, P, ctypes.c_int, P, sz, P]
    lib.pkv_paged_kv_checksum.restype = ctypes.c_int
    lib.pkv_paged_kv_checksum.argtypes = [ctypes.POINTER(CacheDesc), P, i32, P, i32, i32, P, P]
    lib.pkv_copy_blocks.restype = ctypes.c_int
    lib.pkv_copy_blocks.argtypes = [ctypes.POINTER(CacheDesc), P, i64, P]
    lib.pkv_stage_copy.restype = ctypes.c_int
    lib.pkv_stage_copy.argtypes = [P, P, ctypes.c_size_t, P]
    lib.pkv_check_device_status.restype = ctypes.c_int
    lib.pkv_check_device_status.argtypes = [P, ctypes.POINTER(ctypes.c_uint32)]
    lib.pkv_status_string.restype = ctypes.c_char_p
    lib.pkv_status_string.argtypes = [ctypes.c_int]
    lib.pkv_last_error.restype = ctypes.c_char_p
    lib.pkv_last_error.argtypes = []
    lib.pkv_version.restype = i32
    lib.pkv_version.argtypes = []
    return lib


lib = _load()


def _check(status: int) -> None:
    if status != PKV_OK:
        raise PkvError(status, lib.pkv_last_error().decode() or lib.pkv_status_string(status).decode())


def _stream(stream: Optional[torch.cuda.Stream]) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(s.cuda_stream)


def _kv_dtype_of(k_cache: torch.Tensor) -> int:
    if k_cache.dtype == torch.bfloat16:
        return KV_BF16
    if k_cache.dtype in (torch.uint8, torch.float8_e4m3fn):
        return KV_FP8_E4M3
    raise TypeError(f"k_cache dtype {k_cache.dtype} is neither bfloat16 nor E4M3 bytes")


def _cache_desc(k_cache: torch.Tensor, v_cache: torch.Tensor, kv_dtype: Optional[str],
                scales: Optional[torch.Tensor]) -> CacheDesc:
    if k_cache.shape != v_cache.shape or k_cache.dtype != v_cache.dtype:
        raise ValueError("k_cache and v_cache must have the same shape and dtype")
    if k_cache.dim() != 4:
        raise ValueError("caches are [num_blocks, block_size, num_kv_heads, head_dim]")
    if not (k_cache.is_contiguous() and v_cache.is_contiguous()):
        raise ValueError("caches must be contiguous")
    code = _kv_dtype_of(k_cache)
    if kv_dtype is not None and {"bf16": KV_BF16, "e4m3": KV_FP8_E4M3, "fp8": KV_FP8_E4M3}[kv_dtype] != code:
        raise ValueError(f"kv_dtype={kv_dtype} does not match k_cache dtype {k_cache.dtype}")
    if scales is not None:
        if scales.dtype != torch.float32 or not scales.is_contiguous():
            raise ValueError("scales must be a contiguous float32 tensor [2, num_kv_heads]")
    nb, bs, hkv, d = k_cache.shape
    return CacheDesc(k_cache.data_ptr(), v_cache.data_ptr(), nb, bs, hkv, d, code,
                     scales.data_ptr() if scales is not None else None)


def paged_kv_append(k: torch.Tensor, v: torch.Tensor, slot_mapping: torch.Tensor, k_cache: torch.Tensor,
                    v_cache: torch.Tensor, kv_dtype: Optional[str] = None, scales: Optional[torch.Tensor] = None,
                    stream: Optional[torch.cuda.Stream] = None) -> None:
    """Write k, v ([T, Hkv, D] bf16) into the pools at slot_mapping ([T] int64)."""
    desc = _cache_desc(k_cache, v_cache, kv_dtype, scales)
    if k.dtype != torch.bfloat16 or v.dtype != torch.bfloat16:
        raise TypeError("k and v must be bfloat16")
    if not (k.is_contiguous() and v.is_contiguous() and slot_mapping.is_contiguous()):
        raise ValueError("k, v and slot_mapping must be contiguous")
    if slot_mapping.dtype != torch.int64:
        raise TypeError("slot_mapping must be int64")
    T = slot_mapping.shape[0]
    if tuple(k.shape) != (T, desc.num_kv_heads, desc.head_dim) or k.shape != v.shape:
        raise ValueError("k, v must be [num_tokens, num_kv_heads, head_dim]")
    _check(lib.pkv_paged_kv_append(ctypes.byref(desc), k.data_ptr(), v.data_ptr(), slot_mapping.data_ptr(), T,
                                   _stream(stream)))


def copy_blocks(block_pairs: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                scales: Optional[torch.Tensor] = None, stream: Optional[torch.cuda.Stream] = None) -> None:
    """Copy-on-write: for each row (src, dst) of block_pairs ([n, 2] int64), make block dst
    of both pools a copy of block src."""
    desc = _cache_desc(k_cache, v_cache, None, scales)
    if block_pairs.dtype != torch.int64 or block_pairs.dim() != 2 or block_pairs.shape[1] != 2:
        raise ValueError("block_pairs must be an int64 tensor [n, 2]")
    if not block_pairs.is_contiguous():
        raise ValueError("block_pairs must be contiguous")
    _check(lib.pkv_copy_blocks(ctypes.byref(desc), block_pairs.data_ptr(), block_pairs.shape[0], _stream(stream)))


_workspaces: Dict[Tuple[int, int], torch.Tensor] = {}


def workspace_size(batch: int, num_q_heads: int, num_kv_heads: int, head_dim: int, max_context_len: int) -> int:
    return int(lib.pkv_decode_workspace_size(batch, num_q_heads, num_kv_heads, head_dim, max_context_len))


def partition_tokens(batch: int, num_kv_heads: int, max_context_len: int) -> int:
    return int(lib.pkv_decode_partition_tokens(batch, num_kv_heads, max_context_len))


def _workspace(device: torch.device, stream_handle: int, nbytes: int) -> torch.Tensor:
    """A workspace per (device, stream), grown on demand (the decode needs nothing in it
    initialised)."""
    key = (device.index if device.index is not None else torch.cuda.current_device(), stream_handle)
    ws = _workspaces.get(key)
    if ws is None or ws.numel() < nbytes:
        ws = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)
        _workspaces[key] = ws
    return ws


def paged_decode_attention(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, block_tables: torch.Tensor,
                           context_lens: torch.Tensor, softmax_scale: float, out: Optional[torch.Tensor] = None, *,
                           scales: Optional[torch.Tensor] = None, kv_dtype: Optional[str] = None,
                           max_context_len: Optional[int] = None, workspace: Optional[torch.Tensor] = None,
                           stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """Decode attention of q ([B, Hq, D] bf16) over the paged cache.

    block_tables: [B, max_blocks] int32; context_lens: [B] int32.  out: [B, Hq, D] bf16 or
    float32 (allocated as bf16 when None).  max_context_len defaults to the table capacity
    (max_blocks * 16), which needs no device-to-host read.
    """
    desc = _cache_desc(k_cache, v_cache, kv_dtype, scales)
    if q.dtype != torch.bfloat16 or not q.is_contiguous() or q.dim() != 3:
        raise ValueError("q must be a contiguous bfloat16 tensor [B, Hq, D]")
    B, hq, d = q.shape
    if d != desc.head_dim:
        raise ValueError("q head_dim differs from the cache's")
    if block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32:
        raise TypeError("block_tables and context_lens must be int32")
    if not (block_tables.is_contiguous() and context_lens.is_contiguous()):
        raise ValueError("block_tables and context_lens must be contiguous")
    if block_tables.dim() != 2 or block_tables.shape[0] != B or context_lens.shape != (B,):
        raise ValueError("block_tables must be [B, max_blocks] and context_lens [B]")
    max_blocks = block_tables.shape[1]
    if max_context_len is None:
        max_context_len = max_blocks * desc.block_size
    if out is None:
        out = torch.empty((B, hq, d), dtype=torch.bfloat16, device=q.device)
    if out.dtype not in (torch.bfloat16, torch.float32) or tuple(out.shape) != (B, hq, d) or not out.is_contiguous():
        raise ValueError("out must be a contiguous [B, Hq, D] bfloat16 or float32 tensor")
    out_code = OUT_FP32 if out.dtype == torch.float32 else OUT_BF16
    sh = _stream(stream)
    # a size query that fails leaves need at 0; the call below then makes the same check and
    # raises with its status
    need = workspace_size(B, hq, desc.num_kv_heads, d, max_context_len) if B > 0 else 0
    ws_ptr, ws_bytes = None, 0
    if need > 0:
        ws = workspace if workspace is not None else _workspace(q.device, sh, need)
        ws_ptr, ws_bytes = ws.data_ptr(), ws.numel() * ws.element_size()
    _check(lib.pkv_paged_decode_attention(ctypes.byref(desc), q.data_ptr(), block_tables.data_ptr(), max_blocks,
                                          context_lens.data_ptr(), B, hq, max_context_len, float(softmax_scale),
                                          out.data_ptr(), out_code, ws_ptr, ws_bytes, sh))
    return out


def paged_append_decode(k: torch.Tensor, v: torch.Tensor, slot_mapping: torch.Tensor, q: torch.Tensor,
                        k_cache: torch.Tensor, v_cache: torch.Tensor, block_tables: torch.Tensor,
                        context_lens: torch.Tensor, softmax_scale: float, out: Optional[torch.Tensor] = None, *,
                        scales: Optional[torch.Tensor] = None, max_context_len: Optional[int] = None,
                        workspace: Optional[torch.Tensor] = None,
                        stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """Append each sequence's new token (k, v [B, Hkv, D] bf16 at slot_mapping [B] int64, the
    slot of position context_lens[b] - 1) and run decode attention over the cache that holds
    it, in one launch; the same pool and output as paged_kv_append then paged_decode_attention."""
    desc = _cache_desc(k_cache, v_cache, None, scales)
    if q.dtype != torch.bfloat16 or not q.is_contiguous() or q.dim() != 3:
        raise ValueError("q must be a contiguous bfloat16 tensor [B, Hq, D]")
    B, hq, d = q.shape
    if k.dtype != torch.bfloat16 or v.dtype != torch.bfloat16 or not (k.is_contiguous() and v.is_contiguous()):
        raise TypeError("k and v must be contiguous bfloat16")
    if tuple(k.shape) != (B, desc.num_kv_heads, desc.head_dim) or k.shape != v.shape:
        raise ValueError("k, v must be [B, num_kv_heads, head_dim]: one new token per sequence")
    if slot_mapping.dtype != torch.int64 or tuple(slot_mapping.shape) != (B,) or not slot_mapping.is_contiguous():
        raise ValueError("slot_mapping must be a contiguous int64 tensor [B]")
    if block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32:
        raise TypeError("block_tables and context_lens must be int32")
    if not (block_tables.is_contiguous() and context_lens.is_contiguous()):
        raise ValueError("block_tables and context_lens must be contiguous")
    if block_tables.dim() != 2 or block_tables.shape[0] != B or context_lens.shape != (B,):
        raise ValueError("block_tables must be [B, max_blocks] and context_lens [B]")
    max_blocks = block_tables.shape[1]
    if max_context_len is None:
        max_context_len = max_blocks * desc.block_size
    if out is None:
        out = torch.empty((B, hq, d), dtype=torch.bfloat16, device=q.device)
    if out.dtype not in (torch.bfloat16, torch.float32) or tuple(out.shape) != (B, hq, d) or not out.is_contiguous():
        raise ValueError("out must be a contiguous [B, Hq, D] bfloat16 or float32 tensor")
    sh = _stream(stream)
    need = workspace_size(B, hq, desc.num_kv_heads, d, max_context_len) if B > 0 else 0
    ws_ptr, ws_bytes = None, 0
    if need > 0:
        ws = workspace if workspace is not None else _workspace(q.device, sh, need)
        ws_ptr, ws_bytes = ws.data_ptr(), ws.numel() * ws.element_size()
    _check(lib.pkv_paged_append_decode(ctypes.byref(desc), k.data_ptr(), v.data_ptr(), slot_mapping.data_ptr(),
                                       q.data_ptr(), block_tables.data_ptr(), max_blocks, context_lens.data_ptr(), B,
                                       hq, max_context_len, float(softmax_scale), out.data_ptr(),
                                       OUT_FP32 if out.dtype == torch.float32 else OUT_BF16, ws_ptr, ws_bytes, sh))
    return out


def cascade_workspace_size(batch: int, num_q_heads: int, num_kv_heads: int, head_dim: int, max_context_len: int,
                           num_prefixes: int, max_members: int, max_prefix_len: int) -> int:
    return int(lib.pkv_cascade_workspace_size(batch, num_q_heads, num_kv_heads, head_dim, max_context_len,
                                              num_prefixes, max_members, max_prefix_len))


def cascade_decode_attention(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                             prefix_tables: torch.Tensor, prefix_lens: torch.Tensor, member_indptr: torch.Tensor,
                             member_seqs: torch.Tensor, seq_prefix: torch.Tensor, block_tables: torch.Tensor,
                             context_lens: torch.Tensor, softmax_scale: float, out: Optional[torch.Tensor] = None, *,
                             max_members: int, max_prefix_len: Optional[int] = None,
                             max_context_len: Optional[int] = None, scales: Optional[torch.Tensor] = None,
                             workspace: Optional[torch.Tensor] = None,
                             stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """Decode attention where sequences share prefixes: prefix p ([num_prefixes] rows of
    prefix_tables, prefix_lens[p] tokens) is attended once for all its members
    member_seqs[member_indptr[p]:member_indptr[p+1]]; block_tables / context_lens hold each
    sequence's blocks after its prefix (seq_prefix[b] = p, or -1 without a prefix)."""
    desc = _cache_desc(k_cache, v_cache, None, scales)
    if q.dtype != torch.bfloat16 or not q.is_contiguous() or q.dim() != 3:
        raise ValueError("q must be a contiguous bfloat16 tensor [B, Hq, D]")
    B, hq, d = q.shape
    for name, t in (("prefix_tables", prefix_tables), ("prefix_lens", prefix_lens), ("member_indptr", member_indptr),
                    ("member_seqs", member_seqs), ("seq_prefix", seq_prefix), ("block_tables", block_tables),
                    ("context_lens", context_lens)):
        if t.dtype != torch.int32 or not t.is_contiguous():
            raise TypeError(f"{name} must be a contiguous int32 tensor")
    if prefix_tables.dim() != 2 or prefix_lens.shape != (prefix_tables.shape[0],):
        raise ValueError("prefix_tables must be [P, max_prefix_blocks] and prefix_lens [P]")
    P = prefix_tables.shape[0]
    if member_indptr.shape != (P + 1,) or seq_prefix.shape != (B,):
        raise ValueError("member_indptr must be [P + 1] and seq_prefix [B]")
    if block_tables.dim() != 2 or block_tables.shape[0] != B or context_lens.shape != (B,):
        raise ValueError("block_tables must be [B, max_blocks] and context_lens [B]")
    if max_prefix_len is None:
        max_prefix_len = prefix_tables.shape[1] * 16
    if max_context_len is None:
        max_context_len = block_tables.shape[1] * 16
    if out is None:
        out = torch.empty((B, hq, d), dtype=torch.bfloat16, device=q.device)
    if out.dtype not in (torch.bfloat16, torch.float32) or tuple(out.shape) != (B, hq, d) or not out.is_contiguous():
        raise ValueError("out must be a contiguous [B, Hq, D] bfloat16 or float32 tensor")
    px = PrefixDesc(prefix_tables.data_ptr(), prefix_tables.shape[1], prefix_lens.data_ptr(), P,
                    member_indptr.data_ptr(), member_seqs.data_ptr() if member_seqs.numel() else None,
                    max_members, max_prefix_len, seq_prefix.data_ptr())
    sh = _stream(stream)
    need = cascade_workspace_size(B, hq, desc.num_kv_heads, d, max_context_len, P, max_members, max_prefix_len)
    ws_ptr, ws_bytes = None, 0
    if need > 0:
        ws = workspace if workspace is not None else _workspace(q.device, sh, need)
        ws_ptr, ws_bytes = ws.data_ptr(), ws.numel() * ws.element_size()
    _check(lib.pkv_cascade_decode_attention(ctypes.byref(desc), q.data_ptr(), ctypes.byref(px),
                                            block_tables.data_ptr(), block_tables.shape[1], context_lens.data_ptr(),
                                            B, hq, max_context_len, float(softmax_scale), out.data_ptr(),
                                            OUT_FP32 if out.dtype == torch.float32 else OUT_BF16, ws_ptr, ws_bytes,
                                            sh))
    return out


def kv_checksum(k_cache: torch.Tensor, v_cache: torch.Tensor, block_tables: torch.Tensor, context_lens: torch.Tensor,
                out: Optional[torch.Tensor] = None, *, scales: Optional[torch.Tensor] = None,
                max_context_len: Optional[int] = None, stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """Per (sequence, kv head) checksums of the cached K and V read through the block tables
    (int32 [B, Hkv, 2]; the bits are the uint32 of include/pkv.h): a read-only pass with the
    decode's gather, so its time is the ceiling of the decode's reads."""
    desc = _cache_desc(k_cache, v_cache, None, scales)
    if block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32:
        raise TypeError("block_tables and context_lens must be int32")
    if not (block_tables.is_contiguous() and context_lens.is_contiguous()) or block_tables.dim() != 2:
        raise ValueError("block_tables must be a contiguous [B, max_blocks] and context_lens a contiguous [B]")
    B = block_tables.shape[0]
    if out is None:
        out = torch.empty((B, desc.num_kv_heads, 2), dtype=torch.int32, device=k_cache.device)
    if out.dtype != torch.int32 or tuple(out.shape) != (B, desc.num_kv_heads, 2) or not out.is_contiguous():
        raise ValueError("out must be a contiguous int32 tensor [B, num_kv_heads, 2]")
    if max_context_len is None:
        max_context_len = block_tables.shape[1] * desc.block_size
    _check(lib.pkv_paged_kv_checksum(ctypes.byref(desc), block_tables.data_ptr(), block_tables.shape[1],
                                     context_lens.data_ptr(), B, max_context_len, out.data_ptr(), _stream(stream)))
    return out


def stage_copy(dst: torch.Tensor, src: torch.Tensor, stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """Copy src into dst with the SMs (include/pkv.h pkv_stage_copy): either may be a
    page-locked (pinned) CPU tensor or a tensor on the current device; both contiguous, of
    the same number of bytes (a multiple of 16), 16-byte aligned."""
    for name, t in (("dst", dst), ("src", src)):
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
        if t.device.type == "cpu" and not t.is_pinned():
            raise ValueError(f"{name} must be a pinned (page-locked) CPU tensor or a CUDA tensor")
    n = dst.numel() * dst.element_size()
    if src.numel() * src.element_size() != n:
        raise ValueError("dst and src must hold the same number of bytes")
    _check(lib.pkv_stage_copy(dst.data_ptr(), src.data_ptr(), n, _stream(stream)))
    return dst


def check_device_status(stream: Optional[torch.cuda.Stream] = None) -> int:
    """Synchronise the stream; return the device status flags (and clear them)."""
    flags = ctypes.c_uint32(0)
    st = lib.pkv_check_device_status(_stream(stream), ctypes.byref(flags))
    if st not in (PKV_OK, PKV_ERR_DEVICE_CHECK):
        _check(st)
    return int(flags.value)


def version() -> int:
    return int(lib.pkv_version())
