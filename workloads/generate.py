"""Seeded synthetic inputs for paged decode: q, a scattered K/V pool, block tables,
context lengths, the step's new K/V rows and their slot mapping.

This module holds no arithmetic of the method (no attention, no append, no e4m3
encoder of its own): it draws random numbers, hands out block ids through the host
allocator and lays the results out in the shapes the calls take.  Both the CUDA
path and the CPU oracle read what it produces; neither is called from here.

Random streams: one torch CPU generator per (seed, stream tag, chunk), so the data
do not depend on the number of threads used to draw them.
"""
from __future__ import annotations

import math
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass
from typing import Dict, List, Optional

import numpy as np
import torch

from .allocator import BLOCK_SIZE, BlockPool, Sequence_, allocate_private, allocate_with_prefix, \
    blocks_for_tokens
from .configs import Config, get

E4M3_MAX = 448.0  # largest finite OCP E4M3 magnitude, used only to size the per-head scales
_CHUNK = 1 << 22
_STREAMS = {"q": 1, "k_pool": 2, "v_pool": 3, "k_new": 4, "v_new": 5, "pad": 6}


def _chunk_seed(seed: int, tag: int, chunk: int) -> int:
    return (seed * 1_000_003 + tag * 7_919 + chunk * 104_729) % (2**63 - 1)


def randn_bf16(shape, seed: int, tag: str, threads: int = 8) -> torch.Tensor:
    """N(0, 1) values rounded to bf16, drawn in fixed-size chunks with their own seeds."""
    numel = int(np.prod(shape))
    out = torch.empty(numel, dtype=torch.bfloat16)
    nchunks = (numel + _CHUNK - 1) // _CHUNK

    def work(c: int) -> None:
        g = torch.Generator().manual_seed(_chunk_seed(seed, _STREAMS[tag], c))
        lo, hi = c * _CHUNK, min(numel, (c + 1) * _CHUNK)
        out[lo:hi] = torch.randn(hi - lo, generator=g).to(torch.bfloat16)

    if nchunks <= 1:
        for c in range(nchunks):
            work(c)
    else:
        with ThreadPoolExecutor(max_workers=threads) as ex:
            list(ex.map(work, range(nchunks)))
    return out.view(*shape)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """uint16 numpy view of a CPU bf16 tensor (the raw bits, no conversion)."""
    assert t.dtype == torch.bfloat16 and t.device.type == "cpu"
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


@dataclass
class Workload:
    cfg: Config
    seqs: List[Sequence_]
    num_blocks: int
    q: torch.Tensor  # [B, Hq, D] bf16
    k_cache: torch.Tensor  # [NB, 16, Hkv, D] bf16, or uint8 e4m3 codes; state BEFORE the append
    v_cache: torch.Tensor
    k_new: torch.Tensor  # [T, Hkv, D] bf16
    v_new: torch.Tensor
    slot_mapping: torch.Tensor  # [T] int64
    block_tables: torch.Tensor  # [B, M] int32 (entries past a sequence's blocks are valid ids, unused)
    context_lens: torch.Tensor  # [B] int32, including the appended token
    scales: Optional[torch.Tensor]  # [2, Hkv] f32 for e4m3, else None

    @property
    def batch(self) -> int:
        return len(self.seqs)

    @property
    def kv_dtype_code(self) -> int:
        return 1 if self.cfg.kv_dtype == "e4m3" else 0

    @property
    def max_context_len(self) -> int:
        return max(s.length for s in self.seqs)

    def unique_kv_bytes(self) -> int:
        """K+V bytes of every distinct valid (physical block, slot): what one decode step must
        read at least once.  A block shared by several sequences counts once."""
        fill: Dict[int, int] = {}
        for s in self.seqs:
            for j, blk in enumerate(s.blocks):
                valid = min(BLOCK_SIZE, s.length - j * BLOCK_SIZE)
                if valid > fill.get(blk, 0):
                    fill[blk] = valid
        c = self.cfg
        return sum(fill.values()) * 2 * c.hkv * c.d * c.elem_bytes

    def logical_kv_bytes(self) -> int:
        c = self.cfg
        return sum(s.length for s in self.seqs) * 2 * c.hkv * c.d * c.elem_bytes

    def total_tokens(self) -> int:
        return sum(s.length for s in self.seqs)

    def cascade(self) -> CascadeInputs:
        """This step's shared prefixes (the shared-prefix and fork workloads) as cascade
        inputs; other workloads have none."""
        c = self.cfg
        B = self.batch
        if c.kind == "prefix":
            groups, pblk = [list(range(B))], [c.prefix_len // BLOCK_SIZE]
        elif c.kind == "fork":
            groups = [list(range(i * c.samples, (i + 1) * c.samples)) for i in range(c.prompts)]
            pblk = [c.prefix_len // BLOCK_SIZE] * c.prompts
        else:
            groups, pblk = [], []
        return cascade_split(self.seqs, groups, pblk)

    def np(self) -> Dict[str, np.ndarray]:
        """numpy views for the oracle (bf16 as uint16 bits, e4m3 as uint8 codes)."""
        def pool(t):
            return t.numpy().copy() if t.dtype == torch.uint8 else bf16_bits(t).copy()
        return {
            "q": bf16_bits(self.q),
            "k_cache": pool(self.k_cache),
            "v_cache": pool(self.v_cache),
            "k_new": bf16_bits(self.k_new),
            "v_new": bf16_bits(self.v_new),
            "slot_mapping": self.slot_mapping.numpy(),
            "block_tables": self.block_tables.numpy(),
            "context_lens": self.context_lens.numpy(),
            "scales": None if self.scales is None else self.scales.numpy(),
        }


@dataclass
class CascadeInputs:
    """The same decode step split into shared prefixes and per-sequence suffixes."""

    prefix_tables: torch.Tensor  # [P, max_prefix_blocks] int32
    prefix_lens: torch.Tensor    # [P] int32 (multiples of 16)
    member_indptr: torch.Tensor  # [P + 1] int32
    member_seqs: torch.Tensor    # [members] int32
    seq_prefix: torch.Tensor     # [B] int32, -1 without a prefix
    block_tables: torch.Tensor   # [B, max_suffix_blocks] int32: blocks after the prefix
    context_lens: torch.Tensor   # [B] int32: tokens after the prefix
    max_members: int
    max_prefix_len: int


def cascade_split(seqs: List[Sequence_], groups: List[List[int]], prefix_blocks: List[int]) -> CascadeInputs:
    """Cascade inputs for sequences where group i (sequence indices) shares its first
    prefix_blocks[i] blocks (the same physical ids in every member).  Sequences in no group
    keep their whole table."""
    B = len(seqs)
    P = len(groups)
    seq_prefix = [-1] * B
    for i, grp in enumerate(groups):
        for b in grp:
            assert seq_prefix[b] == -1, "a sequence belongs to at most one prefix"
            assert seqs[b].blocks[: prefix_blocks[i]] == seqs[grp[0]].blocks[: prefix_blocks[i]]
            assert seqs[b].length >= prefix_blocks[i] * BLOCK_SIZE
            seq_prefix[b] = i
    mpb = max([1] + list(prefix_blocks))
    ptab = torch.zeros((max(P, 0), mpb), dtype=torch.int32)
    for i, grp in enumerate(groups):
        ptab[i, : prefix_blocks[i]] = torch.tensor(seqs[grp[0]].blocks[: prefix_blocks[i]], dtype=torch.int32)
    suffix = []
    for b, sq in enumerate(seqs):
        nb = prefix_blocks[seq_prefix[b]] if seq_prefix[b] >= 0 else 0
        suffix.append((sq.blocks[nb:], sq.length - nb * BLOCK_SIZE))
    msb = max([1] + [len(bl) for bl, _ in suffix])
    stab = torch.zeros((B, msb), dtype=torch.int32)
    for b, (bl, _) in enumerate(suffix):
        if bl:
            stab[b, : len(bl)] = torch.tensor(bl, dtype=torch.int32)
    indptr = [0]
    for grp in groups:
        indptr.append(indptr[-1] + len(grp))
    return CascadeInputs(
        prefix_tables=ptab, prefix_lens=torch.tensor([n * BLOCK_SIZE for n in prefix_blocks], dtype=torch.int32),
        member_indptr=torch.tensor(indptr, dtype=torch.int32),
        member_seqs=torch.tensor([b for grp in groups for b in grp], dtype=torch.int32),
        seq_prefix=torch.tensor(seq_prefix, dtype=torch.int32), block_tables=stab,
        context_lens=torch.tensor([n for _, n in suffix], dtype=torch.int32),
        max_members=max([0] + [len(grp) for grp in groups]), max_prefix_len=max([0] + list(prefix_blocks)) * BLOCK_SIZE)


def _lengths(cfg: Config, g: torch.Generator) -> List[int]:
    if cfg.kind == "explicit":
        return list(cfg.lens)
    lo, hi = cfg.len_range
    n = cfg.num_seqs
    draws = torch.randint(lo, hi + 1, (n,), generator=g).tolist()
    if cfg.kind == "uniform":
        return draws
    return [cfg.prefix_len + t for t in draws]  # prefix / fork: shared part + private tail


def _build_sequences(cfg: Config, lens: List[int], g: torch.Generator,
                     contiguous: bool = False) -> tuple[BlockPool, List[Sequence_]]:
    bs = BLOCK_SIZE
    if cfg.kind in ("prefix", "fork"):
        assert cfg.prefix_len % bs == 0, "only full blocks are shared"
        pblocks = cfg.prefix_len // bs
        groups = 1 if cfg.kind == "prefix" else cfg.prompts
        used = groups * pblocks + sum(blocks_for_tokens(n, bs) - pblocks for n in lens)
    else:
        used = sum(blocks_for_tokens(n, bs) for n in lens)
    nb = cfg.pool_blocks if cfg.pool_blocks is not None else int(math.ceil(used * (1.0 + cfg.spare_frac)))
    assert nb >= used
    # shuffled: ids come from a seeded permutation, so consecutive logical blocks land
    # anywhere; contiguous: ids in order, each sequence's blocks side by side in the pool
    pool = BlockPool(nb, bs, generator=None if contiguous else g)
    seqs: List[Sequence_] = []
    if cfg.kind in ("explicit", "uniform"):
        seqs = [allocate_private(pool, n) for n in lens]
    elif cfg.kind == "prefix":
        first = allocate_private(pool, lens[0])
        prefix = first.blocks[: cfg.prefix_len // bs]
        seqs = [first] + [allocate_with_prefix(pool, prefix, n) for n in lens[1:]]
    else:  # fork: prompts x samples, samples of one prompt share its full blocks
        for p in range(cfg.prompts):
            chunk = lens[p * cfg.samples:(p + 1) * cfg.samples]
            first = allocate_private(pool, chunk[0])
            prefix = first.blocks[: cfg.prefix_len // bs]
            seqs.append(first)
            seqs.extend(allocate_with_prefix(pool, prefix, n) for n in chunk[1:])
    return pool, seqs


def make_workload(cfg_or_name, seed: Optional[int] = None, lens: Optional[List[int]] = None,
                  threads: int = 8, layout: str = "shuffled") -> Workload:
    """Build one seeded workload.  `lens` overrides the drawn lengths (same structure).
    layout "contiguous" hands out block ids in order instead of shuffled (the same lengths
    and sharing; the pool values then sit at other physical ids)."""
    if layout not in ("shuffled", "contiguous"):
        raise ValueError(f"layout must be 'shuffled' or 'contiguous', not {layout!r}")
    cfg = cfg_or_name if isinstance(cfg_or_name, Config) else get(cfg_or_name)
    seed = cfg.seed if seed is None else seed
    g = torch.Generator().manual_seed(seed)
    drawn = _lengths(cfg, g)
    if lens is not None:
        assert len(lens) == len(drawn)
        drawn = list(lens)
    pool, seqs = _build_sequences(cfg, drawn, g, contiguous=(layout == "contiguous"))
    nb = pool.num_blocks
    B = len(seqs)
    M = max(len(s.blocks) for s in seqs)
    # Unused table entries hold valid (in-bounds) but meaningless ids: a reader that
    # wrongly uses them reads wrong values instead of leaving the pool.
    pad = torch.randint(0, nb, (B, M), generator=torch.Generator().manual_seed(
        _chunk_seed(seed, _STREAMS["pad"], 0)), dtype=torch.int32)
    tables = pad.clone()
    for b, s in enumerate(seqs):
        tables[b, : len(s.blocks)] = torch.tensor(s.blocks, dtype=torch.int32)
    ctx = torch.tensor([s.length for s in seqs], dtype=torch.int32)
    slots = torch.tensor([s.slot(s.length - 1) for s in seqs], dtype=torch.int64)

    shape_pool = (nb, BLOCK_SIZE, cfg.hkv, cfg.d)
    q = randn_bf16((B, cfg.hq, cfg.d), seed, "q", threads)
    kp = randn_bf16(shape_pool, seed, "k_pool", threads)
    vp = randn_bf16(shape_pool, seed, "v_pool", threads)
    kn = randn_bf16((B, cfg.hkv, cfg.d), seed, "k_new", threads)
    vn = randn_bf16((B, cfg.hkv, cfg.d), seed, "v_new", threads)
    scales = None
    if cfg.kv_dtype == "e4m3":
        # One fp32 scale per (K or V, kv head): the head's largest magnitude maps to 448,
        # so the stored pool never saturates.  The pool bytes are made with torch's own
        # float8 cast (input preparation, standing in for the prefill that filled it).
        def quant(x: torch.Tensor) -> tuple[torch.Tensor, torch.Tensor]:
            amax = x.float().abs().amax(dim=(0, 1, 3))
            sc = (amax / E4M3_MAX).to(torch.float32)
            y = (x.float() / sc.view(1, 1, -1, 1)).clamp(-E4M3_MAX, E4M3_MAX)
            return y.to(torch.float8_e4m3fn).view(torch.uint8), sc
        kp, ks = quant(kp)
        vp, vs = quant(vp)
        scales = torch.stack([ks, vs]).contiguous()
    return Workload(cfg=cfg, seqs=seqs, num_blocks=nb, q=q, k_cache=kp, v_cache=vp, k_new=kn,
                    v_new=vn, slot_mapping=slots, block_tables=tables.contiguous(),
                    context_lens=ctx, scales=scales)


def sample_pairs(w: Workload, n: int, seed: int = 7) -> np.ndarray:
    """n distinct (b, hq) pairs, always including the longest and shortest sequences."""
    B, hq = w.batch, w.cfg.hq
    g = torch.Generator().manual_seed(seed)
    lens = w.context_lens
    must = {(int(torch.argmax(lens)), 0), (int(torch.argmin(lens)), hq - 1)}
    picks = set(must)
    total = B * hq
    n = min(n, total)
    perm = torch.randperm(total, generator=g).tolist()
    for p in perm:
        if len(picks) >= n:
            break
        picks.add((p // hq, p % hq))
    return np.array(sorted(picks), dtype=np.int32)
