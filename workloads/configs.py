"""The five seeded synthetic decode workloads.

Shapes stand in for the workloads of the pages: GQA heads shaped like Llama-3-8B
(32 query / 8 KV heads, D 128) and Llama-3.1-70B (64 / 8, D 128) from the model
table of habr.com/ru/articles/1021832 section 2; 16-token blocks (section 4); a
2000-token system prompt shared through the block tables (section 7 "Тот самый
Cache Read"); best-of-8 forks of one prompt (actionbridge.io chapter 8); 32K-128K
contexts (section 2 context table); FP8 KV (section 2, --kv-cache-dtype fp8).
No dataset and no trained weights are involved: every value is N(0, 1) from a seed.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional, Tuple


@dataclass(frozen=True)
class Config:
    name: str
    hq: int
    hkv: int
    d: int
    kv_dtype: str  # "bf16" or "e4m3"
    softmax_scale: float
    seed: int
    kind: str  # "explicit" | "uniform" | "prefix" | "fork"
    lens: Tuple[int, ...] = ()  # explicit
    batch: int = 0  # uniform / prefix
    len_range: Tuple[int, int] = (0, 0)  # uniform lengths, or tail lengths for prefix/fork
    prefix_len: int = 0  # prefix / fork prompt length
    prompts: int = 0  # fork
    samples: int = 0  # fork
    pool_blocks: Optional[int] = None  # fixed pool size (else used blocks + spare)
    spare_frac: float = 0.10

    @property
    def g(self) -> int:
        return self.hq // self.hkv

    @property
    def elem_bytes(self) -> int:
        return 1 if self.kv_dtype == "e4m3" else 2

    @property
    def num_seqs(self) -> int:
        if self.kind == "explicit":
            return len(self.lens)
        if self.kind == "fork":
            return self.prompts * self.samples
        return self.batch

    @property
    def max_len_bound(self) -> int:
        if self.kind == "explicit":
            return max(self.lens)
        if self.kind == "uniform":
            return self.len_range[1]
        return self.prefix_len + self.len_range[1]


CONFIGS = {
    "tiny": Config(name="tiny", hq=8, hkv=2, d=64, kv_dtype="bf16", softmax_scale=1.0 / 8.0,
                   seed=1000, kind="explicit", lens=(17, 33, 64, 100), pool_blocks=64),
    "llama3_8b": Config(name="llama3_8b", hq=32, hkv=8, d=128, kv_dtype="bf16",
                        softmax_scale=1.0 / math.sqrt(128.0), seed=1001, kind="uniform", batch=64,
                        len_range=(512, 4096)),
    "prefix_shared": Config(name="prefix_shared", hq=32, hkv=8, d=128, kv_dtype="bf16",
                            softmax_scale=1.0 / math.sqrt(128.0), seed=1002, kind="prefix",
                            batch=256, prefix_len=2048, len_range=(32, 512)),
    "long_context_70b": Config(name="long_context_70b", hq=64, hkv=8, d=128, kv_dtype="bf16",
                               softmax_scale=1.0 / math.sqrt(128.0), seed=1003, kind="uniform",
                               batch=8, len_range=(32768, 131072)),
    "fp8_fork": Config(name="fp8_fork", hq=32, hkv=8, d=128, kv_dtype="e4m3",
                       softmax_scale=1.0 / math.sqrt(128.0), seed=1004, kind="fork", prompts=16,
                       samples=8, prefix_len=2000, len_range=(1, 256)),
}

ORDER = ["tiny", "llama3_8b", "prefix_shared", "long_context_70b", "fp8_fork"]


def get(name_or_index) -> Config:
    if isinstance(name_or_index, int):
        return CONFIGS[ORDER[name_or_index]]
    return CONFIGS[name_or_index]
