"""Seeded synthetic workloads for paged decode (shared by tests, smoke and bench).

Holds input generation and the host block allocator only; none of the method's
arithmetic lives here.
"""
from .allocator import (BLOCK_SIZE, BlockPool, Sequence_, allocate_private, allocate_with_prefix,
                        blocks_for_tokens, copy_on_write, fork, position_to_block,
                        sampling_block_counts, sampling_token_counts, slot_of, wasted_slots)
from .configs import CONFIGS, ORDER, Config, get
from .generate import CascadeInputs, Workload, bf16_bits, cascade_split, make_workload, randn_bf16, sample_pairs

__all__ = [
    "BLOCK_SIZE", "BlockPool", "Sequence_", "allocate_private", "allocate_with_prefix", "copy_on_write", "fork",
    "blocks_for_tokens", "position_to_block", "sampling_block_counts", "sampling_token_counts",
    "slot_of", "wasted_slots", "CONFIGS", "ORDER", "Config", "get", "Workload", "bf16_bits",
    "make_workload", "randn_bf16", "sample_pairs", "CascadeInputs", "cascade_split",
]
