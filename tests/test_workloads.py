"""Host logic: the block allocator's accounting against the pages' worked examples, and
the structure of the five seeded workloads (no GPU)."""
import numpy as np
import pytest
import torch

import workloads as W
from conftest import golden_kv


def test_allocation_example_from_pages():
    g = golden_kv("allocation_example.txt")
    n = int(g["example_tokens"])
    assert W.blocks_for_tokens(int(g["prefill_tokens"])) == int(g["prefill_blocks"])
    assert W.blocks_for_tokens(n) == int(g["paged_blocks"])
    assert W.blocks_for_tokens(n) * 16 == int(g["paged_slots"])
    assert W.wasted_slots(n) == int(g["paged_waste_slots"])
    assert round(100.0 * W.wasted_slots(n) / (W.blocks_for_tokens(n) * 16), 1) == float(g["paged_waste_pct"])
    assert n - 16 * (W.blocks_for_tokens(n) - 1) == int(g["last_block_fill"])
    naive = int(g["naive_max_seq_len"])
    assert naive - n == int(g["naive_waste_slots"])
    assert round(100.0 * (naive - n) / naive, 1) == float(g["naive_waste_pct"])


def test_allocator_walkthrough_of_the_decode_example():
    # prefill 1024 tokens, then decode 10: the 65th block opens at token 1025
    pool = W.BlockPool(1000, generator=torch.Generator().manual_seed(0))
    seq = W.allocate_private(pool, 1024)
    assert len(seq.blocks) == 64
    for pos in range(1024, 1034):
        j, off = W.position_to_block(pos)
        if j == len(seq.blocks):
            seq.blocks += pool.allocate(1)
        seq.length = pos + 1
    assert len(seq.blocks) == 65 and W.wasted_slots(seq.length) == 6
    assert pool.num_free == 1000 - 65
    assert len(set(seq.blocks)) == 65


def test_prefix_example_from_pages():
    g = golden_kv("allocation_example.txt")
    sp, um = int(g["system_prompt_tokens"]), int(g["user_message_tokens"])
    assert W.blocks_for_tokens(sp) == int(g["system_prompt_blocks"])
    assert W.blocks_for_tokens(um) == int(g["user_message_blocks"])
    assert W.blocks_for_tokens(sp) + W.blocks_for_tokens(um) == int(g["request1_blocks"])
    # a second request shares the prompt's 125 blocks (ref_cnt 2) and owns 13 fresh ones
    pool = W.BlockPool(400, generator=torch.Generator().manual_seed(1))
    r1 = W.allocate_private(pool, sp + um)
    r2 = W.allocate_with_prefix(pool, r1.blocks[:125], sp + um)
    assert r2.blocks[:125] == r1.blocks[:125]
    assert not set(r2.blocks[125:]) & set(r1.blocks)
    assert all(pool.ref_cnt[b] == 2 for b in r1.blocks[:125])
    assert pool.num_free == 400 - 138 - 13


def test_best_of_n_example_from_pages():
    g = golden_kv("allocation_example.txt")
    unshared, shared = W.sampling_token_counts(int(g["best_of_prompt_tokens"]),
                                               int(g["best_of_generated_tokens"]),
                                               int(g["best_of_n"]))
    assert (unshared, shared) == (int(g["best_of_unshared"]), int(g["best_of_shared"]))
    # the same case in 16-token blocks: 8 x 132 vs 125 + 8 x 7
    assert W.sampling_block_counts(2000, 100, 8) == (1056, 181)


def test_release_and_refcounts():
    pool = W.BlockPool(10)
    a = pool.allocate(3)
    pool.share(a)
    pool.release(a)
    assert pool.num_free == 7
    pool.release(a)
    assert pool.num_free == 10
    with pytest.raises(ValueError):
        pool.release(a)
    with pytest.raises(MemoryError):
        pool.allocate(11)


@pytest.mark.parametrize("name", ["tiny", "llama3_8b", "prefix_shared", "fp8_fork"])
def test_workload_structure(name):
    w = W.make_workload(name)
    c = w.cfg
    B = w.batch
    assert w.q.shape == (B, c.hq, c.d) and w.q.dtype == torch.bfloat16
    assert w.k_cache.shape == (w.num_blocks, 16, c.hkv, c.d)
    assert w.block_tables.dtype == torch.int32 and w.context_lens.dtype == torch.int32
    assert w.slot_mapping.dtype == torch.int64 and w.slot_mapping.shape == (B,)
    lens = w.context_lens.tolist()
    tables = w.block_tables.numpy()
    assert tables.min() >= 0 and tables.max() < w.num_blocks
    owners = {}
    for b, s in enumerate(w.seqs):
        assert len(s.blocks) == W.blocks_for_tokens(lens[b])
        assert list(tables[b, : len(s.blocks)]) == s.blocks
        # the new token goes to position len-1 of its own sequence
        pos = lens[b] - 1
        assert int(w.slot_mapping[b]) == s.blocks[pos // 16] * 16 + pos % 16
        for j, blk in enumerate(s.blocks):
            owners.setdefault(blk, set()).add(b)
    # appends never write a block that another sequence also reads
    for b in range(B):
        blk = int(w.slot_mapping[b]) // 16
        assert owners[blk] == {b}
    if name == "tiny":
        assert lens == [17, 33, 64, 100] and w.num_blocks == 64
        assert int(w.slot_mapping[0]) % 16 == 0 and int(w.slot_mapping[2]) % 16 == 15
    if name == "llama3_8b":
        assert min(lens) >= 512 and max(lens) <= 4096
        used = sum(len(s.blocks) for s in w.seqs)
        assert w.num_blocks == int(np.ceil(used * 1.1))
    if name == "prefix_shared":
        prefix = w.seqs[0].blocks[:128]
        assert all(s.blocks[:128] == prefix for s in w.seqs)
        assert all(2048 + 32 <= n <= 2048 + 512 for n in lens)
    if name == "fp8_fork":
        assert w.k_cache.dtype == torch.uint8 and w.scales.shape == (2, c.hkv)
        for p in range(16):
            grp = w.seqs[p * 8:(p + 1) * 8]
            assert all(s.blocks[:125] == grp[0].blocks[:125] for s in grp)
        assert all(2001 <= n <= 2256 for n in lens)
        assert w.unique_kv_bytes() < w.logical_kv_bytes() / 4


def test_workload_is_deterministic():
    a = W.make_workload("llama3_8b")
    b = W.make_workload("llama3_8b")
    assert torch.equal(a.k_cache.view(torch.int16), b.k_cache.view(torch.int16))
    assert torch.equal(a.block_tables, b.block_tables)
    assert torch.equal(a.q.view(torch.int16), b.q.view(torch.int16))
    c = W.make_workload("llama3_8b", seed=5)
    assert not torch.equal(a.block_tables, c.block_tables)


def test_unique_bytes_count_shared_blocks_once():
    w = W.make_workload("prefix_shared")
    per_tok = 2 * 8 * 128 * 2
    tails = sum(n - 2048 for n in w.context_lens.tolist())
    assert w.unique_kv_bytes() == (2048 + tails) * per_tok
    assert w.logical_kv_bytes() == w.total_tokens() * per_tok


def test_fork_and_copy_on_write_accounting():
    pool = W.BlockPool(20, generator=torch.Generator().manual_seed(2))
    a = W.allocate_private(pool, 37)  # 3 blocks, the last holds 5 tokens
    b = W.fork(pool, a)
    assert b.blocks == a.blocks and all(pool.ref_cnt[x] == 2 for x in a.blocks)
    assert pool.num_free == 17
    # b writes into its shared tail block: it gets a fresh copy, a keeps the original
    pair = W.copy_on_write(pool, b, 2)
    assert pair is not None and pair[0] == a.blocks[2] and pair[1] == b.blocks[2] != a.blocks[2]
    assert pool.ref_cnt[a.blocks[2]] == 1 and pool.ref_cnt[b.blocks[2]] == 1
    assert pool.num_free == 16
    # now a's tail is private: no copy
    assert W.copy_on_write(pool, a, 2) is None
    # full shared blocks keep being shared
    assert pool.ref_cnt[a.blocks[0]] == 2


def test_contiguous_layout_keeps_lengths_and_orders_ids():
    s = W.make_workload("llama3_8b")
    c = W.make_workload("llama3_8b", layout="contiguous")
    assert torch.equal(s.context_lens, c.context_lens) and s.num_blocks == c.num_blocks
    nxt = 0
    for seq in c.seqs:  # sequence after sequence, each one's blocks side by side
        assert seq.blocks == list(range(nxt, nxt + len(seq.blocks)))
        nxt += len(seq.blocks)
    assert s.unique_kv_bytes() == c.unique_kv_bytes()
    with pytest.raises(ValueError):
        W.make_workload("tiny", layout="strided")
