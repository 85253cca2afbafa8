"""The cascade call with a workspace of exactly pkv_cascade_workspace_size bytes, on shapes
whose prefix-pass plan takes the most splits: five bf16 prefixes of 76 blocks, 64 members
each with own tails of up to 256 tokens.  The pass's work (2 tiles x 8 kv heads x 76 blocks
per prefix) is under half the decode's, so the planner counts half the SMs as slots, and on
a 152-SM GPU that plan takes 4 splits per prefix where the whole-SM plans take at most 3: the
size query has to cover every plan the call can make.  Sampled rows are checked against the
oracle's plain decode over each sequence's whole table (habr.com/ru/articles/1021832,
section 3: attention over the prefix keys and the own keys combines exactly)."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from gpu_helpers import assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    __graft_entry__.build()
    import paged_kv_cache_17_gb300 as m

    m.check_device_status()
    return m


def build(num_prefixes, members, pblocks, hkv, g, d, own_max, seed):
    gen = torch.Generator().manual_seed(seed)
    owns = [torch.randint(1, own_max + 1, (members,), generator=gen).tolist() for _ in range(num_prefixes)]
    owns[0][0] = own_max  # the longest own context is exactly own_max
    nb = num_prefixes * pblocks + sum(W.blocks_for_tokens(n) for own in owns for n in own) + 8
    pool = W.BlockPool(nb, generator=gen)
    seqs, idx = [], []
    for own in owns:
        prefix = pool.allocate(pblocks)
        idx.append(list(range(len(seqs), len(seqs) + members)))
        for n in own:
            seqs.append(W.Sequence_(pblocks * 16 + n, list(prefix) + pool.allocate(W.blocks_for_tokens(n))))
    c = W.cascade_split(seqs, idx, [pblocks] * num_prefixes)
    kp = W.randn_bf16((nb, 16, hkv, d), seed, "k_pool")
    vp = W.randn_bf16((nb, 16, hkv, d), seed, "v_pool")
    q = W.randn_bf16((len(seqs), hkv * g, d), seed, "q")
    full = torch.zeros((len(seqs), max(len(s.blocks) for s in seqs)), dtype=torch.int32)
    for b, s in enumerate(seqs):
        full[b, : len(s.blocks)] = torch.tensor(s.blocks, dtype=torch.int32)
    lens = torch.tensor([s.length for s in seqs], dtype=torch.int32)
    return c, kp, vp, q, full, lens


def test_workspace_of_the_queried_size_suffices(pkv):
    hkv, g, d, P, members, pblocks, own_max = 8, 4, 128, 5, 64, 76, 256
    c, kp, vp, q, full, lens = build(P, members, pblocks, hkv, g, d, own_max, seed=2600)
    B = q.shape[0]
    mcl = int(c.context_lens.max())
    assert mcl == own_max
    need = pkv.cascade_workspace_size(B, hkv * g, hkv, d, mcl, P, c.max_members, c.max_prefix_len)
    assert need > 0
    dev = "cuda"
    ws = torch.empty(need, dtype=torch.uint8, device=dev)
    out = torch.empty(q.shape, dtype=torch.float32, device=dev)
    pkv.cascade_decode_attention(q.to(dev), kp.to(dev), vp.to(dev), c.prefix_tables.to(dev), c.prefix_lens.to(dev),
                                 c.member_indptr.to(dev), c.member_seqs.to(dev), c.seq_prefix.to(dev),
                                 c.block_tables.to(dev), c.context_lens.to(dev), d ** -0.5, out,
                                 max_members=c.max_members, max_prefix_len=c.max_prefix_len, max_context_len=mcl,
                                 workspace=ws)
    torch.cuda.synchronize()
    assert pkv.check_device_status() == 0
    got = out.cpu().double().numpy()
    # sampled (sequence, query head) rows: every prefix, first and last members, first and last heads
    pairs = np.array([(p * members + m, h) for p in range(P) for m in (0, members - 1) for h in (0, hkv * g - 1)],
                     dtype=np.int32)
    ref = oracle.decode_pairs(W.bf16_bits(q), W.bf16_bits(kp), W.bf16_bits(vp), oracle.KV_BF16, full.numpy(),
                              lens.numpy(), d ** -0.5, pairs, nthreads=4)
    assert_close(got[pairs[:, 0], pairs[:, 1]], ref, "fp32", "sampled rows, workspace of the queried size")
