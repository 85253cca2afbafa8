"""The mma.sync prefix pass of cascade decode -- small member groups of an E4M3 pool, at
most 32 query rows per prefix and kv head -- on shapes beyond the fork workload: one and two
16-row slices with a ragged last slice, head dims 64 and 128, query groups of 1 to 8, one
split longer than the 32 KiB load ring and many short splits, prefixes of different lengths
(the shorter ones get empty splits), members whose whole context is the prefix, scores that
grow along the prefix (rows move their reference max and the output is rescaled), the
tcgen05 pass on the same inputs, repeated calls, and block ids outside the pool (read as
zeros and flagged, by both prefix passes and by the E4M3 decode, whose codes also go straight
from the swizzled tiles into the MMA fragments).  PKV_PREFIX_SPLIT_BLOCKS fixes the blocks
per split.

Reference: the oracle's plain decode over each sequence's whole table -- attention over the
prefix keys and over the own keys combine exactly (habr.com/ru/articles/1021832, section 3,
running max and sum with the rescale exp(m_old - m_new)); the fork shape is actionbridge.io
chapter 8's best-of-8 parallel sampling (the samples share the prompt's blocks)."""
import pytest
import torch

import oracle
import workloads as W
from gpu_helpers import assert_close, e4m3_vmax, fp16_weight_atol
from test_gpu_cascade_tc import env, quant_e4m3, run

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


def build_groups(hkv, g, d, groups, seed, grow=0.0, no_own=0, own_range=(1, 40)):
    """Prefix groups given as (members, prefix blocks); each member owns `own_range` tokens
    after its prefix (the first `no_own` members of every group none).  With grow > 0 the K
    rows of prefix block j are scaled by (1 + grow * j) before rounding, so the running max
    climbs along the prefix.  Returns the cascade inputs, the E4M3 pools with their scales,
    q, and each sequence's whole table and length for the oracle."""
    gen = torch.Generator().manual_seed(seed)
    owns = []
    for members, _ in groups:
        own = torch.randint(own_range[0], own_range[1] + 1, (members,), generator=gen).tolist()
        owns.append([0] * no_own + own[no_own:])
    nb = sum(pb for _, pb in groups) + sum(W.blocks_for_tokens(n) for own in owns for n in own) + 8
    pool = W.BlockPool(nb, generator=gen)
    seqs, idx, prefix_blocks, grow_rows = [], [], [], []
    for (members, pblocks), own in zip(groups, owns):
        prefix = pool.allocate(pblocks)
        grow_rows.append(prefix)
        idx.append(list(range(len(seqs), len(seqs) + members)))
        prefix_blocks.append(pblocks)
        for n in own:
            seqs.append(W.Sequence_(pblocks * 16 + n, list(prefix) + pool.allocate(W.blocks_for_tokens(n))))
    c = W.cascade_split(seqs, idx, prefix_blocks)
    kp = W.randn_bf16((nb, 16, hkv, d), seed, "k_pool").float()
    if grow:
        for prefix in grow_rows:
            for j, blk in enumerate(prefix):
                kp[blk] *= 1.0 + grow * j
    kp = kp.to(torch.bfloat16)
    vp = W.randn_bf16((nb, 16, hkv, d), seed, "v_pool")
    k8, ks = quant_e4m3(kp)
    v8, vs = quant_e4m3(vp)
    scales = torch.stack([ks, vs]).contiguous()
    q = W.randn_bf16((len(seqs), hkv * g, d), seed, "q")
    full = torch.zeros((len(seqs), max(len(s.blocks) for s in seqs)), dtype=torch.int32)
    for b, s in enumerate(seqs):
        full[b, : len(s.blocks)] = torch.tensor(s.blocks, dtype=torch.int32)
    lens = torch.tensor([s.length for s in seqs], dtype=torch.int32)
    return c, k8, v8, scales, q, full, lens


def check(pkv, case, d, what, **knobs):
    c, k8, v8, scales, q, full, lens = case
    scale = d ** -0.5
    with env(**knobs):
        got = run(pkv, c, k8.cuda(), v8.cuda(), q, scale, scales=scales)
    ref = oracle.decode_all(W.bf16_bits(q), k8.numpy(), v8.numpy(), oracle.KV_E4M3, full.numpy(), lens.numpy(),
                            scale, scales=scales.numpy())
    assert_close(got, ref, "fp8", what)
    assert_close(got, ref, fp16_weight_atol(e4m3_vmax(v8.numpy(), scales.numpy())), what + ", fp16 weights")
    return got


# (hkv, g, d, members, prefix blocks, blocks per split): 32 rows in two slices with one split
# of 45 blocks (the ring holds 8); 20 rows (a ragged second slice) in 4-block splits; 12 rows
# in one slice; head dim 64 (a 16-stage ring) with 32 and 10 rows; a group of 1 with 9 rows
@pytest.mark.parametrize("hkv,g,d,members,pblocks,split",
                         [(2, 4, 128, 8, 45, 1000), (2, 4, 128, 5, 45, 4), (3, 4, 128, 3, 30, 7),
                          (2, 8, 64, 4, 50, 1000), (1, 2, 64, 5, 33, 8), (4, 1, 128, 9, 20, 1000)])
def test_slices_and_splits(pkv, hkv, g, d, members, pblocks, split):
    case = build_groups(hkv, g, d, [(members, pblocks)], seed=2000 + members * 7 + d + g)
    check(pkv, case, d, f"hkv={hkv} g={g} d={d} members={members} split={split}",
          PKV_PREFIX_PASS="mma", PKV_PREFIX_SPLIT_BLOCKS=split)


@pytest.mark.parametrize("d", [64, 128])
def test_prefixes_of_different_lengths(pkv, d):
    """Three prefixes of 40, 3 and 17 blocks in 8-block splits: 5 records per member, of
    which the 3-block prefix fills one and the 17-block prefix three (the others are empty
    splits); two members per group have no blocks of their own."""
    case = build_groups(2, 4, d, [(8, 40), (6, 3), (4, 17)], seed=2100 + d, no_own=2)
    check(pkv, case, d, f"prefixes of 40, 3 and 17 blocks d={d}", PKV_PREFIX_PASS="mma", PKV_PREFIX_SPLIT_BLOCKS=8)


@pytest.mark.parametrize("members", [3, 8])
def test_growing_scores_rescale(pkv, members):
    case = build_groups(2, 4, 128, [(members, 36)], seed=2200 + members, grow=0.6)
    check(pkv, case, 128, f"growing scores members={members}", PKV_PREFIX_PASS="mma", PKV_PREFIX_SPLIT_BLOCKS=1000)


@pytest.mark.parametrize("defer", ["0", "1"])
def test_tcgen05_pass_on_the_same_inputs(pkv, defer):
    """The tcgen05 pass and the mma.sync pass on one fork-shaped case (8 members x G 4), with
    the prefix records merged in the decode CTA (0) or by the merge kernel (1): both within
    the oracle's bounds."""
    case = build_groups(2, 4, 128, [(8, 30), (8, 22)], seed=2300)
    for kind in ("mma", "tc"):
        check(pkv, case, 128, f"{kind} pass, defer={defer}", PKV_PREFIX_PASS=kind, PKV_CASCADE_DEFER=defer)


def test_repeated_calls_give_identical_bits(pkv):
    """Ten calls on the same inputs give the same bits: the streams of a slice combine in a
    fixed order, and a ring slot is refilled only after both warps of its stream have read it."""
    c, k8, v8, scales, q, full, lens = build_groups(2, 4, 128, [(8, 60), (7, 41)], seed=2400)
    kd, vd = k8.cuda(), v8.cuda()
    with env(PKV_PREFIX_PASS="mma", PKV_PREFIX_SPLIT_BLOCKS=12):
        outs = [run(pkv, c, kd, vd, q, 128 ** -0.5, scales=scales) for _ in range(10)]
    assert all((o == outs[0]).all() for o in outs[1:]), "repeated calls differ"


def _zero_block_reference(case, d, bad_rows):
    """The oracle's answer when the prefix table entries in `bad_rows` ((prefix, block index)
    pairs) point outside the pool: such a block reads as zeros (K and V), so every sequence
    of that prefix sees a zero block in that place."""
    c, k8, v8, scales, q, full, lens = case
    nb = k8.shape[0]
    kz = torch.cat([k8, torch.zeros_like(k8[:1])])  # block nb: all-zero codes
    vz = torch.cat([v8, torch.zeros_like(v8[:1])])
    full = full.clone()
    for pfx, j in bad_rows:
        members = c.member_seqs[c.member_indptr[pfx]:c.member_indptr[pfx + 1]].tolist()
        for b in members:
            full[b, j] = nb
    return oracle.decode_all(W.bf16_bits(q), kz.numpy(), vz.numpy(), oracle.KV_E4M3, full.numpy(), lens.numpy(),
                             d ** -0.5, scales=scales.numpy())


@pytest.mark.parametrize("kind", ["mma", "tc"])
def test_out_of_pool_prefix_block_reads_zeros_and_is_flagged(pkv, kind):
    """A prefix table entry past the pool (and a negative one) is read as a block of zeros by
    either prefix pass and flagged in the device status; nothing else changes."""
    case = build_groups(2, 4, 128, [(8, 30), (5, 20)], seed=2500)
    c = case[0]
    nb = case[1].shape[0]
    c.prefix_tables[0, 3] = nb
    c.prefix_tables[1, 7] = -1
    d = 128
    with env(PKV_PREFIX_PASS=kind, PKV_PREFIX_SPLIT_BLOCKS=8):
        out = torch.empty(case[4].shape, dtype=torch.float32, device="cuda")
        pkv.cascade_decode_attention(case[4].cuda(), case[1].cuda(), case[2].cuda(), c.prefix_tables.cuda(),
                                     c.prefix_lens.cuda(), c.member_indptr.cuda(), c.member_seqs.cuda(),
                                     c.seq_prefix.cuda(), c.block_tables.cuda(), c.context_lens.cuda(), d ** -0.5, out,
                                     max_members=c.max_members, max_prefix_len=c.max_prefix_len,
                                     max_context_len=max(16, int(c.context_lens.max())), scales=case[3].cuda())
        torch.cuda.synchronize()
    assert pkv.check_device_status() == pkv.DEVFLAG_BAD_BLOCK_ID
    ref = _zero_block_reference(case, d, [(0, 3), (1, 7)])
    got = out.cpu().double().numpy()
    assert_close(got, ref, "fp8", f"{kind} pass, out-of-pool prefix blocks")
    assert_close(got, ref, fp16_weight_atol(e4m3_vmax(case[2].numpy(), case[3].numpy())),
                 f"{kind} pass, out-of-pool prefix blocks, fp16 weights")


def test_e4m3_decode_out_of_pool_block_reads_zeros_and_is_flagged(pkv):
    """The E4M3 decode (codes read straight into the MMA fragments from swizzled tiles) reads
    a block id past the pool, or a negative one, as zeros and flags it."""
    c, k8, v8, scales, q, full, lens = build_groups(2, 4, 128, [(6, 10)], seed=2600, own_range=(20, 70))
    nb = k8.shape[0]
    tb = full.clone()
    tb[0, 2] = nb
    tb[3, 12] = -1
    d = 128
    out = torch.empty(q.shape, dtype=torch.float32, device="cuda")
    pkv.paged_decode_attention(q.cuda(), k8.cuda(), v8.cuda(), tb.cuda(), lens.cuda(), d ** -0.5, out,
                               scales=scales.cuda(), max_context_len=int(lens.max()))
    torch.cuda.synchronize()
    assert pkv.check_device_status() == pkv.DEVFLAG_BAD_BLOCK_ID
    kz = torch.cat([k8, torch.zeros_like(k8[:1])])
    vz = torch.cat([v8, torch.zeros_like(v8[:1])])
    tz = tb.clone()
    tz[0, 2] = nb
    tz[3, 12] = nb
    ref = oracle.decode_all(W.bf16_bits(q), kz.numpy(), vz.numpy(), oracle.KV_E4M3, tz.numpy(), lens.numpy(),
                            d ** -0.5, scales=scales.numpy())
    assert_close(out.cpu().double().numpy(), ref, "fp32", "E4M3 decode, out-of-pool blocks")
