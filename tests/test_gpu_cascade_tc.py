"""The tcgen05 prefix pass of cascade decode on shapes the workload tests do not reach:
several 128-row query tiles with a ragged last tile, one split longer than the load ring
(4 stages of 64 keys in flight, 3 expanded stages for E4M3 pools), a partial last stage,
and scores that keep growing along the prefix, so that rows move their reference max and
the output accumulated in tensor memory is rescaled.  PKV_PREFIX_SPLIT_BLOCKS fixes the
blocks per split so that small cases still run long splits.

Reference: the oracle's plain decode over each sequence's whole table -- attention over the
prefix keys and over the own keys combine exactly (habr.com/ru/articles/1021832, section 3,
running max and sum with the rescale exp(m_old - m_new))."""
import os
from contextlib import contextmanager

import pytest
import torch

import oracle
import workloads as W
from gpu_helpers import assert_close, e4m3_vmax, fp16_weight_atol

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


@contextmanager
def env(**kv):
    old = {k: os.environ.get(k) for k in kv}
    try:
        for k, v in kv.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = str(v)
        yield
    finally:
        for k, v in old.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v


def build(hkv, g, d, members, pblocks, seed, grow=0.0, no_own=0, own_range=(1, 40)):
    """`members` sequences share a prefix of `pblocks` blocks and own `own_range` tokens each (the
    first `no_own` members none: the prefix is their whole context); with grow > 0 the K rows
    of prefix block j are multiplied by (1 + grow * j) before rounding to bf16, so later keys
    score higher and the running max climbs stage after stage."""
    gen = torch.Generator().manual_seed(seed)
    own = torch.randint(own_range[0], own_range[1] + 1, (members,), generator=gen).tolist()
    own = [0] * no_own + own[no_own:]
    nb = pblocks + sum(W.blocks_for_tokens(n) for n in own) + 8
    pool = W.BlockPool(nb, generator=gen)
    prefix = pool.allocate(pblocks)
    seqs = [W.Sequence_(pblocks * 16 + n, list(prefix) + pool.allocate(W.blocks_for_tokens(n))) for n in own]
    c = W.cascade_split(seqs, [list(range(members))], [pblocks])
    kp = W.randn_bf16((nb, 16, hkv, d), seed, "k_pool").float()
    if grow:
        for j, blk in enumerate(prefix):
            kp[blk] *= 1.0 + grow * j
    kp = kp.to(torch.bfloat16)
    vp = W.randn_bf16((nb, 16, hkv, d), seed, "v_pool")
    q = W.randn_bf16((members, hkv * g, d), seed, "q")
    full = torch.zeros((members, max(len(s.blocks) for s in seqs)), dtype=torch.int32)
    for b, s in enumerate(seqs):
        full[b, : len(s.blocks)] = torch.tensor(s.blocks, dtype=torch.int32)
    lens = torch.tensor([s.length for s in seqs], dtype=torch.int32)
    return c, kp, vp, q, full, lens


def quant_e4m3(x):
    sc = (x.float().abs().amax(dim=(0, 1, 3)) / 448.0).to(torch.float32)
    return (x.float() / sc.view(1, 1, -1, 1)).to(torch.float8_e4m3fn).view(torch.uint8), sc


def run(pkv, c, kd, vd, q, scale, scales=None):
    dev = "cuda"
    out = torch.empty(q.shape, dtype=torch.float32, device=dev)
    pkv.cascade_decode_attention(q.to(dev), kd, vd, c.prefix_tables.to(dev), c.prefix_lens.to(dev),
                                 c.member_indptr.to(dev), c.member_seqs.to(dev), c.seq_prefix.to(dev),
                                 c.block_tables.to(dev), c.context_lens.to(dev), scale, out,
                                 max_members=c.max_members, max_prefix_len=c.max_prefix_len,
                                 max_context_len=max(16, int(c.context_lens.max())),
                                 scales=None if scales is None else scales.to(dev))
    torch.cuda.synchronize()
    assert pkv.check_device_status() == 0
    return out.cpu().double().numpy()


# (hkv, g, d, members, prefix blocks, blocks per split): 296 rows = 3 tiles (40 in the last);
# 26 blocks in one split = 7 stages, the last holding 2 blocks; then two splits of 16 + 10
@pytest.mark.parametrize("hkv,g,d,members,pblocks,split",
                         [(2, 8, 128, 37, 26, 1000), (2, 8, 128, 37, 26, 16), (1, 4, 64, 50, 30, 1000),
                          (3, 2, 128, 70, 21, 8)])
def test_tiles_and_long_splits(pkv, hkv, g, d, members, pblocks, split):
    c, kp, vp, q, full, lens = build(hkv, g, d, members, pblocks, seed=100 + members + d)
    scale = d ** -0.5
    with env(PKV_PREFIX_SPLIT_BLOCKS=split):
        got = run(pkv, c, kp.cuda(), vp.cuda(), q, scale)
    ref = oracle.decode_all(W.bf16_bits(q), W.bf16_bits(kp), W.bf16_bits(vp), oracle.KV_BF16, full.numpy(),
                            lens.numpy(), scale)
    assert_close(got, ref, "bf16", f"hkv={hkv} g={g} d={d} members={members} split={split}")
    assert_close(got, ref, "fp32", f"hkv={hkv} g={g} d={d} members={members} split={split}")


@pytest.mark.parametrize("d", [64, 128])
def test_growing_scores_rescale(pkv, d):
    c, kp, vp, q, full, lens = build(2, 4, d, 40, 24, seed=300 + d, grow=0.6)
    scale = d ** -0.5
    with env(PKV_PREFIX_SPLIT_BLOCKS=1000):
        got = run(pkv, c, kp.cuda(), vp.cuda(), q, scale)
    ref = oracle.decode_all(W.bf16_bits(q), W.bf16_bits(kp), W.bf16_bits(vp), oracle.KV_BF16, full.numpy(),
                            lens.numpy(), scale)
    assert_close(got, ref, "bf16", f"growing scores d={d}")
    assert_close(got, ref, "fp32", f"growing scores d={d}")


@pytest.mark.parametrize("d,grow", [(128, 0.0), (64, 0.0), (128, 0.6)])
def test_e4m3_tiles_and_rescale(pkv, d, grow):
    c, kp, vp, q, full, lens = build(2, 8, d, 21, 27, seed=500 + d, grow=grow)
    k8, ks = quant_e4m3(kp)
    v8, vs = quant_e4m3(vp)
    scales = torch.stack([ks, vs]).contiguous()
    scale = d ** -0.5
    with env(PKV_PREFIX_SPLIT_BLOCKS=1000):
        got = run(pkv, c, k8.cuda(), v8.cuda(), q, scale, scales=scales)
    ref = oracle.decode_all(W.bf16_bits(q), k8.numpy(), v8.numpy(), oracle.KV_E4M3, full.numpy(), lens.numpy(),
                            scale, scales=scales.numpy())
    assert_close(got, ref, "fp8", f"e4m3 d={d} grow={grow}")
    assert_close(got, ref, fp16_weight_atol(e4m3_vmax(v8.numpy(), scales.numpy())), f"e4m3 d={d} grow={grow}, fp16 weights")


def test_many_short_splits_are_capped(pkv):
    """A forced split of 4 blocks over a 200-block prefix would give 50 prefix records per
    sequence; the planner caps them at 16 (longer splits) and the result is unchanged."""
    c, kp, vp, q, full, lens = build(1, 4, 128, 9, 200, seed=77)
    scale = 128 ** -0.5
    with env(PKV_PREFIX_SPLIT_BLOCKS=4):
        got = run(pkv, c, kp.cuda(), vp.cuda(), q, scale)
    ref = oracle.decode_all(W.bf16_bits(q), W.bf16_bits(kp), W.bf16_bits(vp), oracle.KV_BF16, full.numpy(),
                            lens.numpy(), scale)
    assert_close(got, ref, "bf16", "capped prefix splits")
    assert_close(got, ref, "fp32", "capped prefix splits")


@pytest.mark.parametrize("fp8", [False, True])
@pytest.mark.parametrize("defer,per_sm", [("0", "1"), ("1", "1"), ("0", "2"), ("1", "2")])
def test_merge_placement_and_prefix_occupancy(pkv, fp8, defer, per_sm):
    """The prefix records merged in the decode CTA (0) or by the merge kernel after it (1),
    with the prefix pass planned for one or two CTAs per SM: the same result, including
    members without blocks of their own (the prefix alone)."""
    c, kp, vp, q, full, lens = build(2, 4, 128, 45, 40, seed=900 + int(fp8), no_own=3)
    scale = 128 ** -0.5
    if fp8:
        k8, ks = quant_e4m3(kp)
        v8, vs = quant_e4m3(vp)
        scales = torch.stack([ks, vs]).contiguous()
        with env(PKV_CASCADE_DEFER=defer, PKV_PREFIX_CTAS_PER_SM=per_sm, PKV_PREFIX_SPLIT_BLOCKS=8):
            got = run(pkv, c, k8.cuda(), v8.cuda(), q, scale, scales=scales)
        ref = oracle.decode_all(W.bf16_bits(q), k8.numpy(), v8.numpy(), oracle.KV_E4M3, full.numpy(), lens.numpy(),
                                scale, scales=scales.numpy())
        assert_close(got, ref, "fp8", f"e4m3 defer={defer} per_sm={per_sm}")
        assert_close(got, ref, fp16_weight_atol(e4m3_vmax(v8.numpy(), scales.numpy())),
                     f"e4m3 defer={defer} per_sm={per_sm}, fp16 weights")
    else:
        with env(PKV_CASCADE_DEFER=defer, PKV_PREFIX_CTAS_PER_SM=per_sm, PKV_PREFIX_SPLIT_BLOCKS=8):
            got = run(pkv, c, kp.cuda(), vp.cuda(), q, scale)
        ref = oracle.decode_all(W.bf16_bits(q), W.bf16_bits(kp), W.bf16_bits(vp), oracle.KV_BF16, full.numpy(),
                                lens.numpy(), scale)
        assert_close(got, ref, "bf16", f"bf16 defer={defer} per_sm={per_sm}")
        assert_close(got, ref, "fp32", f"bf16 defer={defer} per_sm={per_sm}")


@pytest.mark.parametrize("fp8", [False, True])
@pytest.mark.parametrize("defer", ["0", "1"])
def test_prefix_and_suffix_records_beyond_64(pkv, fp8, defer):
    """16 prefix records (4-block splits of a 64-block prefix) plus 16-token partitions of
    1,000-1,200 own tokens (63-75 partitions): 79-91 records per (sequence, kv head), past
    the 64 whose (max, sum) pairs the merge kernel holds in lanes."""
    c, kp, vp, q, full, lens = build(2, 4, 128, 5, 64, seed=1300 + int(fp8), own_range=(1000, 1200))
    scale = 128 ** -0.5
    knobs = dict(PKV_CASCADE_DEFER=defer, PKV_PREFIX_SPLIT_BLOCKS=4, PKV_SPLIT_TOKENS=16)
    if fp8:
        k8, ks = quant_e4m3(kp)
        v8, vs = quant_e4m3(vp)
        scales = torch.stack([ks, vs]).contiguous()
        with env(**knobs):
            got = run(pkv, c, k8.cuda(), v8.cuda(), q, scale, scales=scales)
        ref = oracle.decode_all(W.bf16_bits(q), k8.numpy(), v8.numpy(), oracle.KV_E4M3, full.numpy(), lens.numpy(),
                                scale, scales=scales.numpy())
        assert_close(got, ref, "fp8", f"e4m3 records > 64, defer={defer}")
        assert_close(got, ref, fp16_weight_atol(e4m3_vmax(v8.numpy(), scales.numpy())),
                     f"e4m3 records > 64, defer={defer}, fp16 weights")
    else:
        with env(**knobs):
            got = run(pkv, c, kp.cuda(), vp.cuda(), q, scale)
        ref = oracle.decode_all(W.bf16_bits(q), W.bf16_bits(kp), W.bf16_bits(vp), oracle.KV_BF16, full.numpy(),
                                lens.numpy(), scale)
        assert_close(got, ref, "fp32", f"bf16 records > 64, defer={defer}")
