"""Cascade (two-level) decode on the GPU: shared prefixes attended once for all their
members on the tensor cores, each sequence's own blocks by the decode kernel, merged with
log-sum-exp weights.  The reference is the oracle's plain decode over each sequence's
whole table (prefix blocks, then its own): the split is exact (habr.com/ru/articles/1021832,
section 3).  bf16 pools: the prefix pass feeds its tensor-core P V product the softmax
weights as a bf16 hi + lo pair (about 16 significant bits), so fp32 outputs are held to the
fp32-output tolerance (1e-4 + 1e-4 |ref|) as well as the bf16-KV one.  E4M3 pools: the
weights enter as fp16, so besides the 3e-2 bound of E4M3 KV the output must stay within
2^-10 max|V| (+1e-4) of the oracle, the rounding bound of fp16 weights."""
import os
from contextlib import contextmanager

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from gpu_helpers import (assert_close, e4m3_vmax, fp16_weight_atol, oracle_pools_after_append, split_tokens,
                         to_dev)

pytestmark = pytest.mark.gpu
NT = os.cpu_count() or 4


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
            os.environ[k] = str(v)
        yield
    finally:
        for k, v in old.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v


def run_cascade(pkv, q, kd, vd, c: W.CascadeInputs, scale, out_dtype=torch.float32):
    dev = q.device
    out = torch.empty(q.shape, dtype=out_dtype, device=dev)
    pkv.cascade_decode_attention(q, kd, vd, c.prefix_tables.to(dev), c.prefix_lens.to(dev), c.member_indptr.to(dev),
                                 c.member_seqs.to(dev), c.seq_prefix.to(dev), c.block_tables.to(dev),
                                 c.context_lens.to(dev), scale, out, max_members=c.max_members,
                                 max_prefix_len=c.max_prefix_len,
                                 max_context_len=max(16, int(c.context_lens.max())))
    torch.cuda.synchronize()
    return out


def test_prefix_shared_workload(pkv):
    w = W.make_workload("prefix_shared")
    t = to_dev(w)
    pkv.paged_kv_append(t["k_new"], t["v_new"], t["slot_mapping"], t["k_cache"], t["v_cache"])
    c = w.cascade()
    out = run_cascade(pkv, t["q"], t["k_cache"], t["v_cache"], c, w.cfg.softmax_scale)
    assert pkv.check_device_status() == 0
    a, kc, vc = oracle_pools_after_append(w)
    ref = oracle.decode_all(a["q"], kc, vc, oracle.KV_BF16, a["block_tables"], a["context_lens"],
                            w.cfg.softmax_scale, nthreads=NT)
    got = out.cpu().double().numpy()
    assert_close(got, ref, "fp32", "cascade prefix_shared (every row)")
    assert_close(got, ref, "bf16", "cascade prefix_shared (every row)")
    # and the plain decode over the whole tables gives the same answer within tolerance
    plain = torch.empty_like(out)
    pkv.paged_decode_attention(t["q"], t["k_cache"], t["v_cache"], t["block_tables"], t["context_lens"],
                               w.cfg.softmax_scale, plain, max_context_len=int(w.context_lens.max()))
    torch.cuda.synchronize()
    assert_close(got, plain.cpu().double().numpy(), "fp32", "cascade vs plain decode")


def build_case(hkv, g, d, seed):
    """Seven sequences over a 96-block pool: prefix A (3 blocks: a partial 64-key stage) for
    sequences 0, 2, 5; prefix B (9 blocks) for 1, 3, 6; sequence 4 has none; sequence 5's
    own part is empty; sequence 6 owns one partial block."""
    nb = 96
    gen = torch.Generator().manual_seed(seed)
    pool = W.BlockPool(nb, generator=gen)
    pa, pb = pool.allocate(3), pool.allocate(9)
    own = {0: 37, 1: 100, 2: 16, 3: 250, 4: 77, 5: 0, 6: 5}
    seqs = []
    for b in range(7):
        pre = pa if b in (0, 2, 5) else (pb if b in (1, 3, 6) else [])
        blocks = list(pre) + pool.allocate(W.blocks_for_tokens(own[b]))
        seqs.append(W.Sequence_(len(pre) * 16 + own[b], blocks))
    c = W.cascade_split(seqs, [[0, 2, 5], [1, 3, 6]], [3, 9])
    hq = hkv * g
    kp = W.randn_bf16((nb, 16, hkv, d), seed, "k_pool")
    vp = W.randn_bf16((nb, 16, hkv, d), seed, "v_pool")
    q = W.randn_bf16((7, hq, d), seed, "q")
    full = torch.zeros((7, max(len(s.blocks) for s in seqs)), dtype=torch.int32)
    for b, s in enumerate(seqs):
        full[b, : len(s.blocks)] = torch.tensor(s.blocks, dtype=torch.int32)
    lens = torch.tensor([s.length for s in seqs], dtype=torch.int32)
    return c, kp, vp, q, full, lens


@pytest.mark.parametrize("hkv,g,d", [(2, 4, 128), (1, 8, 128), (4, 1, 64), (2, 2, 64), (3, 8, 64)])
def test_edge_cases(pkv, hkv, g, d):
    c, kp, vp, q, full, lens = build_case(hkv, g, d, seed=11 + g + d)
    scale = d ** -0.5
    out = run_cascade(pkv, q.cuda(), kp.cuda(), vp.cuda(), c, scale)
    assert pkv.check_device_status() == 0
    ref = oracle.decode_all(W.bf16_bits(q), W.bf16_bits(kp), W.bf16_bits(vp), oracle.KV_BF16, full.numpy(),
                            lens.numpy(), scale)
    assert_close(out.cpu().double().numpy(), ref, "bf16", f"cascade edges hkv={hkv} g={g} d={d}")
    assert_close(out.cpu().double().numpy(), ref, "fp32", f"cascade edges hkv={hkv} g={g} d={d}")


@pytest.mark.parametrize("defer", ["0", "1"])
@pytest.mark.parametrize("split", [16, 64])
def test_split_suffixes_merge_with_prefix(pkv, split, defer):
    """Suffixes in several partitions, merged with the prefix records in the merge kernel
    either way; defer=1 also sends single-partition suffixes there."""
    c, kp, vp, q, full, lens = build_case(2, 4, 128, seed=5)
    with split_tokens(split), env(PKV_CASCADE_DEFER=defer):
        out = run_cascade(pkv, q.cuda(), kp.cuda(), vp.cuda(), c, 0.1, out_dtype=torch.bfloat16)
    assert pkv.check_device_status() == 0
    ref = oracle.decode_all(W.bf16_bits(q), W.bf16_bits(kp), W.bf16_bits(vp), oracle.KV_BF16, full.numpy(),
                            lens.numpy(), 0.1)
    assert_close(out.cpu().double().numpy(), ref, "bf16", f"cascade split {split} defer {defer}")


@pytest.mark.parametrize("hkv,g,d", [(2, 4, 128), (1, 8, 128), (4, 1, 64)])
def test_cascade_on_cuda_core_decode(pkv, hkv, g, d):
    """The cascade with the CUDA-core decode form (PKV_DECODE_CUDA_CORES=1) for the
    sequences' own blocks: it merges the prefix records itself."""
    c, kp, vp, q, full, lens = build_case(hkv, g, d, seed=31 + g + d)
    scale = d ** -0.5
    with env(PKV_DECODE_CUDA_CORES=1):
        out = run_cascade(pkv, q.cuda(), kp.cuda(), vp.cuda(), c, scale)
    assert pkv.check_device_status() == 0
    ref = oracle.decode_all(W.bf16_bits(q), W.bf16_bits(kp), W.bf16_bits(vp), oracle.KV_BF16, full.numpy(),
                            lens.numpy(), scale)
    assert_close(out.cpu().double().numpy(), ref, "bf16", f"cascade on CUDA cores hkv={hkv} g={g} d={d}")
    assert_close(out.cpu().double().numpy(), ref, "fp32", f"cascade on CUDA cores hkv={hkv} g={g} d={d}")


def test_no_prefixes_is_plain_decode(pkv):
    w = W.make_workload("tiny")
    t = to_dev(w)
    c = w.cascade()
    assert c.prefix_tables.shape[0] == 0
    out = run_cascade(pkv, t["q"], t["k_cache"], t["v_cache"], c, w.cfg.softmax_scale)
    plain = torch.empty_like(out)
    pkv.paged_decode_attention(t["q"], t["k_cache"], t["v_cache"], t["block_tables"], t["context_lens"],
                               w.cfg.softmax_scale, plain)
    torch.cuda.synchronize()
    assert torch.equal(out, plain)


def test_fp8_fork_workload(pkv):
    w = W.make_workload("fp8_fork")
    t = to_dev(w)
    pkv.paged_kv_append(t["k_new"], t["v_new"], t["slot_mapping"], t["k_cache"], t["v_cache"], scales=t["scales"])
    c = w.cascade()
    dev = t["q"].device
    out = torch.empty(t["q"].shape, dtype=torch.float32, device=dev)
    pkv.cascade_decode_attention(t["q"], t["k_cache"], t["v_cache"], c.prefix_tables.to(dev), c.prefix_lens.to(dev),
                                 c.member_indptr.to(dev), c.member_seqs.to(dev), c.seq_prefix.to(dev),
                                 c.block_tables.to(dev), c.context_lens.to(dev), w.cfg.softmax_scale, out,
                                 max_members=c.max_members, max_prefix_len=c.max_prefix_len,
                                 max_context_len=max(16, int(c.context_lens.max())), scales=t["scales"])
    torch.cuda.synchronize()
    assert pkv.check_device_status() == 0
    a, kc, vc = oracle_pools_after_append(w)
    ref = oracle.decode_all(a["q"], kc, vc, oracle.KV_E4M3, a["block_tables"], a["context_lens"],
                            w.cfg.softmax_scale, scales=a["scales"], nthreads=NT)
    got = out.cpu().double().numpy()
    assert_close(got, ref, "fp8", "cascade fp8_fork (every row)")
    assert_close(got, ref, fp16_weight_atol(e4m3_vmax(vc, a["scales"])), "cascade fp8_fork, fp16-weight bound")


@pytest.mark.parametrize("d", [64, 128])
def test_fp8_edge_cases(pkv, d):
    c, kp, vp, q, full, lens = build_case(2, 4, d, seed=7 + d)
    # quantise the pool with per-head scales (the harness's rule: max |x| -> 448)
    def quant(x):
        sc = (x.float().abs().amax(dim=(0, 1, 3)) / 448.0).to(torch.float32)
        return (x.float() / sc.view(1, 1, -1, 1)).to(torch.float8_e4m3fn).view(torch.uint8), sc
    k8, ks = quant(kp)
    v8, vs = quant(vp)
    scales = torch.stack([ks, vs]).contiguous()
    scale = d ** -0.5
    dev = "cuda"
    out = torch.empty(q.shape, dtype=torch.float32, device=dev)
    pkv.cascade_decode_attention(q.cuda(), k8.cuda(), v8.cuda(), c.prefix_tables.cuda(), c.prefix_lens.cuda(),
                                 c.member_indptr.cuda(), c.member_seqs.cuda(), c.seq_prefix.cuda(),
                                 c.block_tables.cuda(), c.context_lens.cuda(), scale, out, max_members=c.max_members,
                                 max_prefix_len=c.max_prefix_len, max_context_len=max(16, int(c.context_lens.max())),
                                 scales=scales.cuda())
    torch.cuda.synchronize()
    assert pkv.check_device_status() == 0
    ref = oracle.decode_all(W.bf16_bits(q), k8.numpy(), v8.numpy(), oracle.KV_E4M3, full.numpy(), lens.numpy(),
                            scale, scales=scales.numpy())
    got = out.cpu().double().numpy()
    assert_close(got, ref, "fp8", f"cascade fp8 edges d={d}")
    assert_close(got, ref, fp16_weight_atol(e4m3_vmax(v8.numpy(), scales.numpy())),
                 f"cascade fp8 edges d={d}, fp16-weight bound")


def test_cascade_shared_prefix_bitwise_consistent(pkv):
    """The shared-prefix workload's consistency variant through the cascade call: the same q
    for every member gives identical output bits (ml-canon.vercel.app/54-prefix-caching-cacheblend.html,
    "Идея и механизм": the prefix KV is identical across requests), with no own blocks and
    with bit-equal own blocks; members 0 and 200 sit in different 128-row tiles of the
    prefix pass."""
    w = W.make_workload("prefix_shared")
    t = to_dev(w)
    c = w.cascade()
    B = w.batch
    q = t["q"][:1].expand(B, -1, -1).contiguous()
    dev = q.device
    args = dict(max_members=c.max_members, max_prefix_len=c.max_prefix_len)

    def run(lens):
        out = torch.empty(q.shape, dtype=torch.float32, device=dev)
        pkv.cascade_decode_attention(q, t["k_cache"], t["v_cache"], c.prefix_tables.to(dev), c.prefix_lens.to(dev),
                                     c.member_indptr.to(dev), c.member_seqs.to(dev), c.seq_prefix.to(dev),
                                     c.block_tables.to(dev), lens.to(dev), w.cfg.softmax_scale, out,
                                     max_context_len=max(16, int(lens.max())), **args)
        torch.cuda.synchronize()
        assert pkv.check_device_status() == 0
        return out

    out = run(torch.zeros_like(c.context_lens))
    assert all(torch.equal(out[0], out[i]) for i in range(1, B)), "prefix-only outputs differ"
    b0, b1 = 0, 200
    lens = c.context_lens.clone()
    n = int(min(lens[b0], lens[b1]))
    lens[b0] = lens[b1] = n
    for j in range((n + 15) // 16):
        src, dst = int(c.block_tables[b0, j]), int(c.block_tables[b1, j])
        t["k_cache"][dst] = t["k_cache"][src]
        t["v_cache"][dst] = t["v_cache"][src]
    out2 = run(lens)
    assert torch.equal(out2[b0], out2[b1]), "equal suffixes, different bits"


@pytest.mark.parametrize("name", ["prefix_shared", "fp8_fork"])
def test_repeated_calls_give_identical_bits(pkv, name):
    """Ten calls back to back on the same inputs (the workspace reused) give the same bits
    and stay within the oracle's bound each time.  The ring stages of the decode are read
    through the generic proxy and refilled by TMA; a missing proxy fence before a stage's
    release once let a refill land under a pending read, wrong in a few rows per call."""
    from test_gpu_cascade_tc import run

    w = W.make_workload(name)
    t = to_dev(w)
    c = w.cascade()
    outs = [run(pkv, c, t["k_cache"], t["v_cache"], t["q"], w.cfg.softmax_scale, scales=t["scales"])
            for _ in range(10)]
    assert all((o == outs[0]).all() for o in outs[1:]), "repeated calls differ"
    a, kc, vc = oracle_pools_after_append(w, append=False)
    ref = oracle.decode_all(a["q"], kc, vc, w.kv_dtype_code, a["block_tables"], a["context_lens"],
                            w.cfg.softmax_scale, scales=a["scales"], nthreads=NT)
    if w.cfg.kv_dtype == "e4m3":
        assert_close(outs[0], ref, fp16_weight_atol(e4m3_vmax(vc, a["scales"])), f"{name}, repeated")
    else:
        assert_close(outs[0], ref, "fp32", f"{name}, repeated")
