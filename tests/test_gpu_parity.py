"""Parity of the CUDA path (through the C ABI) with the CPU oracle, on the GPU.

Append: bit-exact over the whole pool.  Decode: element by element against the fp64
oracle -- within the bf16-KV tolerance (|err| <= 2e-3 + 1e-2 |ref|) for bf16 output,
3e-2 absolute for E4M3 KV, and a tighter 1e-4 + 1e-4 |ref| for fp32 output (the kernel's
own fp32 arithmetic).  Full outputs on every workload, the long-context one included, in
the launch configuration the benchmark uses.
"""
import os

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from gpu_helpers import (assert_close, gpu_step, oracle_pools_after_append, pool_bits, split_tokens, to_dev)

pytestmark = pytest.mark.gpu
NT = os.cpu_count() or 4


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    __graft_entry__.build()
    import paged_kv_cache_17_gb300 as pkv

    pkv.check_device_status()
    yield pkv
    torch.cuda.synchronize()


def _check_flags(expect=0):
    import paged_kv_cache_17_gb300 as pkv

    assert pkv.check_device_status() == expect


# ------------------------------------------------------------------ append

@pytest.mark.parametrize("name", W.ORDER)
def test_append_bit_exact(name):
    w = W.make_workload(name)
    t, _ = gpu_step(w)
    _, kc, vc = oracle_pools_after_append(w)
    assert np.array_equal(pool_bits(t["k_cache"]), kc), "K pool differs from the oracle"
    assert np.array_equal(pool_bits(t["v_cache"]), vc), "V pool differs from the oracle"
    _check_flags()


def test_append_e4m3_saturates_and_skips_negative_slots():
    import paged_kv_cache_17_gb300 as pkv

    hkv, d, nb = 2, 128, 4
    g = torch.Generator().manual_seed(3)
    k = (torch.randn(6, hkv, d, generator=g) * 300).to(torch.bfloat16)  # beyond +-448 * scale
    v = (torch.randn(6, hkv, d, generator=g) * 0.01).to(torch.bfloat16)
    slots = torch.tensor([0, 17, -1, 63, 5, -7], dtype=torch.int64)
    scales = torch.tensor([[0.5, 2.0], [0.001, 0.01]], dtype=torch.float32)
    kc = torch.zeros(nb, 16, hkv, d, dtype=torch.uint8)
    vc = torch.zeros_like(kc)
    kd, vd = kc.cuda(), vc.cuda()
    pkv.paged_kv_append(k.cuda(), v.cuda(), slots.cuda(), kd, vd, kv_dtype="e4m3", scales=scales.cuda())
    torch.cuda.synchronize()
    kb = W.bf16_bits(k)
    vb = W.bf16_bits(v)
    kn, vn = kc.numpy().copy(), vc.numpy().copy()
    oracle.append(kn, vn, kb, vb, slots.numpy(), oracle.KV_E4M3, scales.numpy())
    assert np.array_equal(kd.cpu().numpy(), kn) and np.array_equal(vd.cpu().numpy(), vn)
    assert (kn.reshape(-1, hkv, d) == 0x7E).any() and (kn.reshape(-1, hkv, d) == 0xFE).any()
    _check_flags()


# ------------------------------------------------------------------ decode, full outputs

@pytest.mark.parametrize("name", ["tiny", "llama3_8b", "prefix_shared", "fp8_fork"])
def test_decode_full_parity(name):
    w = W.make_workload(name)
    t, out32 = gpu_step(w, out_dtype=torch.float32)
    a, kc, vc = oracle_pools_after_append(w)
    ref = oracle.decode_all(a["q"], kc, vc, w.kv_dtype_code, a["block_tables"], a["context_lens"],
                            w.cfg.softmax_scale, scales=a["scales"], nthreads=NT)
    got = out32.cpu().double().numpy()
    assert_close(got, ref, "fp32", f"{name} fp32 out")
    if w.cfg.kv_dtype == "e4m3":
        assert_close(got, ref, "fp8", f"{name} e4m3 KV")
    # bf16 output of the same step (the pool already holds the appended tokens)
    _, out16 = gpu_step(w, out_dtype=torch.bfloat16, append=False, t=t)
    assert_close(out16.cpu().double().numpy(), ref, "bf16", f"{name} bf16 out")
    _check_flags()


def test_decode_long_context_full():
    """Full-size 70B-shaped long-context step (8 sequences of 32K-128K tokens), default
    partitioning as benchmarked: every (b, hq) row against the oracle, bf16 output (the
    bench's) at the bf16-KV tolerance and fp32 output at the fp32 one."""
    w = W.make_workload("long_context_70b")
    t, out16 = gpu_step(w, out_dtype=torch.bfloat16)
    _, out32 = gpu_step(w, out_dtype=torch.float32, append=False, t=t)
    a, kc, vc = oracle_pools_after_append(w)
    ref = oracle.decode_all(a["q"], kc, vc, 0, a["block_tables"], a["context_lens"], w.cfg.softmax_scale,
                            nthreads=NT)
    assert_close(out16.cpu().double().numpy(), ref, "bf16", "long context bf16 out")
    assert_close(out32.cpu().double().numpy(), ref, "fp32", "long context fp32 out")
    _check_flags()


# ------------------------------------------------------------------ partitions / edges

@pytest.mark.parametrize("split", [16, 32, 48, 256])
def test_decode_multi_partition(split):
    cfg = W.Config(name="mixed", hq=32, hkv=8, d=128, kv_dtype="bf16", softmax_scale=0.088, seed=77,
                   kind="uniform", batch=12, len_range=(1, 900))
    w = W.make_workload(cfg)
    with split_tokens(split):
        _, out = gpu_step(w)
    a, kc, vc = oracle_pools_after_append(w)
    ref = oracle.decode_all(a["q"], kc, vc, 0, a["block_tables"], a["context_lens"], cfg.softmax_scale,
                            nthreads=NT)
    assert_close(out.cpu().double().numpy(), ref, "fp32", f"split {split}")
    _check_flags()


@pytest.mark.parametrize("split", [None, 16, 64])
@pytest.mark.parametrize("d,g", [(64, 1), (64, 2), (64, 4), (64, 8), (128, 1), (128, 2), (128, 4), (128, 8)])
def test_e4m3_decode_every_group_size_and_partitions(d, g, split):
    """The E4M3 decode reads its codes from 128-byte (D = 128) or 64-byte (D = 64) swizzled
    tiles straight into the MMA fragments (head-dim permutation for K, byte-permuted token
    pairs for V): every query-group instance, one partition per sequence and 16- or 64-token
    partitions (the merge kernel), lengths 1..300 with partial last blocks."""
    hkv = 2
    cfg = W.Config(name="e4m3_groups", hq=hkv * g, hkv=hkv, d=d, kv_dtype="e4m3", softmax_scale=1.0 / np.sqrt(d),
                   seed=400 + d + 10 * g, kind="uniform", batch=10, len_range=(1, 300))
    w = W.make_workload(cfg)
    with split_tokens(split):
        _, out = gpu_step(w)
    a, kc, vc = oracle_pools_after_append(w)
    ref = oracle.decode_all(a["q"], kc, vc, oracle.KV_E4M3, a["block_tables"], a["context_lens"], cfg.softmax_scale,
                            scales=a["scales"], nthreads=NT)
    got = out.cpu().double().numpy()
    assert_close(got, ref, "fp8", f"e4m3 d={d} g={g} split={split}")
    assert_close(got, ref, "fp32", f"e4m3 d={d} g={g} split={split}")
    _check_flags()


@pytest.mark.parametrize("d,g,kv", [(64, 1, "bf16"), (64, 2, "bf16"), (64, 4, "e4m3"), (64, 8, "bf16"),
                                    (128, 1, "e4m3"), (128, 2, "bf16"), (128, 4, "bf16"), (128, 8, "e4m3")])
def test_decode_edge_lengths_all_variants(d, g, kv):
    hkv = 2
    lens = [1, 15, 16, 17, 31, 33, 63, 64, 65, 127, 128, 129, 200, 0]
    cfg = W.Config(name="edges", hq=hkv * g, hkv=hkv, d=d, kv_dtype=kv, softmax_scale=1.0 / np.sqrt(d),
                   seed=5 + d + g, kind="explicit", lens=tuple(lens))
    # len 0 has no block to append into: build the workload with len 1 there, then mark it empty
    w = W.make_workload(cfg, lens=[max(n, 1) for n in lens])
    w.context_lens[-1] = 0
    w.slot_mapping[-1] = -1
    with split_tokens(64):
        _, out = gpu_step(w)
    a, kc, vc = oracle_pools_after_append(w)
    ref = oracle.decode_all(a["q"], kc, vc, w.kv_dtype_code, a["block_tables"], a["context_lens"],
                            cfg.softmax_scale, scales=a["scales"], nthreads=NT)
    got = out.cpu().double().numpy()
    assert np.all(got[-1] == 0.0), "empty sequence must give zeros"
    assert_close(got, ref, "fp32", f"edges d={d} g={g} {kv}")
    _check_flags()


def test_decode_table_capacity_and_tiny_partitions():
    # every sequence fills its table row completely (len == max_blocks * 16)
    cfg = W.Config(name="cap", hq=16, hkv=4, d=128, kv_dtype="bf16", softmax_scale=0.1, seed=9,
                   kind="explicit", lens=(512, 512, 512))
    w = W.make_workload(cfg)
    assert w.block_tables.shape[1] * 16 == 512
    for split in (16, 512, None):
        with split_tokens(split):
            _, out = gpu_step(w, append=False)
        a, kc, vc = oracle_pools_after_append(w, append=False)
        ref = oracle.decode_all(a["q"], kc, vc, 0, a["block_tables"], a["context_lens"], 0.1, nthreads=NT)
        assert_close(out.cpu().double().numpy(), ref, "fp32", f"capacity split {split}")
    _check_flags()


# ------------------------------------------------------------------ determinism / invariances

def test_decode_bitwise_deterministic_and_placement_invariant():
    w = W.make_workload("llama3_8b")
    t = to_dev(w)
    _, o1 = gpu_step(w, t=t)
    _, o2 = gpu_step(w, append=False, t=t)
    assert torch.equal(o1, o2), "two runs differ"
    # move every physical block to another place; rewrite the tables accordingly
    nb = w.num_blocks
    perm = torch.randperm(nb, generator=torch.Generator().manual_seed(11)).cuda()
    k2 = torch.empty_like(t["k_cache"])
    v2 = torch.empty_like(t["v_cache"])
    k2[perm] = t["k_cache"]
    v2[perm] = t["v_cache"]
    t2 = dict(t, k_cache=k2, v_cache=v2, block_tables=perm[t["block_tables"].long()].int().contiguous())
    _, o3 = gpu_step(w, append=False, t=t2)
    assert torch.equal(o1, o3), "output depends on physical placement"
    _check_flags()


def test_prefix_shared_outputs_bitwise_consistent():
    """Sequences that read the same prefix blocks with the same q give identical bits
    (prefix KV identical across requests: ml-canon.vercel.app prefix-caching card)."""
    w = W.make_workload("prefix_shared")
    t = to_dev(w)
    B = w.batch
    t["q"] = t["q"][:1].expand(B, -1, -1).contiguous()
    t["context_lens"] = torch.full((B,), 2048, dtype=torch.int32, device="cuda")
    _, out = gpu_step(w, append=False, t=t)
    assert all(torch.equal(out[0], out[i]) for i in range(1, B)), "shared-prefix outputs differ"
    # two sequences whose private tails hold equal bits also agree bit for bit
    t["context_lens"] = w.context_lens.cuda()
    s0, s1 = w.seqs[0], w.seqs[1]
    n = min(s0.length, s1.length)
    t["context_lens"][0] = n
    t["context_lens"][1] = n
    for j in range(128, (n + 15) // 16):
        t["k_cache"][s1.blocks[j]] = t["k_cache"][s0.blocks[j]]
        t["v_cache"][s1.blocks[j]] = t["v_cache"][s0.blocks[j]]
    _, out2 = gpu_step(w, append=False, t=t)
    assert torch.equal(out2[0], out2[1])
    _check_flags()


# ------------------------------------------------------------------ device-side checks

def test_device_checks_flag_bad_inputs_without_faulting():
    import paged_kv_cache_17_gb300 as pkv

    w = W.make_workload("tiny")
    t = to_dev(w)
    nb = w.num_blocks
    # a slot past the pool is skipped and flagged; the pool is left untouched
    before = t["k_cache"].clone()
    bad = t["slot_mapping"].clone()
    bad[0] = nb * 16 + 3
    bad[1:] = -1
    pkv.paged_kv_append(t["k_new"], t["v_new"], bad, t["k_cache"], t["v_cache"])
    assert pkv.check_device_status() == pkv.DEVFLAG_BAD_SLOT
    assert torch.equal(before, t["k_cache"])
    # a block id just past the pool (and a negative one) read as zeros and are flagged
    tb = t["block_tables"].clone()
    tb[0, 0] = nb
    tb[1, 0] = -1
    out = torch.empty(w.q.shape, dtype=torch.float32, device="cuda")
    pkv.paged_decode_attention(t["q"], t["k_cache"], t["v_cache"], tb, t["context_lens"], 0.125, out)
    assert pkv.check_device_status() == pkv.DEVFLAG_BAD_BLOCK_ID
    assert torch.isfinite(out).all()
    # a context length beyond the table capacity is clamped and flagged
    cl = t["context_lens"].clone()
    cl[2] = 10_000
    pkv.paged_decode_attention(t["q"], t["k_cache"], t["v_cache"], t["block_tables"], cl, 0.125, out)
    assert pkv.check_device_status() == pkv.DEVFLAG_BAD_CONTEXT_LEN
    assert pkv.check_device_status() == 0


def test_workspace_needs_no_initialisation():
    """A workspace full of garbage (NaN bit patterns) gives the same, correct output: every
    partial record the merge reads was written by the same call."""
    import paged_kv_cache_17_gb300 as pkv

    w = W.make_workload("llama3_8b")
    t = to_dev(w)
    B, hq, hkv, d = w.batch, w.cfg.hq, w.cfg.hkv, w.cfg.d
    with split_tokens(256):
        need = pkv.workspace_size(B, hq, hkv, d, 4096)
        assert need > 0
        ws = torch.full((need,), 0xFF, dtype=torch.uint8, device="cuda")
        out = torch.empty(w.q.shape, dtype=torch.float32, device="cuda")
        outs = []
        for _ in range(2):
            pkv.paged_decode_attention(t["q"], t["k_cache"], t["v_cache"], t["block_tables"], t["context_lens"],
                                       w.cfg.softmax_scale, out, max_context_len=4096, workspace=ws)
            torch.cuda.synchronize()
            outs.append(out.clone())
            ws.fill_(0xFF)
    assert torch.equal(outs[0], outs[1]) and bool(torch.isfinite(outs[0]).all())
    a, kc, vc = oracle_pools_after_append(w, append=False)
    pairs = W.sample_pairs(w, 24, seed=2)
    ref = oracle.decode_pairs(a["q"], kc, vc, 0, a["block_tables"], a["context_lens"], w.cfg.softmax_scale, pairs,
                              nthreads=NT)
    assert_close(outs[0].cpu().double().numpy()[pairs[:, 0], pairs[:, 1]], ref, "fp32", "garbage workspace")
    small = torch.zeros(need // 2, dtype=torch.uint8, device="cuda")
    with split_tokens(256):
        with pytest.raises(pkv.PkvError) as ei:
            pkv.paged_decode_attention(t["q"], t["k_cache"], t["v_cache"], t["block_tables"], t["context_lens"],
                                       w.cfg.softmax_scale, out, max_context_len=4096, workspace=small)
    assert ei.value.status == pkv.PKV_ERR_WORKSPACE


@pytest.mark.parametrize("name", ["llama3_8b", "fp8_fork"])
def test_repeated_decodes_give_identical_bits(name):
    """Ten plain decodes back to back on the same inputs give the same bits (the ring's
    generic-proxy reads are fenced before TMA refills their stage)."""
    w = W.make_workload(name)
    t = to_dev(w)
    outs = [gpu_step(w, append=False, t=t)[1].cpu() for _ in range(10)]
    assert all(torch.equal(o, outs[0]) for o in outs[1:]), "repeated decodes differ"
    _check_flags()
