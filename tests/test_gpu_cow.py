"""Copy-on-write on the GPU: the block copy against the oracle (bit-exact), and a fork whose
two sequences both append into their shared tail block (the pages' copy-on-write
paragraph: the writer gets a copy, the original stays untouched), decoded afterwards."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from gpu_helpers import assert_close, pool_bits

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


def disjoint_pairs(nb, n, seed):
    perm = torch.randperm(nb, generator=torch.Generator().manual_seed(seed))
    return torch.stack([perm[:n], perm[n:2 * n]], dim=1).contiguous()  # no dst is a src


@pytest.mark.parametrize("name", ["llama3_8b", "fp8_fork", "tiny"])
def test_copy_blocks_bit_exact(pkv, name):
    w = W.make_workload(name)
    kd, vd = w.k_cache.cuda(), w.v_cache.cuda()
    n = min(300, w.num_blocks // 2)
    pairs = disjoint_pairs(w.num_blocks, n, 5)
    pairs[0, 1] = pairs[0, 0] if n > 1 else pairs[0, 1]  # one self-copy: a no-op
    sc = None if w.scales is None else w.scales.cuda()
    pkv.copy_blocks(pairs.cuda(), kd, vd, scales=sc)
    torch.cuda.synchronize()
    a = w.np()
    kc, vc = a["k_cache"], a["v_cache"]
    assert oracle.copy_blocks(kc, vc, pairs.numpy()) == 0
    assert np.array_equal(pool_bits(kd), kc) and np.array_equal(pool_bits(vd), vc)
    assert pkv.check_device_status() == 0
    # a pair outside the pool is skipped and flagged; nothing else moves
    bad = torch.tensor([[0, w.num_blocks], [-3, 1]], dtype=torch.int64).cuda()
    before = kd.clone()
    pkv.copy_blocks(bad, kd, vd, scales=sc)
    assert pkv.check_device_status() == pkv.DEVFLAG_BAD_BLOCK_ID
    assert torch.equal(before, kd)


def test_fork_copy_on_write_then_append_and_decode(pkv):
    hkv, hq, d, nb = 2, 8, 64, 32
    g = torch.Generator().manual_seed(21)
    pool = W.BlockPool(nb, generator=g)
    a = W.allocate_private(pool, 37)  # tokens 0..36 cached; tail block holds 5
    b = W.fork(pool, a)               # a second sample of the same prompt
    kp = W.randn_bf16((nb, 16, hkv, d), 7, "k_pool")
    vp = W.randn_bf16((nb, 16, hkv, d), 7, "v_pool")
    knew = W.randn_bf16((2, hkv, d), 7, "k_new")
    vnew = W.randn_bf16((2, hkv, d), 7, "v_new")
    q = W.randn_bf16((2, hq, d), 7, "q")
    # both samples append token 37 into logical block 2, which they share: b copies first
    pair = W.copy_on_write(pool, b, 2)
    assert pair is not None and W.copy_on_write(pool, a, 2) is None
    a.length = b.length = 38
    slots = torch.tensor([a.slot(37), b.slot(37)], dtype=torch.int64)
    tables = torch.tensor([a.blocks, b.blocks], dtype=torch.int32)
    lens = torch.tensor([38, 38], dtype=torch.int32)
    # GPU: copy, append, decode
    kd, vd = kp.cuda(), vp.cuda()
    pkv.copy_blocks(torch.tensor([pair], dtype=torch.int64).cuda(), kd, vd)
    pkv.paged_kv_append(knew.cuda(), vnew.cuda(), slots.cuda(), kd, vd)
    out = torch.empty((2, hq, d), dtype=torch.float32, device="cuda")
    pkv.paged_decode_attention(q.cuda(), kd, vd, tables.cuda(), lens.cuda(), 0.125, out)
    torch.cuda.synchronize()
    assert pkv.check_device_status() == 0
    # oracle: the same three steps on the host
    kc, vc = W.bf16_bits(kp).copy(), W.bf16_bits(vp).copy()
    assert oracle.copy_blocks(kc, vc, np.array([pair])) == 0
    assert oracle.append(kc, vc, W.bf16_bits(knew), W.bf16_bits(vnew), slots.numpy(), oracle.KV_BF16) == 0
    assert np.array_equal(pool_bits(kd), kc) and np.array_equal(pool_bits(vd), vc)
    ref = oracle.decode_all(W.bf16_bits(q), kc, vc, oracle.KV_BF16, tables.numpy(), lens.numpy(), 0.125)
    assert_close(out.cpu().double().numpy(), ref, "fp32", "fork + copy-on-write")
    # the shared history is the same bits in both copies; the appended tokens differ
    src, dst = pair
    assert np.array_equal(kc[dst, :5], kc[src, :5]) and not np.array_equal(kc[dst, 5], kc[src, 5])
