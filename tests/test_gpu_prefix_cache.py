"""The host prefix cache feeding the GPU path: a second request with the same 2000-token
system prompt reuses the first request's 125 cached blocks (habr.com/ru/articles/1021832,
section 7, worked example) and only its 200 new tokens are appended; a repeat of the
first request reuses 137 blocks and recomputes its last, partial block.  Decode over the
resulting block tables must equal the oracle over each request's contiguous K/V."""
import random

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


def tokens(n, seed):
    r = random.Random(seed)
    return [r.randrange(0, 128256) for _ in range(n)]


def test_prefix_cache_hits_feed_decode(pkv):
    from paged_kv_cache_17_gb300.block_manager import BlockManager

    hkv, hq, d, nb, sp, um = 2, 8, 64, 160, 2000, 200
    system, user1, user2 = tokens(sp, 1), tokens(um, 2), tokens(um, 3)
    r1, r2 = system + user1, system + user2
    # K/V rows by position: the system prompt's rows are shared; each user message has its own
    ks, vs = W.randn_bf16((sp, hkv, d), 5, "k_new"), W.randn_bf16((sp, hkv, d), 5, "v_new")
    k1, v1 = W.randn_bf16((um, hkv, d), 6, "k_new"), W.randn_bf16((um, hkv, d), 6, "v_new")
    k2, v2 = W.randn_bf16((um, hkv, d), 7, "k_new"), W.randn_bf16((um, hkv, d), 7, "v_new")
    pool_k, pool_v = W.randn_bf16((nb, 16, hkv, d), 5, "k_pool"), W.randn_bf16((nb, 16, hkv, d), 5, "v_pool")
    kd, vd = pool_k.cuda(), pool_v.cuda()
    kc, vc = W.bf16_bits(pool_k).copy(), W.bf16_bits(pool_v).copy()

    def append(blocks, first_pos, k, v):
        slots = torch.tensor([blocks[p // 16] * 16 + p % 16 for p in range(first_pos, first_pos + k.shape[0])],
                             dtype=torch.int64)
        pkv.paged_kv_append(k.cuda(), v.cuda(), slots.cuda(), kd, vd)
        assert oracle.append(kc, vc, W.bf16_bits(k), W.bf16_bits(v), slots.numpy(), oracle.KV_BF16) == 0

    mgr = BlockManager(nb)
    # request 1: empty cache, all 138 blocks computed, full ones cached, then released
    assert mgr.get_computed_blocks(r1) == []
    b1 = mgr.allocate(138)
    append(b1, 0, torch.cat([ks, k1]), torch.cat([vs, v1]))
    assert mgr.cache_full_blocks(r1, b1) == 137
    mgr.free(b1)
    # request 2: the system prompt's 125 blocks hit, 13 fresh blocks take the new tokens
    h2 = mgr.get_computed_blocks(r2)
    assert h2 == b1[:125]
    b2 = h2 + mgr.allocate(13)
    append(b2, sp, k2, v2)
    # request 3 repeats request 1: 137 blocks hit, the partial last block is recomputed
    h3 = mgr.get_computed_blocks(r1)
    assert h3 == b1[:137]
    b3 = h3 + mgr.allocate(1)
    assert b3[-1] not in b1[:137] and b3[-1] not in b2
    append(b3, 137 * 16, k1[137 * 16 - sp:], v1[137 * 16 - sp:])
    assert [mgr.ref_count(b) for b in b1[:125]] == [2] * 125

    q = W.randn_bf16((2, hq, d), 5, "q")
    tables = torch.tensor([b2, b3], dtype=torch.int32)
    lens = torch.tensor([sp + um, sp + um], dtype=torch.int32)
    out = torch.empty((2, hq, d), dtype=torch.float32, device="cuda")
    pkv.paged_decode_attention(q.cuda(), kd, vd, tables.cuda(), lens.cuda(), 0.125, out)
    torch.cuda.synchronize()
    assert pkv.check_device_status() == 0
    assert np.array_equal(pool_bits(kd), kc) and np.array_equal(pool_bits(vd), vc)
    got = out.cpu().double().numpy()
    ref = oracle.decode_all(W.bf16_bits(q), kc, vc, oracle.KV_BF16, tables.numpy(), lens.numpy(), 0.125)
    assert_close(got, ref, "fp32", "decode over prefix-cache tables")
    # and against each request's K/V as one contiguous sequence, never paged
    qf = q.double().numpy()
    for b, (kk, vv) in enumerate(((torch.cat([ks, k2]), torch.cat([vs, v2])),
                                  (torch.cat([ks, k1]), torch.cat([vs, v1])))):
        K, V = kk.double().numpy(), vv.double().numpy()
        for h in range(hq):
            ref_c = oracle.attention_one(qf[b, h], K[:, h // (hq // hkv)], V[:, h // (hq // hkv)], 0.125)
            assert_close(got[b, h], ref_c, "fp32", f"request {b + 2} head {h} vs contiguous")
