"""The read-only checksum pass (pkv_paged_kv_checksum) against its definition, on the GPU.

Per (sequence b, kv head h): x_t = XOR of the 32-bit words of row t of K (or V), checksum =
XOR over t < len of rotl32(x_t, t mod 32), the rows found through the block table (the
gather of habr.com/ru/articles/1021832, section 4).  The reference below computes it with
numpy from the host copy of the pool; it must match bit for bit, for bf16 and E4M3 pools,
both head sizes, one or many partitions per sequence."""
import numpy as np
import pytest
import torch

import workloads as W
from gpu_helpers import split_tokens, to_dev

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


def checksum_ref(pool: torch.Tensor, tables: np.ndarray, lens: np.ndarray) -> np.ndarray:
    nb, bs, hkv, d = pool.shape
    words = pool.contiguous().view(torch.uint8).numpy().reshape(nb * bs, hkv, -1).view(np.uint32)
    x = np.bitwise_xor.reduce(words, axis=2)  # [slot, kv head]
    out = np.zeros((len(lens), hkv), dtype=np.uint32)
    for b, n in enumerate(lens):
        t = np.arange(n)
        rows = x[tables[b, t // 16].astype(np.int64) * 16 + t % 16]
        r = (t & 31).astype(np.uint32)[:, None]
        rot = (rows << r) | (rows >> ((np.uint32(32) - r) & np.uint32(31)))
        out[b] = np.bitwise_xor.reduce(rot, axis=0) if n else 0
    return out


TINY_E4M3 = W.Config(name="tiny_e4m3", hq=8, hkv=2, d=64, kv_dtype="e4m3", softmax_scale=1.0 / 8.0, seed=1010,
                     kind="explicit", lens=(17, 33, 64, 100), pool_blocks=64)


@pytest.mark.parametrize("cfg", ["tiny", TINY_E4M3, "llama3_8b", "fp8_fork"],
                         ids=["tiny", "tiny_e4m3", "llama3_8b", "fp8_fork"])
@pytest.mark.parametrize("split", [None, 16])
def test_checksum_matches_definition(pkv, cfg, split):
    w = W.make_workload(cfg)
    t = to_dev(w)
    with split_tokens(split):
        got = pkv.kv_checksum(t["k_cache"], t["v_cache"], t["block_tables"], t["context_lens"], scales=t["scales"],
                              max_context_len=int(w.context_lens.max()))
        torch.cuda.synchronize()
    assert pkv.check_device_status() == 0
    got = got.cpu().numpy().view(np.uint32)
    tables, lens = w.block_tables.numpy(), w.context_lens.numpy()
    assert np.array_equal(got[:, :, 0], checksum_ref(w.k_cache, tables, lens)), "K checksums differ"
    assert np.array_equal(got[:, :, 1], checksum_ref(w.v_cache, tables, lens)), "V checksums differ"


def test_checksum_placement_invariant_and_flags_bad_ids(pkv):
    w = W.make_workload("tiny")
    t = to_dev(w)
    base = pkv.kv_checksum(t["k_cache"], t["v_cache"], t["block_tables"], t["context_lens"]).clone()
    perm = torch.randperm(w.num_blocks, generator=torch.Generator().manual_seed(5)).cuda()
    k2, v2 = torch.empty_like(t["k_cache"]), torch.empty_like(t["v_cache"])
    k2[perm], v2[perm] = t["k_cache"], t["v_cache"]
    moved = pkv.kv_checksum(k2, v2, perm[t["block_tables"].long()].int().contiguous(), t["context_lens"])
    assert torch.equal(base, moved)
    assert pkv.check_device_status() == 0
    tb = t["block_tables"].clone()
    tb[0, 0] = w.num_blocks  # outside the pool: read as zeros and flagged
    pkv.kv_checksum(t["k_cache"], t["v_cache"], tb, t["context_lens"])
    assert pkv.check_device_status() == pkv.DEVFLAG_BAD_BLOCK_ID
