"""The fused decode step (pkv_paged_append_decode) on the GPU: one launch that appends each
sequence's new token and attends over the cache that holds it (habr.com/ru/articles/1021832,
section 1: a decode step appends the new token's K, V and attends over the whole cache).

It must leave the pool and the output bit for bit as the two calls do (append, then
decode), and agree with the oracle; partitions of 16 tokens put the new token's block in a
later partition than the first; sequences without a new token (slot < 0) and a slot that is
not the table's position len - 1 are covered too."""
import os

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from gpu_helpers import assert_close, oracle_pools_after_append, pool_bits, split_tokens, to_dev

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


def two_calls(pkv, w, t, slots, out_dtype=torch.float32):
    pkv.paged_kv_append(t["k_new"], t["v_new"], slots, t["k_cache"], t["v_cache"], scales=t["scales"])
    out = torch.empty(t["q"].shape, dtype=out_dtype, device="cuda")
    pkv.paged_decode_attention(t["q"], t["k_cache"], t["v_cache"], t["block_tables"], t["context_lens"],
                               w.cfg.softmax_scale, out, scales=t["scales"], max_context_len=int(w.context_lens.max()))
    torch.cuda.synchronize()
    return out


def fused(pkv, w, t, slots, out_dtype=torch.float32):
    out = torch.empty(t["q"].shape, dtype=out_dtype, device="cuda")
    pkv.paged_append_decode(t["k_new"], t["v_new"], slots, t["q"], t["k_cache"], t["v_cache"], t["block_tables"],
                            t["context_lens"], w.cfg.softmax_scale, out, scales=t["scales"],
                            max_context_len=int(w.context_lens.max()))
    torch.cuda.synchronize()
    return out


TINY_E4M3 = W.Config(name="tiny_e4m3", hq=8, hkv=2, d=64, kv_dtype="e4m3", softmax_scale=1.0 / 8.0, seed=1010,
                     kind="explicit", lens=(17, 33, 64, 100), pool_blocks=64)


@pytest.mark.parametrize("cfg,split", [("tiny", None), (TINY_E4M3, None), ("tiny", 16), ("llama3_8b", None),
                                       ("llama3_8b", 16), ("fp8_fork", None), ("long_context_70b", None)],
                         ids=["tiny", "tiny_e4m3", "tiny-16", "llama3_8b", "llama3_8b-16", "fp8_fork", "long_context"])
def test_fused_step_equals_the_two_calls_and_the_oracle(pkv, cfg, split):
    w = W.make_workload(cfg)
    assert w.k_new.shape[0] == w.batch  # one new token per sequence, in batch order
    with split_tokens(split):
        t1, t2 = to_dev(w), to_dev(w)
        ref_out = two_calls(pkv, w, t1, t1["slot_mapping"])
        got_out = fused(pkv, w, t2, t2["slot_mapping"])
    assert pkv.check_device_status() == 0
    assert np.array_equal(pool_bits(t1["k_cache"]), pool_bits(t2["k_cache"])), "K pools differ"
    assert np.array_equal(pool_bits(t1["v_cache"]), pool_bits(t2["v_cache"])), "V pools differ"
    assert torch.equal(ref_out, got_out), "fused output differs from the two calls"
    if w.cfg.name in ("tiny", "tiny_e4m3", "llama3_8b"):
        a, kc, vc = oracle_pools_after_append(w)
        assert np.array_equal(pool_bits(t2["k_cache"]), kc) and np.array_equal(pool_bits(t2["v_cache"]), vc)
        ref = oracle.decode_all(a["q"], kc, vc, w.kv_dtype_code, a["block_tables"], a["context_lens"],
                                w.cfg.softmax_scale, scales=a["scales"], nthreads=NT)
        assert_close(got_out.cpu().double().numpy(), ref, "fp32", f"fused {w.cfg.name}")


def test_fused_step_without_new_tokens_and_with_a_wrong_slot(pkv):
    w = W.make_workload("tiny")
    t1, t2 = to_dev(w), to_dev(w)
    slots = t1["slot_mapping"].clone()
    slots[1] = -1  # sequence 1 appends nothing this step
    ref_out = two_calls(pkv, w, t1, slots)
    got_out = fused(pkv, w, t2, slots)
    assert pkv.check_device_status() == 0
    assert np.array_equal(pool_bits(t1["k_cache"]), pool_bits(t2["k_cache"]))
    assert torch.equal(ref_out, got_out)
    # a slot that is not the table's position len - 1: stored, flagged
    bad = t2["slot_mapping"].clone()
    bad[2] = bad[2] + 1 if int(w.context_lens[2]) % 16 != 0 else bad[2] - 1
    fused(pkv, w, t2, bad)
    assert pkv.check_device_status() == pkv.DEVFLAG_BAD_SLOT
