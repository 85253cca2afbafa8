"""The log-sum-exp merge of many partial records per (sequence, kv head), on the GPU.

A split context leaves one record (running max, running sum, unnormalised output) per
partition, and a shared prefix up to 16 more; the merge kernel reads the (max, sum) pairs of
the first 64 records two per lane and walks the rest in a loop (habr.com/ru/articles/1021832,
section 3: the parts of a split key set combine exactly through their maxima and sums).
These cases go past 64 records: 16-token partitions over 1,100-3,000-token contexts
(70-188 records), and one 200,000-token context at the default partitioning (the
Llama-3-70B-sized context of the actionbridge.io chapter 8 H2O paragraph; with 8 kv heads it
is split into more than 64 partitions).  Every output row is compared with the oracle.
"""
import os

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from gpu_helpers import assert_close, gpu_step, oracle_pools_after_append, split_tokens

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


@pytest.mark.parametrize("g,kv", [(8, "bf16"), (4, "bf16"), (8, "e4m3"), (4, "e4m3")])
def test_merge_more_than_64_partition_records(_lib, g, kv):
    cfg = W.Config(name="records", hq=8 * g, hkv=8, d=128, kv_dtype=kv, softmax_scale=128 ** -0.5, seed=300 + g,
                   kind="uniform", batch=6, len_range=(1100, 3000))
    w = W.make_workload(cfg)
    with split_tokens(16):
        _, out = gpu_step(w)
    lens = w.context_lens.numpy()
    assert int((-(-lens // 16)).min()) > 64, "every sequence must leave more than 64 records"
    a, kc, vc = oracle_pools_after_append(w)
    ref = oracle.decode_all(a["q"], kc, vc, w.kv_dtype_code, a["block_tables"], a["context_lens"], cfg.softmax_scale,
                            scales=a["scales"], nthreads=NT)
    got = out.cpu().double().numpy()
    assert_close(got, ref, "fp32", f"{kv} g={g}, 16-token partitions")
    if kv == "e4m3":
        assert_close(got, ref, "fp8", f"{kv} g={g}, 16-token partitions")
    assert _lib.check_device_status() == 0


def test_decode_200k_token_context_default_partitions(_lib):
    cfg = W.Config(name="ctx200k", hq=64, hkv=8, d=128, kv_dtype="bf16", softmax_scale=128 ** -0.5, seed=1200,
                   kind="explicit", lens=(200_000,))
    w = W.make_workload(cfg)
    split = _lib.partition_tokens(1, 8, 200_000)
    assert -(-200_000 // split) > 64, f"{split}-token partitions leave at most 64 records"
    t, out16 = gpu_step(w, out_dtype=torch.bfloat16)
    _, out32 = gpu_step(w, out_dtype=torch.float32, append=False, t=t)
    a, kc, vc = oracle_pools_after_append(w)
    ref = oracle.decode_all(a["q"], kc, vc, 0, a["block_tables"], a["context_lens"], cfg.softmax_scale, nthreads=NT)
    assert_close(out32.cpu().double().numpy(), ref, "fp32", "200K context, fp32 out")
    assert_close(out16.cpu().double().numpy(), ref, "bf16", "200K context, bf16 out")
    assert _lib.check_device_status() == 0
