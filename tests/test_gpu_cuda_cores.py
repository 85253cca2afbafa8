"""The CUDA-core decode kernel (selected with PKV_DECODE_CUDA_CORES=1; by default every pool
takes the tensor-core form) against the oracle, on the cases that cover its variants: full
workloads, every head_dim / group size, partial blocks, forced partitions, E4M3 pools and
the cascade merge."""
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
def cuda_cores():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    __graft_entry__.build()
    import paged_kv_cache_17_gb300 as pkv

    pkv.check_device_status()
    old = os.environ.get("PKV_DECODE_CUDA_CORES")
    os.environ["PKV_DECODE_CUDA_CORES"] = "1"
    yield pkv
    torch.cuda.synchronize()
    if old is None:
        os.environ.pop("PKV_DECODE_CUDA_CORES", None)
    else:
        os.environ["PKV_DECODE_CUDA_CORES"] = old


@pytest.mark.parametrize("name", ["tiny", "llama3_8b"])
def test_full_parity(cuda_cores, name):
    w = W.make_workload(name)
    _, out = gpu_step(w)
    a, kc, vc = oracle_pools_after_append(w)
    ref = oracle.decode_all(a["q"], kc, vc, 0, a["block_tables"], a["context_lens"], w.cfg.softmax_scale, nthreads=NT)
    assert_close(out.cpu().double().numpy(), ref, "fp32", f"cuda cores {name}")
    assert cuda_cores.check_device_status() == 0


@pytest.mark.parametrize("d,g", [(64, 1), (64, 8), (128, 2), (128, 4), (128, 8)])
def test_edge_lengths(cuda_cores, d, g):
    hkv = 2
    lens = [1, 15, 16, 17, 33, 64, 65, 129, 200, 0]
    cfg = W.Config(name="edges", hq=hkv * g, hkv=hkv, d=d, kv_dtype="bf16", softmax_scale=1.0 / np.sqrt(d),
                   seed=15 + d + g, kind="explicit", lens=tuple(lens))
    w = W.make_workload(cfg, lens=[max(n, 1) for n in lens])
    w.context_lens[-1] = 0
    w.slot_mapping[-1] = -1
    with split_tokens(48):
        _, out = gpu_step(w)
    a, kc, vc = oracle_pools_after_append(w)
    ref = oracle.decode_all(a["q"], kc, vc, 0, a["block_tables"], a["context_lens"], cfg.softmax_scale, nthreads=NT)
    got = out.cpu().double().numpy()
    assert np.all(got[-1] == 0.0)
    assert_close(got, ref, "fp32", f"cuda cores edges d={d} g={g}")
    assert cuda_cores.check_device_status() == 0


def test_cascade_merge(cuda_cores):
    from test_gpu_cascade import build_case, run_cascade

    c, kp, vp, q, full, lens = build_case(2, 4, 128, seed=9)
    out = run_cascade(cuda_cores, q.cuda(), kp.cuda(), vp.cuda(), c, 0.1)
    assert cuda_cores.check_device_status() == 0
    ref = oracle.decode_all(W.bf16_bits(q), W.bf16_bits(kp), W.bf16_bits(vp), oracle.KV_BF16, full.numpy(),
                            lens.numpy(), 0.1)
    assert_close(out.cpu().double().numpy(), ref, "bf16", "cuda cores cascade")
    assert_close(out.cpu().double().numpy(), ref, "fp32", "cuda cores cascade")


@pytest.mark.parametrize("name", ["fp8_fork"])
def test_e4m3_workload(cuda_cores, name):
    w = W.make_workload(name)
    _, out = gpu_step(w)
    a, kc, vc = oracle_pools_after_append(w)
    ref = oracle.decode_all(a["q"], kc, vc, oracle.KV_E4M3, a["block_tables"], a["context_lens"],
                            w.cfg.softmax_scale, scales=a["scales"], nthreads=NT)
    got = out.cpu().double().numpy()
    assert_close(got, ref, "fp8", f"cuda cores {name}")
    # the CUDA-core form widens the codes exactly and computes in fp32 throughout
    assert_close(got, ref, "fp32", f"cuda cores {name}")
    assert cuda_cores.check_device_status() == 0
