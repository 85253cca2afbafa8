"""Failure detection on the GPU without a fault: a pipeline wait that runs out is reported
through the device status word, the call returns, and the next call is correct.

Every wait in the decode kernels is bounded (about a second); when one runs out the kernel
sets PKV_DEVFLAG_WAIT_TIMEOUT and unwinds, and its producer still waits for every copy it
issued, so no copy is in flight when a CTA exits.  Two test-only knobs make the consumers'
wait for a K/V stage run out: PKV_TEST_CONSUMER_WAIT_CYCLES shortens that wait to about
10 us, and PKV_TEST_PRODUCER_DELAY_CYCLES holds the producer back for about 2 ms before its
first load, so the stages are still unfilled when the consumers give up.  The cases use
partitions no longer than the load ring, so the producer never waits for a stage the
consumers would have freed.
"""
import os
from contextlib import contextmanager

import pytest
import torch

import oracle
import workloads as W
from gpu_helpers import assert_close, oracle_pools_after_append, to_dev

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


TINY_E4M3 = W.Config(name="tiny_e4m3", hq=8, hkv=2, d=64, kv_dtype="e4m3", softmax_scale=1.0 / 8.0, seed=1010,
                     kind="explicit", lens=(17, 33, 64, 100), pool_blocks=64)


@pytest.mark.parametrize("cfg", ["tiny", TINY_E4M3], ids=["bf16", "e4m3"])
def test_consumer_wait_runs_out_then_next_call_is_exact(pkv, cfg):
    w = W.make_workload(cfg)
    assert int(w.context_lens.max()) <= 8 * 16  # every partition fits the load ring
    t = to_dev(w)
    out = torch.empty(w.q.shape, dtype=torch.float32, device="cuda")

    def decode():
        pkv.paged_decode_attention(t["q"], t["k_cache"], t["v_cache"], t["block_tables"], t["context_lens"],
                                   w.cfg.softmax_scale, out, scales=t["scales"],
                                   max_context_len=int(w.context_lens.max()))

    assert pkv.check_device_status() == 0
    with env(PKV_TEST_CONSUMER_WAIT_CYCLES=20000, PKV_TEST_PRODUCER_DELAY_CYCLES=4000000):
        decode()  # enqueues and returns: the failure is data, not an error of the call
    assert pkv.check_device_status() == pkv.DEVFLAG_WAIT_TIMEOUT
    assert pkv.check_device_status() == 0  # reading the word cleared it
    # the context is still usable, and a normal call gives the oracle's answer
    out.fill_(float("nan"))
    decode()
    torch.cuda.synchronize()
    assert pkv.check_device_status() == 0
    a, kc, vc = oracle_pools_after_append(w, append=False)
    ref = oracle.decode_all(a["q"], kc, vc, w.kv_dtype_code, a["block_tables"], a["context_lens"],
                            w.cfg.softmax_scale, scales=a["scales"], nthreads=NT)
    assert_close(out.cpu().double().numpy(), ref, "fp32", f"{w.cfg.name} after a timed-out call")
