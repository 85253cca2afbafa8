"""The decode entry point that allocates nothing, against the regular one (GPU).

pkv_paged_decode_attention_noalloc is for callers that cannot allocate device memory when
they run a decode step (an allocator that holds all device memory, a serving loop that
forbids allocation after start-up, a C caller without an allocator): its workspace is a
fixed array inside the library.  These tests call it through the C ABI and compare its
output with pkv_paged_decode_attention given a caller-provided workspace, on two calls in a
row, and with the fp64 oracle; check that a call needing more scratch than the array holds
is refused; and check that refused arguments get the same status and message from both
entry points.  This file is collected last on purpose.
"""
import ctypes
import os

import pytest
import torch

import oracle
import workloads as W
from gpu_helpers import assert_close, oracle_pools_after_append, split_tokens, to_dev

NT = os.cpu_count() or 4

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__

    __graft_entry__.build()
    import paged_kv_cache_17_gb300 as m

    return m


def call_noalloc(pkv, t, w, out, max_len):
    desc = pkv._cache_desc(t["k_cache"], t["v_cache"], None, t["scales"])
    return pkv.lib.pkv_paged_decode_attention_noalloc(
        ctypes.byref(desc), t["q"].data_ptr(), t["block_tables"].data_ptr(), t["block_tables"].shape[1],
        t["context_lens"].data_ptr(), w.batch, w.cfg.hq, max_len, float(w.cfg.softmax_scale), out.data_ptr(),
        pkv.OUT_FP32 if out.dtype == torch.float32 else pkv.OUT_BF16, torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("name", ["llama3_8b", "fp8_fork", "tiny"])
def test_noalloc_matches_workspace_entry_point_twice(pkv, name):
    w = W.make_workload(name)
    t = to_dev(w)
    max_len = int(w.context_lens.max())
    ref = torch.empty(w.q.shape, dtype=torch.float32, device="cuda")
    pkv.paged_decode_attention(t["q"], t["k_cache"], t["v_cache"], t["block_tables"], t["context_lens"],
                               w.cfg.softmax_scale, ref, scales=t["scales"], max_context_len=max_len)
    torch.cuda.synchronize()
    ref_np = ref.cpu().double().numpy()
    for _ in range(2):  # the second call finds the scratch as the first one left it
        out = torch.full(w.q.shape, float("nan"), dtype=torch.float32, device="cuda")
        st = call_noalloc(pkv, t, w, out, max_len)
        assert st == pkv.PKV_OK, pkv.lib.pkv_last_error().decode()
        torch.cuda.synchronize()
        assert_close(out.cpu().double().numpy(), ref_np, "fp32", f"{name} without allocation")
    assert pkv.check_device_status() == 0
    # and against the oracle directly (the pools hold no appended token: none was appended)
    a, kc, vc = oracle_pools_after_append(w, append=False)
    want = oracle.decode_all(a["q"], kc, vc, w.kv_dtype_code, a["block_tables"], a["context_lens"],
                             w.cfg.softmax_scale, scales=a["scales"], nthreads=NT)
    got = out.cpu().double().numpy()
    assert_close(got, want, "fp32", f"{name} without allocation vs oracle")
    if w.cfg.kv_dtype == "e4m3":
        assert_close(got, want, "fp8", f"{name} without allocation vs oracle")


def test_noalloc_refuses_more_scratch_than_it_holds(pkv):
    # 16-token partitions of 64 sequences x 8 kv heads x 128K tokens need far more than
    # 32 MiB; the call must fail on the host, before anything is enqueued (the pointers
    # below are never dereferenced).
    desc = pkv.CacheDesc(0x100000, 0x200000, 1 << 20, 16, 8, 128, pkv.KV_BF16, None)
    with split_tokens(16):
        st = pkv.lib.pkv_paged_decode_attention_noalloc(ctypes.byref(desc), 0x300000, 0x400000, 8192, 0x500000, 64,
                                                        64, 131072, 0.088, 0x600000, pkv.OUT_BF16, None)
    assert st == pkv.PKV_ERR_WORKSPACE
    assert b"no-allocation" in pkv.lib.pkv_last_error()


def test_noalloc_refusals_match_the_regular_entry_point(pkv):
    """Arguments the regular call refuses get the same status and message here (the
    pointers are never dereferenced: every case fails on the host)."""

    def both(desc, batch=4, hq=8, max_blocks=7, max_len=100):
        args = (ctypes.byref(desc), 0x60000, 0x80000, max_blocks, 0x90000, batch, hq, max_len, 0.125, 0x70000,
                pkv.OUT_BF16)
        st_reg = pkv.lib.pkv_paged_decode_attention(*args, None, 0, None)
        msg_reg = pkv.lib.pkv_last_error()
        st_na = pkv.lib.pkv_paged_decode_attention_noalloc(*args, None)
        msg_na = pkv.lib.pkv_last_error()
        return st_reg, st_na, msg_reg, msg_na

    def desc(**kw):
        base = dict(k_cache=0x10000, v_cache=0x20000, num_blocks=64, block_size=16, num_kv_heads=2, head_dim=64,
                    kv_dtype=pkv.KV_BF16, scales=None)
        base.update(kw)
        return pkv.CacheDesc(**base)

    cases = [
        (dict(), dict(hq=12), pkv.PKV_ERR_UNSUPPORTED),           # query group of 6
        (dict(head_dim=96), dict(), pkv.PKV_ERR_UNSUPPORTED),     # head_dim not 64 / 128
        (dict(block_size=8), dict(batch=0), pkv.PKV_ERR_UNSUPPORTED),  # bad pool, empty batch
        (dict(), dict(hq=5), pkv.PKV_ERR_INVALID_ARG),            # not a multiple of the kv heads
        (dict(), dict(max_len=113), pkv.PKV_ERR_INVALID_ARG),     # beyond the table capacity
        (dict(), dict(batch=0), pkv.PKV_OK),                      # empty batch, valid pool: nothing to do
    ]
    for dkw, ckw, want in cases:
        st_reg, st_na, msg_reg, msg_na = both(desc(**dkw), **ckw)
        assert st_reg == want, (dkw, ckw, st_reg, msg_reg)
        assert st_na == st_reg and msg_na == msg_reg, (dkw, ckw, st_na, msg_na, msg_reg)
