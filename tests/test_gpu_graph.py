"""The decode step captured in a CUDA graph: the fused append + decode call (split sequences,
so the merge kernel too) and the cascade call are captured once and replayed; each replay
gives the bits of the same call run eagerly on the same inputs.  The calls allocate nothing
and never synchronise the host (workspaces are passed in), and their programmatic dependent
launches become graph edges."""
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

    return m


def _fresh(w):
    return to_dev(w)


@pytest.mark.parametrize("cfg,split", [("tiny", 16), ("llama3_8b", None), ("fp8_fork", None)])
def test_fused_step_in_a_graph(pkv, cfg, split):
    w = W.make_workload(cfg)
    mx = int(w.context_lens.max())
    with split_tokens(split):
        # eager reference: the same call on its own copy of the inputs
        te = _fresh(w)
        ref = torch.empty(te["q"].shape, dtype=torch.float32, device="cuda")
        pkv.paged_append_decode(te["k_new"], te["v_new"], te["slot_mapping"], te["q"], te["k_cache"], te["v_cache"],
                                te["block_tables"], te["context_lens"], w.cfg.softmax_scale, ref, scales=te["scales"],
                                max_context_len=mx)
        torch.cuda.synchronize()
        tg = _fresh(w)
        out = torch.empty_like(ref)
        B, hq, d = tg["q"].shape
        ws = torch.empty(max(1, pkv.workspace_size(B, hq, w.cfg.hkv, d, mx)), dtype=torch.uint8, device="cuda")
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):  # warm-up outside the capture (first-call attribute setting)
            pkv.paged_append_decode(tg["k_new"], tg["v_new"], tg["slot_mapping"], tg["q"], tg["k_cache"],
                                    tg["v_cache"], tg["block_tables"], tg["context_lens"], w.cfg.softmax_scale, out,
                                    scales=tg["scales"], max_context_len=mx, workspace=ws)
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        tg = _fresh(w)  # the warm-up appended: start again from the step's inputs
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            pkv.paged_append_decode(tg["k_new"], tg["v_new"], tg["slot_mapping"], tg["q"], tg["k_cache"],
                                    tg["v_cache"], tg["block_tables"], tg["context_lens"], w.cfg.softmax_scale, out,
                                    scales=tg["scales"], max_context_len=mx, workspace=ws)
        for _ in range(3):  # the append stores the same rows each time: every replay is the same step
            out.zero_()
            g.replay()
            torch.cuda.synchronize()
            assert pkv.check_device_status() == 0
            assert torch.equal(out, ref), f"graph replay differs from the eager call ({cfg})"
        assert torch.equal(tg["k_cache"], te["k_cache"]) and torch.equal(tg["v_cache"], te["v_cache"])


def test_cascade_call_in_a_graph(pkv):
    w = W.make_workload("fp8_fork")
    c = w.cascade()
    t = _fresh(w)
    dev = "cuda"
    ct = {k: getattr(c, k).to(dev) for k in ("prefix_tables", "prefix_lens", "member_indptr", "member_seqs",
                                             "seq_prefix", "block_tables", "context_lens")}
    mx = max(16, int(c.context_lens.max()))
    B, hq, d = t["q"].shape
    ws = torch.empty(pkv.cascade_workspace_size(B, hq, w.cfg.hkv, d, mx, c.prefix_tables.shape[0], c.max_members,
                                                c.max_prefix_len), dtype=torch.uint8, device=dev)

    def call(out):
        pkv.cascade_decode_attention(t["q"], t["k_cache"], t["v_cache"], ct["prefix_tables"], ct["prefix_lens"],
                                     ct["member_indptr"], ct["member_seqs"], ct["seq_prefix"], ct["block_tables"],
                                     ct["context_lens"], w.cfg.softmax_scale, out, max_members=c.max_members,
                                     max_prefix_len=c.max_prefix_len, max_context_len=mx, scales=t["scales"],
                                     workspace=ws)

    ref = torch.empty(t["q"].shape, dtype=torch.float32, device=dev)
    call(ref)
    torch.cuda.synchronize()
    out = torch.empty_like(ref)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        call(out)
    for _ in range(3):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert pkv.check_device_status() == 0
        assert torch.equal(out, ref), "graph replay of the cascade call differs from the eager call"
