"""The C-ABI library without a GPU: it builds, loads, exports every symbol that
include/pkv.h declares, and rejects bad arguments on the host before any CUDA call."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def pkv():
    import __graft_entry__

    __graft_entry__.build()
    import paged_kv_cache_17_gb300 as m

    return m


def header_functions(name):
    text = open(os.path.join(ROOT, "include", name)).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pkv_[a-z0-9_]+)\s*\(", text)))


def test_header_symbols_are_exported(pkv):
    from paged_kv_cache_17_gb300 import block_manager

    headers = sorted(f for f in os.listdir(os.path.join(ROOT, "include")) if f.endswith(".h"))
    assert headers == ["pkv.h", "pkv_block_manager.h"]
    lib = ctypes.CDLL(pkv.LIB_PATH)
    for h, bound in (("pkv.h", pkv.EXPORTED_SYMBOLS), ("pkv_block_manager.h", block_manager.EXPORTED_SYMBOLS)):
        names = header_functions(h)
        assert len(names) >= 9
        for n in names:
            assert hasattr(lib, n), f"{n} declared in include/{h} but not exported"
        assert set(names) == set(bound)


def test_version_and_status_strings(pkv):
    assert pkv.version() == 100
    for code in range(6):
        assert pkv.lib.pkv_status_string(code)
    assert pkv.lib.pkv_status_string(99) == b"unknown status"


def desc(pkv, **kw):
    base = dict(k_cache=0x10000, v_cache=0x20000, num_blocks=64, block_size=16, num_kv_heads=2, head_dim=64,
                kv_dtype=0, scales=None)
    base.update(kw)
    return pkv.CacheDesc(**base)


def append(pkv, d, k=0x30000, v=0x40000, slots=0x50000, n=4):
    return pkv.lib.pkv_paged_kv_append(ctypes.byref(d) if d is not None else None, k, v, slots, n, None)


def decode(pkv, d, batch=4, hq=8, max_blocks=7, max_len=100, q=0x60000, out=0x70000, scale=0.125):
    return pkv.lib.pkv_paged_decode_attention(ctypes.byref(d), q, 0x80000, max_blocks, 0x90000, batch, hq,
                                              max_len, scale, out, 0, None, 0, None)


def last(pkv):
    return pkv.lib.pkv_last_error().decode()


def test_append_rejects_bad_arguments_on_host(pkv):
    assert append(pkv, None) == pkv.PKV_ERR_INVALID_ARG
    assert append(pkv, desc(pkv, block_size=32)) == pkv.PKV_ERR_UNSUPPORTED and "block_size" in last(pkv)
    assert append(pkv, desc(pkv, head_dim=96)) == pkv.PKV_ERR_UNSUPPORTED
    assert append(pkv, desc(pkv, k_cache=0x10008)) == pkv.PKV_ERR_INVALID_ARG and "aligned" in last(pkv)
    assert append(pkv, desc(pkv, v_cache=None)) == pkv.PKV_ERR_INVALID_ARG
    assert append(pkv, desc(pkv, num_blocks=0)) == pkv.PKV_ERR_INVALID_ARG
    assert append(pkv, desc(pkv, num_blocks=1 << 28)) == pkv.PKV_ERR_INVALID_ARG
    assert append(pkv, desc(pkv, kv_dtype=1)) == pkv.PKV_ERR_INVALID_ARG and "scales" in last(pkv)
    assert append(pkv, desc(pkv, scales=0xA0000)) == pkv.PKV_ERR_INVALID_ARG
    assert append(pkv, desc(pkv, kv_dtype=7)) == pkv.PKV_ERR_INVALID_ARG
    assert append(pkv, desc(pkv), n=-1) == pkv.PKV_ERR_INVALID_ARG
    assert append(pkv, desc(pkv), n=0) == pkv.PKV_OK  # nothing to do, no CUDA call
    assert append(pkv, desc(pkv), k=0x30004) == pkv.PKV_ERR_INVALID_ARG
    assert append(pkv, desc(pkv), slots=0x50004) == pkv.PKV_ERR_INVALID_ARG
    assert append(pkv, desc(pkv), slots=None) == pkv.PKV_ERR_INVALID_ARG


def test_decode_rejects_bad_arguments_on_host(pkv):
    d = desc(pkv)
    assert decode(pkv, d, batch=0) == pkv.PKV_OK  # empty batch: no CUDA call
    assert decode(pkv, d, q=None) == pkv.PKV_ERR_INVALID_ARG
    assert decode(pkv, d, q=0x60008) == pkv.PKV_ERR_INVALID_ARG
    assert decode(pkv, d, out=0x70004) == pkv.PKV_ERR_INVALID_ARG
    assert decode(pkv, d, max_len=113) == pkv.PKV_ERR_INVALID_ARG and "max_blocks_per_seq" in last(pkv)
    assert decode(pkv, d, max_blocks=0) == pkv.PKV_ERR_INVALID_ARG
    assert decode(pkv, d, hq=6) == pkv.PKV_ERR_UNSUPPORTED and "group size" in last(pkv)
    assert decode(pkv, d, hq=5) == pkv.PKV_ERR_INVALID_ARG
    assert decode(pkv, d, batch=70000) == pkv.PKV_ERR_INVALID_ARG
    assert decode(pkv, d, scale=float("inf")) == pkv.PKV_ERR_INVALID_ARG
    assert decode(pkv, desc(pkv, head_dim=256)) == pkv.PKV_ERR_UNSUPPORTED
    assert pkv.lib.pkv_decode_workspace_size(4, 6, 2, 64, 100) == 0 and "group size" in last(pkv)


def test_binding_fails_loudly_without_library(tmp_path, monkeypatch):
    """The product path has no fallback: a missing library is an import error."""
    import importlib.util

    src = os.path.join(ROOT, "paged_kv_cache_17_gb300", "__init__.py")
    spec = importlib.util.spec_from_file_location("pkv_nolib", src)
    mod = importlib.util.module_from_spec(spec)
    monkeypatch.setattr(os.path, "exists", lambda p: False)
    with pytest.raises(ImportError):
        spec.loader.exec_module(mod)


def test_noalloc_refusals_match_the_regular_entry_point_on_host(pkv):
    """The entry point without a workspace refuses what the regular one refuses, with the
    same status and message, before any CUDA call."""
    cases = [
        (dict(), dict(hq=12), pkv.PKV_ERR_UNSUPPORTED),                 # query group of 6
        (dict(head_dim=96), dict(), pkv.PKV_ERR_UNSUPPORTED),           # head_dim not 64 / 128
        (dict(block_size=8), dict(batch=0), pkv.PKV_ERR_UNSUPPORTED),   # bad pool, empty batch
        (dict(), dict(hq=5), pkv.PKV_ERR_INVALID_ARG),                  # not a multiple of the kv heads
        (dict(), dict(max_len=113), pkv.PKV_ERR_INVALID_ARG),           # beyond the table capacity
        (dict(), dict(q=0x60008), pkv.PKV_ERR_INVALID_ARG),             # misaligned q
        (dict(), dict(batch=0), pkv.PKV_OK),                            # empty batch: nothing to do
    ]
    for dkw, ckw, want in cases:
        kw = dict(batch=4, hq=8, max_blocks=7, max_len=100, q=0x60000)
        kw.update(ckw)
        args = (ctypes.byref(desc(pkv, **dkw)), kw["q"], 0x80000, kw["max_blocks"], 0x90000, kw["batch"], kw["hq"],
                kw["max_len"], 0.125, 0x70000, 0)
        st_reg = pkv.lib.pkv_paged_decode_attention(*args, None, 0, None)
        msg_reg = last(pkv)
        st_na = pkv.lib.pkv_paged_decode_attention_noalloc(*args, None)
        assert st_reg == want, (dkw, ckw, st_reg, msg_reg)
        assert st_na == st_reg and last(pkv) == msg_reg, (dkw, ckw, st_na, last(pkv), msg_reg)


def test_stage_copy_refuses_bad_arguments_on_host(pkv):
    """The staging copy checks its pointers and size before any CUDA call."""
    sc = pkv.lib.pkv_stage_copy
    assert sc(0x10000, 0x20000, 0, None) == pkv.PKV_OK  # nothing to copy
    assert sc(None, 0x20000, 16, None) == pkv.PKV_ERR_INVALID_ARG
    assert sc(0x10000, None, 16, None) == pkv.PKV_ERR_INVALID_ARG
    assert sc(0x10008, 0x20000, 16, None) == pkv.PKV_ERR_INVALID_ARG and "aligned" in last(pkv)
    assert sc(0x10000, 0x20004, 16, None) == pkv.PKV_ERR_INVALID_ARG
    assert sc(0x10000, 0x20000, 24, None) == pkv.PKV_ERR_INVALID_ARG and "multiple of 16" in last(pkv)
    assert sc(0x10000, 0x10010, 64, None) == pkv.PKV_ERR_INVALID_ARG and "overlap" in last(pkv)
    assert sc(0x10010, 0x10000, 64, None) == pkv.PKV_ERR_INVALID_ARG
