"""Host prefix cache (no GPU): the oracle model pinned to the pages' properties and worked
example, then the library's C++ block manager checked against the model, operation by
operation, and its SHA-256 against hashlib."""
import random

import numpy as np
import pytest

from conftest import golden_kv
from oracle import prefix_cache as orc


@pytest.fixture(scope="module")
def bm():
    import __graft_entry__

    __graft_entry__.build()
    from paged_kv_cache_17_gb300 import block_manager as m

    return m


def prompt(n, seed):
    r = random.Random(seed)
    return [r.randrange(0, 128256) for _ in range(n)]


# ------------------------------------------------------------------ pins of the model

def test_chain_covers_the_whole_prefix():
    t = prompt(16 * 12, 1)
    h = orc.chain_hashes(t)
    assert len(h) == 12 and len(set(h)) == 12
    # one token changed in block 5: blocks 0..4 keep their hashes, 5.. all change
    u = list(t)
    u[5 * 16 + 3] += 1
    g = orc.chain_hashes(u)
    assert g[:5] == h[:5] and all(a != b for a, b in zip(g[5:], h[5:]))
    # one token changed in block 0 changes every hash
    u = list(t)
    u[0] += 1
    assert all(a != b for a, b in zip(orc.chain_hashes(u), h))
    # the same 16 tokens at another position hash differently (the parent differs)
    rep = t[:16] * 3
    hr = orc.chain_hashes(rep)
    assert len(set(hr)) == 3
    # a later suffix does not move earlier hashes; a partial last block gets none
    assert orc.chain_hashes(t + prompt(40, 2))[:12] == h
    assert len(orc.chain_hashes(t + [7] * 15)) == 12


def test_salt_enters_first_block_only():
    t = prompt(64, 3)
    plain = orc.chain_hashes(t)
    assert orc.chain_hashes(t, salt=b"") == plain
    a = orc.chain_hashes(t, salt=b"tenant-a")
    b = orc.chain_hashes(t, salt=b"tenant-b")
    assert all(x != y for x, y in zip(a, plain)) and all(x != y for x, y in zip(a, b))
    assert orc.chain_hashes(t, salt=b"tenant-a") == a
    # blocks after the first see the salt only through their parent
    assert orc.block_hash(a[0], t[16:32]) == a[1]


def release(m, blocks):
    (m.release if isinstance(m, orc.PrefixCacheModel) else m.free)(blocks)


def run_page_example(model_cls):
    g = golden_kv("prefix_cache_example.txt")
    sp, um = int(g["system_prompt_tokens"]), int(g["user_message_tokens"])
    system = prompt(sp, 10)
    r1 = system + prompt(um, 11)
    r2 = system + prompt(um, 12)
    m = model_cls(400)
    hits1 = m.get_computed_blocks(r1)
    assert len(hits1) == int(g["request1_hits"])
    need = -(-len(r1) // 16)
    assert need == int(g["request1_blocks"])
    blocks1 = hits1 + m.allocate(need - len(hits1))
    assert m.cache_full_blocks(r1, blocks1) == len(r1) // 16  # every full block cached
    release(m, blocks1)
    assert m.num_free == 400
    hits2 = m.get_computed_blocks(r2)
    assert len(hits2) == int(g["request2_hits"]) == int(g["system_prompt_blocks"])
    assert hits2 == blocks1[:125]
    new = -(-len(r2) // 16) - len(hits2)
    assert new == int(g["request2_new_blocks"])
    fresh = m.allocate(new)
    assert not set(fresh) & set(blocks1[:125])
    # an exact repeat of a cached prompt still computes its last token
    m2 = model_cls(400)
    b = m2.allocate(125)
    m2.cache_full_blocks(system, b)
    cap = int(g["hit_cap_tokens_short_by"])
    assert len(m2.get_computed_blocks(system)) == (sp - cap) // 16 == 124
    assert len(m2.get_computed_blocks(system + [1])) == 125


def test_page_example_on_the_model():
    run_page_example(orc.PrefixCacheModel)


def test_lru_eviction_on_the_model():
    m = orc.PrefixCacheModel(6)
    a = m.allocate(3)
    ta = prompt(48, 20)
    assert m.cache_full_blocks(ta, a) == 3
    m.release(a)  # tail first: queue = 3, 4, 5, a2, a1, a0
    assert m.free == [3, 4, 5, a[2], a[1], a[0]]
    # a hit takes a freed cached block back out of the queue
    assert m.get_computed_blocks(ta[:33]) == a[:2]
    assert m.free == [3, 4, 5, a[2]]
    # four new blocks: three never used, then the least recently freed cached one (evicted)
    got = m.allocate(4)
    assert got == [3, 4, 5, a[2]] and a[2] not in m.hash_of
    m.release(a[:2])
    # the evicted block's hash no longer hits: the walk stops after two blocks
    assert m.get_computed_blocks(ta + [0]) == a[:2]


def test_copy_on_write_on_the_model():
    m = orc.PrefixCacheModel(8)
    a = m.allocate(2)
    assert m.copy_on_write(a[1]) == (a[1], False)  # private, uncached: write in place
    m.share(a)
    new, copy = m.copy_on_write(a[1])
    assert copy and new not in a and m.ref[a[1]] == 1 and m.ref[new] == 1
    t = prompt(32, 5)
    m.cache_full_blocks(t, a)
    new2, copy2 = m.copy_on_write(a[0])  # shared and cached
    assert copy2 and m.ref[a[0]] == 1
    m.release([a[0]])
    new3, copy3 = m.copy_on_write(a[1])  # held alone but cached: immutable, so copy
    assert copy3 and m.ref[a[1]] == 0 and a[1] in m.free and a[1] in m.hash_of


# ------------------------------------------------------------------ the library against the model

def test_sha256_matches_hashlib(bm):
    import hashlib

    r = random.Random(0)
    for n in list(range(0, 130)) + [1000, 4096, 100003]:
        data = bytes(r.randrange(256) for _ in range(n))
        assert bm.sha256(data) == hashlib.sha256(data).digest(), n


def test_chain_hashes_match_the_model(bm):
    for n, salt, seed in ((0, None, bytes(32)), (15, None, bytes(32)), (16, None, bytes(32)),
                          (2200, None, bytes(32)), (100, b"x", bytes(range(32))), (64, b"tenant", bytes(32))):
        t = prompt(n, n)
        assert bm.chain_hashes(t, 16, seed, salt) == orc.chain_hashes(t, 16, seed, salt)
    t = prompt(40, 9)
    assert bm.chain_hashes(t, 5) == orc.chain_hashes(t, 5)


def test_page_example_on_the_library(bm):
    class Lib(bm.BlockManager):
        pass

    run_page_example(Lib)


def state(m_lib, m_orc):
    n = len(m_orc.ref)
    assert [m_lib.ref_count(i) for i in range(n)] == m_orc.ref
    assert m_lib.free_queue() == m_orc.free
    assert m_lib.num_cached == len(m_orc.table)
    for i in range(n):
        assert m_lib.block_hash(i) == m_orc.hash_of.get(i)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_random_operations_match_the_model(bm, seed):
    r = random.Random(seed)
    nb = 48
    lib_m, orc_m = bm.BlockManager(nb), orc.PrefixCacheModel(nb)
    prompts = [prompt(r.randrange(20, 200), 100 + i) for i in range(4)]
    salts = [None, b"a"]
    live = []  # (tokens, salt, blocks) of running requests
    for step in range(400):
        op = r.random()
        if op < 0.45:  # a new request: lookup, allocate the rest, cache its full blocks
            base = r.choice(prompts)
            toks = base[: r.randrange(1, len(base) + 1)] + prompt(r.randrange(0, 40), 1000 + step)
            salt = r.choice(salts)
            h_lib = lib_m.get_computed_blocks(toks, salt)
            h_orc = orc_m.get_computed_blocks(toks, salt)
            assert h_lib == h_orc
            need = -(-len(toks) // 16) - len(h_lib)
            try:
                got_o = orc_m.allocate(need)
            except MemoryError:
                with pytest.raises(Exception):
                    lib_m.allocate(need)
                lib_m.free(h_lib)
                orc_m.release(h_orc)
                state(lib_m, orc_m)
                continue
            got_l = lib_m.allocate(need)
            assert got_l == got_o
            blocks = h_lib + got_l
            assert lib_m.cache_full_blocks(toks, blocks, salt) == orc_m.cache_full_blocks(toks, blocks, salt)
            live.append((toks, salt, blocks))
        elif op < 0.75 and live:  # a request finishes
            _, _, blocks = live.pop(r.randrange(len(live)))
            lib_m.free(blocks)
            orc_m.release(blocks)
        elif op < 0.85 and live:  # fork: share all blocks of a running request
            toks, salt, blocks = r.choice(live)
            lib_m.share(blocks)
            orc_m.share(blocks)
            live.append((toks, salt, list(blocks)))
        elif op < 0.95 and live:  # a writer into its last block
            i = r.randrange(len(live))
            toks, salt, blocks = live[i]
            if orc_m.num_free == 0:
                continue
            res_o = orc_m.copy_on_write(blocks[-1])
            res_l = lib_m.copy_on_write(blocks[-1])
            assert res_l == res_o
            blocks = blocks[:-1] + [res_o[0]]
            live[i] = (toks, salt, blocks)
        else:  # invalid release: both refuse and nothing changes
            held = [b for b in range(nb) if orc_m.ref[b] == 0]
            if held:
                with pytest.raises(Exception):
                    orc_m.release([held[0]])
                with pytest.raises(Exception):
                    lib_m.free([held[0]])
        state(lib_m, orc_m)
    for _, _, blocks in live:
        lib_m.free(blocks)
        orc_m.release(blocks)
    state(lib_m, orc_m)
    assert lib_m.num_free == nb


def test_library_errors_change_nothing(bm):
    m = bm.BlockManager(8)
    a = m.allocate(3)
    with pytest.raises(bm.PkvError):
        m.allocate(6)
    assert m.num_free == 5
    with pytest.raises(bm.PkvError):
        m.free([a[0], a[0]])  # held once, released twice
    assert m.ref_count(a[0]) == 1
    with pytest.raises(bm.PkvError):
        m.free([99])
    with pytest.raises(bm.PkvError):
        m.share([7])  # not held
    with pytest.raises(bm.PkvError):
        m.cache_full_blocks(prompt(64, 1), a)  # four full blocks, a table of three
    assert m.num_cached == 0
    m.cache_full_blocks(prompt(48, 1), a)
    with pytest.raises(bm.PkvError):
        m.cache_full_blocks(prompt(48, 2), a)  # a cached block is immutable: no other hash
    assert m.block_hash(a[0]) == orc.chain_hashes(prompt(48, 1))[0]
    with pytest.raises(bm.PkvError):
        bm.BlockManager(-1)
    with pytest.raises(ValueError):
        bm.BlockManager(4, seed=b"short")
    assert m.lookup(orc.chain_hashes(prompt(48, 1))[2]) == a[2] and m.lookup(bytes(32)) == -1
