"""Pins of the CPU oracle to things other than itself (no GPU needed).

Each group below would fail for a plausible mistake in the oracle: a dropped or
inverted softmax scale, a wrong sign in the exponent, a transposed q/K operand, a
wrong GQA head map, swapped block/offset indexing in the gather, a wrong e4m3
exponent bias or tie rule, a scale multiplied instead of divided on quantisation.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from conftest import golden_rows

rng = np.random.default_rng(12345)


def bf16(x):
    """fp64 array -> (uint16 bf16 bits, exact fp64 value of those bits) via torch's cast."""
    t = torch.tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)
    bits = t.view(torch.int16).numpy().view(np.uint16).copy()
    return bits, t.to(torch.float64).numpy()


def make_paged(n_seqs, lens, hkv, d, nb, seed=0, hq=None):
    """A tiny scattered pool + tables + the dense per-sequence K/V they encode."""
    g = torch.Generator().manual_seed(seed)
    perm = torch.randperm(nb, generator=g).tolist()
    M = max((n + 15) // 16 for n in lens)
    tables = np.zeros((n_seqs, M), dtype=np.int32)
    used = 0
    for b, n in enumerate(lens):
        nbk = (n + 15) // 16
        tables[b, :nbk] = perm[used:used + nbk]
        tables[b, nbk:] = perm[-1]  # in-bounds filler
        used += nbk
    kbits, kval = bf16(rng.standard_normal((nb, 16, hkv, d)))
    vbits, vval = bf16(rng.standard_normal((nb, 16, hkv, d)))
    return tables, kbits, kval, vbits, vval


# ----------------------------------------------------------------- attention definition

def sdpa_ref(q, K, V, scale, g):
    """torch's scaled_dot_product_attention in fp64 with GQA (library routine)."""
    qt = torch.tensor(q).unsqueeze(0).unsqueeze(2)  # [1, Hq, 1, D]
    kt = torch.tensor(K).unsqueeze(0)  # [1, Hkv, n, D]
    vt = torch.tensor(V).unsqueeze(0)
    kt = kt.repeat_interleave(g, dim=1)
    vt = vt.repeat_interleave(g, dim=1)
    out = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=scale)
    return out[0, :, 0, :].numpy()


@pytest.mark.parametrize("hq,hkv,d,lens", [(8, 2, 64, [17, 33, 64, 100]), (4, 4, 32, [1, 5, 16]),
                                           (16, 2, 16, [40, 7])])
def test_decode_matches_torch_sdpa(hq, hkv, d, lens):
    nb = sum((n + 15) // 16 for n in lens) + 5
    tables, kbits, kval, vbits, vval = make_paged(len(lens), lens, hkv, d, nb, seed=hq + d)
    qbits, qval = bf16(rng.standard_normal((len(lens), hq, d)))
    scale = 1.0 / math.sqrt(d)
    out = oracle.decode_all(qbits, kbits, vbits, oracle.KV_BF16, tables,
                            np.array(lens, dtype=np.int32), scale)
    for b, n in enumerate(lens):
        pos = np.arange(n)
        blk = tables[b, pos // 16]
        K = kval[blk, pos % 16].transpose(1, 0, 2)  # [Hkv, n, D] by torch-free fancy indexing
        V = vval[blk, pos % 16].transpose(1, 0, 2)
        ref = sdpa_ref(qval[b], K, V, scale, hq // hkv)
        np.testing.assert_allclose(out[b], ref, rtol=1e-12, atol=1e-12)


def test_len_one_returns_v0():
    q = rng.standard_normal(8)
    K = rng.standard_normal((1, 8))
    V = rng.standard_normal((1, 8))
    np.testing.assert_array_equal(oracle.attention_one(q, K, V, 0.3), V[0])


def test_equal_keys_give_mean_of_v():
    q = rng.standard_normal(16)
    K = np.tile(rng.standard_normal(16), (37, 1))
    V = rng.standard_normal((37, 16))
    np.testing.assert_allclose(oracle.attention_one(q, K, V, 0.7), V.mean(axis=0), rtol=0, atol=1e-13)


def test_zero_scale_gives_mean_of_v():
    q = rng.standard_normal(16)
    K = rng.standard_normal((23, 16))
    V = rng.standard_normal((23, 16))
    np.testing.assert_allclose(oracle.attention_one(q, K, V, 0.0), V.mean(axis=0), atol=1e-13)


def test_two_token_closed_form():
    # softmax over two scores is a logistic function of their difference.
    q = rng.standard_normal(12)
    K = rng.standard_normal((2, 12))
    V = rng.standard_normal((2, 12))
    scale = 0.37
    s0, s1 = scale * q @ K[0], scale * q @ K[1]
    w0 = 1.0 / (1.0 + math.exp(s1 - s0))
    expect = w0 * V[0] + (1.0 - w0) * V[1]
    np.testing.assert_allclose(oracle.attention_one(q, K, V, scale), expect, rtol=1e-13, atol=1e-14)


def test_dominant_key_selects_its_value():
    q = np.zeros(8)
    q[0] = 1.0
    K = np.zeros((5, 8))
    K[3, 0] = 1.0
    V = rng.standard_normal((5, 8))
    out = oracle.attention_one(q, K, V, 1000.0)  # weights of the others: e^-1000
    np.testing.assert_allclose(out, V[3], rtol=0, atol=1e-15)
    # reversing the sign of q makes key 3 the least likely one
    out2 = oracle.attention_one(-q, K, V, 1000.0)
    np.testing.assert_allclose(out2, V[[0, 1, 2, 4]].mean(axis=0), atol=1e-13)


def test_shift_of_all_keys_and_token_permutation_are_invariances():
    q = rng.standard_normal(16)
    K = rng.standard_normal((29, 16))
    V = rng.standard_normal((29, 16))
    base = oracle.attention_one(q, K, V, 0.25)
    shifted = oracle.attention_one(q, K + rng.standard_normal(16), V, 0.25)
    np.testing.assert_allclose(shifted, base, rtol=1e-11, atol=1e-12)
    p = rng.permutation(29)
    np.testing.assert_allclose(oracle.attention_one(q, K[p], V[p], 0.25), base, rtol=1e-12, atol=1e-13)


def test_linear_in_v():
    q = rng.standard_normal(16)
    K = rng.standard_normal((19, 16))
    V1 = rng.standard_normal((19, 16))
    V2 = rng.standard_normal((19, 16))
    a = oracle.attention_one(q, K, V1, 0.5)
    b = oracle.attention_one(q, K, V2, 0.5)
    np.testing.assert_allclose(oracle.attention_one(q, K, 2.0 * V1 - V2, 0.5), 2.0 * a - b,
                               rtol=1e-12, atol=1e-12)


def test_empty_sequence_gives_zeros():
    out = oracle.attention_one(np.ones(4), np.zeros((0, 4)), np.zeros((0, 4)), 1.0)
    np.testing.assert_array_equal(out, np.zeros(4))


def test_online_softmax_tiling_is_exact():
    """The tiling argument of habr.com/ru/articles/1021832 section 3 ("Tiling и online
    softmax": running max m, running sum l, rescale by exp(m_old - m_new); the result
    is identical to full attention).  Restated here in fp64 over 16-token tiles and
    over split partitions merged with their log-sum-exp; it must equal the oracle."""
    d, n = 32, 301
    q = rng.standard_normal(d)
    K = rng.standard_normal((n, d))
    V = rng.standard_normal((n, d))
    scale = 1.0 / math.sqrt(d)
    ref = oracle.attention_one(q, K, V, scale)

    def partial(lo, hi):
        m, l, acc = -math.inf, 0.0, np.zeros(d)
        for j in range(lo, hi, 16):
            s = scale * K[j:min(hi, j + 16)] @ q
            m_new = max(m, s.max())
            p = np.exp(s - m_new)
            alpha = math.exp(m - m_new)
            l = l * alpha + p.sum()
            acc = acc * alpha + p @ V[j:min(hi, j + 16)]
            m = m_new
        return m, l, acc

    m, l, acc = partial(0, n)
    np.testing.assert_allclose(acc / l, ref, rtol=1e-12, atol=1e-13)
    for P in (16, 64, 128, 256):
        parts = [partial(lo, min(n, lo + P)) for lo in range(0, n, P)]
        M = max(p[0] for p in parts)
        num = sum(math.exp(p[0] - M) * p[2] for p in parts)
        den = sum(math.exp(p[0] - M) * p[1] for p in parts)
        np.testing.assert_allclose(num / den, ref, rtol=1e-12, atol=1e-13)


# ----------------------------------------------------------------- paging / gather

def test_gather_follows_page_example_table():
    rows = golden_rows("paging_example.txt")
    table = {int(r[1]): int(r[2]) for r in rows if r[0] == "table"}
    hkv, d, nb = 1, 4, 1000
    row = np.zeros(70, dtype=np.int32)
    for lb, pb in table.items():
        row[lb] = pb
    row[63], row[64] = 5, 6
    pool = np.zeros((nb, 16, hkv, d), dtype=np.uint16)
    # mark every slot with a distinct bf16 pattern derived from (block, slot)
    blk = np.arange(nb)[:, None]
    off = np.arange(16)[None, :]
    marks = (blk * 16 + off).astype(np.float32)
    bits, _ = bf16(marks)
    pool[:, :, 0, :] = bits[:, :, None]
    got = oracle.gather(pool, oracle.KV_BF16, row, 65 * 16, 0)
    for lb, pb in table.items():
        for off_ in range(16):
            expect = np.float32(pb * 16 + off_)
            assert got[lb * 16 + off_, 0] == float(torch.tensor(expect).bfloat16().float())
    # token numbers of the page (1-based) -> (logical block, slot 1-based)
    for r in rows:
        if r[0] != "token":
            continue
        tok, lb, slot1 = int(r[1]), int(r[2]), int(r[3])
        assert W.position_to_block(tok - 1) == (lb, slot1 - 1)


def test_gather_invariant_under_physical_permutation():
    lens = [45, 3, 16]
    nb = 12
    tables, kbits, _, vbits, _ = make_paged(3, lens, 2, 8, nb, seed=3)
    qbits, _ = bf16(rng.standard_normal((3, 4, 8)))
    cl = np.array(lens, dtype=np.int32)
    base = oracle.decode_all(qbits, kbits, vbits, oracle.KV_BF16, tables, cl, 0.3)
    perm = rng.permutation(nb)  # physical block i moves to perm[i]
    k2 = np.empty_like(kbits)
    v2 = np.empty_like(vbits)
    k2[perm] = kbits
    v2[perm] = vbits
    t2 = perm[tables].astype(np.int32)
    moved = oracle.decode_all(qbits, k2, v2, oracle.KV_BF16, t2, cl, 0.3)
    np.testing.assert_array_equal(moved, base)


def test_shared_blocks_give_bitwise_identical_outputs():
    # two sequences reading the same physical blocks with the same q: identical bits
    lens = [40, 40]
    nb = 8
    tables, kbits, _, vbits, _ = make_paged(2, [40, 1], 2, 8, nb, seed=5)
    tables = np.stack([tables[0], tables[0]])
    q1, _ = bf16(rng.standard_normal((1, 4, 8)))
    q = np.concatenate([q1, q1])
    out = oracle.decode_all(q, kbits, vbits, oracle.KV_BF16, tables, np.array(lens, np.int32), 0.5)
    assert out[0].tobytes() == out[1].tobytes()


# ----------------------------------------------------------------- append

def test_append_bf16_is_bit_copy_and_lands_at_position():
    w = W.make_workload("tiny")
    a = w.np()
    k, v = a["k_cache"].copy(), a["v_cache"].copy()
    rc = oracle.append(k, v, a["k_new"], a["v_new"], a["slot_mapping"], oracle.KV_BF16)
    assert rc == 0
    changed = np.argwhere((k != a["k_cache"]).any(axis=(2, 3)))
    for b, s in enumerate(w.seqs):
        pos = s.length - 1
        row = a["block_tables"][b]
        got = oracle.gather(k, oracle.KV_BF16, row, s.length, 1)[pos]
        expect = np.array([oracle.bf16_to_f64(x) for x in a["k_new"][b, 1]])
        np.testing.assert_array_equal(got, expect)
        blk, off = s.blocks[pos // 16], pos % 16
        assert (k[blk, off] == a["k_new"][b]).all() and (v[blk, off] == a["v_new"][b]).all()
    # nothing else moved: exactly one (block, slot) per sequence changed
    assert len({(int(r[0]), int(r[1])) for r in changed}) <= w.batch


def test_append_negative_slot_is_skipped_and_out_of_range_reported():
    k = np.zeros((2, 16, 1, 4), np.uint16)
    v = np.zeros_like(k)
    new = np.full((2, 1, 4), 0x3F80, np.uint16)  # bf16 1.0
    assert oracle.append(k, v, new, new, np.array([-1, 17], np.int64), oracle.KV_BF16) == 0
    assert (k[1, 1] == 0x3F80).all() and k.sum() == 0x3F80 * 4
    assert oracle.append(k, v, new, new, np.array([32, 0], np.int64), oracle.KV_BF16) == -1


def test_append_e4m3_matches_torch_float8_cast():
    """Quantise-on-write x -> RNE(x / scale) to E4M3 (saturating) against torch's own
    float8_e4m3fn cast (an independent library conversion) on in-range values."""
    hkv, d, T = 4, 32, 40
    x = rng.standard_normal((T, hkv, d)) * rng.uniform(0.2, 3.0, size=(1, hkv, 1))
    kbits, kval = bf16(x)
    vbits, vval = bf16(-x * 0.5)
    scales = np.stack([np.abs(kval).max(axis=(0, 2)) / 400.0,
                       np.abs(vval).max(axis=(0, 2)) / 300.0]).astype(np.float32)
    k = np.zeros((3, 16, hkv, d), np.uint8)
    v = np.zeros_like(k)
    slots = np.arange(T, dtype=np.int64)
    assert oracle.append(k, v, kbits, vbits, slots, oracle.KV_E4M3, scales) == 0
    for src, sc, pool in ((kval, scales[0], k), (vval, scales[1], v)):
        y = torch.tensor(src.astype(np.float32)) / torch.tensor(sc).view(1, -1, 1)
        ref = y.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        got = pool.reshape(-1, hkv, d)[:T]
        np.testing.assert_array_equal(got, ref)


# ----------------------------------------------------------------- e4m3 codec

def test_e4m3_decode_matches_spec_codes():
    for code_hex, val in golden_rows("e4m3_codes.txt"):
        got = oracle.e4m3_decode(int(code_hex, 16))
        if val == "nan":
            assert math.isnan(got)
        else:
            assert got == float(val) and math.copysign(1.0, got) == math.copysign(1.0, float(val))


def test_e4m3_decode_all_codes_match_torch():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for c in range(256):
        got = oracle.e4m3_decode(c)
        if math.isnan(ref[c]):
            assert math.isnan(got)
        else:
            assert got == ref[c], c


def test_e4m3_encode_round_trips_every_finite_code():
    for c in range(256):
        x = oracle.e4m3_decode(c)
        if math.isnan(x):
            continue
        assert oracle.e4m3_encode(x) == c, hex(c)


def test_e4m3_encode_ties_to_even_and_saturates():
    # midpoints between neighbouring codes go to the code with an even mantissa
    for c in range(0, 0x7E):
        lo, hi = oracle.e4m3_decode(c), oracle.e4m3_decode(c + 1)
        mid = (lo + hi) / 2.0
        if float(np.float32(mid)) != mid:
            continue
        expect = c if c % 2 == 0 else c + 1
        assert oracle.e4m3_encode(mid) == expect, hex(c)
        assert oracle.e4m3_encode(-mid) == 0x80 | expect
        # just off the midpoint rounds to the nearer side
        assert oracle.e4m3_encode(np.nextafter(np.float32(mid), np.float32(0))) == c
        assert oracle.e4m3_encode(np.nextafter(np.float32(mid), np.float32(1e9))) == c + 1
    for big in (448.0, 449.0, 464.0, 480.0, 1e6, float("inf")):
        assert oracle.e4m3_encode(big) == 0x7E
        assert oracle.e4m3_encode(-big) == 0xFE
    assert oracle.e4m3_encode(float("nan")) & 0x7F == 0x7F
    assert oracle.e4m3_encode(2.0 ** -10) == 0x00  # half of the smallest subnormal: tie to 0
    assert oracle.e4m3_encode(-(2.0 ** -11)) == 0x80


def test_e4m3_encode_matches_torch_on_random_values():
    x = (rng.standard_normal(20000) * np.exp(rng.uniform(-9, 6, 20000))).astype(np.float32)
    x = np.clip(x, -448, 448)
    ref = torch.tensor(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(oracle.e4m3_encode_array(x), ref)


def test_e4m3_paged_decode_uses_scaled_codes():
    # decode through an e4m3 pool equals decode over the dequantised values
    hkv, d, lens = 2, 16, [20, 7]
    nb = 4
    codes = rng.integers(0, 256, size=(nb, 16, hkv, d)).astype(np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x00  # no NaNs in a pool
    scales = np.array([[0.5, 0.25], [2.0, 0.125]], dtype=np.float32)
    tables = np.array([[2, 0], [3, 1]], dtype=np.int32)
    qbits, qval = bf16(rng.standard_normal((2, 4, d)))
    out = oracle.decode_all(qbits, codes, codes, oracle.KV_E4M3, tables, np.array(lens, np.int32),
                            0.2, scales=scales)
    dec = np.vectorize(oracle.e4m3_decode)(codes)
    for b, n in enumerate(lens):
        pos = np.arange(n)
        blk = tables[b, pos // 16]
        K = dec[blk, pos % 16].transpose(1, 0, 2) * scales[0][:, None, None]
        V = dec[blk, pos % 16].transpose(1, 0, 2) * scales[1][:, None, None]
        ref = sdpa_ref(qval[b], K, V, 0.2, 2)
        np.testing.assert_allclose(out[b], ref, rtol=1e-12, atol=1e-12)


# ----------------------------------------------------------------- KV size formula

def test_kv_bytes_per_token_matches_pages():
    for label, L, hkv, d, q, expect in golden_rows("kv_bytes_per_token.txt"):
        assert oracle.kv_bytes_per_token(int(L), int(hkv), int(d), int(q)) == int(expect), label


def test_kv_bytes_per_context_matches_pages():
    per_tok = oracle.kv_bytes_per_token(80, 8, 128, 2)
    for ctx, gib in golden_rows("kv_bytes_per_context.txt"):
        assert per_tok * int(ctx) == pytest.approx(float(gib) * 2**30, rel=1e-12)


def test_workload_byte_accounting_uses_the_formula():
    # per-token, per-layer bytes for the workload shapes follow the same formula
    for name, expect in (("tiny", 512), ("llama3_8b", 4096), ("long_context_70b", 4096),
                         ("fp8_fork", 2048)):
        c = W.get(name)
        assert oracle.kv_bytes_per_token(1, c.hkv, c.d, c.elem_bytes) == expect


# ----------------------------------------------------------------- copy-on-write

def test_copy_blocks_invariants():
    """A copied block equals its source bit for bit, the source and every other block stay
    untouched (the pages' copy-on-write: the original remains as it was)."""
    nb = 10
    k = rng.integers(0, 2**16, size=(nb, 16, 2, 8), dtype=np.uint16)
    v = rng.integers(0, 2**16, size=(nb, 16, 2, 8), dtype=np.uint16)
    k0, v0 = k.copy(), v.copy()
    pairs = np.array([[1, 7], [4, 4], [2, 9]], dtype=np.int64)
    assert oracle.copy_blocks(k, v, pairs) == 0
    for src, dst in ((1, 7), (2, 9)):
        assert np.array_equal(k[dst], k0[src]) and np.array_equal(v[dst], v0[src])
    untouched = [i for i in range(nb) if i not in (7, 9)]
    assert np.array_equal(k[untouched], k0[untouched]) and np.array_equal(v[untouched], v0[untouched])
    # out-of-range pairs are skipped and reported
    assert oracle.copy_blocks(k, v, np.array([[0, nb], [-1, 3]], dtype=np.int64)) == -1
    assert np.array_equal(k[[0, 3]], k0[[0, 3]])
    # e4m3 pools copy the same way
    k8 = rng.integers(0, 256, size=(4, 16, 2, 8), dtype=np.uint8)
    v8 = k8.copy()
    ref = k8[3].copy()
    assert oracle.copy_blocks(k8, v8, np.array([[3, 0]], dtype=np.int64)) == 0
    assert np.array_equal(k8[0], ref)
