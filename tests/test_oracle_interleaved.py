"""Pins of the oracle's one-pool record layout (each physical block one record,
K array then V array): the record's byte layout against offsets computed by
hand from C's struct rule, and each operation against the two-pool oracle on
the records' members. CPU only."""

import numpy as np
import pytest

import oracle
from oracle import interleaved as il


def test_record_size_and_member_offsets():
    for elem, esz in ((np.float16, 2), (np.uint8, 1)):
        dt = il.kv_block_dtype(16, 8, 128, elem)
        E = 16 * 8 * 128
        assert dt.itemsize == 2 * E * esz
        assert dt.fields["K"][1] == 0
        assert dt.fields["V"][1] == E * esz


def _check_addresses(record_dtype):
    """Element (b, member, t, h, d) of the pool sits at element index
    b*2E + member*E + (t*H + h)*D + d of the raw buffer (E = BS*H*D)."""
    NB, BS, H, D = 5, 4, 3, 8
    E = BS * H * D
    dt = record_dtype(BS, H, D)
    raw = np.arange(NB * dt.itemsize // 2, dtype=np.uint16)
    kv = raw.view(np.float16).view(dt)
    assert kv.shape == (NB,)
    kb = kv["K"].view(np.uint16)
    vb = kv["V"].view(np.uint16)
    for b in range(NB):
        for t in range(BS):
            for h in range(H):
                for d in range(D):
                    off = (t * H + h) * D + d
                    assert kb[b, t, h, d] == b * 2 * E + off
                    assert vb[b, t, h, d] == b * 2 * E + E + off


def test_record_element_addresses_brute_force():
    _check_addresses(il.kv_block_dtype)


@pytest.mark.parametrize("mutant", ["v_first", "padded", "v_one_row_early", "one_member_wide"])
def test_wrong_record_layouts_are_caught(mutant):
    def record(BS, H, D):
        shp = (BS, H, D)
        if mutant == "v_first":
            return np.dtype({"names": ["K", "V"], "formats": [(np.float16, shp)] * 2,
                             "offsets": [BS * H * D * 2, 0]})
        if mutant == "padded":
            return np.dtype({"names": ["K", "V"], "formats": [(np.float16, shp)] * 2,
                             "offsets": [0, BS * H * D * 2 + 16],
                             "itemsize": 2 * BS * H * D * 2 + 16})
        if mutant == "v_one_row_early":
            return np.dtype({"names": ["K", "V"], "formats": [(np.float16, shp)] * 2,
                             "offsets": [0, (BS - 1) * H * D * 2],
                             "itemsize": 2 * BS * H * D * 2})
        return np.dtype([("K", np.float16, (BS, H, D + 1)), ("V", np.float16, (BS, H, D))])

    with pytest.raises((AssertionError, IndexError, ValueError)):
        _check_addresses(record)


def _pools(rng, NB=9, BS=16, H=2, D=16):
    k = rng.standard_normal((NB, BS, H, D)).astype(np.float16)
    v = rng.standard_normal((NB, BS, H, D)).astype(np.float16)
    return k, v


def test_make_and_split_round_trip():
    rng = np.random.default_rng(1)
    k, v = _pools(rng)
    kv = il.make_kv_pool(k, v)
    k2, v2 = il.split_kv_pool(kv)
    assert np.array_equal(k2.view(np.uint16), k.view(np.uint16))
    assert np.array_equal(v2.view(np.uint16), v.view(np.uint16))


def test_append_matches_two_pool_append_and_touches_only_the_slots():
    rng = np.random.default_rng(2)
    k, v = _pools(rng)
    kv = il.make_kv_pool(k, v)
    T = 7
    kn = rng.standard_normal((T, 2, 16)).astype(np.float16)
    vn = rng.standard_normal((T, 2, 16)).astype(np.float16)
    slots = np.array([0, 17, -1, 143, 100, 31, 64], np.int32)
    got = il.append_kv_interleaved(kv, kn, vn, slots)
    ek, ev = oracle.append_kv(k, v, kn, vn, slots)
    gk, gv = il.split_kv_pool(got)
    assert np.array_equal(gk.view(np.uint16), ek.view(np.uint16))
    assert np.array_equal(gv.view(np.uint16), ev.view(np.uint16))
    # raw bytes: nothing outside the written rows of the two members changes
    changed = (got.view(np.uint8) != kv.view(np.uint8)).reshape(9, 2, 16, -1).any(axis=-1)
    written = np.zeros((9, 2, 16), bool)
    for s in slots[slots >= 0]:
        written[s // 16, :, s % 16] = True
    assert not (changed & ~written).any()


def test_copy_blocks_copies_whole_records():
    rng = np.random.default_rng(3)
    k, v = _pools(rng)
    kv = il.make_kv_pool(k, v)
    pairs = [(1, 4), (6, 0), (2, 7)]
    got = il.copy_blocks_interleaved(kv, pairs)
    ek, ev = oracle.copy_blocks(k, v, pairs)
    gk, gv = il.split_kv_pool(got)
    assert np.array_equal(gk.view(np.uint16), ek.view(np.uint16))
    assert np.array_equal(gv.view(np.uint16), ev.view(np.uint16))
    raw = got.view(np.uint8).reshape(9, -1)
    assert np.array_equal(raw[4], kv.view(np.uint8).reshape(9, -1)[1])


def test_attention_over_records_equals_two_pool_attention():
    rng = np.random.default_rng(4)
    k, v = _pools(rng, NB=12)
    kv = il.make_kv_pool(k, v)
    table = np.array([[3, 7, 1, -1], [11, 0, -1, -1]], np.int32)
    lens = [40, 17]
    q = rng.standard_normal((2, 4, 16)).astype(np.float16)
    got = il.decode_attention_interleaved(q, kv, table, lens, np.float32(0.25))
    exp = oracle.decode_attention(q, k, v, table, lens, np.float32(0.25))
    assert np.array_equal(got, exp)
    # swapping the members changes the result: the V member is the values
    swapped = il.make_kv_pool(v, k)
    other = il.decode_attention_interleaved(q, swapped, table, lens, np.float32(0.25))
    assert not np.allclose(other, exp)


def test_fp8_records():
    rng = np.random.default_rng(5)
    k = rng.integers(0, 0x7F, (6, 16, 2, 32), dtype=np.uint8)
    v = rng.integers(0x80, 0xFF, (6, 16, 2, 32), dtype=np.uint8)
    kv = il.make_kv_pool(k, v)
    assert kv.dtype.itemsize == 2 * 16 * 2 * 32
    ks = np.array([0.01, 0.02], np.float32)
    vs = np.array([0.03, 0.005], np.float32)
    table = np.array([[5, 2], [0, 1]], np.int32)
    q = rng.standard_normal((2, 2, 32)).astype(np.float16)
    got = il.decode_attention_interleaved_fp8(q, kv, ks, vs, table, [30, 9], np.float32(0.2))
    exp = oracle.decode_attention_fp8(q, k, v, ks, vs, table, [30, 9], np.float32(0.2))
    assert np.array_equal(got, exp)
