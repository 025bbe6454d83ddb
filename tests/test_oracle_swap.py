"""Pins of the oracle block manager's swapping and of the block move between
pools, to facts outside them: conservation of device and host blocks, blocks
shared with other tables staying on the device, a swap-out/swap-in round trip
restoring a sequence's tokens byte for byte through the pools, all-or-nothing
refusals, and a swapped-out sequence refusing appends. CPU only."""

import numpy as np
import pytest

import oracle
from oracle.allocator import BlockAllocator, OutOfBlocks


def _mgr(nb=20, bs=4, host=12):
    a = BlockAllocator(nb, bs)
    a.add_host_pool(host)
    return a


def _conserved(a):
    free, ref = a.export_state()
    hfree, nsw, _, _ = a.export_host_state()
    # every device block is free xor referenced; every host block free xor held
    assert sorted(free + [b for b, r in enumerate(ref) if r > 0]) == list(range(a.num_blocks))
    held = sorted(h for hs in a.host_tables.values() for h in hs)
    assert sorted(hfree + held) == list(range(a.num_host_blocks))
    assert nsw == len(a.host_tables)


def test_swap_out_and_in_conserve_blocks():
    a = _mgr()
    a.add_seq(1, 10)           # 3 blocks
    a.add_seq(2, 5)            # 2 blocks
    free0 = len(a.free)
    pairs = a.swap_out(1)
    assert [d for d, _ in pairs] == [0, 1, 2] and [h for _, h in pairs] == [0, 1, 2]
    assert len(a.free) == free0 + 3
    assert a.seq_len(1) == 10
    _conserved(a)
    back = a.swap_in(1)
    assert [h for h, _ in back] == [0, 1, 2]
    assert len(a.table(1)) == 3 and a.seq_len(1) == 10
    assert a.export_host_state()[0] == list(range(3, 12)) + [0, 1, 2]   # FIFO return
    _conserved(a)


def test_shared_blocks_stay_on_device_for_other_holders():
    a = _mgr()
    a.add_seq(0, 8)             # blocks 0, 1
    a.fork(0, 1)
    a.swap_out(1)
    assert a.table(0) == [0, 1]
    _, ref = a.export_state()
    assert ref[0] == 1 and ref[1] == 1            # only sequence 0 holds them now
    assert 0 not in a.free and 1 not in a.free
    a.swap_in(1)
    assert set(a.table(1)).isdisjoint({0, 1})     # private copies, sharing not restored
    _conserved(a)


def test_refusals_change_nothing():
    a = _mgr(nb=10, bs=4, host=2)
    a.add_seq(1, 12)            # 3 blocks, host pool holds 2
    before = (a.export_state(), a.export_host_state())
    with pytest.raises(OutOfBlocks):
        a.swap_out(1)
    assert (a.export_state(), a.export_host_state()[:3]) == (before[0], before[1][:3])
    a2 = _mgr(nb=4, bs=4, host=4)
    a2.add_seq(1, 12)           # 3 of 4 device blocks
    a2.swap_out(1)
    a2.add_seq(2, 8)            # 2 blocks: 2 left free
    with pytest.raises(OutOfBlocks):
        a2.swap_in(1)           # needs 3
    assert 1 in a2.host_tables
    _conserved(a2)


def test_swapped_sequence_refuses_use_and_frees_host_blocks():
    a = _mgr()
    a.add_seq(1, 6)
    a.swap_out(1)
    with pytest.raises(ValueError):
        a.append_slot(1)
    with pytest.raises(ValueError):
        a.fork(1, 5)
    with pytest.raises(ValueError):
        a.swap_out(1)
    a.free_seq(1)
    assert len(a.export_host_state()[0]) == 12
    _conserved(a)


def test_round_trip_restores_the_tokens():
    """Tokens written through the manager's slots survive a swap-out, a reuse
    of the freed device blocks by another sequence, and a swap-in into other
    blocks: attention over the restored table equals attention before."""
    rng = np.random.default_rng(0)
    nb, bs, H, D = 16, 4, 2, 8
    a = _mgr(nb=nb, bs=bs, host=8)
    kp = rng.standard_normal((nb, bs, H, D)).astype(np.float16)
    vp = rng.standard_normal((nb, bs, H, D)).astype(np.float16)
    hk = np.zeros((8, bs, H, D), np.float16)
    hv = np.zeros((8, bs, H, D), np.float16)
    a.add_seq(1, 9)
    q = rng.standard_normal((1, 4, D)).astype(np.float16)
    table = np.array([a.table(1)], np.int32)
    before = oracle.decode_attention(q, kp, vp, table, [9], np.float32(0.3))
    pairs = a.swap_out(1)
    hk, hv = oracle.swap_blocks(kp, vp, hk, hv, pairs)
    a.add_seq(2, 12)                                # takes the freed blocks
    for b in a.table(2):
        kp[b] = np.float16(np.nan)
        vp[b] = np.float16(np.nan)
    back = a.swap_in(1)
    kp, vp = oracle.swap_blocks(hk, hv, kp, vp, back)
    table = np.array([a.table(1)], np.int32)
    after = oracle.decode_attention(q, kp, vp, table, [9], np.float32(0.3))
    assert np.array_equal(before, after)
    for (h, d), (d0, _) in zip(back, pairs):
        assert h == pairs[[p[1] for p in pairs].index(h)][1]
    _conserved(a)


def test_swap_blocks_moves_whole_blocks_only():
    rng = np.random.default_rng(1)
    sk = rng.integers(0, 256, (5, 4, 2, 8), dtype=np.uint8)
    sv = rng.integers(0, 256, (5, 4, 2, 8), dtype=np.uint8)
    dk = np.zeros((3, 4, 2, 8), np.uint8)
    dv = np.ones((3, 4, 2, 8), np.uint8)
    k, v = oracle.swap_blocks(sk, sv, dk, dv, [(4, 0), (1, 2)])
    assert np.array_equal(k[0], sk[4]) and np.array_equal(v[2], sv[1])
    assert np.array_equal(k[1], dk[1]) and np.array_equal(v[1], dv[1])
