"""The reference block manager against the pages' rules and printed figures."""

import numpy as np
import pytest

import oracle
from oracle import BlockAllocator, OutOfBlocks
from tests.oracle_pins import golden


def _token_by_token_blocks(length, bs):
    """Blocks held after `length` one-token appends, counted by simulation:
    a new block is opened whenever the current one is full (or none exists)."""
    blocks, fill = 0, bs
    for _ in range(length):
        if fill == bs:
            blocks += 1
            fill = 0
        fill += 1
    return blocks


@pytest.mark.parametrize("bs", [1, 8, 16, 32])
def test_blocks_needed_matches_simulation(bs):
    for L in list(range(0, 70)) + [100, 2040, 4096, 32768]:
        assert oracle.blocks_needed(L, bs) == _token_by_token_blocks(L, bs)


def test_add_seq_and_growth_agree_with_simulation():
    a = BlockAllocator(64, 16)
    a.add_seq(0, 0)
    for L in range(1, 130):
        a.append_slot(0)
        assert len(a.table(0)) == _token_by_token_blocks(L, 16)
    b = BlockAllocator(64, 16)
    b.add_seq(0, 129)
    assert len(b.table(0)) == len(a.table(0))


def test_printed_capacity_figures():
    g = golden("capacity_figures.json")
    r = g["blocks_for_request"]
    assert oracle.blocks_needed(r["tokens"], r["block_size"]) == r["blocks"]
    n = g["naive_slab_waste"]
    w = oracle.naive_slab_waste([n["tokens"]], n["slab_tokens"])
    assert abs(w - n["waste_approx"]) <= n["abs_tol"]
    c = g["capacity_question"]
    assert oracle.concurrent_sequences(c["pool_blocks"], c["context_tokens"],
                                       c["block_size"]) == c["sequences"]
    # the allocator itself admits exactly that many before running out
    a = BlockAllocator(c["pool_blocks"], c["block_size"])
    admitted = 0
    with pytest.raises(OutOfBlocks):
        while True:
            a.add_seq(admitted, c["context_tokens"])
            admitted += 1
    assert admitted == c["sequences"]


def test_waste_below_one_block_per_sequence():
    g = golden("capacity_figures.json")["paged_waste_bound"]
    rng = np.random.default_rng(5)
    lens = rng.integers(1, 5000, size=300)
    a = BlockAllocator(int(sum(-(-L // 16) for L in lens)), 16)
    for i, L in enumerate(lens):
        a.add_seq(i, int(L))
        empty = len(a.table(i)) * 16 - int(L)
        assert 0 <= empty < 16 * g["max_partial_blocks_per_sequence"]
    assert oracle.paged_internal_waste(lens, 16) < g["aggregate_waste_below"]


def test_worked_mapping_reproduced_by_allocator():
    """Free list starting 7, 2, 9 hands request A exactly the pictured blocks."""
    g = golden("worked_block_table.json")
    order = g["logical_to_physical"] + [b for b in range(10) if b not in g["logical_to_physical"]]
    a = BlockAllocator(g["physical_blocks_pictured"], 16, order)
    a.add_seq(0, 40)
    assert a.table(0) == g["logical_to_physical"]


def test_sharing_picture_reproduced_by_allocator():
    """A shares its first block with B (fork after one full block); both then
    grow: A -> [3,7,1], B -> [3,9], refcount(3) = 2."""
    g = golden("sharing_picture.json")
    order = [3, 7, 1, 9] + [b for b in range(10) if b not in (3, 7, 1, 9)]
    a = BlockAllocator(10, 16, order)
    a.add_seq(0, 16)
    a.fork(0, 1)
    for _ in range(32):
        a.append_slot(0)
    s, src, dst = a.append_slot(1)
    assert (src, dst) == (-1, -1)            # full shared block: grow, no copy
    assert a.table(0) == g["seq_A"] and a.table(1) == g["seq_B"]
    free, ref = a.export_state()
    assert ref[g["shared_block"]] == g["refcount_of_shared"]
    assert a.stats()["shared"] == 1


def test_copy_on_write_of_partial_shared_block():
    a = BlockAllocator(20, 4)
    a.add_seq(0, 6)                           # blocks [0, 1], block 1 half full
    for c in (1, 2):
        a.fork(0, c)
    r1 = a.append_slot(1)
    assert r1[1:] == (1, 2) and r1[0] == 2 * 4 + 2
    r2 = a.append_slot(2)
    assert r2[1:] == (1, 3)
    r0 = a.append_slot(0)                     # last holder writes in place
    assert r0 == (1 * 4 + 2, -1, -1)
    free, ref = a.export_state()
    assert ref[0] == 3 and ref[1] == 1 and ref[2] == 1 and ref[3] == 1
    assert a.stats()["cow_copies"] == 2


def test_shared_prefix_first_step_counts():
    """128 sequences on one prefix ending in a partial block: the first step
    copies the shared block for 127 of them and the last writes in place."""
    a = BlockAllocator(400, 16)
    a.add_seq(0, 2040)
    for c in range(1, 128):
        a.fork(0, c)
    pairs = [a.append_slot(i)[1:] for i in range(128)]
    copies = [p for p in pairs if p[0] >= 0]
    assert len(copies) == 127 and pairs[-1] == (-1, -1)
    assert len({d for _, d in copies}) == 127
    free, ref = a.export_state()
    assert sum(ref) == sum(len(a.table(i)) for i in range(128))


def test_fifo_free_list_and_invariants():
    rng = np.random.default_rng(9)
    nb = 200
    order = rng.permutation(nb).tolist()
    a = BlockAllocator(nb, 8, order)
    live = []
    for k in range(2000):
        if rng.random() < 0.55:
            try:
                a.add_seq(k, int(rng.integers(0, 60)))
                live.append(k)
            except OutOfBlocks:
                pass
        elif live:
            victim = live.pop(int(rng.integers(len(live))))
            before = a.table(victim)
            tail_before = list(a.free)
            a.free_seq(victim)
            assert list(a.free) == tail_before + before     # freed to the back, in order
        free, ref = a.export_state()
        used = [b for b in range(nb) if ref[b] > 0]
        assert sorted(free + used) == list(range(nb))
        assert sum(ref) == sum(len(a.table(s)) for s in live)


def test_out_of_blocks_is_all_or_nothing():
    a = BlockAllocator(4, 4)
    a.add_seq(0, 12)
    state = a.export_state()
    with pytest.raises(OutOfBlocks):
        a.add_seq(1, 8)
    assert a.export_state() == state and a.stats()["alloc_failures"] == 1
    a.add_seq(1, 4)
    with pytest.raises(OutOfBlocks):
        a.append_slot(1)                      # needs a new block, none left
    assert a.seq_len(1) == 4
    a.fork(0, 2)
    a.free_seq(1)
    a.append_slot(0)                          # block 2 of seq 0 is full? len 12 -> new block
    with pytest.raises(OutOfBlocks):
        a.append_slot(2)                      # seq 2 shares a full last block -> needs a new one


def test_bad_arguments():
    with pytest.raises(ValueError):
        BlockAllocator(0, 16)
    with pytest.raises(ValueError):
        BlockAllocator(4, 16, [0, 1, 1, 2])
    a = BlockAllocator(4, 16)
    a.add_seq(0, 1)
    with pytest.raises(ValueError):
        a.add_seq(0, 1)
    with pytest.raises(ValueError):
        a.fork(5, 6)


def test_shared_prefix_of_the_sharing_picture():
    """Document 04 §3: A -> [3,7,1] and B -> [3,9] share block 3; both attend
    it whole, so the batch's shared prefix is [3]. A sequence that does not
    fill block 3 yet shares no whole block."""
    g = golden("sharing_picture.json")
    order = [3, 7, 1, 9] + [b for b in range(10) if b not in (3, 7, 1, 9)]
    a = BlockAllocator(10, 16, order)
    a.add_seq(0, 16)
    a.fork(0, 1)
    for _ in range(32):
        a.append_slot(0)
    a.append_slot(1)
    assert a.table(0) == g["seq_A"] and a.table(1) == g["seq_B"]
    assert a.shared_prefix([0, 1]) == [g["shared_block"]]
    assert a.shared_prefix([1, 0]) == [g["shared_block"]]
    # a third sequence holding block 3 with only 10 of its 16 tokens
    b = BlockAllocator(10, 16, order)
    b.add_seq(0, 10)
    b.fork(0, 1)
    b.append_slot(0)                           # copy-on-write: seq 0 moves off block 3
    assert b.table(1) == [3] and b.table(0) != [3]
    assert b.shared_prefix([0, 1]) == []
    assert oracle.shared_prefix_blocks([[3, 7, 1], [3, 9]], [40, 10], 16) == []


def test_shared_prefix_special_cases():
    assert oracle.shared_prefix_blocks([], [], 16) == []
    # one sequence: its whole blocks (the worked mapping, 40 tokens = 2 whole)
    assert oracle.shared_prefix_blocks([[7, 2, 9]], [40], 16) == [7, 2]
    assert oracle.shared_prefix_blocks([[7, 2, 9]], [48], 16) == [7, 2, 9]
    # no common first block
    assert oracle.shared_prefix_blocks([[1, 2], [2, 1]], [32, 32], 16) == []


def test_shared_prefix_invariants_under_random_forks():
    """After random forks and appends: every returned block sits at the same
    place in every table and is held by at least as many references as there
    are sequences (reference counts are kept apart from the tables), every
    sequence attends it whole, and no longer run has all three properties."""
    rng = np.random.default_rng(12)
    for trial in range(200):
        bs = int(rng.choice([1, 2, 4, 16]))
        a = BlockAllocator(600, bs)
        a.add_seq(0, int(rng.integers(0, 6 * bs)))
        live = [0]
        for nid in range(1, int(rng.integers(2, 7))):
            parent = int(rng.choice(live))
            a.fork(parent, nid)
            live.append(nid)
            for s in live:
                for _ in range(int(rng.integers(0, 2 * bs))):
                    a.append_slot(s)
        batch = [int(s) for s in rng.permutation(live)[:int(rng.integers(1, len(live) + 1))]]
        pre = a.shared_prefix(batch)
        k = len(pre)
        _, ref = a.export_state()
        for j, blk in enumerate(pre):
            assert all(a.table(s)[j] == blk for s in batch)
            assert ref[blk] >= len(batch)
        assert all(a.seq_len(s) >= k * bs for s in batch)
        longer = all(len(a.table(s)) > k and a.seq_len(s) >= (k + 1) * bs for s in batch) and \
            len({a.table(s)[k] for s in batch}) == 1
        assert not longer
