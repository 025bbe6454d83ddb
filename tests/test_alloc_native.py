"""The native block manager (libpa pa_alloc_*) against the oracle's, bit for
bit: free-list order, reference counts, tables, slots, copy-on-write pairs and
counters after every operation."""

import numpy as np
import pytest

import oracle
import synthetic


def _same(native, ref, seqs):
    assert native.export_state() == ref.export_state()
    for s in seqs:
        assert native.table(s) == ref.table(s)
        assert native.seq_len(s) == ref.seq_len(s)
    ns, rs = native.stats(), ref.stats()
    for k in ("free", "used", "shared", "cow_copies", "alloc_failures", "total_refs",
              "num_seqs", "num_blocks"):
        assert ns[k] == rs[k], k


def test_random_ops_with_forks_and_copy_on_write(libpa):
    rng = np.random.default_rng(31)
    nb, bs = 300, 8
    order = rng.permutation(nb).tolist()
    nat = libpa.BlockAllocator(nb, bs, order)
    ref = oracle.BlockAllocator(nb, bs, order)
    live = []
    next_id = 0
    for step in range(3000):
        r = rng.random()
        if r < 0.25 or not live:
            L = int(rng.integers(0, 50))
            ok_n = ok_r = True
            try:
                nat.add_seq(next_id, L)
            except libpa.OutOfBlocksError:
                ok_n = False
            try:
                ref.add_seq(next_id, L)
            except oracle.OutOfBlocks:
                ok_r = False
            assert ok_n == ok_r
            if ok_n:
                live.append(next_id)
            next_id += 1
        elif r < 0.35:
            parent = live[int(rng.integers(len(live)))]
            nat.fork(parent, next_id)
            ref.fork(parent, next_id)
            live.append(next_id)
            next_id += 1
        elif r < 0.8:
            s = live[int(rng.integers(len(live)))]
            try:
                got = nat.append_slot(s)
            except libpa.OutOfBlocksError:
                got = None
            try:
                exp = ref.append_slot(s)
            except oracle.OutOfBlocks:
                exp = None
            assert got == exp
        else:
            s = live.pop(int(rng.integers(len(live))))
            nat.free_seq(s)
            ref.free_seq(s)
        if step % 50 == 0:
            _same(nat, ref, live)
    _same(nat, ref, live)
    assert ref.stats()["cow_copies"] > 10 and ref.stats()["alloc_failures"] > 0


def test_churned_placement_matches(libpa):
    b = synthetic.config3_mha_lognormal(num_seqs=40, num_heads=1, head_dim=8, churn_ops=2000)
    nat = libpa.BlockAllocator(b.num_blocks, b.block_size, b.free_order)
    ref = oracle.BlockAllocator(b.num_blocks, b.block_size, b.free_order)
    for op in b.churn:
        if op.kind == "alloc":
            nat.add_seq(op.owner, op.nblocks * b.block_size)
            ref.add_seq(op.owner, op.nblocks * b.block_size)
        else:
            nat.free_seq(op.owner)
            ref.free_seq(op.owner)
    for i, L in enumerate(b.prefill_lens):
        nat.add_seq(i, int(L))
        ref.add_seq(i, int(L))
    slots, pairs = nat.append_slots(list(range(40)))
    exp = [ref.append_slot(i) for i in range(40)]
    assert slots == [e[0] for e in exp] and pairs == [] and all(e[1] == -1 for e in exp)
    _same(nat, ref, range(40))
    table, lens = nat.build_tables(list(range(40)), 600, fill=-1)
    assert table.tolist() == ref.dense_table(range(40), 600, fill=-1)
    assert lens.tolist() == [ref.seq_len(i) for i in range(40)]


def test_shared_prefix_step_pairs_match(libpa):
    nat = libpa.BlockAllocator(400, 16)
    ref = oracle.BlockAllocator(400, 16)
    for a in (nat, ref):
        a.add_seq(0, 2040)
        for c in range(1, 128):
            a.fork(0, c)
    slots, pairs = nat.append_slots(list(range(128)))
    exp = [ref.append_slot(i) for i in range(128)]
    assert slots == [e[0] for e in exp]
    assert pairs == [(e[1], e[2]) for e in exp if e[1] >= 0]
    assert len(pairs) == 127
    _same(nat, ref, range(128))


def test_out_of_blocks_leaves_state(libpa):
    nat = libpa.BlockAllocator(4, 4)
    nat.add_seq(0, 12)
    before = nat.export_state()
    with pytest.raises(libpa.OutOfBlocksError):
        nat.add_seq(1, 8)
    assert nat.export_state() == before and nat.stats()["alloc_failures"] == 1
    with pytest.raises(libpa.PaError):
        nat.add_seq(0, 1)          # duplicate id
    with pytest.raises(libpa.PaError):
        libpa.BlockAllocator(4, 4, [0, 1, 1, 2])
    slots, pairs = nat.append_slots([])
    assert slots == [] and pairs == []
    table, lens = nat.build_tables([], 5)
    assert table.shape == (0, 5) and lens.shape == (0,)


def test_batched_append_stops_at_failure(libpa):
    nat = libpa.BlockAllocator(3, 2)
    nat.add_seq(0, 2)
    nat.add_seq(1, 2)
    with pytest.raises(libpa.OutOfBlocksError):
        nat.append_slots([0, 1])     # seq 0 takes the last block, seq 1 fails
    assert nat.seq_len(0) == 3 and nat.seq_len(1) == 2


def test_random_ops_with_swapping(libpa):
    """Native block manager against the oracle's under random adds, forks,
    appends, frees, swap-outs and swap-ins: identical results, refusals and
    state (device and host free lists, reference counts) after every op."""
    rng = np.random.default_rng(77)
    nb, bs, nh = 200, 8, 120
    order = rng.permutation(nb).tolist()
    horder = rng.permutation(nh).tolist()
    nat = libpa.BlockAllocator(nb, bs, order)
    ref = oracle.BlockAllocator(nb, bs, order)
    nat.add_host_pool(nh, horder)
    ref.add_host_pool(nh, horder)
    resident, swapped = [], []
    next_id = 0

    def both(fn_n, fn_r):
        try:
            a = fn_n()
        except libpa.OutOfBlocksError:
            a = "oob"
        try:
            b = fn_r()
        except oracle.OutOfBlocks:
            b = "oob"
        assert a == b
        return a

    for step in range(3000):
        r = rng.random()
        if r < 0.2 or not (resident or swapped):
            L = int(rng.integers(0, 60))
            if both(lambda: nat.add_seq(next_id, L), lambda: ref.add_seq(next_id, L)) != "oob":
                resident.append(next_id)
            next_id += 1
        elif r < 0.28 and resident:
            p = resident[int(rng.integers(len(resident)))]
            both(lambda: nat.fork(p, next_id), lambda: ref.fork(p, next_id))
            resident.append(next_id)
            next_id += 1
        elif r < 0.6 and resident:
            s = resident[int(rng.integers(len(resident)))]
            both(lambda: nat.append_slot(s), lambda: ref.append_slot(s))
        elif r < 0.72 and resident:
            s = resident[int(rng.integers(len(resident)))]
            got = both(lambda: nat.swap_out(s), lambda: ref.swap_out(s))
            if got != "oob":
                resident.remove(s)
                swapped.append(s)
        elif r < 0.84 and swapped:
            s = swapped[int(rng.integers(len(swapped)))]
            got = both(lambda: nat.swap_in(s), lambda: ref.swap_in(s))
            if got != "oob":
                swapped.remove(s)
                resident.append(s)
        else:
            pool = resident + swapped
            if not pool:
                continue
            s = pool[int(rng.integers(len(pool)))]
            nat.free_seq(s)
            ref.free_seq(s)
            (resident if s in resident else swapped).remove(s)
        assert nat.export_state() == ref.export_state()
        assert nat.export_host_state() == ref.export_host_state()
    assert nat.stats() == ref.stats()
    assert nat.export_host_state()[2] > 20 and nat.export_host_state()[3] > 10


def test_swapped_sequence_is_refused(libpa):
    a = libpa.BlockAllocator(16, 4)
    a.add_host_pool(8)
    a.add_seq(1, 6)
    a.swap_out(1)
    for call in (lambda: a.append_slot(1), lambda: a.fork(1, 2), lambda: a.table(1),
                 lambda: a.build_tables([1], 4), lambda: a.swap_out(1)):
        with pytest.raises(libpa.PaError):
            call()
    assert a.seq_len(1) == 6
    a.swap_in(1)
    assert len(a.table(1)) == 2


def test_shared_prefix_matches_oracle(libpa):
    """pa_alloc_shared_prefix against the oracle's definition after random
    forks and appends, for random batches (order and subset)."""
    rng = np.random.default_rng(44)
    for trial in range(150):
        bs = int(rng.choice([1, 4, 16]))
        nat, ref = libpa.BlockAllocator(800, bs), oracle.BlockAllocator(800, bs)
        L0 = int(rng.integers(0, 8 * bs))
        nat.add_seq(0, L0)
        ref.add_seq(0, L0)
        live = [0]
        for nid in range(1, int(rng.integers(2, 8))):
            parent = int(rng.choice(live))
            nat.fork(parent, nid)
            ref.fork(parent, nid)
            live.append(nid)
            for s in live:
                for _ in range(int(rng.integers(0, 2 * bs))):
                    assert nat.append_slot(s) == ref.append_slot(s)
        batch = [int(s) for s in rng.permutation(live)[:int(rng.integers(0, len(live) + 1))]]
        got = nat.shared_prefix(batch)
        assert got.dtype == np.int32 and got.tolist() == ref.shared_prefix(batch)


def test_shared_prefix_of_a_forked_prompt(libpa):
    """128 sequences forked from a 2040-token prompt, after their first
    append: the 127 whole prompt blocks are shared, the partial one was
    copied on write."""
    a = libpa.BlockAllocator(400, 16)
    a.add_seq(0, 2040)
    for c in range(1, 128):
        a.fork(0, c)
    a.append_slots(list(range(128)))
    pre = a.shared_prefix(list(range(128)))
    assert pre.tolist() == a.table(0)[:127]


def test_shared_prefix_refusals(libpa):
    a = libpa.BlockAllocator(8, 4)
    a.add_seq(0, 8)
    with pytest.raises(libpa.PaError):
        a.shared_prefix([0, 5])                 # unknown sequence
    a.add_host_pool(8)
    a.fork(0, 1)
    a.swap_out(1)
    with pytest.raises(libpa.PaError):
        a.shared_prefix([0, 1])                 # swapped out
    assert a.shared_prefix([]).tolist() == []
    assert a.shared_prefix([0]).tolist() == a.table(0)


def test_shared_prefix_capacity_reports_the_length_needed(libpa):
    """A buffer too small for the run: PA_ERR_INVALID_ARG, the length needed
    in *num_blocks, the caller's buffer untouched and the manager unchanged."""
    import ctypes
    from paged_kv_cache_40_gb300._lib import STATUS_NAMES
    a = libpa.BlockAllocator(64, 4, list(range(63, -1, -1)))
    a.add_seq(0, 22)                            # 5 whole blocks + 2 tokens
    a.fork(0, 1)
    before = a.export_state()
    ids = np.array([0, 1], np.int64)
    buf = np.full(8, -7, np.int32)
    k = ctypes.c_int(-1)
    L = libpa.lib()
    st = L.pa_alloc_shared_prefix(a._h, ids.ctypes.data, 2, buf.ctypes.data, 3, ctypes.byref(k))
    assert STATUS_NAMES[st] == "PA_ERR_INVALID_ARG"
    assert k.value == 5
    assert (buf == -7).all()
    k.value = -1
    st = L.pa_alloc_shared_prefix(a._h, ids.ctypes.data, 2, None, 0, ctypes.byref(k))
    assert STATUS_NAMES[st] == "PA_ERR_INVALID_ARG" and k.value == 5
    assert L.pa_alloc_shared_prefix(a._h, ids.ctypes.data, 2, buf.ctypes.data, 5,
                                    ctypes.byref(k)) == 0
    assert k.value == 5 and buf[:5].tolist() == a.table(0)[:5] and (buf[5:] == -7).all()
    assert a.export_state() == before


def _oracle_step(ref, ids, max_blocks, fill=-1):
    slots, pairs = [], []
    for s in ids:
        sl, cs, cd = ref.append_slot(s)
        slots.append(sl)
        if cs >= 0:
            pairs.append((cs, cd))
    return slots, pairs, np.asarray(ref.dense_table(ids, max_blocks, fill), np.int32)


def test_plan_step_matches_the_oracle_step_by_step(libpa):
    """One call per step (slots, copy-on-write pairs, tables, lengths) equals
    the oracle's block manager appending the batch in order and tabling it,
    over steps of a forked batch (shared blocks, copies, in-place writes) and
    random growth."""
    rng = np.random.default_rng(44)
    nb, bs = 400, 8
    order = rng.permutation(nb).tolist()
    nat = libpa.BlockAllocator(nb, bs, order)
    ref = oracle.BlockAllocator(nb, bs, order)
    for a in (nat, ref):
        a.add_seq(0, 29)
        a.add_seq(1, 16)
        a.add_seq(2, 0)
        a.fork(0, 3)
        a.fork(0, 4)
        a.fork(1, 5)
    ids = [4, 0, 1, 2, 3, 5]
    mb = 12
    for step in range(40):
        batch = [s for s in ids if rng.random() < 0.8]
        slots, pairs, table, lens = nat.plan_step(batch, mb)
        es, ep, et = _oracle_step(ref, batch, mb)
        assert slots.tolist() == es, step
        assert [tuple(p) for p in pairs.tolist()] == ep, step
        assert table.tolist() == et.tolist(), step
        assert lens.tolist() == [ref.seq_len(s) for s in batch], step
        _same(nat, ref, ids)
    assert nat.stats()["cow_copies"] > 0


def test_plan_step_into_caller_buffers(libpa):
    """Outputs land in preallocated arrays (as the pinned input buffers of a
    step), pairs first rows only; the first step of 128 forks of a 2040-token
    prompt makes 127 copies and one in-place write."""
    a = libpa.BlockAllocator(400, 16)
    a.add_seq(0, 2040)
    for c in range(1, 128):
        a.fork(0, c)
    n, mb = 128, 130
    bufs = (np.full(n, -9, np.int32), np.full((n, 2), -9, np.int32),
            np.full((n, mb), -9, np.int32), np.full(n, -9, np.int32))
    slots, pairs, table, lens = a.plan_step(list(range(n)), mb, fill=-1, out=bufs)
    assert slots.base is bufs[0] or slots.ctypes.data == bufs[0].ctypes.data
    assert len(pairs) == 127 and pairs.ctypes.data == bufs[1].ctypes.data
    assert (bufs[1][127:] == -9).all()
    assert (lens == 2041).all() and (bufs[3] == 2041).all()
    assert (table[:, 128:] == -1).all()
    prompt_last = a.table(127)[127]       # the last holder wrote in place
    assert all(p[0] == prompt_last for p in pairs.tolist())


def test_plan_step_refusals_change_nothing(libpa):
    a = libpa.BlockAllocator(6, 4, list(range(6)))
    a.add_seq(0, 8)      # 2 blocks, full: grows on append
    a.add_seq(1, 6)      # 2 blocks
    a.fork(1, 2)         # shares 1's blocks: the append of 1 or 2 copies
    before, st = a.export_state(), a.stats()
    with pytest.raises(libpa.PaError):
        a.plan_step([0, 7], 4)              # unknown sequence
    with pytest.raises(libpa.PaError):
        a.plan_step([0, 1, 0], 4)           # listed twice
    with pytest.raises(libpa.PaError):
        a.plan_step([0], 2)                 # 3 blocks after the append
    assert a.export_state() == before
    a.add_seq(3, 4)      # takes the last two free blocks... one block
    a.add_seq(4, 4)
    before = a.export_state()
    # 0 grows (1 block) and 1 copies (1 block): 2 needed, 0 free
    with pytest.raises(libpa.OutOfBlocksError):
        a.plan_step([0, 1, 2], 4)
    assert a.export_state() == before
    assert a.stats()["alloc_failures"] == st["alloc_failures"] + 1
    # 2 then 1: 2 copies (refcount 2 -> 1), 1 writes in place: 1 block; still 0 free
    with pytest.raises(libpa.OutOfBlocksError):
        a.plan_step([2], 4)
    a.free_seq(4)
    slots, pairs, table, lens = a.plan_step([2, 1], 4)
    assert len(pairs) == 1 and lens.tolist() == [7, 7]
