"""Shared prefix + copy-on-write over many decode steps, GPU vs oracle.

128 sequences share a 2040-token prefix (the last shared block holds 8
tokens). Every step each active sequence appends one token -- the first step
copies the partial shared block for 127 sequences and the last holder writes
in place -- and then attends. Sequence i retires after its own number of
steps. Checked: the native block manager against the oracle's after every
step (bit-exact), the pools after the first and the last step (bit-exact),
and attention at the first step and at each sequence's last step."""

import numpy as np
import pytest

import oracle
import synthetic
from tests.gpu_helpers import assert_close_attention

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def run_shared_prefix(pa, w, heads_first=(0, 13, 31), heads_last=None):
    S, BS = w.num_seqs, w.block_size
    nat = pa.BlockAllocator(w.num_blocks, BS, w.free_order)
    ref = oracle.BlockAllocator(w.num_blocks, BS, w.free_order)
    for a in (nat, ref):
        a.add_seq(0, w.prefix_len)
        for c in range(1, S):
            a.fork(0, c)
    assert nat.stats()["shared"] == -(-w.prefix_len // BS)
    kp, vp = w.k_pool, w.v_pool
    dk, dv = dev(kp), dev(vp)
    mb = -(-(w.prefix_len + int(w.steps.max())) // BS)
    remaining = w.steps.copy()
    active = list(range(S))
    step = 0
    while active:
        q, kn, vn = w.step_inputs(step, len(active))
        slots, pairs = nat.append_slots(active)
        exp = [ref.append_slot(s) for s in active]
        assert slots == [e[0] for e in exp]
        assert pairs == [(e[1], e[2]) for e in exp if e[1] >= 0]
        if step == 0:
            assert len(pairs) == S - 1
        pairs_np = np.asarray(pairs, np.int32).reshape(-1, 2)
        if len(pairs):
            kp, vp = oracle.copy_blocks(kp, vp, pairs_np)
            pa.pa_copy_blocks(dk, dv, dev(pairs_np))
        kp, vp = oracle.append_kv(kp, vp, kn, vn, np.asarray(slots, np.int32))
        pa.pa_append_kv(dev(kn), dev(vn), dk, dv, dev(np.asarray(slots, np.int32)))
        table, lens = nat.build_tables(active, mb)
        assert table.tolist() == ref.dense_table(active, mb)
        out = pa.pa_decode_attention(dev(q), dk, dv, dev(table), dev(lens), float(w.scale))
        retiring = [j for j, s in enumerate(active) if remaining[s] == 1]
        rows = list(range(len(active))) if step == 0 else retiring
        heads = heads_first if step == 0 else heads_last
        heads = None if heads is None else list(heads)
        if rows:
            got = out.cpu().numpy()
            e = oracle.decode_attention(q, kp, vp, table, lens, w.scale, seqs=rows, heads=heads)
            hs = list(range(w.num_q_heads)) if heads is None else list(heads)
            assert_close_attention(got[np.ix_(rows, hs)], e[np.ix_(rows, hs)], f"step {step}")
        if step == 0:
            torch.cuda.synchronize()
            assert np.array_equal(dk.cpu().numpy().view(np.uint16), kp.view(np.uint16))
            assert np.array_equal(dv.cpu().numpy().view(np.uint16), vp.view(np.uint16))
        for j in retiring:
            nat.free_seq(active[j])
            ref.free_seq(active[j])
        assert nat.export_state() == ref.export_state()
        for s in active:
            remaining[s] -= 1
        active = [s for s in active if remaining[s] > 0]
        step += 1
    torch.cuda.synchronize()
    assert np.array_equal(dk.cpu().numpy().view(np.uint16), kp.view(np.uint16))
    assert np.array_equal(dv.cpu().numpy().view(np.uint16), vp.view(np.uint16))
    assert pa.pa_device_error() == 0
    assert nat.stats()["used"] == 0 and nat.stats()["free"] == w.num_blocks
    return step


def test_shared_prefix_small(libpa):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    w = synthetic.config4_shared_prefix(num_seqs=9, prefix_len=70, max_steps=40)
    steps = run_shared_prefix(libpa, w, heads_first=None, heads_last=None)
    assert steps == int(w.steps.max())


def test_shared_prefix_full_size(libpa):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    w = synthetic.config4_shared_prefix()
    run_shared_prefix(libpa, w, heads_last=[0, 17, 31])
