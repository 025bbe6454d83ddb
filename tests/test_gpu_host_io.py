"""Host-memory paths of a decode step on the GPU: the attention calls write
their output straight into pinned host memory (through its device mapping),
bit-equal to a device output, pageable host memory is refused before any
launch, and a step whose inputs are packed into one buffer and uploaded with
one copy gives the same pools and output as the unpacked step."""

import ctypes

import numpy as np
import pytest

import oracle
import synthetic
from tests.gpu_helpers import assert_close_attention, poison_unread_rows

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def pa(libpa):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return libpa


def d(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _case(seed=3, BS=16):
    rng = np.random.default_rng(seed)
    lens = [1, 40, 300, 1000, 17]
    S, Hkv, G, D = len(lens), 2, 4, 128
    mb = max(-(-L // BS) for L in lens)
    nb = sum(-(-L // BS) for L in lens) + 3
    perm = rng.permutation(nb)
    table = -np.ones((S, mb), np.int32)
    pos = 0
    for i, L in enumerate(lens):
        n = -(-L // BS)
        table[i, :n] = perm[pos:pos + n]
        pos += n
    q = rng.standard_normal((S, G * Hkv, D)).astype(np.float16)
    kp = rng.standard_normal((nb, BS, Hkv, D)).astype(np.float16)
    vp = rng.standard_normal((nb, BS, Hkv, D)).astype(np.float16)
    kp, vp = poison_unread_rows(kp, vp, table, lens, BS)
    return q, kp, vp, table, np.asarray(lens, np.int32)


def test_output_into_pinned_host_memory(pa):
    q, kp, vp, table, lens = _case()
    args = (d(q), d(kp), d(vp), d(table), d(lens), 0.088)
    dev = pa.pa_decode_attention(*args)
    host = torch.empty(q.shape, dtype=torch.float16).pin_memory()
    pa.pa_decode_attention(*args, out=host)
    fixed_host = torch.empty(q.shape, dtype=torch.float16).pin_memory()
    pa.pa_decode_attention_fixed_scratch(*args, out=fixed_host)
    torch.cuda.synchronize()
    assert torch.equal(host, dev.cpu())
    assert torch.equal(fixed_host, dev.cpu())
    exp = oracle.decode_attention(q, kp, vp, table, lens, np.float32(0.088))
    assert_close_attention(host.numpy(), exp, "output in pinned host memory")


def test_fp8_and_shared_prefix_outputs_into_pinned_host_memory(pa):
    rng = np.random.default_rng(9)
    q, kp, vp, table, lens = _case(seed=9)
    k8 = synthetic.fp8_codes(rng, kp.shape)
    v8 = synthetic.fp8_codes(rng, vp.shape)
    ks = np.full(2, 0.01, np.float32)
    vs = np.full(2, 0.02, np.float32)
    a8 = (d(q), d(k8), d(v8), d(ks), d(vs), d(table), d(lens), 0.088)
    dev8 = pa.pa_decode_attention_fp8(*a8)
    host8 = torch.empty(q.shape, dtype=torch.float16).pin_memory()
    pa.pa_decode_attention_fp8(*a8, out=host8)
    # shared prefix: every table starts with the same two blocks
    t2 = table.copy()
    t2[:, :2] = table[3, :2]
    lens2 = np.maximum(lens, 33).astype(np.int32)
    for i in range(len(lens2)):
        need = -(-int(lens2[i]) // 16)
        for j in range(need):
            if t2[i, j] < 0:
                t2[i, j] = table[3, j]
    prefix = d(t2[0, :2].copy())
    ap = (d(q), d(kp), d(vp), prefix, d(t2), d(lens2), 0.088)
    devp = pa.pa_decode_attention_shared_prefix(*ap)
    hostp = torch.empty(q.shape, dtype=torch.float16).pin_memory()
    pa.pa_decode_attention_shared_prefix(*ap, out=hostp)
    torch.cuda.synchronize()
    assert torch.equal(host8, dev8.cpu())
    assert torch.equal(hostp, devp.cpu())


def test_pageable_output_is_refused_before_launch(pa):
    q, kp, vp, table, lens = _case()
    host = torch.empty(q.shape, dtype=torch.float16)           # not pinned
    with pytest.raises(ValueError):
        pa.pa_decode_attention(d(q), d(kp), d(vp), d(table), d(lens), 0.1, out=host)
    # the library refuses it too (the binding is not the only guard)
    lib = pa.lib()
    S, Hq, D = q.shape
    nb, BS, Hkv, _ = kp.shape
    dq, dk, dv, dt, dl = d(q), d(kp), d(vp), d(table), d(lens)
    ws = pa.alloc_workspace(S, Hq, Hkv, D, BS, table.shape[1])
    pageable = np.zeros(q.size, np.float16)
    st = lib.pa_decode_attention(
        ctypes.c_void_p(dq.data_ptr()), ctypes.c_void_p(dk.data_ptr()),
        ctypes.c_void_p(dv.data_ptr()), ctypes.c_void_p(dt.data_ptr()),
        ctypes.c_void_p(dl.data_ptr()), S, Hq, Hkv, D, BS, table.shape[1], nb, 0,
        ctypes.c_float(0.1), ctypes.c_void_p(pageable.ctypes.data), ctypes.c_void_p(ws.data_ptr()),
        ws.numel(), 0, None)
    assert st == 1 and b"pinned" in lib.pa_last_error()


def test_packed_inputs_step_matches_unpacked(pa):
    """One decode step of the copy-on-write batch (127 copies) with its inputs
    packed and uploaded in one copy, the output written to pinned host memory."""
    from paged_kv_cache_40_gb300.engine import DecodeBatchRunner, SharedPrefixRunner
    w = synthetic.config4_shared_prefix()
    a = SharedPrefixRunner(w)
    a.plan_step()
    a.run_step()
    b = SharedPrefixRunner(w)
    b.plan_step()
    b.pack_inputs()
    host = torch.empty(b.out.shape, dtype=torch.float16).pin_memory()
    b.out = host
    assert b.upload_inputs() == b.host_arena.numel()
    b.run_step()
    torch.cuda.synchronize()
    assert torch.equal(a.k_pool, b.k_pool) and torch.equal(a.v_pool, b.v_pool)
    assert torch.equal(a.out.cpu(), host)
    assert pa.pa_device_error() == 0
    # the plain runner on the GQA batch, several uploads of the same step
    g = synthetic.config2_gqa_batch(num_seqs=9, lo=1, hi=700)
    r1 = DecodeBatchRunner(g)
    r1.plan_step()
    r1.run_step()
    r2 = DecodeBatchRunner(g)
    r2.plan_step()
    r2.pack_inputs()
    for _ in range(3):
        r2.upload_inputs()
        r2.run_step()
    torch.cuda.synchronize()
    assert torch.equal(r1.out, r2.out)
    # then the same runner with its inputs moved to host memory (as the
    # benchmark times both paths one after the other)
    assert r2.host_inputs() == sum(t.numel() * t.element_size()
                                   for t in r2.packed_host.values())
    r2.run_step()
    torch.cuda.synchronize()
    assert torch.equal(r1.out, r2.out)


def test_inputs_read_from_pinned_host_memory(pa):
    """A step whose every input (q, new K/V rows, slots, copy pairs, tables,
    lengths, the prefix block list) lives in pinned host memory gives the
    same pools and output, bit for bit, as the step with device inputs."""
    from paged_kv_cache_40_gb300.engine import DecodeBatchRunner, SharedPrefixRunner
    g = synthetic.config2_gqa_batch(num_seqs=11, lo=1, hi=900)
    a = DecodeBatchRunner(g)
    a.plan_step()
    a.run_step()
    b = DecodeBatchRunner(g)
    b.plan_step()
    assert b.host_inputs() > 0 and not b.q.is_cuda and b.q.is_pinned()
    b.out = torch.empty(b.out.shape, dtype=torch.float16).pin_memory()
    b.run_step()
    torch.cuda.synchronize()
    assert torch.equal(a.k_pool, b.k_pool) and torch.equal(a.v_pool, b.v_pool)
    assert torch.equal(a.out.cpu(), b.out)
    # copy-on-write pairs and the shared prefix's block list from host memory
    w = synthetic.config4_shared_prefix()
    c = SharedPrefixRunner(w)
    c.plan_step()
    c.run_step()
    e = SharedPrefixRunner(w)
    e.plan_step()
    e.host_inputs()
    assert not e.d_pairs.is_cuda and not e.d_prefix.is_cuda
    e.run_step()
    torch.cuda.synchronize()
    assert torch.equal(c.k_pool, e.k_pool) and torch.equal(c.out, e.out)
    assert pa.pa_device_error() == 0


def test_fp8_step_inputs_from_pinned_host_memory(pa):
    from paged_kv_cache_40_gb300.engine import DecodeBatchRunner
    g = synthetic.config2_gqa_batch(num_seqs=7, lo=1, hi=600)
    c8 = synthetic.fp8_cache(g)
    kw = dict(kv_dtype="fp8", k_pool=c8.k_pool, v_pool=c8.v_pool, k_scale=c8.k_scale,
              v_scale=c8.v_scale)
    a = DecodeBatchRunner(g, **kw)
    a.plan_step()
    a.run_step()
    b = DecodeBatchRunner(g, **kw)
    b.plan_step()
    b.host_inputs()
    b.k_scale = b.k_scale.cpu().pin_memory()
    b.v_scale = b.v_scale.cpu().pin_memory()
    b.run_step()
    torch.cuda.synchronize()
    assert torch.equal(a.k_pool, b.k_pool) and torch.equal(a.out, b.out)


def test_pageable_inputs_and_host_pools_are_refused(pa):
    q, kp, vp, table, lens = _case()
    with pytest.raises(ValueError):
        pa.pa_decode_attention(torch.from_numpy(q), d(kp), d(vp), d(table), d(lens), 0.1)
    with pytest.raises(ValueError):
        pa.pa_decode_attention(d(q), torch.from_numpy(kp).pin_memory(),
                               torch.from_numpy(vp).pin_memory(), d(table), d(lens), 0.1)
    # the library itself refuses a pageable table and a pinned host pool
    lib = pa.lib()
    S, Hq, D = q.shape
    nb, BS, Hkv, _ = kp.shape
    dq, dk, dv, dl = d(q), d(kp), d(vp), d(lens)
    ws = pa.alloc_workspace(S, Hq, Hkv, D, BS, table.shape[1])
    out = torch.empty(q.shape, dtype=torch.float16, device="cuda")
    pageable_table = np.ascontiguousarray(table)
    vp_ = lambda t: ctypes.c_void_p(t.data_ptr())
    st = lib.pa_decode_attention(vp_(dq), vp_(dk), vp_(dv),
                                 ctypes.c_void_p(pageable_table.ctypes.data), vp_(dl), S, Hq, Hkv, D,
                                 BS, table.shape[1], nb, 0, ctypes.c_float(0.1), vp_(out), vp_(ws),
                                 ws.numel(), 0, None)
    assert st == 1 and b"pinned" in lib.pa_last_error()
    host_pool = torch.from_numpy(kp).pin_memory()
    st = lib.pa_decode_attention(vp_(dq), vp_(host_pool), vp_(dv), vp_(d(table)), vp_(dl), S, Hq,
                                 Hkv, D, BS, table.shape[1], nb, 0, ctypes.c_float(0.1), vp_(out),
                                 vp_(ws), ws.numel(), 0, None)
    assert st == 1 and b"device memory" in lib.pa_last_error()


def test_steps_planned_in_place_match_the_oracle(pa):
    """A decode loop whose steps the block manager plans with one call each
    straight into pinned host memory (two rotating buffer sets, the kernels
    reading them in place), the sequences growing by a token a step: slots,
    copy-on-write pairs, tables, lengths and the pools bit-exact with the
    oracle's block manager and cache operations, attention within tolerance,
    over steps that grow blocks."""
    import dataclasses
    from paged_kv_cache_40_gb300.engine import DecodeBatchRunner
    rng = np.random.default_rng(12)
    lens0 = rng.integers(14, 40, size=6, endpoint=True)
    steps = 20
    nb = sum(-(-(int(L) + steps + 1) // 16) for L in lens0) + 4   # room for the growth
    b = synthetic.make_batch("planned", rng, lens0, 32, 8, 128, 16, nb, seed=12)
    mb = max(-(-(int(L) + steps + 1) // b.block_size) for L in b.prefill_lens)
    run = DecodeBatchRunner(b, max_blocks=mb)
    run.host_planned(sets=2)
    ref = oracle.BlockAllocator(b.num_blocks, b.block_size, b.free_order)
    for i, L in enumerate(b.prefill_lens):
        ref.add_seq(i, int(L))
    kp, vp = b.k_pool.copy(), b.v_pool.copy()
    ids = list(range(b.num_seqs))
    for k in range(steps):
        plan = run.plan_step_host()
        slots, pairs = [], []
        for s_ in ids:
            sl, cs, cd = ref.append_slot(s_)
            slots.append(sl)
            if cs >= 0:
                pairs.append((cs, cd))
        table = np.asarray(ref.dense_table(ids, mb), np.int32)
        lens = np.asarray([ref.seq_len(s_) for s_ in ids], np.int32)
        assert plan.slots.tolist() == slots and plan.cow_pairs.tolist() == [list(p) for p in pairs]
        assert plan.block_table.tolist() == table.tolist()
        assert plan.seq_lens.tolist() == lens.tolist()
        run.run_step()
        torch.cuda.synchronize()
        assert pa.pa_device_error() == 0
        if pairs:
            kp, vp = oracle.copy_blocks(kp, vp, np.asarray(pairs, np.int32))
        kp, vp = oracle.append_kv(kp, vp, b.k_new, b.v_new, np.asarray(slots, np.int32))
        assert np.array_equal(run.k_pool.cpu().numpy().view(np.uint16), kp.view(np.uint16))
        assert np.array_equal(run.v_pool.cpu().numpy().view(np.uint16), vp.view(np.uint16))
        exp = oracle.decode_attention(b.q, kp, vp, table, lens, b.scale)
        assert_close_attention(run.out.cpu().numpy(), exp, f"planned step {k}")


def test_one_call_steps_match_the_oracle(pa):
    """pa_decode_step (plan, copy-on-write copies, append and attention in one
    library call, the plan written into pinned host memory the kernels read in
    place) over steps of a batch with forked sequences (shared blocks, so the
    first steps copy): plans, pools and outputs against the oracle."""
    from paged_kv_cache_40_gb300.engine import DecodeBatchRunner
    rng = np.random.default_rng(21)
    lens0 = rng.integers(14, 40, size=5, endpoint=True)
    lens0[1] = 21                       # a partial last block: the fork's first append copies
    steps = 12
    nb = sum(-(-(int(L) + steps + 1) // 16) for L in lens0) * 2 + 8
    b = synthetic.make_batch("one-call", rng, lens0, 16, 4, 128, 16, nb, seed=21)
    mb = max(-(-(int(L) + steps + 1) // 16) for L in lens0) + 1
    run = DecodeBatchRunner(b, max_blocks=mb)
    ref = oracle.BlockAllocator(b.num_blocks, b.block_size, b.free_order)
    for i, L in enumerate(b.prefill_lens):
        ref.add_seq(i, int(L))
    # sequence 4 becomes a fork of sequence 1: its blocks are shared
    run.alloc.free_seq(4)
    run.alloc.fork(1, 4)
    ref.free_seq(4)
    ref.fork(1, 4)
    run.host_planned(sets=2)
    run.prepare_native_steps()
    kp, vp = b.k_pool.copy(), b.v_pool.copy()
    ids = list(range(b.num_seqs))
    copies = 0
    for k in range(steps):
        plan = run.run_native_step()
        slots, pairs = [], []
        for s_ in ids:
            sl, cs, cd = ref.append_slot(s_)
            slots.append(sl)
            if cs >= 0:
                pairs.append((cs, cd))
        table = np.asarray(ref.dense_table(ids, mb), np.int32)
        lens = np.asarray([ref.seq_len(s_) for s_ in ids], np.int32)
        torch.cuda.synchronize()
        assert pa.pa_device_error() == 0
        assert plan.slots.tolist() == slots and plan.cow_pairs.tolist() == [list(p) for p in pairs]
        assert plan.block_table.tolist() == table.tolist()
        assert plan.seq_lens.tolist() == lens.tolist()
        copies += len(pairs)
        if pairs:
            kp, vp = oracle.copy_blocks(kp, vp, np.asarray(pairs, np.int32))
        kp, vp = oracle.append_kv(kp, vp, b.k_new, b.v_new, np.asarray(slots, np.int32))
        assert np.array_equal(run.k_pool.cpu().numpy().view(np.uint16), kp.view(np.uint16))
        assert np.array_equal(run.v_pool.cpu().numpy().view(np.uint16), vp.view(np.uint16))
        exp = oracle.decode_attention(b.q, kp, vp, table, lens, b.scale)
        assert_close_attention(run.out.cpu().numpy(), exp, f"one-call step {k}")
    assert copies >= 1


def test_one_call_fp8_steps_match_the_oracle(pa):
    """pa_decode_step_fp8 over steps of a batch with a forked sequence: the
    plans, the E4M3 pools (bit-exact: copies, then each new row quantized with
    its KV head's scale) and the outputs against the oracle."""
    from paged_kv_cache_40_gb300.engine import DecodeBatchRunner
    rng = np.random.default_rng(23)
    lens0 = rng.integers(14, 40, size=5, endpoint=True)
    lens0[2] = 37                       # a partial last block: the fork's first append copies
    steps = 10
    nb = sum(-(-(int(L) + steps + 1) // 16) for L in lens0) * 2 + 8
    b = synthetic.make_batch("one-call-fp8", rng, lens0, 16, 4, 128, 16, nb, seed=23)
    c = synthetic.fp8_cache(b, seed=24)
    mb = max(-(-(int(L) + steps + 1) // 16) for L in lens0) + 1
    run = DecodeBatchRunner(b, max_blocks=mb, kv_dtype="fp8", k_pool=c.k_pool, v_pool=c.v_pool,
                            k_scale=c.k_scale, v_scale=c.v_scale)
    ref = oracle.BlockAllocator(b.num_blocks, b.block_size, b.free_order)
    for i, L in enumerate(b.prefill_lens):
        ref.add_seq(i, int(L))
    run.alloc.free_seq(4)
    run.alloc.fork(2, 4)
    ref.free_seq(4)
    ref.fork(2, 4)
    run.host_planned(sets=2)
    run.prepare_native_steps()
    kp, vp = c.k_pool.copy(), c.v_pool.copy()
    ids = list(range(b.num_seqs))
    copies = 0
    for k in range(steps):
        plan = run.run_native_step()
        slots, pairs = [], []
        for s_ in ids:
            sl, cs, cd = ref.append_slot(s_)
            slots.append(sl)
            if cs >= 0:
                pairs.append((cs, cd))
        table = np.asarray(ref.dense_table(ids, mb), np.int32)
        lens = np.asarray([ref.seq_len(s_) for s_ in ids], np.int32)
        torch.cuda.synchronize()
        assert pa.pa_device_error() == 0
        assert plan.slots.tolist() == slots and plan.cow_pairs.tolist() == [list(p) for p in pairs]
        assert plan.block_table.tolist() == table.tolist()
        assert plan.seq_lens.tolist() == lens.tolist()
        copies += len(pairs)
        if pairs:
            kp, vp = oracle.copy_blocks(kp, vp, np.asarray(pairs, np.int32))
        kp, vp = oracle.append_kv_fp8(kp, vp, b.k_new, b.v_new, np.asarray(slots, np.int32),
                                      c.k_scale, c.v_scale)
        assert np.array_equal(run.k_pool.cpu().numpy(), kp)
        assert np.array_equal(run.v_pool.cpu().numpy(), vp)
        exp = oracle.decode_attention_fp8(b.q, kp, vp, c.k_scale, c.v_scale, table, lens, b.scale)
        assert_close_attention(run.out.cpu().numpy(), exp, f"one-call fp8 step {k}")
    assert copies >= 1


def test_one_call_steps_queued_behind_slow_work(pa):
    """Steps enqueued back to back with no wait, each behind slow device work,
    so the host plans far ahead of the device over two rotating sets of plan
    buffers that the kernels read in place: no set may be rewritten before the
    kernels that read it have run (the runner waits for them), so every step
    appends its own row. The pools after all steps are bit-exact with the
    oracle's block manager replayed over the same steps, and the last output
    matches the oracle's attention."""
    from paged_kv_cache_40_gb300.engine import DecodeBatchRunner
    rng = np.random.default_rng(25)
    lens0 = rng.integers(14, 40, size=6, endpoint=True)
    steps = 16
    nb = sum(-(-(int(L) + steps + 1) // 16) for L in lens0) + 8
    b = synthetic.make_batch("queued", rng, lens0, 16, 4, 128, 16, nb, seed=25)
    mb = max(-(-(int(L) + steps + 1) // 16) for L in lens0) + 1
    run = DecodeBatchRunner(b, max_blocks=mb)
    ref = oracle.BlockAllocator(b.num_blocks, b.block_size, b.free_order)
    for i, L in enumerate(b.prefill_lens):
        ref.add_seq(i, int(L))
    run.host_planned(sets=2)
    run.prepare_native_steps()
    slow = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")
    torch.cuda.synchronize()
    for k in range(steps):
        slow.fill_(k & 0xFF)            # about 0.1 ms of device work ahead of each step
        run.run_native_step()
    torch.cuda.synchronize()
    assert pa.pa_device_error() == 0
    kp, vp = b.k_pool.copy(), b.v_pool.copy()
    ids = list(range(b.num_seqs))
    for k in range(steps):
        slots, pairs = [], []
        for s_ in ids:
            sl, cs, cd = ref.append_slot(s_)
            slots.append(sl)
            if cs >= 0:
                pairs.append((cs, cd))
        if pairs:
            kp, vp = oracle.copy_blocks(kp, vp, np.asarray(pairs, np.int32))
        kp, vp = oracle.append_kv(kp, vp, b.k_new, b.v_new, np.asarray(slots, np.int32))
    assert np.array_equal(run.k_pool.cpu().numpy().view(np.uint16), kp.view(np.uint16))
    assert np.array_equal(run.v_pool.cpu().numpy().view(np.uint16), vp.view(np.uint16))
    table = np.asarray(ref.dense_table(ids, mb), np.int32)
    lens = np.asarray([ref.seq_len(s_) for s_ in ids], np.int32)
    exp = oracle.decode_attention(b.q, kp, vp, table, lens, b.scale)
    assert_close_attention(run.out.cpu().numpy(), exp, "queued one-call steps")
