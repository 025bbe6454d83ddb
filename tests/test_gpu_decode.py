"""Paged decode attention on the GPU (through the C ABI) against the fp64
oracle, on the seeded workloads and on edge cases. Pool rows no sequence may
read are NaN-poisoned, so any read outside a sequence's tokens fails."""

import dataclasses
import math

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


def _poisoned(batch):
    """Batch with unread pool rows set to NaN (placement computed by the oracle)."""
    ref = oracle.decode_step(batch, compute_attention=False)
    kp, vp = poison_unread_rows(batch.k_pool, batch.v_pool, ref.block_table, ref.seq_lens,
                                batch.block_size)
    return dataclasses.replace(batch, k_pool=kp, v_pool=vp)


def run_and_compare(pa, batch, partition_tokens=0, seqs=None, heads=None, poison=True):
    from paged_kv_cache_40_gb300.engine import DecodeBatchRunner
    if poison:
        batch = _poisoned(batch)
    ref = oracle.decode_step(batch, compute_attention=False)
    run = DecodeBatchRunner(batch, partition_tokens=partition_tokens)
    plan = run.plan_step()
    # host slot assignment: bit-exact with the oracle's block manager
    assert plan.slots.tolist() == ref.slot_mapping.tolist()
    assert plan.cow_pairs.tolist() == ref.cow_pairs.tolist()
    assert plan.block_table.tolist() == ref.block_table.tolist()
    assert plan.seq_lens.tolist() == ref.seq_lens.tolist()
    assert run.alloc.export_state() == ref.allocator.export_state()
    run.run_step()
    torch.cuda.synchronize()
    assert pa.pa_device_error() == 0
    # append (and copy) results: bit-exact pools
    assert np.array_equal(run.k_pool.cpu().numpy().view(np.uint16), ref.k_pool.view(np.uint16))
    assert np.array_equal(run.v_pool.cpu().numpy().view(np.uint16), ref.v_pool.view(np.uint16))
    out = run.out.cpu().numpy()
    exp = oracle.decode_attention(batch.q, ref.k_pool, ref.v_pool, ref.block_table,
                                  ref.seq_lens, batch.scale, seqs=seqs, heads=heads)
    S = batch.num_seqs
    si = list(range(S)) if seqs is None else list(seqs)
    hi = list(range(batch.num_q_heads)) if heads is None else list(heads)
    assert_close_attention(out[np.ix_(si, hi)], exp[np.ix_(si, hi)], batch.name)
    return run, ref


def test_tiny_config(pa):
    run_and_compare(pa, synthetic.config1_tiny())


@pytest.mark.parametrize("partition", [0, 16, 32, 128, 512])
def test_gqa_small_several_partitions(pa, partition):
    b = synthetic.config2_gqa_batch(num_seqs=7, lo=1, hi=1100)
    run_and_compare(pa, b, partition_tokens=partition)


def test_gqa_batch_full_size(pa):
    """64 sequences U[128,2048], 32q/8kv, D=128, BS=16: every output checked."""
    run_and_compare(pa, synthetic.config2_gqa_batch())


def test_mha_lognormal_small_churned(pa):
    b = synthetic.config3_mha_lognormal(num_seqs=12, churn_ops=800)
    run_and_compare(pa, b)


def test_mha_lognormal_full_size_sampled(pa):
    b = synthetic.config3_mha_lognormal()
    rng = np.random.default_rng(0)
    seqs = sorted(rng.choice(b.num_seqs, 12, replace=False).tolist())
    seqs.append(int(np.argmax(b.prefill_lens)))          # the longest sequence too
    # every head of the sampled sequences: KV heads 0-7, 8-15, 16-23 and 24-31
    # are the kernel's four head groups, each chunked separately at this size
    run_and_compare(pa, b, seqs=sorted(set(seqs)))


@pytest.mark.parametrize("bs", [8, 16, 32])
def test_long_context_small(pa, bs):
    b = synthetic.config5_long_context(block_size=bs, num_seqs=3, seq_len=3000)
    run_and_compare(pa, b)


@pytest.mark.parametrize("bs", [8, 16, 32])
def test_long_context_full_size_sampled(pa, bs):
    """16 x 32768 tokens, 64 q / 8 KV heads: every head of three sequences,
    with every pool row no sequence reads poisoned."""
    b = synthetic.config5_long_context(block_size=bs)
    run_and_compare(pa, b, seqs=[0, 9, 15])


# ---------------------------------------------------------------- edge cases --
def _direct(pa, q, kp, vp, table, lens, scale, partition=0):
    d = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    out = pa.pa_decode_attention(d(q), d(kp), d(vp), d(table.astype(np.int32)),
                                 d(np.asarray(lens, np.int32)), scale,
                                 partition_tokens=partition)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def _random_case(seed, S, Hq, Hkv, D, BS, lens, nb_extra=3):
    rng = np.random.default_rng(seed)
    mb = max(1, max(-(-L // BS) for L in lens))
    need = sum(-(-L // BS) for L in lens)
    nb = need + nb_extra
    perm = rng.permutation(nb)
    table = -np.ones((S, mb), np.int32)
    pos = 0
    for i, L in enumerate(lens):
        n = -(-L // BS)
        table[i, :n] = perm[pos:pos + n]
        pos += n
    q = rng.standard_normal((S, Hq, D)).astype(np.float16)
    kp = rng.standard_normal((nb, BS, Hkv, D)).astype(np.float16)
    vp = rng.standard_normal((nb, BS, Hkv, D)).astype(np.float16)
    kp, vp = poison_unread_rows(kp, vp, table, lens, BS)
    return q, kp, vp, table


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("BS", [8, 16, 32])
@pytest.mark.parametrize("G", [1, 2, 4, 8])
def test_shape_matrix(pa, D, BS, G):
    Hkv = 2
    lens = [1, BS - 1, BS, BS + 1, 255, 256, 257, 700]
    q, kp, vp, table = _random_case(D * 100 + BS * 10 + G, len(lens), G * Hkv, Hkv, D, BS, lens)
    scale = np.float32(1 / math.sqrt(D))
    got = _direct(pa, q, kp, vp, table, lens, scale)
    exp = oracle.decode_attention(q, kp, vp, table, lens, scale)
    assert_close_attention(got, exp, f"D{D} BS{BS} G{G}")
    assert pa.pa_device_error() == 0


def test_zero_length_gives_zeros(pa):
    lens = [0, 5, 0, 40]
    q, kp, vp, table = _random_case(5, 4, 8, 2, 128, 16, [1, 5, 1, 40])
    got = _direct(pa, q, kp, vp, table, lens, np.float32(0.1))
    assert not got[0].any() and not got[2].any()
    exp = oracle.decode_attention(q, kp, vp, table, lens, np.float32(0.1))
    assert_close_attention(got, exp, "zero length")


@pytest.mark.parametrize("partition", [16, 48, 256, 512])
def test_partition_sizes_agree(pa, partition):
    lens = [1, 300, 1000, 4097]
    q, kp, vp, table = _random_case(9, 4, 16, 4, 128, 16, lens)
    got = _direct(pa, q, kp, vp, table, lens, np.float32(0.088), partition)
    exp = oracle.decode_attention(q, kp, vp, table, lens, np.float32(0.088))
    assert_close_attention(got, exp, f"partition {partition}")


def test_large_scores_stay_finite(pa):
    lens = [600]
    q, kp, vp, table = _random_case(11, 1, 4, 1, 128, 16, lens)
    q = (q.astype(np.float32) * 40).astype(np.float16)
    got = _direct(pa, q, kp, vp, table, lens, np.float32(1.0))
    exp = oracle.decode_attention(q, kp, vp, table, lens, np.float32(1.0))
    assert np.isfinite(got).all()
    assert_close_attention(got, exp, "large scores")


def test_workspace_reuse_and_repeat(pa):
    """One workspace serves repeated calls and calls with other lengths: the
    partial results of split sequences never leak from one call into the
    next."""
    from paged_kv_cache_40_gb300 import alloc_workspace
    lens_a = [3000, 20, 1500]
    lens_b = [10, 2900, 700]
    q, kp, vp, table = _random_case(13, 3, 8, 2, 128, 16, [3000, 2900, 1500])
    d = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    ws = alloc_workspace(3, 8, 2, 128, 16, table.shape[1])
    dq, dk, dv, dt = d(q), d(kp), d(vp), d(table)
    for lens in (lens_a, lens_a, lens_b, lens_a):
        out = pa.pa_decode_attention(dq, dk, dv, dt, d(np.asarray(lens, np.int32)), 0.0884,
                                     workspace=ws)
        torch.cuda.synchronize()
        exp = oracle.decode_attention(q, kp, vp, table, lens, np.float32(0.0884))
        assert_close_attention(out.cpu().numpy(), exp, f"reuse {lens}")
    # a completed call leaves every arrival counter word (8 bytes per sequence
    # and KV head, at the start of the workspace) back at zero
    assert not ws[: 3 * 2 * 8].view(torch.int64).cpu().any()
    ws.fill_(255)                   # garbage in the workspace must not matter
    lens = lens_b
    out = pa.pa_decode_attention(dq, dk, dv, dt, d(np.asarray(lens, np.int32)), 0.0884,
                                 workspace=ws)
    torch.cuda.synchronize()
    exp = oracle.decode_attention(q, kp, vp, table, lens, np.float32(0.0884))
    assert_close_attention(out.cpu().numpy(), exp, "garbage workspace")


def test_bad_block_id_is_reported_not_faulted(pa):
    lens = [40, 40]
    q, kp, vp, table = _random_case(17, 2, 4, 4, 64, 16, lens)
    table = table.copy()
    table[1, 1] = 10_000_000            # far outside the pool
    table[0, 2] = -5
    _direct(pa, q, kp, vp, table, lens, np.float32(0.125))
    with pytest.raises(pa.PaError) as e:
        pa.pa_device_error()
    assert e.value.flags & pa.PA_DEVERR_BAD_BLOCK
    assert pa.pa_device_error() == 0     # cleared


def test_length_beyond_table_is_reported(pa):
    q, kp, vp, table = _random_case(19, 1, 4, 4, 64, 16, [32])
    _direct(pa, q, kp, vp, table, [33], np.float32(0.125))   # table holds 2 blocks
    with pytest.raises(pa.PaError) as e:
        pa.pa_device_error()
    assert e.value.flags & pa.PA_DEVERR_BAD_LEN


def test_lengths_written_by_the_kernel_just_before(pa):
    """A serving loop that bumps the lengths on the device right before the
    attention call: the attention kernel (a programmatic dependent of that
    kernel) must read the new lengths, never the old ones. Lengths cross
    block boundaries, so a stale read would change the result."""
    # from L - 4 to L: 29 -> 33, 60 -> 64, 13 -> 17, 2045 -> 2049 cross blocks
    lens_end = [31, 33, 64, 1200, 2049, 17, 5, 500]
    q, kp, vp, table = _random_case(23, len(lens_end), 32, 8, 128, 16, lens_end)
    d = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    dq, dk, dv, dt = d(q), d(kp), d(vp), d(table)
    steps = 4
    lens_dev = d(np.asarray([L - steps for L in lens_end], np.int32))
    for k in range(steps):
        lens_dev.add_(1)                 # the kernel just before the attention call
        out = pa.pa_decode_attention(dq, dk, dv, dt, lens_dev, np.float32(0.088))
        lens_now = [L - steps + k + 1 for L in lens_end]
        torch.cuda.synchronize()
        assert lens_dev.cpu().tolist() == lens_now
        exp = oracle.decode_attention(q, kp, vp, table, lens_now, np.float32(0.088))
        assert_close_attention(out.cpu().numpy(), exp, f"lengths bumped, step {k}")
    assert pa.pa_device_error() == 0


# ------------------------------------------- append + attention, one kernel --
def _append_case(seed, D=128, BS=16, G=4, hkv=2, S=9):
    rng = np.random.default_rng(seed)
    lens0 = rng.integers(1, 90, size=S, endpoint=True)
    nb = sum(-(-(int(L) + 1) // BS) for L in lens0) + 12
    b = synthetic.make_batch(f"append-attend-{seed}", rng, lens0, G * hkv, hkv, D, BS, nb,
                             seed=seed)
    ref = oracle.decode_step(b, compute_attention=False)
    return b, ref


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


@pytest.mark.parametrize("D,BS,G,hkv", [(128, 16, 4, 2), (64, 8, 1, 3), (128, 32, 8, 1),
                                        (128, 16, 2, 16)])
def test_append_attention_equals_append_then_attention(pa, D, BS, G, hkv):
    """pa_decode_append_attention gives the pools pa_append_kv gives
    (bit-exact) and the output of pa_decode_attention after it (bit-equal:
    the same kernel reads the same rows), with every row past a length
    poisoned; 16 KV heads make two head groups, each writing its part."""
    b, ref = _append_case(40 + D + BS + G + hkv, D, BS, G, hkv)
    kp, vp = poison_unread_rows(b.k_pool, b.v_pool, ref.block_table, ref.seq_lens, BS)
    # the rows the append writes are poisoned too: only the append fills them
    for s, slot in enumerate(ref.slot_mapping.tolist()):
        kp[slot // BS, slot % BS] = np.float16(np.nan)
        vp[slot // BS, slot % BS] = np.float16(np.nan)
    args = (_dev(b.q), _dev(b.k_new), _dev(b.v_new), _dev(ref.slot_mapping))
    tab, lens = _dev(ref.block_table), _dev(ref.seq_lens)
    k1, v1 = _dev(kp), _dev(vp)
    out1 = pa.pa_decode_append_attention(*args, k1, v1, tab, lens, float(b.scale))
    k2, v2 = _dev(kp), _dev(vp)
    pa.pa_append_kv(args[1], args[2], k2, v2, args[3])
    out2 = pa.pa_decode_attention(args[0], k2, v2, tab, lens, float(b.scale))
    torch.cuda.synchronize()
    assert pa.pa_device_error() == 0
    assert torch.equal(k1.view(torch.int16), k2.view(torch.int16))
    assert torch.equal(v1.view(torch.int16), v2.view(torch.int16))
    ek, ev = oracle.append_kv(kp, vp, b.k_new, b.v_new, ref.slot_mapping)
    assert np.array_equal(k1.cpu().numpy().view(np.uint16), ek.view(np.uint16))
    assert np.array_equal(v1.cpu().numpy().view(np.uint16), ev.view(np.uint16))
    assert torch.equal(out1, out2)
    exp = oracle.decode_attention(b.q, ek, ev, ref.block_table, ref.seq_lens, b.scale)
    assert_close_attention(out1.cpu().numpy(), exp, f"append+attention D{D} BS{BS} G{G}")


def test_append_attention_slot_checks(pa):
    """A negative slot writes nothing (the pool's row is attended); a slot
    that is not the row of the sequence's last token (another row, or past
    the pool) is not written and sets PA_DEVERR_BAD_SLOT."""
    b, ref = _append_case(77)
    BS = b.block_size
    slots = ref.slot_mapping.copy()
    kp, vp = b.k_pool.copy(), b.v_pool.copy()
    base_k, base_v = _dev(kp), _dev(vp)
    # sequence 0: negative slot; its last row keeps the pool's value
    slots[0] = -1
    tab, lens = _dev(ref.block_table), _dev(ref.seq_lens)
    out = pa.pa_decode_append_attention(_dev(b.q), _dev(b.k_new), _dev(b.v_new), _dev(slots),
                                        base_k, base_v, tab, lens, float(b.scale))
    torch.cuda.synchronize()
    assert pa.pa_device_error() == 0
    ek, ev = oracle.append_kv(kp, vp, b.k_new, b.v_new, slots)
    assert np.array_equal(base_k.cpu().numpy().view(np.uint16), ek.view(np.uint16))
    exp = oracle.decode_attention(b.q, ek, ev, ref.block_table, ref.seq_lens, b.scale)
    assert_close_attention(out.cpu().numpy(), exp, "negative slot")
    # sequence 1: the slot of another row of its last block; sequence 2: past the pool
    for bad in (ref.slot_mapping[1] ^ 1 if BS > 1 else ref.slot_mapping[1] + BS,
                b.num_blocks * BS + 3):
        slots2 = ref.slot_mapping.copy()
        who = 1 if bad < b.num_blocks * BS else 2
        slots2[who] = bad
        k3, v3 = _dev(kp), _dev(vp)
        pa.pa_decode_append_attention(_dev(b.q), _dev(b.k_new), _dev(b.v_new), _dev(slots2),
                                      k3, v3, tab, lens, float(b.scale))
        with pytest.raises(pa.PaError) as e:
            pa.pa_device_error()
        assert e.value.flags & pa.PA_DEVERR_BAD_SLOT
        # that sequence's row was not written anywhere; the others were
        good = ref.slot_mapping.copy()
        good[who] = -1
        ek3, _ = oracle.append_kv(kp, vp, b.k_new, b.v_new, good)
        assert np.array_equal(k3.cpu().numpy().view(np.uint16), ek3.view(np.uint16))
