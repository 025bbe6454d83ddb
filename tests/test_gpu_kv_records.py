"""The one-pool record layout on the GPU (each physical block one record, its K
rows then its V rows), through the C ABI with the pool's block stride, against
the oracle's record-pool operations: append, block copy and swaps bit for bit
over the raw records, attention within the attention tolerance and bit-equal
to the same kernel over two separate pools. Rows no sequence may read are
NaN-poisoned in both members."""

import math

import numpy as np
import pytest

import oracle
import synthetic
from tests.gpu_helpers import assert_close_attention, poison_unread_rows, used_rows_mask

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def pa(libpa):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return libpa


def d(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _raw(records):
    """Oracle record array -> its raw element array [NB][2][BS][H][D]."""
    dt = records.dtype
    bs, h, dd = dt["K"].shape
    elem = dt["K"].base
    return records.view(elem).reshape(len(records), 2, bs, h, dd)


def _device_records(pa, kp, vp):
    """A device record pool holding the blocks of two host pools, and its views."""
    kv = d(_raw(oracle.make_kv_pool(kp, vp)))
    k, v = pa.kv_views(kv)
    return kv, k, v


def _same_bits(dev_kv, records):
    a = dev_kv.cpu().numpy()
    b = _raw(records)
    if a.dtype == np.float16:
        a, b = a.view(np.uint16), b.view(np.uint16)
    return np.array_equal(a, b)


# ------------------------------------------------------------ cache writes --
@pytest.mark.parametrize("shape", [(40, 16, 8, 128), (33, 8, 4, 64), (9, 32, 2, 128)])
def test_append_records_bit_exact(pa, shape):
    nb, bs, h, dd = shape
    rng = np.random.default_rng(nb)
    kp = rng.standard_normal(shape).astype(np.float16)
    vp = rng.standard_normal(shape).astype(np.float16)
    T = 13
    slots = rng.choice(nb * bs, T, replace=False).astype(np.int32)
    slots[2] = -1
    kn = rng.standard_normal((T, h, dd)).astype(np.float16)
    vn = rng.standard_normal((T, h, dd)).astype(np.float16)
    kv, k, v = _device_records(pa, kp, vp)
    pa.pa_append_kv(d(kn), d(vn), k, v, d(slots))
    torch.cuda.synchronize()
    exp = oracle.append_kv_interleaved(oracle.make_kv_pool(kp, vp), kn, vn, slots)
    assert _same_bits(kv, exp)
    assert pa.pa_device_error() == 0


def test_copy_blocks_records_bit_exact(pa):
    rng = np.random.default_rng(7)
    shape = (12, 16, 4, 128)
    kp = rng.standard_normal(shape).astype(np.float16)
    vp = rng.standard_normal(shape).astype(np.float16)
    pairs = np.array([[1, 4], [6, 0], [2, 11], [9, 3]], np.int32)
    kv, k, v = _device_records(pa, kp, vp)
    pa.pa_copy_blocks(k, v, d(pairs))
    torch.cuda.synchronize()
    assert _same_bits(kv, oracle.copy_blocks_interleaved(oracle.make_kv_pool(kp, vp), pairs))


def test_overlapping_member_views_are_refused(pa):
    kv = pa.kv_block_pool(4, 16, 2, 64)
    k, _ = pa.kv_views(kv)
    with pytest.raises(pa.PaError):
        pa.pa_copy_blocks(k, k, d(np.array([[0, 1]], np.int32)))


# ---------------------------------------------------------------- attention --
def _case(seed, S, Hq, Hkv, D, BS, lens, nb_extra=3):
    rng = np.random.default_rng(seed)
    mb = max(1, max(-(-L // BS) for L in lens))
    nb = sum(-(-L // BS) for L in lens) + nb_extra
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
@pytest.mark.parametrize("G", [1, 4, 8])
def test_records_shape_matrix(pa, D, BS, G):
    Hkv = 2
    lens = [1, BS - 1, BS, BS + 1, 255, 256, 257, 700]
    q, kp, vp, table = _case(D * 100 + BS * 10 + G + 1, len(lens), G * Hkv, Hkv, D, BS, lens)
    scale = np.float32(1 / math.sqrt(D))
    _, k, v = _device_records(pa, kp, vp)
    got = pa.pa_decode_attention(d(q), k, v, d(table), d(np.asarray(lens, np.int32)), scale)
    two = pa.pa_decode_attention(d(q), d(kp), d(vp), d(table), d(np.asarray(lens, np.int32)),
                                 scale)
    torch.cuda.synchronize()
    exp = oracle.decode_attention_interleaved(q, oracle.make_kv_pool(kp, vp), table, lens, scale)
    assert_close_attention(got.cpu().numpy(), exp, f"records D{D} BS{BS} G{G}")
    assert torch.equal(got, two)
    assert pa.pa_device_error() == 0


def test_records_fixed_scratch_and_partitions(pa):
    lens = [1, 300, 1000, 4097]
    q, kp, vp, table = _case(9, 4, 16, 4, 128, 16, lens)
    _, k, v = _device_records(pa, kp, vp)
    dq, dt, dl = d(q), d(table), d(np.asarray(lens, np.int32))
    exp = oracle.decode_attention_interleaved(q, oracle.make_kv_pool(kp, vp), table, lens,
                                              np.float32(0.088))
    for part in (0, 16, 256):
        got = pa.pa_decode_attention(dq, k, v, dt, dl, 0.088, partition_tokens=part)
        torch.cuda.synchronize()
        assert_close_attention(got.cpu().numpy(), exp, f"records partition {part}")
        if part != 16:      # one-block chunks need more than the fixed 16 MiB of scratch
            fixed = pa.pa_decode_attention_fixed_scratch(dq, k, v, dt, dl, 0.088,
                                                         partition_tokens=part)
            torch.cuda.synchronize()
            assert torch.equal(got, fixed)


def _step_and_compare(pa, batch, partition_tokens=0, seqs=None):
    """One decode step (append, copy-on-write, attend) on a record pool via
    the engine, against the oracle's step on the same batch."""
    from paged_kv_cache_40_gb300.engine import DecodeBatchRunner
    ref = oracle.decode_step(batch, compute_attention=False)
    run = DecodeBatchRunner(batch, partition_tokens=partition_tokens, layout="records")
    plan = run.plan_step()
    assert plan.block_table.tolist() == ref.block_table.tolist()
    run.run_step()
    torch.cuda.synchronize()
    assert pa.pa_device_error() == 0
    assert _same_bits(run.kv_pool, oracle.make_kv_pool(ref.k_pool, ref.v_pool))
    exp = oracle.decode_attention_interleaved(batch.q, oracle.make_kv_pool(ref.k_pool, ref.v_pool),
                                              ref.block_table, ref.seq_lens, batch.scale,
                                              seqs=seqs)
    out = run.out.cpu().numpy()
    si = list(range(batch.num_seqs)) if seqs is None else list(seqs)
    assert_close_attention(out[si], exp[si], f"records step {batch.name}")
    return run


def _poisoned(batch):
    import dataclasses
    ref = oracle.decode_step(batch, compute_attention=False)
    kp, vp = poison_unread_rows(batch.k_pool, batch.v_pool, ref.block_table, ref.seq_lens,
                                batch.block_size)
    return dataclasses.replace(batch, k_pool=kp, v_pool=vp)


def test_records_step_tiny(pa):
    _step_and_compare(pa, _poisoned(synthetic.config1_tiny()))


@pytest.mark.parametrize("partition", [0, 16, 128])
def test_records_step_gqa_small(pa, partition):
    b = _poisoned(synthetic.config2_gqa_batch(num_seqs=7, lo=1, hi=1100))
    _step_and_compare(pa, b, partition)


def test_records_step_mha_churned(pa):
    b = _poisoned(synthetic.config3_mha_lognormal(num_seqs=12, churn_ops=800))
    _step_and_compare(pa, b)


def test_records_gqa_batch_full_size(pa):
    """The 64-sequence GQA batch (lengths U[128, 2048], 32q/8kv, D=128,
    BS=16) in the record layout, as the benchmark's record-layout line runs
    it: sampled sequences against the oracle, every output bit-equal to the
    two-pool run."""
    from paged_kv_cache_40_gb300.engine import DecodeBatchRunner
    b = _poisoned(synthetic.config2_gqa_batch())
    run = _step_and_compare(pa, b, seqs=[0, 17, 40, 63])
    two = DecodeBatchRunner(b)
    two.plan_step()
    two.run_step()
    torch.cuda.synchronize()
    assert torch.equal(run.out, two.out)


# ---------------------------------------------------------------- fp8 cache --
def test_records_fp8_append_copy_attend(pa):
    rng = np.random.default_rng(40)
    S, Hq, Hkv, D, BS = 5, 16, 4, 128, 16
    lens = [30, 15, 200, 1, 77]
    mb = max(-(-L // BS) for L in lens)
    nb = sum(-(-L // BS) for L in lens) + 4
    perm = rng.permutation(nb)
    table = -np.ones((S, mb), np.int32)
    pos = 0
    for i, L in enumerate(lens):
        n = -(-L // BS)
        table[i, :n] = perm[pos:pos + n]
        pos += n
    kp = synthetic.fp8_codes(rng, (nb, BS, Hkv, D))
    vp = synthetic.fp8_codes(rng, (nb, BS, Hkv, D))
    ks = rng.uniform(0.002, 0.02, Hkv).astype(np.float32)
    vs = rng.uniform(0.002, 0.02, Hkv).astype(np.float32)
    # the new token of each sequence goes to its last row (length already counts it)
    slots = np.array([int(table[i, (L - 1) // BS]) * BS + (L - 1) % BS for i, L in enumerate(lens)],
                     np.int32)
    kn = rng.standard_normal((S, Hkv, D)).astype(np.float16)
    vn = rng.standard_normal((S, Hkv, D)).astype(np.float16)
    free = [b for b in range(nb) if b not in set(table[table >= 0].tolist())]
    pairs = np.array([[int(table[2, 0]), free[0]], [int(table[4, 0]), free[1]]], np.int32)
    kv, k, v = _device_records(pa, kp, vp)
    pa.pa_copy_blocks_fp8(k, v, d(pairs))
    pa.pa_append_kv_fp8(d(kn), d(vn), k, v, d(slots), d(ks), d(vs))
    q = rng.standard_normal((S, Hq, D)).astype(np.float16)
    out = pa.pa_decode_attention_fp8(d(q), k, v, d(ks), d(vs), d(table),
                                     d(np.asarray(lens, np.int32)), np.float32(0.09))
    torch.cuda.synchronize()
    # oracle: copy, then the quantizing append on the two members, as records
    ck, cv = oracle.copy_blocks(kp, vp, pairs)
    ek, ev = oracle.append_kv_fp8(ck, cv, kn, vn, slots, ks, vs)
    exp_records = oracle.make_kv_pool(ek, ev)
    assert _same_bits(kv, exp_records)
    exp = oracle.decode_attention_interleaved_fp8(q, exp_records, ks, vs, table, lens,
                                                  np.float32(0.09))
    assert_close_attention(out.cpu().numpy(), exp, "fp8 records")
    assert pa.pa_device_error() == 0


# ------------------------------------------------------------ shared prefix --
@pytest.mark.parametrize("BS", [16, 32])
def test_records_shared_prefix(pa, BS):
    rng = np.random.default_rng(BS)
    S, Hkv, G, P = 6, 2, 4, 5
    suffix = [0, 1, BS - 1, BS, 3 * BS + 5, 200]
    lens = [P * BS + s for s in suffix]
    priv = [-(-s // BS) for s in suffix]
    nb = P + sum(priv) + 4
    perm = rng.permutation(nb).astype(np.int32)
    prefix = perm[:P]
    table = -np.ones((S, P + max(priv) + 1), np.int32)
    pos = P
    for i in range(S):
        table[i, :P] = prefix
        table[i, P:P + priv[i]] = perm[pos:pos + priv[i]]
        pos += priv[i]
    q = rng.standard_normal((S, G * Hkv, 128)).astype(np.float16)
    kp = rng.standard_normal((nb, BS, Hkv, 128)).astype(np.float16)
    vp = rng.standard_normal((nb, BS, Hkv, 128)).astype(np.float16)
    kp, vp = poison_unread_rows(kp, vp, table, lens, BS)
    _, k, v = _device_records(pa, kp, vp)
    scale = np.float32(1 / math.sqrt(128))
    got = pa.pa_decode_attention_shared_prefix(d(q), k, v, d(prefix), d(table),
                                               d(np.asarray(lens, np.int32)), scale)
    torch.cuda.synchronize()
    exp = oracle.decode_attention_interleaved(q, oracle.make_kv_pool(kp, vp), table, lens, scale)
    assert_close_attention(got.cpu().numpy(), exp, f"records shared prefix BS{BS}")
    assert pa.pa_device_error() == 0


# ------------------------------------------------------------------ swapping --
def test_records_swap_whole_records_and_members(pa):
    """Out to a pinned host record pool as whole records, back as K/V members
    into fresh device blocks; and members of a record pool into two dense
    pinned pools."""
    rng = np.random.default_rng(11)
    shape = (10, 16, 2, 128)
    kp = rng.standard_normal(shape).astype(np.float16)
    vp = rng.standard_normal(shape).astype(np.float16)
    kv, k, v = _device_records(pa, kp, vp)
    host = pa.kv_block_pool(6, 16, 2, 128, device="cpu").pin_memory()
    out_pairs = np.array([[3, 0], [7, 5], [1, 2]], np.int32)
    pa.pa_swap_blocks(kv, None, host, None, d(out_pairs))
    torch.cuda.synchronize()
    zeros = np.zeros((6,) + shape[1:], np.float16)
    hk_exp, hv_exp = oracle.swap_blocks(kp, vp, zeros, zeros, out_pairs)
    assert _same_bits(host, oracle.make_kv_pool(hk_exp, hv_exp))
    # back as members into other device blocks, pairs in pinned host memory
    in_pairs = np.array([[0, 8], [5, 9], [2, 4]], np.int32)
    hk, hv = pa.kv_views(host)
    pa.pa_swap_blocks(hk, hv, k, v, torch.from_numpy(in_pairs).pin_memory())
    torch.cuda.synchronize()
    dk_exp, dv_exp = oracle.swap_blocks(hk_exp, hv_exp, kp, vp, in_pairs)
    assert _same_bits(kv, oracle.make_kv_pool(dk_exp, dv_exp))
    # record members into two dense pinned pools
    sk = torch.zeros((4,) + shape[1:], dtype=torch.float16).pin_memory()
    sv = torch.zeros((4,) + shape[1:], dtype=torch.float16).pin_memory()
    pa.pa_swap_blocks(k, v, sk, sv, d(np.array([[9, 3], [8, 0]], np.int32)))
    torch.cuda.synchronize()
    z4 = np.zeros((4,) + shape[1:], np.float16)
    ek, ev = oracle.swap_blocks(dk_exp, dv_exp, z4, z4, [[9, 3], [8, 0]])
    assert np.array_equal(sk.numpy().view(np.uint16), ek.view(np.uint16))
    assert np.array_equal(sv.numpy().view(np.uint16), ev.view(np.uint16))
    assert pa.pa_device_error() == 0


def test_unread_rows_mask_covers_both_members(pa):
    """The poisoning used above reaches both members of a record: a read of
    an unread K or V row would show as NaN."""
    q, kp, vp, table = _case(3, 2, 4, 2, 64, 16, [20, 33])
    rec = _raw(oracle.make_kv_pool(kp, vp))
    keep = used_rows_mask(table, [20, 33], kp.shape[0], 16)
    assert np.isnan(rec[:, 0][~keep].astype(np.float32)).all()
    assert np.isnan(rec[:, 1][~keep].astype(np.float32)).all()
